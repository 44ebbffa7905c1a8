"""GB300-native paged KV-cache decode attention (GQA / MQA / MHA and MLA).

Thin Python binding over ``libkvattn.so`` (C ABI, ``include/kvattn.h``).
Functions keep the C names and only marshal arguments: torch tensors become
device pointers, the current torch stream becomes the CUDA stream.  Every step
of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback -- if the library cannot be built or loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

from . import _build

KVATTN_OK = 0
KVATTN_ERR_INVALID_ARG = 1
KVATTN_ERR_UNSUPPORTED = 2
KVATTN_ERR_CUDA = 3
KVATTN_ERR_WORKSPACE = 4

KVATTN_DEVERR_BLOCK_ID = 1
KVATTN_DEVERR_SEQ_LEN = 2
KVATTN_DEVERR_POSITION = 4
KVATTN_DEVERR_TIMEOUT = 8

KVATTN_GQA = 0
KVATTN_MLA = 1
KVATTN_BF16 = 0
KVATTN_FP8_E4M3 = 1

EXPORTED = [
    "kvattn_status_string", "kvattn_abi_version", "kvattn_page_bytes", "kvattn_cell_bytes",
    "kvattn_append", "kvattn_decode_workspace_bytes", "kvattn_default_num_ctas",
    "kvattn_decode_gqa", "kvattn_decode_mla", "kvattn_combine", "kvattn_decode_gqa_noalloc",
    "kvattn_decode_gqa_multi", "kvattn_mla_absorb_q", "kvattn_mla_up_v", "kvattn_mla_prefill",
]

KVATTN_NOALLOC_SCRATCH_BYTES = 8 << 20


class KvattnError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class kvattn_cache(ctypes.Structure):
    """Mirror of ``struct kvattn_cache`` in include/kvattn.h."""
    _fields_ = [
        ("kind", ctypes.c_int32), ("dtype", ctypes.c_int32), ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32), ("h_kv", ctypes.c_int32), ("d_h", ctypes.c_int32),
        ("d_c", ctypes.c_int32), ("d_rope", ctypes.c_int32), ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float), ("reserved", ctypes.c_int32), ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p), ("latent", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB


def load_library(build: bool = True) -> ctypes.CDLL:
    """Load libkvattn.so, building it with nvcc first if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libkvattn.so not found at {_build.LIB}; run __graft_entry__.build()")
        _lib = open_library(_build.LIB)
        return _lib


def open_library(path: str) -> ctypes.CDLL:
    """Load a build of the library at `path` with every entry point's ctypes
    signature set (load_library() does this for libkvattn.so)."""
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    CP = ctypes.POINTER(kvattn_cache)
    sig = {
        "kvattn_status_string": (ctypes.c_char_p, [i32]),
        "kvattn_abi_version": (i32, []),
        "kvattn_page_bytes": (i64, [CP]),
        "kvattn_cell_bytes": (i64, [i32, i32, i32, i32, i32, i32, i32]),
        "kvattn_append": (i32, [CP, P, P, i64, P, P, P, i32, i32, P, P]),
        "kvattn_decode_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "kvattn_default_num_ctas": (i32, [i32, i32, i32, i32, i32]),
        "kvattn_decode_gqa": (i32, [P, CP, P, P, i32, i32, i32, i32, i32, f32, P, P, P, sz,
                                    i32, P, P]),
        "kvattn_decode_mla": (i32, [P, CP, P, P, i32, i32, i32, i32, i32, f32, P, P, P, sz,
                                    i32, P, P]),
        "kvattn_combine": (i32, [P, P, P, P, i32, i32, i32, P, P, P]),
        "kvattn_decode_gqa_noalloc": (i32, [P, CP, P, P, i32, i32, i32, i32, i32, f32, P, P,
                                            i32, P, P]),
        "kvattn_decode_gqa_multi": (i32, [P, CP, P, P, i32, i32, i32, i32, i32, i32, f32, P,
                                          P, P, sz, i32, P, P]),
        "kvattn_mla_absorb_q": (i32, [P, P, P, i32, i32, i32, i32, i32, P, P, P]),
        "kvattn_mla_up_v": (i32, [P, P, i32, i32, i32, i32, P, P, P]),
        "kvattn_mla_prefill": (i32, [P, P, CP, P, P, i32, i32, i32, i32, i32, i32, P, P, f32,
                                     P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(fn: str, status: int):
    if status != KVATTN_OK:
        raise KvattnError(fn, status, kvattn_status_string(status))


# ---- the C entry points, same names ----------------------------------------

def kvattn_status_string(status: int) -> str:
    return load_library().kvattn_status_string(int(status)).decode()


def kvattn_abi_version() -> int:
    return int(load_library().kvattn_abi_version())


def kvattn_page_bytes(cache: kvattn_cache) -> int:
    return int(load_library().kvattn_page_bytes(ctypes.byref(cache)))


def kvattn_cell_bytes(kind, num_layers, h_kv, d_h, d_c, d_rope, elem_bytes) -> int:
    return int(load_library().kvattn_cell_bytes(kind, num_layers, h_kv, d_h, d_c, d_rope, elem_bytes))


def kvattn_decode_workspace_bytes(kind, batch, h, h_kv, dv, num_ctas=0) -> int:
    return int(load_library().kvattn_decode_workspace_bytes(kind, batch, h, h_kv, dv, num_ctas))


def kvattn_default_num_ctas(kind, dtype, h, h_kv, d_h) -> int:
    return int(load_library().kvattn_default_num_ctas(kind, dtype, h, h_kv, d_h))


def kvattn_append(cache: kvattn_cache, k_or_ckv, v_or_kr, seq_idx, pos, block_table,
                  err=None, stream=None):
    n = int(seq_idx.numel())
    batch, max_blocks = block_table.shape
    _check("kvattn_append", load_library().kvattn_append(
        ctypes.byref(cache), _ptr(k_or_ckv), _ptr(v_or_kr), n, _ptr(seq_idx), _ptr(pos),
        _ptr(block_table), int(batch), int(max_blocks), _ptr(err), _stream(stream)))


def kvattn_decode_gqa(q, cache: kvattn_cache, block_table, seq_lens, h, h_kv, d_h, scale,
                      out, lse, workspace, num_ctas=0, err=None, stream=None):
    batch, max_blocks = block_table.shape
    _check("kvattn_decode_gqa", load_library().kvattn_decode_gqa(
        _ptr(q), ctypes.byref(cache), _ptr(block_table), _ptr(seq_lens), int(batch),
        int(max_blocks), int(h), int(h_kv), int(d_h), float(scale), _ptr(out), _ptr(lse),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()) if workspace is not None else 0,
        int(num_ctas), _ptr(err), _stream(stream)))


def kvattn_decode_gqa_multi(q, cache: kvattn_cache, block_table, seq_lens, q_len, h, h_kv, d_h,
                            scale, out, lse, workspace, num_ctas=0, err=None, stream=None):
    """q_len new tokens per sequence ([batch][q_len][h][d_h] q, out and lse
    rows [batch][q_len][h]), causal among the new tokens."""
    batch, max_blocks = block_table.shape
    _check("kvattn_decode_gqa_multi", load_library().kvattn_decode_gqa_multi(
        _ptr(q), ctypes.byref(cache), _ptr(block_table), _ptr(seq_lens), int(batch),
        int(max_blocks), int(q_len), int(h), int(h_kv), int(d_h), float(scale), _ptr(out),
        _ptr(lse), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()) if workspace is not None else 0,
        int(num_ctas), _ptr(err), _stream(stream)))


def kvattn_decode_gqa_noalloc(q, cache: kvattn_cache, block_table, seq_lens, h, h_kv, d_h,
                              scale, out, lse, num_ctas=0, err=None, stream=None):
    """kvattn_decode_gqa without a workspace: for callers that cannot provide
    device memory.  The scratch is a fixed array inside the library
    (KVATTN_NOALLOC_SCRATCH_BYTES per GPU); larger problems are rejected, and
    calls that overlap on the GPU race on it."""
    batch, max_blocks = block_table.shape
    _check("kvattn_decode_gqa_noalloc", load_library().kvattn_decode_gqa_noalloc(
        _ptr(q), ctypes.byref(cache), _ptr(block_table), _ptr(seq_lens), int(batch),
        int(max_blocks), int(h), int(h_kv), int(d_h), float(scale), _ptr(out), _ptr(lse),
        int(num_ctas), _ptr(err), _stream(stream)))


def kvattn_decode_mla(q_absorbed, cache: kvattn_cache, block_table, seq_lens, h, d_c, d_rope,
                      scale, out, lse, workspace, num_ctas=0, err=None, stream=None):
    batch, max_blocks = block_table.shape
    _check("kvattn_decode_mla", load_library().kvattn_decode_mla(
        _ptr(q_absorbed), ctypes.byref(cache), _ptr(block_table), _ptr(seq_lens), int(batch),
        int(max_blocks), int(h), int(d_c), int(d_rope), float(scale), _ptr(out), _ptr(lse),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()) if workspace is not None else 0,
        int(num_ctas), _ptr(err), _stream(stream)))


def kvattn_mla_absorb_q(q_nope, q_rope, w_uk, q_absorbed, err=None, stream=None):
    """q_nope [B][h][d_hc], q_rope [B][h][d_rope], w_uk [h][d_hc][d_c] (bf16 bits)
    -> q_absorbed [B][h][d_c + d_rope] bf16 bits."""
    batch, h, d_hc = q_nope.shape
    d_c = int(w_uk.shape[2])
    d_rope = int(q_rope.shape[2]) if q_rope is not None else 0
    _check("kvattn_mla_absorb_q", load_library().kvattn_mla_absorb_q(
        _ptr(q_nope), _ptr(q_rope), _ptr(w_uk), int(batch), int(h), int(d_hc), d_c, d_rope,
        _ptr(q_absorbed), _ptr(err), _stream(stream)))


def kvattn_mla_up_v(u_tilde, w_uv, v, err=None, stream=None):
    """u_tilde [B][h][d_c] float32, w_uv [h][d_v][d_c] bf16 bits -> v [B][h][d_v] float32."""
    batch, h, d_c = u_tilde.shape
    d_v = int(w_uv.shape[1])
    _check("kvattn_mla_up_v", load_library().kvattn_mla_up_v(
        _ptr(u_tilde), _ptr(w_uv), int(batch), int(h), int(d_c), d_v, _ptr(v), _ptr(err),
        _stream(stream)))


def kvattn_mla_prefill(q_nope, q_rope, cache: kvattn_cache, block_table, seq_lens, w_uk, w_uv,
                       scale, out, lse, err=None, stream=None):
    """Explicit-form MLA prefill of q_len new tokens per sequence (already in the
    cache, causal among them): q_nope [B][q_len][h][128], q_rope [B][q_len][h][64]
    bf16 bits, w_uk / w_uv [h][128][512] bf16 bits -> out [B][q_len][h][128],
    lse [B][q_len][h] float32."""
    batch, q_len, h, d_hc = q_nope.shape
    d_v = int(w_uv.shape[1])
    _check("kvattn_mla_prefill", load_library().kvattn_mla_prefill(
        _ptr(q_nope), _ptr(q_rope), ctypes.byref(cache), _ptr(block_table), _ptr(seq_lens),
        int(batch), int(block_table.shape[1]), int(q_len), int(h), int(d_hc), d_v, _ptr(w_uk),
        _ptr(w_uv), float(scale), _ptr(out), _ptr(lse), _ptr(err), _stream(stream)))


def kvattn_combine(part_out, part_lse, split_first, split_count, rows_per_unit, dv, out, lse,
                   stream=None):
    n_units = int(split_first.numel())
    _check("kvattn_combine", load_library().kvattn_combine(
        _ptr(part_out), _ptr(part_lse), _ptr(split_first), _ptr(split_count), n_units,
        int(rows_per_unit), int(dv), _ptr(out), _ptr(lse), _stream(stream)))


# ---- device memory helpers (torch allocates; the library never does) ---------

@dataclass
class PagedCache:
    """One layer's paged pools held as torch tensors, plus the C descriptor."""
    kind: int
    dtype: int
    num_blocks: int
    block_size: int
    h_kv: int = 0
    d_h: int = 0
    d_c: int = 0
    d_rope: int = 0
    k_scale: float = 1.0
    v_scale: float = 1.0
    k: object = None
    v: object = None
    latent: object = None

    @classmethod
    def allocate_gqa(cls, num_blocks, block_size, h_kv, d_h, dtype=KVATTN_BF16, k_scale=1.0,
                     v_scale=1.0, device="cuda", fill_bits=None):
        import torch
        tdt = torch.uint8 if dtype == KVATTN_FP8_E4M3 else torch.int16
        shape = (num_blocks, h_kv, block_size, d_h)
        k = torch.empty(shape, dtype=tdt, device=device)
        v = torch.empty(shape, dtype=tdt, device=device)
        if fill_bits is not None:
            k.fill_(_signed(fill_bits, tdt))
            v.fill_(_signed(fill_bits, tdt))
        return cls(KVATTN_GQA, dtype, num_blocks, block_size, h_kv=h_kv, d_h=d_h, k_scale=k_scale,
                   v_scale=v_scale, k=k, v=v)

    @classmethod
    def allocate_mla(cls, num_blocks, block_size, d_c=512, d_rope=64, dtype=KVATTN_BF16,
                     k_scale=1.0, v_scale=1.0, device="cuda", fill_bits=None):
        """MLA latent pool; for an E4M3 pool k_scale scales the c_KV codes and
        v_scale the k_R codes."""
        import torch
        tdt = torch.uint8 if dtype == KVATTN_FP8_E4M3 else torch.int16
        lat = torch.empty((num_blocks, block_size, d_c + d_rope), dtype=tdt, device=device)
        if fill_bits is not None:
            lat.fill_(_signed(fill_bits, tdt))
        return cls(KVATTN_MLA, dtype, num_blocks, block_size, d_c=d_c, d_rope=d_rope,
                   k_scale=k_scale, v_scale=v_scale, latent=lat)

    def descriptor(self) -> kvattn_cache:
        return kvattn_cache(self.kind, self.dtype, self.num_blocks, self.block_size, self.h_kv,
                            self.d_h, self.d_c, self.d_rope, self.k_scale, self.v_scale, 0,
                            _ptr(self.k), _ptr(self.v), _ptr(self.latent))


def _signed(bits: int, tdt) -> int:
    import torch
    if tdt == torch.int16 and bits >= 1 << 15:
        return bits - (1 << 16)
    return bits


def workspace_for(kind, batch, h, h_kv, dv, num_ctas=0, device="cuda"):
    """Allocate a decode workspace with torch (256-byte aligned)."""
    import torch
    n = kvattn_decode_workspace_bytes(kind, batch, h, h_kv, dv, num_ctas)
    if n <= 0:
        raise KvattnError("kvattn_decode_workspace_bytes", KVATTN_ERR_INVALID_ARG, "no workspace size")
    return torch.empty(n, dtype=torch.uint8, device=device)
