"""Float64 CPU oracle for paged decode attention -- test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg and reference arm (``bench.py --impl reference``) may import this
package.  The product path (the CUDA library and
its binding) never imports it, and it imports nothing from the product.

The arithmetic lives in ``kvattn_oracle.c`` (plain C, double precision,
OpenMP over heads when available); this module compiles it with gcc and wraps
it with ctypes, marshalling numpy arrays.  Page citations are on each C
function.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvattn_oracle.c")
_LIB = os.path.join(_HERE, "libkvattn_oracle.so")
_lock = threading.Lock()
_lib = None

FMT_BF16, FMT_E4M3, FMT_F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC,
            "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, i32, f64, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
        sig = {
            "kvo_num_threads": (i32, []),
            "kvo_bf16_to_double": (f64, [ctypes.c_uint16]),
            "kvo_e4m3_decode": (f64, [ctypes.c_uint8]),
            "kvo_e4m3_encode": (ctypes.c_uint8, [f32]),
            "kvo_quantize_e4m3": (None, [P, i64, f32, P]),
            "kvo_cell_bytes_gqa": (i64, [i64, i64, i64, i64, i64]),
            "kvo_cell_bytes_mla": (i64, [i64, i64, i64, i64]),
            "kvo_page_bytes": (i64, [i64, i64, i64, i64, i64]),
            "kvo_blocks_for": (i64, [i64, i64]),
            "kvo_intensity_gqa": (f64, [f64, f64]),
            "kvo_intensity_mla": (f64, [f64, f64, f64, f64]),
            "kvo_slot_block": (i64, [P, i32, i32, i32, i64]),
            "kvo_gqa_pool_offset": (i64, [P, i32, i32, i32, i32, i32, i64, i32]),
            "kvo_mla_pool_offset": (i64, [P, i32, i32, i32, i32, i64]),
            "kvo_gqa_decode": (i32, [P, P, P, i32, f64, f64, i64, i32, i32, i32, f64, P, P]),
            "kvo_mla_decode": (i32, [P, P, i32, i64, i32, i32, i32, f64, P, P]),
            "kvo_mla_decode_e4m3": (i32, [P, P, i64, i32, i32, i32, f64, f64, f64, P, P]),
            "kvo_mla_absorb_query": (None, [P, P, i32, i32, i32, P]),
            "kvo_mla_apply_wuv": (None, [P, P, i32, i32, i32, P]),
            "kvo_mla_explicit": (i32, [P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, f64, P, P]),
            "kvo_mla_prefill": (i32, [P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, i32, f64, P,
                                      P]),
            "kvo_lse_combine": (None, [P, P, i32, i32, i32, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().kvo_num_threads())


# ---- element formats -------------------------------------------------------

def bf16_to_double(bits: int) -> float:
    return float(_load().kvo_bf16_to_double(int(bits)))


def e4m3_decode(code: int) -> float:
    return float(_load().kvo_e4m3_decode(int(code)))


def e4m3_encode(x: float) -> int:
    return int(_load().kvo_e4m3_encode(float(x)))


def quantize_e4m3(x_bf16: np.ndarray, scale: float) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().kvo_quantize_e4m3(_ptr(x), x.size, float(scale), _ptr(out))
    return out


# ---- sizing ----------------------------------------------------------------

def cell_bytes_gqa(L, h_kv, d_k, d_v, b) -> int:
    return int(_load().kvo_cell_bytes_gqa(L, h_kv, d_k, d_v, b))


def cell_bytes_mla(L, d_c, d_rope, b) -> int:
    return int(_load().kvo_cell_bytes_mla(L, d_c, d_rope, b))


def page_bytes(num_heads, block_size, head_size, head_size_v, b) -> int:
    return int(_load().kvo_page_bytes(num_heads, block_size, head_size, head_size_v, b))


def blocks_for(length, block_size) -> int:
    return int(_load().kvo_blocks_for(length, block_size))


def intensity_gqa(g, b) -> float:
    return float(_load().kvo_intensity_gqa(g, b))


def intensity_mla(h, r_kv, d_rope, b) -> float:
    return float(_load().kvo_intensity_mla(h, r_kv, d_rope, b))


# ---- paged placement -------------------------------------------------------

def gqa_pool_offset(block_table, bs, h_kv, d, b, t, kvh) -> int:
    bt = _c(block_table, np.int32)
    return int(_load().kvo_gqa_pool_offset(_ptr(bt), bt.shape[1], bs, h_kv, d, b, t, kvh))


def mla_pool_offset(block_table, bs, width, b, t) -> int:
    bt = _c(block_table, np.int32)
    return int(_load().kvo_mla_pool_offset(_ptr(bt), bt.shape[1], bs, width, b, t))


def expected_gqa_pool(k_tokens: np.ndarray, seq_idx, pos, block_table, num_blocks, bs,
                      fill) -> np.ndarray:
    """Pool contents after placing token n's vectors k_tokens[n] ([h_kv, d])
    at (seq_idx[n], pos[n]); untouched elements hold ``fill``.  Follows
    kvo_gqa_pool_offset for every (token, kv head)."""
    n_tok, h_kv, d = k_tokens.shape
    pool = np.full(num_blocks * h_kv * bs * d, fill, dtype=k_tokens.dtype)
    bt = _c(block_table, np.int32)
    lib = _load()
    for n in range(n_tok):
        for kvh in range(h_kv):
            off = lib.kvo_gqa_pool_offset(_ptr(bt), bt.shape[1], bs, h_kv, d,
                                          int(seq_idx[n]), int(pos[n]), kvh)
            pool[off:off + d] = k_tokens[n, kvh]
    return pool.reshape(num_blocks, h_kv, bs, d)


def expected_mla_pool(rows: np.ndarray, seq_idx, pos, block_table, num_blocks, bs,
                      fill) -> np.ndarray:
    n_tok, width = rows.shape
    pool = np.full(num_blocks * bs * width, fill, dtype=rows.dtype)
    bt = _c(block_table, np.int32)
    lib = _load()
    for n in range(n_tok):
        off = lib.kvo_mla_pool_offset(_ptr(bt), bt.shape[1], bs, width, int(seq_idx[n]), int(pos[n]))
        pool[off:off + width] = rows[n]
    return pool.reshape(num_blocks, bs, width)


# ---- attention -------------------------------------------------------------

def gqa_decode(q_bf16, k, v, scale, fmt=FMT_BF16, k_scale=1.0, v_scale=1.0):
    """One sequence: q [h, d] bf16 bits; k, v [s, h_kv, d] (bf16 bits, E4M3
    codes or float64 by ``fmt``).  Returns (out [h, d], lse [h]) float64."""
    q = _c(q_bf16, np.uint16)
    dt = {FMT_BF16: np.uint16, FMT_E4M3: np.uint8, FMT_F64: np.float64}[fmt]
    k = _c(k, dt)
    v = _c(v, dt)
    h, d = q.shape
    s, h_kv, d2 = k.shape
    assert d2 == d and v.shape == k.shape
    out = np.empty((h, d), dtype=np.float64)
    lse = np.empty(h, dtype=np.float64)
    rc = _load().kvo_gqa_decode(_ptr(q), _ptr(k), _ptr(v), fmt, float(k_scale), float(v_scale),
                                s, h, h_kv, d, float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("kvo_gqa_decode: bad shape")
    return out, lse


def gqa_decode_multi(q_bf16, k, v, scale, fmt=FMT_BF16, k_scale=1.0, v_scale=1.0):
    """q_len new tokens of one sequence, causal among themselves (speculative
    verification: "MLA：为什么一份 Latent 可以代替多头 KV Cache", section
    "正确性验证应该从两种实现互证", item 5).  q [q_len, h, d] bf16 bits; k, v
    [s, h_kv, d] hold every cached token, the new ones last.  Token j sits at
    position s - q_len + j and attends to positions [0, s - q_len + j]: its row
    is the single-token decode over that prefix.  A token whose position would
    be negative sees nothing (out 0, lse -inf).  Returns (out [q_len, h, d],
    lse [q_len, h]) float64."""
    q = np.asarray(q_bf16)
    q_len, h, d = q.shape
    s = np.asarray(k).shape[0]
    out = np.zeros((q_len, h, d), dtype=np.float64)
    lse = np.full((q_len, h), -np.inf, dtype=np.float64)
    for j in range(q_len):
        n = s - q_len + j + 1
        if n > 0:
            out[j], lse[j] = gqa_decode(q[j], np.asarray(k)[:n], np.asarray(v)[:n], scale, fmt,
                                        k_scale, v_scale)
    return out, lse


def mla_decode(q, rows, d_c, scale, fmt=FMT_BF16):
    """One sequence: q [h, d_c + d_rope], rows [s, d_c + d_rope] (bf16 bits or
    float64).  Returns (out [h, d_c], lse [h]) float64."""
    dt = {FMT_BF16: np.uint16, FMT_F64: np.float64}[fmt]
    q = _c(q, dt)
    rows = _c(rows, dt)
    h, w = q.shape
    s = rows.shape[0]
    assert rows.shape[1] == w
    out = np.empty((h, d_c), dtype=np.float64)
    lse = np.empty(h, dtype=np.float64)
    rc = _load().kvo_mla_decode(_ptr(q), _ptr(rows), fmt, s, h, d_c, w - d_c, float(scale),
                                _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("kvo_mla_decode: bad shape")
    return out, lse


def mla_decode_e4m3(q, codes, d_c, scale, c_scale, r_scale):
    """One sequence over an FP8-E4M3 latent cache: q [h, d_c + d_rope] bf16
    bits, codes [s, d_c + d_rope] uint8; the c_KV codes decode times c_scale,
    the k_R codes times r_scale.  Returns (out [h, d_c], lse [h]) float64."""
    q = _c(q, np.uint16)
    codes = _c(codes, np.uint8)
    h, w = q.shape
    s = codes.shape[0]
    assert codes.shape[1] == w
    out = np.empty((h, d_c), dtype=np.float64)
    lse = np.empty(h, dtype=np.float64)
    rc = _load().kvo_mla_decode_e4m3(_ptr(q), _ptr(codes), s, h, d_c, w - d_c, float(c_scale),
                                     float(r_scale), float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("kvo_mla_decode_e4m3: bad shape")
    return out, lse


def mla_absorb_query(q_c, w_uk):
    q_c = _c(q_c, np.float64)
    w_uk = _c(w_uk, np.float64)
    h, d_hc, d_c = w_uk.shape
    out = np.empty((h, d_c), dtype=np.float64)
    _load().kvo_mla_absorb_query(_ptr(q_c), _ptr(w_uk), h, d_hc, d_c, _ptr(out))
    return out


def mla_apply_wuv(u_tilde, w_uv):
    u_tilde = _c(u_tilde, np.float64)
    w_uv = _c(w_uv, np.float64)
    h, d_v, d_c = w_uv.shape
    out = np.empty((h, d_v), dtype=np.float64)
    _load().kvo_mla_apply_wuv(_ptr(u_tilde), _ptr(w_uv), h, d_v, d_c, _ptr(out))
    return out


def mla_explicit(q_c, q_r, c, k_r, w_uk, w_uv, scale):
    arrs = [_c(a, np.float64) for a in (q_c, q_r, c, k_r, w_uk, w_uv)]
    q_c, q_r, c, k_r, w_uk, w_uv = arrs
    h, d_hc, d_c = w_uk.shape
    d_v = w_uv.shape[1]
    s, d_r = k_r.shape
    u = np.empty((h, d_v), dtype=np.float64)
    lse = np.empty(h, dtype=np.float64)
    rc = _load().kvo_mla_explicit(*[_ptr(a) for a in arrs], s, h, d_c, d_r, d_hc, d_v,
                                  float(scale), _ptr(u), _ptr(lse))
    if rc != 0:
        raise ValueError("kvo_mla_explicit: bad shape")
    return u, lse


def mla_prefill(q_c, q_r, c, k_r, w_uk, w_uv, scale):
    """Explicit-form MLA over the last q_len rows as new tokens, causal among
    them.  q_c [q_len, h, d_hc], q_r [q_len, h, d_r], c [s, d_c], k_r [s, d_r],
    w_uk [h, d_hc, d_c], w_uv [h, d_v, d_c] (float64 or anything numpy casts).
    Returns (out [q_len, h, d_v], lse [q_len, h]) float64."""
    arrs = [_c(a, np.float64) for a in (q_c, q_r, c, k_r, w_uk, w_uv)]
    q_c, q_r, c, k_r, w_uk, w_uv = arrs
    q_len, h, d_hc = q_c.shape
    d_c = w_uk.shape[2]
    d_v = w_uv.shape[1]
    s, d_r = k_r.shape
    assert q_r.shape == (q_len, h, d_r) and c.shape == (s, d_c) and w_uk.shape == (h, d_hc, d_c)
    out = np.empty((q_len, h, d_v), dtype=np.float64)
    lse = np.empty((q_len, h), dtype=np.float64)
    rc = _load().kvo_mla_prefill(*[_ptr(a) for a in arrs], s, q_len, h, d_c, d_r, d_hc, d_v,
                                 float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("kvo_mla_prefill: bad shape")
    return out, lse


def lse_combine(part_o, part_lse):
    """part_o [W, n, dv], part_lse [W, n] -> (out [n, dv], lse [n])."""
    part_o = _c(part_o, np.float64)
    part_lse = _c(part_lse, np.float64)
    W, n, dv = part_o.shape
    out = np.empty((n, dv), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    _load().kvo_lse_combine(_ptr(part_o), _ptr(part_lse), W, n, dv, _ptr(out), _ptr(lse))
    return out, lse
