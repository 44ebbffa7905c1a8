"""Seeded synthetic workloads for paged decode attention.

This module draws random numbers and lays them out in memory; it holds none of
the attention arithmetic.  Both sides of every comparison read what it makes:
the CUDA library (through the Python binding) and the float64 oracle.

Values are drawn with ``numpy.random.default_rng`` (PCG64) in float32 and
rounded to bfloat16 bit patterns (round to nearest even), so the GPU and the
oracle consume identical stored bytes.  Each array comes from its own stream,
keyed by ``(seed, crc32(name))``, so changing one shape does not reshuffle the
others.

The shapes follow the models the pages use as running examples:
Llama-3-8B and Llama-3-70B ("The KV cache size formula", mlinterviewnotes
§2.1; "MHA → MQA → GQA → MLA", §3.5) and DeepSeek-V3's MLA latent of
kv_lora_rank 512 plus a 64-wide decoupled RoPE key ("Multi-Head Latent
Attention (MLA): Mathematical Foundations ...", section "What the Inference
Engine Caches").
"""
from __future__ import annotations

import math
import zlib
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BF16_NAN = 0x7FC0   # quiet NaN bit pattern used to poison unused pool slots
E4M3_NAN = 0x7F     # the E4M3 NaN code (S.1111.111), same purpose for FP8 pools

# name -> recipe.  "lens" is (kind, args): fixed list, integer-uniform range
# (inclusive) or log-uniform range rounded to the nearest integer.
WORKLOADS = {
    # tiny GQA, contiguous cache (identity block table)
    "tiny": dict(kind="gqa", B=2, h=8, h_kv=2, d=64, lens=("fixed", [37, 100]),
                 bs=16, table="identity", kv_dtype="bf16", q_std=1.0),
    # Llama-3-8B decode layer
    "llama3_8b": dict(kind="gqa", B=64, h=32, h_kv=8, d=128, lens=("uniform", 512, 8192),
                      bs=16, table="permuted", kv_dtype="bf16", q_std=1.0),
    # Llama-3-70B decode layer, single GPU, bf16 and FP8-E4M3 caches
    "llama3_70b": dict(kind="gqa", B=32, h=64, h_kv=8, d=128, lens=("fixed", [8192] * 32),
                       bs=16, table="permuted", kv_dtype="bf16", q_std=1.0),
    "llama3_70b_fp8": dict(kind="gqa", B=32, h=64, h_kv=8, d=128, lens=("fixed", [8192] * 32),
                           bs=16, table="permuted", kv_dtype="fp8", q_std=1.0),
    # DeepSeek-V3 MLA absorbed decode layer
    "deepseek_v3_mla": dict(kind="mla", B=64, h=128, d_c=512, d_rope=64,
                            lens=("fixed", [4096] * 64), bs=64, table="permuted",
                            kv_dtype="bf16", q_std=1.0 / 24.0,
                            scale=1.0 / math.sqrt(192.0)),
    # the same layer over an FP8-E4M3 latent cache (per-tensor scales, one for
    # c_KV and one for k_R, each amax / 448)
    "deepseek_v3_mla_fp8": dict(kind="mla", B=64, h=128, d_c=512, d_rope=64,
                                lens=("fixed", [4096] * 64), bs=64, table="permuted",
                                kv_dtype="fp8", q_std=1.0 / 24.0,
                                scale=1.0 / math.sqrt(192.0)),
    # long ragged contexts that need split-KV: GQA-8 and MQA on the same lengths
    "long_gqa8": dict(kind="gqa", B=16, h=64, h_kv=8, d=128, lens=("loguniform", 1024, 131072),
                      bs=16, table="permuted", kv_dtype="bf16", q_std=1.0),
    "long_mqa": dict(kind="gqa", B=16, h=32, h_kv=1, d=128, lens=("loguniform", 1024, 131072),
                     bs=16, table="permuted", kv_dtype="bf16", q_std=1.0),
}


def rng_for(seed: int, stream: str) -> np.random.Generator:
    """Independent PCG64 stream keyed by (seed, name)."""
    return np.random.default_rng([int(seed), zlib.crc32(stream.encode())])


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (no NaN inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, n: int, std: float = 1.0,
                chunk: int = 1 << 24) -> np.ndarray:
    """n draws of N(0, std^2), rounded to bf16, generated in bounded chunks."""
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = bf16_bits(x)
    return out


def draw_lengths(spec, batch: int, seed: int) -> np.ndarray:
    kind = spec[0]
    rng = rng_for(seed, "lens")
    if kind == "fixed":
        vals = list(spec[1])
        if len(vals) != batch:
            vals = [vals[i % len(vals)] for i in range(batch)]
        return np.asarray(vals, dtype=np.int32)
    if kind == "uniform":
        return rng.integers(spec[1], spec[2] + 1, size=batch).astype(np.int32)
    if kind == "loguniform":
        u = rng.uniform(math.log(spec[1]), math.log(spec[2]), size=batch)
        return np.rint(np.exp(u)).astype(np.int32)
    raise ValueError(f"unknown length recipe {spec!r}")


def cdiv(a, b):
    return -(-a // b)


@dataclass
class Workload:
    name: str
    kind: str                 # "gqa" or "mla"
    B: int
    h: int
    h_kv: int                 # 1 for MLA (one shared latent row per token)
    d: int                    # GQA head dim; MLA row width d_c + d_rope
    d_c: int
    d_rope: int
    block_size: int
    kv_dtype: str             # "bf16" or "fp8"
    scale: float              # softmax scale applied to q.k
    seq_lens: np.ndarray      # int32 [B]
    cu_seqlens: np.ndarray    # int64 [B+1], token offsets into the packed K/V arrays
    q: np.ndarray             # uint16 bf16 bits [B, h, d]
    k: Optional[np.ndarray]   # GQA: uint16 [S_tot, h_kv, d]
    v: Optional[np.ndarray]   # GQA: uint16 [S_tot, h_kv, d]
    c_kv: Optional[np.ndarray]  # MLA: uint16 [S_tot, d_c]
    k_r: Optional[np.ndarray]   # MLA: uint16 [S_tot, d_rope]
    block_table: np.ndarray   # int32 [B, max_blocks]; -1 marks unused entries
    num_blocks: int           # pool size in blocks (used + spare)
    k_scale: float = 1.0      # FP8 per-tensor scales (float32 values)
    v_scale: float = 1.0
    meta: dict = field(default_factory=dict)

    @property
    def g(self) -> int:
        return self.h // self.h_kv

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "fp8" else 2

    @property
    def dv(self) -> int:
        return self.d_c if self.kind == "mla" else self.d

    def kv_bytes(self) -> int:
        """Algorithmic KV bytes one decode reads: every cached element of every
        context token exactly once."""
        if self.kind == "mla":
            return self.total_tokens * (self.d_c + self.d_rope) * self.elem_bytes
        return self.total_tokens * self.h_kv * 2 * self.d * self.elem_bytes

    def flops(self) -> int:
        """Attention FLOPs one decode performs (q.k and p.v, 2 per MAC)."""
        if self.kind == "mla":
            return self.total_tokens * 2 * self.h * ((self.d_c + self.d_rope) + self.d_c)
        return self.total_tokens * self.h_kv * 4 * self.g * self.d

    def seq_slice(self, b: int) -> slice:
        return slice(int(self.cu_seqlens[b]), int(self.cu_seqlens[b + 1]))

    def append_indices(self):
        """(seq_idx, pos) int32 arrays that place every packed token at its
        position: token n of sequence b goes to position n - cu[b]."""
        seq_idx = np.repeat(np.arange(self.B, dtype=np.int32), self.seq_lens.astype(np.int64))
        pos = (np.arange(self.total_tokens, dtype=np.int64)
               - np.repeat(self.cu_seqlens[:-1], self.seq_lens.astype(np.int64))).astype(np.int32)
        return seq_idx, pos


def make_block_table(seq_lens: np.ndarray, bs: int, how: str, seed: int,
                     spare_frac: float = 0.02, max_blocks: Optional[int] = None):
    """Block table for the given lengths: "identity" gives each sequence
    consecutive blocks (a contiguous cache); "permuted" hands out a random
    permutation of a pool that holds exactly the blocks needed plus
    ``spare_frac`` never-referenced spare blocks."""
    nb = cdiv(seq_lens.astype(np.int64), bs)
    used = int(nb.sum())
    mb = int(max(1, nb.max() if len(nb) else 1)) if max_blocks is None else int(max_blocks)
    table = np.full((len(seq_lens), mb), -1, dtype=np.int32)
    if how == "identity":
        num_blocks = max(used, 1)
        ids = np.arange(used, dtype=np.int32)
    elif how == "permuted":
        spare = int(math.ceil(used * spare_frac)) + 1
        num_blocks = used + spare
        ids = rng_for(seed, "table").permutation(num_blocks)[:used].astype(np.int32)
    else:
        raise ValueError(how)
    off = 0
    for b, n in enumerate(nb):
        table[b, :n] = ids[off:off + n]
        off += int(n)
    return table, num_blocks


def make_workload(name: str, seed: int = 0, batch: Optional[int] = None,
                  lens=None, block_size: Optional[int] = None, table: Optional[str] = None,
                  q_scale: float = 1.0, heads: Optional[int] = None) -> Workload:
    """Build a named workload.  ``batch``/``lens``/``block_size``/``table``
    override the recipe (smaller parity cases of the same shapes);
    ``q_scale`` multiplies the query spread (large-logit stress cases);
    ``heads`` (MLA only) draws queries for fewer query heads."""
    r = dict(WORKLOADS[name])
    B = int(batch if batch is not None else r["B"])
    if lens is not None:
        seq_lens = np.asarray(lens, dtype=np.int32)
        B = len(seq_lens)
    else:
        seq_lens = draw_lengths(r["lens"], B, seed)
    bs = int(block_size if block_size is not None else r["bs"])
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(seq_lens.astype(np.int64))
    S = int(cu[-1])
    table_kind = table if table is not None else r["table"]
    bt, num_blocks = make_block_table(seq_lens, bs, table_kind, seed)

    if r["kind"] == "mla":
        d_c, d_rope, h = r["d_c"], r["d_rope"], int(heads or r["h"])
        d = d_c + d_rope
        q = normal_bf16(rng_for(seed, "q"), B * h * d, r["q_std"] * q_scale).reshape(B, h, d)
        c_kv = normal_bf16(rng_for(seed, "c_kv"), S * d_c).reshape(S, d_c)
        k_r = normal_bf16(rng_for(seed, "k_r"), S * d_rope).reshape(S, d_rope)
        wl = Workload(name=name, kind="mla", B=B, h=h, h_kv=1, d=d, d_c=d_c, d_rope=d_rope,
                      block_size=bs, kv_dtype=r["kv_dtype"], scale=float(r["scale"]),
                      seq_lens=seq_lens, cu_seqlens=cu, q=q, k=None, v=None,
                      c_kv=c_kv, k_r=k_r, block_table=bt, num_blocks=num_blocks)
        if wl.kv_dtype == "fp8":
            # per-tensor scales amax / 448 in float32: k_scale for c_KV, v_scale for k_R
            wl.k_scale = fp8_scale(c_kv)
            wl.v_scale = fp8_scale(k_r)
        return wl

    if heads is not None:
        raise ValueError("heads overrides the query heads of MLA workloads only")
    h, h_kv, d = r["h"], r["h_kv"], r["d"]
    q = normal_bf16(rng_for(seed, "q"), B * h * d, r["q_std"] * q_scale).reshape(B, h, d)
    k = normal_bf16(rng_for(seed, "k"), S * h_kv * d).reshape(S, h_kv, d)
    v = normal_bf16(rng_for(seed, "v"), S * h_kv * d).reshape(S, h_kv, d)
    wl = Workload(name=name, kind="gqa", B=B, h=h, h_kv=h_kv, d=d, d_c=0, d_rope=0,
                  block_size=bs, kv_dtype=r["kv_dtype"], scale=1.0 / math.sqrt(d),
                  seq_lens=seq_lens, cu_seqlens=cu, q=q, k=k, v=v, c_kv=None, k_r=None,
                  block_table=bt, num_blocks=num_blocks)
    if wl.kv_dtype == "fp8":
        wl.k_scale = fp8_scale(k)
        wl.v_scale = fp8_scale(v)
    return wl


def fp8_scale(bits: np.ndarray) -> float:
    """Per-tensor E4M3 scale = amax / 448 (448 is the largest finite E4M3
    value), evaluated in float32 over the stored bf16 values."""
    amax = np.float32(np.abs(bf16_to_f32(bits)).max()) if bits.size else np.float32(1.0)
    return float(amax / np.float32(448.0)) if amax > 0 else 1.0


def multi_token_queries(wl: Workload, q_len: int, seed: int = 0) -> np.ndarray:
    """Queries of q_len new tokens per sequence for a GQA workload (speculative
    verification): [B][q_len][h][d] bf16 bits, drawn like the single-token q.
    The new tokens are the last q_len cached tokens of each sequence."""
    assert wl.kind == "gqa"
    r = WORKLOADS[wl.name]
    n = wl.B * q_len * wl.h * wl.d
    return normal_bf16(rng_for(seed, f"q_multi{q_len}"), n, r["q_std"]).reshape(
        wl.B, q_len, wl.h, wl.d)


@dataclass
class MlaProjections:
    """Inputs of the per-head projections around MLA decode (bf16 bits)."""
    q_nope: np.ndarray        # [B][h][d_hc]  q^C ~ N(0, 1)
    q_rope: np.ndarray        # [B][h][d_rope] q^R ~ N(0, 1/(d_c + d_rope))
    w_uk: np.ndarray          # [h][d_hc][d_c] ~ N(0, 1/(d_hc (d_c + d_rope)))
    w_uv: np.ndarray          # [h][d_v][d_c] ~ N(0, 1/d_c)


def mla_projections(B: int, h: int = 128, d_hc: int = 128, d_c: int = 512, d_rope: int = 64,
                    d_v: int = 128, seed: int = 0) -> MlaProjections:
    """Random weights and un-absorbed queries shaped like DeepSeek-V3's MLA.
    The spreads make W_UK^T q^C ~ N(0, 1/(d_c + d_rope)), the spread of the
    absorbed query in the MLA decode workload."""
    w = d_c + d_rope
    return MlaProjections(
        q_nope=normal_bf16(rng_for(seed, "q_nope"), B * h * d_hc).reshape(B, h, d_hc),
        q_rope=normal_bf16(rng_for(seed, "q_rope"), B * h * d_rope, w ** -0.5).reshape(B, h, d_rope),
        w_uk=normal_bf16(rng_for(seed, "w_uk"), h * d_hc * d_c, (d_hc * w) ** -0.5).reshape(h, d_hc, d_c),
        w_uv=normal_bf16(rng_for(seed, "w_uv"), h * d_v * d_c, d_c ** -0.5).reshape(h, d_v, d_c))


def prefill_queries(B: int, q_len: int, h: int = 128, d_hc: int = 128, d_rope: int = 64,
                    seed: int = 0, q_scale: float = 1.0):
    """Un-absorbed queries of q_len new tokens per sequence for the explicit-form
    MLA prefill, spread like mla_projections' single-token queries:
    q_nope [B][q_len][h][d_hc], q_rope [B][q_len][h][d_rope] bf16 bits."""
    w = 512 + d_rope
    q_nope = normal_bf16(rng_for(seed, f"pf_q_nope{q_len}"), B * q_len * h * d_hc, q_scale)
    q_rope = normal_bf16(rng_for(seed, f"pf_q_rope{q_len}"), B * q_len * h * d_rope,
                         q_scale * w ** -0.5)
    return q_nope.reshape(B, q_len, h, d_hc), q_rope.reshape(B, q_len, h, d_rope)


def plant_needle(wl: Workload, b: int, head: int, t: int, strength: float = 30.0):
    """Overwrite K[t] of sequence b (the KV head that ``head`` reads) with
    ``strength * q/|q|`` so that one key dominates the softmax of that head."""
    assert wl.kind == "gqa"
    qv = bf16_to_f32(wl.q[b, head]).astype(np.float64)
    vec = strength * qv / np.linalg.norm(qv)
    wl.k[int(wl.cu_seqlens[b]) + t, head // wl.g] = bf16_bits(vec.astype(np.float32))


def plant_needle_mla(wl: Workload, b: int, head: int, t: int, strength: float = 300.0):
    """Overwrite latent row t of sequence b with ``strength * q~/|q~|`` of one
    head, so that row dominates that head's softmax."""
    assert wl.kind == "mla"
    qv = bf16_to_f32(wl.q[b, head]).astype(np.float64)
    vec = (strength * qv / np.linalg.norm(qv)).astype(np.float32)
    n = int(wl.cu_seqlens[b]) + t
    wl.c_kv[n] = bf16_bits(vec[: wl.d_c])
    wl.k_r[n] = bf16_bits(vec[wl.d_c:])
