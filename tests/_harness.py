"""Shared test plumbing: put a workload on the GPU through the C ABI, run the
oracle on the same stored values, and measure the difference."""
from __future__ import annotations

import numpy as np

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300.device import GpuWorkload, dev_bits  # noqa: F401
from kv_cache_decode_paged_gb300 import inputs

# Parity tolerances of the decode outputs: bf16 caches max |err| <= 2e-2 and
# relative RMS <= 1e-2; FP8 caches max |err| <= 5e-2.
TOL_ABS_BF16 = 2e-2
TOL_RELRMS = 1e-2
TOL_ABS_FP8 = 5e-2
TOL_LSE = 2e-2


def oracle_seq(oracle, wl: inputs.Workload, b: int):
    """Oracle output for sequence b on the stored values (bf16 or E4M3 codes)."""
    sl = wl.seq_slice(b)
    if wl.kind == "mla":
        if wl.kv_dtype == "fp8":
            return oracle.mla_decode_e4m3(wl.q[b], mla_codes(oracle, wl, sl), wl.d_c, wl.scale,
                                          wl.k_scale, wl.v_scale)
        rows = np.concatenate([wl.c_kv[sl], wl.k_r[sl]], axis=1)
        return oracle.mla_decode(wl.q[b], rows, wl.d_c, wl.scale)
    if wl.kv_dtype == "fp8":
        kc = oracle.quantize_e4m3(wl.k[sl], wl.k_scale)
        vc = oracle.quantize_e4m3(wl.v[sl], wl.v_scale)
        return oracle.gqa_decode(wl.q[b], kc, vc, wl.scale, fmt=oracle.FMT_E4M3,
                                 k_scale=wl.k_scale, v_scale=wl.v_scale)
    return oracle.gqa_decode(wl.q[b], wl.k[sl], wl.v[sl], wl.scale)


def mla_codes(oracle, wl: inputs.Workload, sl):
    """The stored E4M3 latent rows of tokens sl: c_KV codes (scale k_scale)
    then k_R codes (scale v_scale)."""
    return np.concatenate([oracle.quantize_e4m3(wl.c_kv[sl], wl.k_scale),
                           oracle.quantize_e4m3(wl.k_r[sl], wl.v_scale)], axis=1)


def oracle_all(oracle, wl, seqs=None):
    seqs = range(wl.B) if seqs is None else seqs
    outs, lses = {}, {}
    for b in seqs:
        outs[b], lses[b] = oracle_seq(oracle, wl, b)
    return outs, lses


def errors(got: np.ndarray, ref: np.ndarray):
    """(max |err|, relative RMS = ||got - ref||_2 / ||ref||_2)."""
    d = got.astype(np.float64) - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d) / den) if den > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def assert_parity(out, lse, ref_out: dict, ref_lse: dict, fp8=False):
    seqs = sorted(ref_out)
    got = np.stack([out[b] for b in seqs])
    ref = np.stack([ref_out[b] for b in seqs])
    max_abs, rel = errors(got, ref)
    assert np.isfinite(got).all(), "non-finite output"
    tol = TOL_ABS_FP8 if fp8 else TOL_ABS_BF16
    assert max_abs <= tol, f"max |err| {max_abs:.3e} > {tol}"
    assert rel <= TOL_RELRMS, f"relative RMS {rel:.3e} > {TOL_RELRMS}"
    gl = np.stack([lse[b] for b in seqs])
    rl = np.stack([ref_lse[b] for b in seqs])
    fin = np.isfinite(rl)
    assert (np.isneginf(gl) == np.isneginf(rl)).all()
    if fin.any():
        assert np.abs(gl[fin] - rl[fin]).max() <= TOL_LSE
    return max_abs, rel


def oracle_multi(oracle, wl: inputs.Workload, qm: np.ndarray, seqs=None):
    """Oracle rows of a multi-token decode: qm [B][q_len][h][d] bf16 bits."""
    seqs = range(wl.B) if seqs is None else seqs
    outs, lses = {}, {}
    for b in seqs:
        sl = wl.seq_slice(b)
        if wl.kv_dtype == "fp8":
            kc = oracle.quantize_e4m3(wl.k[sl], wl.k_scale)
            vc = oracle.quantize_e4m3(wl.v[sl], wl.v_scale)
            outs[b], lses[b] = oracle.gqa_decode_multi(qm[b], kc, vc, wl.scale, fmt=oracle.FMT_E4M3,
                                                       k_scale=wl.k_scale, v_scale=wl.v_scale)
        else:
            outs[b], lses[b] = oracle.gqa_decode_multi(qm[b], wl.k[sl], wl.v[sl], wl.scale)
    return outs, lses
