"""Explicit-form ("MHA mode") MLA prefill on the GPU vs the float64 oracle.

q_len new tokens per sequence, already in the paged latent cache, attend
causally with per-head keys [W_UK c | k_R] and values W_UV c expanded from the
latent ("MLA：为什么一份 Latent 可以代替多头 KV Cache", sections "MHA Mode" and
"Prefill 为什么未必使用与 Decode 相同的吸收方式").  The oracle is the plain
definition in float64 (oracle.mla_prefill, pinned on the CPU against causal
SDPA); the GPU keeps the expanded keys and values in bf16."""
import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from _harness import GpuWorkload, TOL_ABS_BF16, TOL_RELRMS, TOL_LSE, dev_bits, errors

pytestmark = pytest.mark.gpu


def _run(wl, q_len, h, seed=0, q_scale=1.0, poison=True):
    import torch
    g = GpuWorkload(wl, poison=poison)
    qn, qr = inputs.prefill_queries(wl.B, q_len, h=h, seed=seed, q_scale=q_scale)
    pj = inputs.mla_projections(1, h=h, seed=seed)
    out = torch.full((wl.B, q_len, h, 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((wl.B, q_len, h), float("nan"), dtype=torch.float32, device="cuda")
    g.err.zero_()
    kv.kvattn_mla_prefill(dev_bits(qn), dev_bits(qr), g.cache.descriptor(), g.bt, g.seq_lens,
                          dev_bits(pj.w_uk), dev_bits(pj.w_uv), wl.scale, out, lse, err=g.err)
    torch.cuda.synchronize()
    return g, qn, qr, pj, out.cpu().numpy(), lse.cpu().numpy()


def _oracle(oracle, wl, b, qn, qr, pj, heads):
    f64 = lambda bits: inputs.bf16_to_f32(bits).astype(np.float64)
    sl = wl.seq_slice(b)
    return oracle.mla_prefill(f64(qn[b][:, heads]), f64(qr[b][:, heads]), f64(wl.c_kv[sl]),
                              f64(wl.k_r[sl]), f64(pj.w_uk[heads]), f64(pj.w_uv[heads]), wl.scale)


def _check(oracle, wl, q_len, h, heads, **kw):
    g, qn, qr, pj, out, lse = _run(wl, q_len, h, **kw)
    assert g.err_bits() == 0
    assert np.isfinite(out).all()
    got, ref, gl, rl = [], [], [], []
    for b in range(wl.B):
        ro, rls = _oracle(oracle, wl, b, qn, qr, pj, heads)
        got.append(out[b][:, heads])
        ref.append(ro)
        gl.append(lse[b][:, heads])
        rl.append(rls)
    got, ref, gl, rl = map(np.stack, (got, ref, gl, rl))
    max_abs, rel = errors(got, ref)
    assert max_abs <= TOL_ABS_BF16, max_abs
    assert rel <= TOL_RELRMS, rel
    assert (np.isneginf(gl) == np.isneginf(rl)).all()
    fin = np.isfinite(rl)
    if fin.any():
        assert np.abs(gl[fin] - rl[fin]).max() <= TOL_LSE
    return out, lse


def test_one_tile_of_new_tokens(oracle):
    wl = inputs.make_workload("deepseek_v3_mla", lens=[70, 200], heads=8)
    _check(oracle, wl, 16, 8, list(range(8)))


def test_two_query_tiles_ragged(oracle):
    # 130 new tokens: a full tile of 128 and a ragged one of 2; prefixes cross
    # several 128-row tiles and end inside a page
    wl = inputs.make_workload("deepseek_v3_mla", lens=[300, 1000, 130], heads=4)
    _check(oracle, wl, 130, 4, list(range(4)))


def test_sequences_shorter_than_the_chunk(oracle):
    # 5 new tokens in sequences of 3, 0 and 17 rows: tokens without a position
    # see nothing (out 0, lse -inf), an empty sequence is all such tokens
    wl = inputs.make_workload("deepseek_v3_mla", lens=[3, 0, 17], heads=4)
    out, lse = _check(oracle, wl, 5, 4, list(range(4)))
    assert (out[0, :2] == 0).all() and np.isneginf(lse[0, :2]).all()
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()


def test_large_logits(oracle):
    # queries 8x larger: peaked softmax, the lazy rescale of O is exercised
    wl = inputs.make_workload("deepseek_v3_mla", lens=[900, 2000], heads=4)
    _check(oracle, wl, 40, 4, list(range(4)), q_scale=8.0)


def test_last_token_equals_absorbed_decode(oracle):
    # the last new token sees the whole sequence: its output equals the absorbed
    # path (query absorption, decode over the latent, value up-projection)
    import torch
    wl = inputs.make_workload("deepseek_v3_mla", lens=[777, 2048])
    h = wl.h
    g, qn, qr, pj, out, lse = _run(wl, 8, h)
    q_abs = torch.empty((wl.B, h, 576), dtype=torch.int16, device="cuda")
    kv.kvattn_mla_absorb_q(dev_bits(np.ascontiguousarray(qn[:, -1])),
                           dev_bits(np.ascontiguousarray(qr[:, -1])), dev_bits(pj.w_uk), q_abs,
                           err=g.err)
    g.q = q_abs
    u, l_dec = g.decode()
    ut = torch.from_numpy(u).cuda()
    v = torch.empty((wl.B, h, 128), dtype=torch.float32, device="cuda")
    kv.kvattn_mla_up_v(ut, dev_bits(pj.w_uv), v, err=g.err)
    torch.cuda.synchronize()
    assert g.err_bits() == 0
    vn = v.cpu().numpy()
    max_abs, rel = errors(out[:, -1], vn.astype(np.float64))
    assert max_abs <= TOL_ABS_BF16 and rel <= TOL_RELRMS, (max_abs, rel)
    assert np.abs(lse[:, -1] - l_dec).max() <= TOL_LSE


def test_deepseek_v3_shape_sampled_heads(oracle):
    # all 128 heads, 2 sequences of 4096 cached rows, a 256-token chunk; the
    # oracle checks three heads of every new token
    wl = inputs.make_workload("deepseek_v3_mla", lens=[4096, 3000])
    _check(oracle, wl, 256, 128, [0, 77, 127])
