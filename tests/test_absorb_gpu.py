"""Per-head MLA projections on the GPU (query absorption, value up-projection)
against the float64 oracle, and the whole absorbed layer against the oracle's
explicit form."""
import math

import numpy as np
import pytest
import torch

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from _harness import GpuWorkload, assert_parity, dev_bits, errors

pytestmark = pytest.mark.gpu

# Elementwise bounds from the arithmetic.  Absorption: products of bf16 values
# are exact in float32; a K-term float32 sum is within K * 2^-23 * sum|terms|
# (taken generously for the tensor core's accumulation order); the result is
# then rounded to bf16 (unit roundoff 2^-8).  Up-projection: u~ is rounded to
# bf16 first (2^-8 of each |w u| term), then the same K-term float32 sum.
def absorb_bound(ref, absdot, k):
    return 2.0 ** -8 * np.abs(ref) + (1 + 2.0 ** -8) * k * 2.0 ** -23 * absdot


def up_bound(absdot, k):
    return (2.0 ** -8 + k * 2.0 ** -23) * absdot * (1 + 2.0 ** -8)


def f32(bits):
    return inputs.bf16_to_f32(bits).astype(np.float64)


def run_absorb(pj, err):
    B, h, d_hc = pj.q_nope.shape
    d_c, d_rope = pj.w_uk.shape[2], pj.q_rope.shape[2]
    q_abs = torch.full((B, h, d_c + d_rope), -1, dtype=torch.int16, device="cuda")  # NaN bits
    kv.kvattn_mla_absorb_q(dev_bits(pj.q_nope), dev_bits(pj.q_rope) if d_rope else None,
                           dev_bits(pj.w_uk), q_abs, err=err)
    torch.cuda.synchronize()
    return q_abs.cpu().numpy().view(np.uint16)


# d_c 512 is one pair of 256-column parts, 256 a single part, 768 a pair and
# a single; q^R of 136 is copied in two passes, 0 means no q^R at all
@pytest.mark.parametrize("B,h,d_c,d_rope", [(1, 128, 512, 64), (64, 128, 512, 64), (130, 16, 512, 64),
                                            (3, 1, 512, 64), (5, 3, 256, 136), (4, 2, 768, 64),
                                            (6, 2, 512, 0)])
def test_absorb_q(oracle, B, h, d_c, d_rope):
    pj = inputs.mla_projections(B, h=h, d_c=d_c, d_rope=d_rope, seed=B + h)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_absorb(pj, err)
    assert int(err.item()) == 0
    d_c = pj.w_uk.shape[2]
    w = f32(pj.w_uk)
    for b in range(B):
        qc = f32(pj.q_nope[b])
        ref = oracle.mla_absorb_query(qc, w)
        absdot = np.einsum("hj,hjc->hc", np.abs(qc), np.abs(w))
        g = f32(got[b, :, :d_c])
        bad = np.abs(g - ref) > absorb_bound(ref, absdot, qc.shape[1])
        assert not bad.any(), f"row {b}: {bad.sum()} elements outside the bound"
        # q^R is copied bit for bit behind the absorbed part
        np.testing.assert_array_equal(got[b, :, d_c:], pj.q_rope[b])


# d_c = 512 holds all of W_UV,i at once; 1024 refills the four-chunk ring;
# 128 and 384 are one and three chunks
@pytest.mark.parametrize("B,h,d_c", [(1, 128, 512), (64, 128, 512), (131, 8, 512), (5, 4, 1024),
                                     (9, 3, 128), (2, 2, 384)])
def test_up_v(oracle, B, h, d_c):
    pj = inputs.mla_projections(B, h=h, d_c=d_c, seed=7 * B + h)
    rng = inputs.rng_for(B, "u_tilde")
    d_v = pj.w_uv.shape[1]
    u = (rng.standard_normal((B, h, d_c), dtype=np.float32) * np.float32(0.05))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    v = torch.full((B, h, d_v), float("nan"), dtype=torch.float32, device="cuda")
    kv.kvattn_mla_up_v(torch.from_numpy(u).cuda(), dev_bits(pj.w_uv), v, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = v.cpu().numpy().astype(np.float64)
    w = f32(pj.w_uv)
    for b in range(B):
        ub = u[b].astype(np.float64)
        ref = oracle.mla_apply_wuv(ub, w)
        absdot = np.einsum("hc,hvc->hv", np.abs(ub), np.abs(w))
        bad = np.abs(got[b] - ref) > up_bound(absdot, d_c)
        assert not bad.any(), f"row {b}: {bad.sum()} elements outside the bound"
    max_abs, rel = errors(got, np.stack([oracle.mla_apply_wuv(u[b].astype(np.float64), w)
                                         for b in range(B)]))
    assert rel <= 1e-2


def test_empty_batch_and_bad_shapes():
    pj = inputs.mla_projections(2, h=4)
    q_abs = torch.empty((2, 4, 576), dtype=torch.int16, device="cuda")
    with pytest.raises(kv.KvattnError) as e:   # d_hc = 64 is not built
        kv.kvattn_mla_absorb_q(dev_bits(pj.q_nope[:, :, :64]), dev_bits(pj.q_rope),
                               dev_bits(pj.w_uk[:, :64]), q_abs)
    assert e.value.status == kv.KVATTN_ERR_UNSUPPORTED
    lib = kv.load_library()
    assert lib.kvattn_mla_up_v(None, None, 0, 4, 512, 128, None, None, None) == 0


@pytest.mark.parametrize("lens", [[200, 64, 1, 700]])
def test_absorbed_layer_equals_explicit_form(oracle, lens):
    """absorb -> append/decode -> up-projection on the GPU against the oracle's
    explicit (un-absorbed) MLA, which expands k = W_UK c and v = W_UV c."""
    wl = inputs.make_workload("deepseek_v3_mla", lens=lens)
    B, h = wl.B, wl.h
    pj = inputs.mla_projections(B, h=h, seed=3)
    g = GpuWorkload(wl)
    err = g.err
    q_abs = torch.empty((B, h, wl.d), dtype=torch.int16, device="cuda")
    kv.kvattn_mla_absorb_q(dev_bits(pj.q_nope), dev_bits(pj.q_rope), dev_bits(pj.w_uk), q_abs,
                           err=err)
    g.q = q_abs
    u_t, lse = g.decode()
    v = torch.empty((B, h, pj.w_uv.shape[1]), dtype=torch.float32, device="cuda")
    kv.kvattn_mla_up_v(torch.from_numpy(u_t).cuda(), dev_bits(pj.w_uv), v, err=err)
    torch.cuda.synchronize()
    assert g.err_bits() == 0
    got = v.cpu().numpy()
    ref_o, ref_l = {}, {}
    w_uk, w_uv = f32(pj.w_uk), f32(pj.w_uv)
    for b in range(B):
        sl = wl.seq_slice(b)
        ref_o[b], ref_l[b] = oracle.mla_explicit(f32(pj.q_nope[b]), f32(pj.q_rope[b]),
                                                 f32(wl.c_kv[sl]), f32(wl.k_r[sl]), w_uk, w_uv,
                                                 wl.scale)
    assert_parity({b: got[b] for b in range(B)}, {b: lse[b] for b in range(B)}, ref_o, ref_l)
