"""The bounded-wait abort path of the GQA decode kernels, run on the GPU.

Every wait of the decode kernels on an mbarrier gives up after a time limit,
reports KVATTN_DEVERR_TIMEOUT in the caller's error word and ends the kernel
(stop issuing, wait for the copies still landing, exit), so that a lost copy or
a protocol bug costs one wrong result instead of a hung GPU.  The library's
own build never takes that path, so this test builds a variant of it
(`_build.build_wait_test`): every main-loop wait gives up after 2 ms (the
drains on the way out keep their full limit), and the producer
of CTA 0 neither loads nor signals chunk 3 of its walk, as if that copy never
landed.  Nothing faults and nothing waits without a limit: the consumer's wait
on that stage runs out, and the rest of CTA 0 follows the abort path.

Checks: the call returns, the stream synchronises within a second, the error
word holds the timeout bit and nothing else, the sequences that other CTAs
walked are still right, and afterwards the library's own build decodes the
same cache correctly in the same context.

The same build drops tile 3 of CTA 0's walk in the tcgen05 kernel (units of
many rows: 8 new tokens on Llama-3-70B shapes, bf16 and E4M3 caches): the
first producer warp issues none of that tile's loads, so its barrier never
completes and the score issuer, the softmax warps and then every other role
of CTA 0 take the abort path, the producers draining with the full limit.

And the MLA decode's CTA pair (bf16 and E4M3 latent caches): rank 0 of pair
0 arms tile 3's barrier but loads nothing, so its score MMAs never run, the
peer waits in vain for that tile's partial scores, and both ranks abort,
drain the exchange and meet at the final cluster barrier.

And the explicit-form MLA prefill: the CTA of (query tile 0, head 0,
sequence 0) arms chunk 3 of its expansion but loads nothing; its MMA issuer
and compute warps time out and it drains, while the other (head, sequence)
CTAs finish normally.

And the two per-head projection GEMMs around the MLA decode: the CTA of
head 0 arms part 1 of W_UK (query absorption) or chunk 3 of W_UV (value
up-projection) but loads nothing; it times out and drains, and the other
heads' results are right.
"""
import ctypes
import time

import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import _build, inputs
from kv_cache_decode_paged_gb300.device import GpuWorkload, dev_bits

from _harness import (TOL_ABS_BF16, TOL_LSE, TOL_RELRMS, assert_parity, errors, oracle_all,
                      oracle_multi)

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_ends_the_kernel_with_a_timeout(oracle):
    import torch
    lib = kv.open_library(_build.build_wait_test())
    # 8 sequences of 1024 tokens over 8 CTAs: the planner gives each CTA the
    # same number of pages, in (sequence, KV head, page) order, so CTA 0
    # walks sequence 0 and no other.
    wl = inputs.make_workload("llama3_8b", lens=[1024] * 8)
    g = GpuWorkload(wl)
    ws = g.workspace(num_ctas=8)
    out = torch.full((wl.B, wl.h, wl.d), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((wl.B, wl.h), float("nan"), dtype=torch.float32, device="cuda")
    g.err.zero_()
    torch.cuda.synchronize()
    desc = g.cache.descriptor()
    t0 = time.monotonic()
    status = lib.kvattn_decode_gqa(
        g.q.data_ptr(), ctypes.byref(desc), g.bt.data_ptr(), g.seq_lens.data_ptr(), wl.B,
        wl.max_blocks, wl.h, wl.h_kv, wl.d, wl.scale, out.data_ptr(), lse.data_ptr(),
        ws.data_ptr(), ws.numel() * ws.element_size(), 8, g.err.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == kv.KVATTN_OK
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert elapsed < 1.0, f"aborted decode took {elapsed:.3f} s"
    assert g.err_bits() == kv.KVATTN_DEVERR_TIMEOUT

    # the CTAs that walked other sequences finished normally
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    keep = range(2, wl.B)
    ref_out, ref_lse = oracle_all(oracle, wl, seqs=keep)
    assert_parity(o, l, ref_out, ref_lse)

    # the context is intact: the library's own build decodes the same cache
    g.err.zero_()
    o2, l2 = g.decode(num_ctas=8)
    assert g.err_bits() == 0
    ref_out, ref_lse = oracle_all(oracle, wl)
    assert_parity(o2, l2, ref_out, ref_lse)
    assert np.isfinite(o2).all()


@pytest.mark.parametrize("name", ["llama3_70b", "llama3_70b_fp8"])
def test_tc_wait_that_runs_out_ends_the_kernel_with_a_timeout(oracle, name):
    import torch
    lib = kv.open_library(_build.build_wait_test())
    # 8 sequences of 1024 tokens, 8 KV heads, over 8 CTAs: CTA c owns pages
    # [c T / 8, (c + 1) T / 8) of the (sequence, KV head, page) order, so CTA 0
    # walks the eight units of sequence 0 and no other.  8 new tokens: 64 rows
    # per unit, the tcgen05 kernel.
    wl = inputs.make_workload(name, lens=[1024] * 8)
    q_len = 8
    qm = inputs.multi_token_queries(wl, q_len)
    g = GpuWorkload(wl)
    q = dev_bits(qm)
    ws = kv.workspace_for(kv.KVATTN_GQA, wl.B, wl.h * q_len, wl.h_kv, wl.d, 8, "cuda")
    out = torch.full((wl.B, q_len, wl.h, wl.d), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((wl.B, q_len, wl.h), float("nan"), dtype=torch.float32, device="cuda")
    g.err.zero_()
    torch.cuda.synchronize()
    desc = g.cache.descriptor()
    t0 = time.monotonic()
    status = lib.kvattn_decode_gqa_multi(
        q.data_ptr(), ctypes.byref(desc), g.bt.data_ptr(), g.seq_lens.data_ptr(), wl.B,
        wl.max_blocks, q_len, wl.h, wl.h_kv, wl.d, wl.scale, out.data_ptr(), lse.data_ptr(),
        ws.data_ptr(), ws.numel() * ws.element_size(), 8, g.err.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == kv.KVATTN_OK
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert elapsed < 1.0, f"aborted decode took {elapsed:.3f} s"
    assert g.err_bits() == kv.KVATTN_DEVERR_TIMEOUT

    fp8 = wl.kv_dtype == "fp8"
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    ref_out, ref_lse = oracle_multi(oracle, wl, qm, seqs=range(1, wl.B))
    assert_parity(o, l, ref_out, ref_lse, fp8=fp8)

    # the library's own build decodes the same cache in the same context
    g.err.zero_()
    o2, l2 = g.decode_multi(qm, num_ctas=8)
    assert g.err_bits() == 0
    ref_out, ref_lse = oracle_multi(oracle, wl, qm)
    assert_parity(o2, l2, ref_out, ref_lse, fp8=fp8)


@pytest.mark.parametrize("name", ["deepseek_v3_mla", "deepseek_v3_mla_fp8"])
def test_mla_pair_wait_that_runs_out_ends_the_kernel_with_a_timeout(oracle, name):
    import torch
    lib = kv.open_library(_build.build_wait_test())
    # 8 sequences of 1024 tokens on 8 CTA pairs: one pair per sequence (no
    # split, no merge), so pair 0 (CTAs 0 and 1) walks sequence 0 alone
    wl = inputs.make_workload(name, lens=[1024] * 8)
    g = GpuWorkload(wl)
    ws = g.workspace(num_ctas=8)
    out = torch.full((wl.B, wl.h, wl.d_c), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((wl.B, wl.h), float("nan"), dtype=torch.float32, device="cuda")
    g.err.zero_()
    torch.cuda.synchronize()
    desc = g.cache.descriptor()
    t0 = time.monotonic()
    status = lib.kvattn_decode_mla(
        g.q.data_ptr(), ctypes.byref(desc), g.bt.data_ptr(), g.seq_lens.data_ptr(), wl.B,
        wl.max_blocks, wl.h, wl.d_c, wl.d_rope, wl.scale, out.data_ptr(), lse.data_ptr(),
        ws.data_ptr(), ws.numel() * ws.element_size(), 8, g.err.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == kv.KVATTN_OK
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert elapsed < 2.0, f"aborted decode took {elapsed:.3f} s"
    assert g.err_bits() == kv.KVATTN_DEVERR_TIMEOUT

    fp8 = wl.kv_dtype == "fp8"
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    ref_out, ref_lse = oracle_all(oracle, wl, seqs=range(1, wl.B))
    assert_parity(o, l, ref_out, ref_lse, fp8=fp8)

    g.err.zero_()
    o2, l2 = g.decode(num_ctas=8)
    assert g.err_bits() == 0
    ref_out, ref_lse = oracle_all(oracle, wl)
    assert_parity(o2, l2, ref_out, ref_lse, fp8=fp8)


def test_prefill_wait_that_runs_out_ends_the_kernel_with_a_timeout(oracle):
    import torch
    lib = kv.open_library(_build.build_wait_test())
    h, q_len = 4, 16
    wl = inputs.make_workload("deepseek_v3_mla", lens=[300, 200], heads=h)
    g = GpuWorkload(wl)
    qn, qr = inputs.prefill_queries(wl.B, q_len, h=h)
    pj = inputs.mla_projections(1, h=h)
    dq, dr, wk, wv = (dev_bits(x) for x in (qn, qr, pj.w_uk, pj.w_uv))

    def run(call):
        out = torch.full((wl.B, q_len, h, 128), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((wl.B, q_len, h), float("nan"), dtype=torch.float32, device="cuda")
        g.err.zero_()
        torch.cuda.synchronize()
        t0 = time.monotonic()
        call(out, lse)
        torch.cuda.synchronize()
        return out.cpu().numpy(), lse.cpu().numpy(), time.monotonic() - t0

    desc = g.cache.descriptor()
    o, l, elapsed = run(lambda out, lse: lib.kvattn_mla_prefill(
        dq.data_ptr(), dr.data_ptr(), ctypes.byref(desc), g.bt.data_ptr(), g.seq_lens.data_ptr(),
        wl.B, wl.max_blocks, q_len, h, 128, 128, wk.data_ptr(), wv.data_ptr(), wl.scale,
        out.data_ptr(), lse.data_ptr(), g.err.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    assert elapsed < 1.0, f"aborted prefill took {elapsed:.3f} s"
    assert g.err_bits() == kv.KVATTN_DEVERR_TIMEOUT

    f64 = lambda bits: inputs.bf16_to_f32(bits).astype(np.float64)

    def check(o, l, skip):
        for b in range(wl.B):
            sl = wl.seq_slice(b)
            ref_o, ref_l = oracle.mla_prefill(f64(qn[b]), f64(qr[b]), f64(wl.c_kv[sl]),
                                              f64(wl.k_r[sl]), f64(pj.w_uk), f64(pj.w_uv),
                                              wl.scale)
            for hd in range(h):
                if (b, hd) == skip:
                    continue
                got = o[b][:, hd]
                assert np.isfinite(got).all()
                max_abs, rel = errors(got, ref_o[:, hd])
                assert max_abs <= TOL_ABS_BF16 and rel <= TOL_RELRMS, (b, hd, max_abs, rel)
                assert np.abs(l[b][:, hd] - ref_l[:, hd]).max() <= TOL_LSE

    # every (sequence, head) but the aborted CTA's is right
    check(o, l, skip=(0, 0))

    # the library's own build, same context: all of them
    o2, l2, _ = run(lambda out, lse: kv.kvattn_mla_prefill(
        dq, dr, g.cache.descriptor(), g.bt, g.seq_lens, wk, wv, wl.scale, out, lse, err=g.err))
    assert g.err_bits() == 0
    check(o2, l2, skip=None)


def _absorb_bounds_ok(oracle, got, pj, heads):
    f32 = lambda bits: inputs.bf16_to_f32(bits).astype(np.float64)
    w = f32(pj.w_uk)
    d_c = pj.w_uk.shape[2]
    for b in range(pj.q_nope.shape[0]):
        qc = f32(pj.q_nope[b])
        ref = oracle.mla_absorb_query(qc, w)
        absdot = np.einsum("hj,hjc->hc", np.abs(qc), np.abs(w))
        # products exact in float32, a K-term float32 sum, then bf16 rounding
        bound = 2.0 ** -8 * np.abs(ref) + (1 + 2.0 ** -8) * qc.shape[1] * 2.0 ** -23 * absdot
        g = f32(got[b, :, :d_c])
        assert not (np.abs(g - ref) > bound)[heads].any(), b
        np.testing.assert_array_equal(got[b, heads, d_c:], pj.q_rope[b, heads])


def test_absorb_wait_that_runs_out_ends_the_kernel_with_a_timeout(oracle):
    import torch
    lib = kv.open_library(_build.build_wait_test())
    B, h = 4, 4
    pj = inputs.mla_projections(B, h=h, seed=11)
    qn, qr, wk = dev_bits(pj.q_nope), dev_bits(pj.q_rope), dev_bits(pj.w_uk)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_abs = torch.full((B, h, 576), -1, dtype=torch.int16, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    status = lib.kvattn_mla_absorb_q(qn.data_ptr(), qr.data_ptr(), wk.data_ptr(), B, h, 128, 512,
                                     64, q_abs.data_ptr(), err.data_ptr(),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == kv.KVATTN_OK
    torch.cuda.synchronize()
    assert time.monotonic() - t0 < 1.0
    assert int(err.item()) == kv.KVATTN_DEVERR_TIMEOUT
    _absorb_bounds_ok(oracle, q_abs.cpu().numpy().view(np.uint16), pj, slice(1, h))

    err.zero_()
    q_abs.fill_(-1)
    kv.kvattn_mla_absorb_q(qn, qr, wk, q_abs, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _absorb_bounds_ok(oracle, q_abs.cpu().numpy().view(np.uint16), pj, slice(0, h))


def test_up_v_wait_that_runs_out_ends_the_kernel_with_a_timeout(oracle):
    import torch
    lib = kv.open_library(_build.build_wait_test())
    B, h, d_c = 4, 4, 512
    pj = inputs.mla_projections(B, h=h, d_c=d_c, seed=13)
    d_v = pj.w_uv.shape[1]
    u = inputs.rng_for(B, "u_tilde").standard_normal((B, h, d_c), dtype=np.float32) * np.float32(0.05)
    ud, wv = torch.from_numpy(u).cuda(), dev_bits(pj.w_uv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    v = torch.full((B, h, d_v), float("nan"), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.monotonic()
    status = lib.kvattn_mla_up_v(ud.data_ptr(), wv.data_ptr(), B, h, d_c, d_v, v.data_ptr(),
                                 err.data_ptr(),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == kv.KVATTN_OK
    torch.cuda.synchronize()
    assert time.monotonic() - t0 < 1.0
    assert int(err.item()) == kv.KVATTN_DEVERR_TIMEOUT
    w = inputs.bf16_to_f32(pj.w_uv).astype(np.float64)

    def check(got, heads):
        for b in range(B):
            ub = u[b].astype(np.float64)
            ref = oracle.mla_apply_wuv(ub, w)
            absdot = np.einsum("hc,hvc->hv", np.abs(ub), np.abs(w))
            # u~ rounded to bf16, then a K-term float32 sum
            bound = (2.0 ** -8 + d_c * 2.0 ** -23) * absdot * (1 + 2.0 ** -8)
            assert not (np.abs(got[b] - ref) > bound)[heads].any(), b

    check(v.cpu().numpy().astype(np.float64), slice(1, h))
    err.zero_()
    v.fill_(float("nan"))
    kv.kvattn_mla_up_v(ud, wv, v, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check(v.cpu().numpy().astype(np.float64), slice(0, h))
