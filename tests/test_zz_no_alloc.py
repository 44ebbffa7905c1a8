"""kvattn_decode_gqa_noalloc, called through the C ABI.

This entry point serves callers that cannot give the library device memory
(plugin or custom-op interfaces that pass only inputs and outputs, runtimes
whose memory all belongs to their own pool, paths where cudaMalloc is not
allowed): its scratch is a fixed array inside the library.  Its results must
match kvattn_decode_gqa (which takes a caller workspace) within the parity
tolerance, on consecutive calls that reuse the same array.

The file name sorts last so a run that stops at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from kv_cache_decode_paged_gb300.device import GpuWorkload

pytestmark = pytest.mark.gpu

TOL_ABS = 2e-2     # same bounds as the oracle parity tests (bf16 cache)
TOL_RELRMS = 1e-2


def _call_noalloc(lib, g, out, lse, num_ctas=0):
    import torch
    wl = g.wl
    desc = g.cache.descriptor()
    return lib.kvattn_decode_gqa_noalloc(
        g.q.data_ptr(), ctypes.byref(desc), g.bt.data_ptr(), g.seq_lens.data_ptr(), wl.B,
        wl.max_blocks, wl.h, wl.h_kv, wl.d, wl.scale, out.data_ptr(), lse.data_ptr(), num_ctas,
        g.err.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(got, ref):
    d = got.astype(np.float64) - ref.astype(np.float64)
    rel = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)
    return np.abs(d).max() <= TOL_ABS and rel <= TOL_RELRMS


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    import torch
    lib = kv.load_library()
    # two different problems back to back: the second call finds the first
    # call's plan and partials still in the shared array
    cases = [inputs.make_workload("llama3_8b", lens=[4000, 37, 1024, 0, 777]),
             inputs.make_workload("long_mqa", lens=[9000, 129, 2])]
    for wl in cases:
        g = GpuWorkload(wl)
        ref_out, ref_lse = g.decode()                    # caller-workspace entry point
        out = torch.full((wl.B, wl.h, wl.d), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((wl.B, wl.h), float("nan"), dtype=torch.float32, device="cuda")
        g.err.zero_()
        assert _call_noalloc(lib, g, out, lse) == kv.KVATTN_OK
        torch.cuda.synchronize()
        assert g.err_bits() == 0
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert np.isfinite(o).all()
        assert _close(o, ref_out)
        fin = np.isfinite(ref_lse)
        assert (np.isneginf(l) == np.isneginf(ref_lse)).all()
        assert np.abs(l[fin] - ref_lse[fin]).max() <= TOL_ABS


def test_noalloc_back_to_back_calls_with_split_units():
    # Two problems enqueued one right after the other on one stream, with no
    # synchronisation between them, both split over 8 CTAs so that each runs
    # its combine over partials in the shared array.  The second call's planner
    # must not overwrite the plan or the partials while the first call's
    # combine still reads them; each result is checked against its own
    # caller-workspace result after one final synchronisation.
    import torch
    lib = kv.load_library()
    cases = [inputs.make_workload("llama3_8b", lens=[4000, 37, 1024, 0, 777]),
             inputs.make_workload("llama3_70b", lens=[3000, 2500, 64])]
    gs = [GpuWorkload(wl) for wl in cases]
    refs = [g.decode(num_ctas=8) for g in gs]
    outs = []
    for g in gs:
        wl = g.wl
        g.err.zero_()
        outs.append((torch.full((wl.B, wl.h, wl.d), float("nan"), dtype=torch.float32,
                                device="cuda"),
                     torch.full((wl.B, wl.h), float("nan"), dtype=torch.float32, device="cuda")))
    torch.cuda.synchronize()
    for g, (out, lse) in zip(gs, outs):
        assert _call_noalloc(lib, g, out, lse, num_ctas=8) == kv.KVATTN_OK
    torch.cuda.synchronize()
    for g, (out, lse), (ref_out, ref_lse) in zip(gs, outs, refs):
        assert g.err_bits() == 0
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        assert np.isfinite(o).all()
        assert _close(o, ref_out)
        fin = np.isfinite(ref_lse)
        assert (np.isneginf(l) == np.isneginf(ref_lse)).all()
        assert np.abs(l[fin] - ref_lse[fin]).max() <= TOL_ABS


def test_noalloc_rejects_problems_beyond_the_scratch():
    import torch
    lib = kv.load_library()
    # 2048 sequences x 8 KV heads x 4 rows x 128 floats of partials needs far
    # more than the built-in scratch; real buffers of the stated sizes, all
    # lengths zero, so nothing could be read out of bounds even if it ran
    B, h, h_kv, d = 2048, 32, 8, 128
    need = kv.kvattn_decode_workspace_bytes(kv.KVATTN_GQA, B, h, h_kv, d, 304)
    assert need > kv.KVATTN_NOALLOC_SCRATCH_BYTES
    cache = kv.PagedCache.allocate_gqa(1, 16, h_kv, d)
    q = torch.zeros((B, h, d), dtype=torch.int16, device="cuda")
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    sl = torch.zeros((B,), dtype=torch.int32, device="cuda")
    out = torch.zeros((B, h, d), dtype=torch.float32, device="cuda")
    lse = torch.zeros((B, h), dtype=torch.float32, device="cuda")
    desc = cache.descriptor()
    st = lib.kvattn_decode_gqa_noalloc(q.data_ptr(), ctypes.byref(desc), bt.data_ptr(),
                                       sl.data_ptr(), B, 1, h, h_kv, d, 0.1, out.data_ptr(),
                                       lse.data_ptr(), 304, None, None)
    assert st == kv.KVATTN_ERR_WORKSPACE
