"""The bounded-wait abort path of the GQA decode kernel, run on the GPU.

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
"""
import ctypes
import time

import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import _build, inputs
from kv_cache_decode_paged_gb300.device import GpuWorkload

from _harness import assert_parity, oracle_all

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
