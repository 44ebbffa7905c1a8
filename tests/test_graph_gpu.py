"""Decode calls captured once in a CUDA graph and replayed.

A decode call only enqueues kernels on the current stream (planner, decode,
combine; the device set-up it needs runs once, on the first uncaptured call),
so it can be captured in a CUDA graph.  Small batches are launch-bound, and a
serving loop replays the captured step instead of paying every launch again.
A replay must give what the direct call gives, and must follow new values
written into the captured buffers between replays.
"""
import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from _harness import GpuWorkload, assert_parity, oracle_all

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,lens", [
    ("tiny", None),
    ("llama3_8b", [700, 33, 2049, 0]),
    ("long_mqa", [9000, 129]),
    ("deepseek_v3_mla", [70, 129, 1000]),
])
def test_graph_replay_matches_direct_call_and_follows_new_queries(oracle, name, lens):
    import torch
    wl = inputs.make_workload(name, lens=lens) if lens else inputs.make_workload(name)
    g = GpuWorkload(wl)
    ref_out, ref_lse = g.decode()            # direct call (and the one-time set-up)
    ws = g.workspace()
    dv = wl.d if wl.kind == "gqa" else wl.d_c
    out = torch.full((wl.B, wl.h, dv), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((wl.B, wl.h), float("nan"), dtype=torch.float32, device="cuda")
    desc = g.cache.descriptor()

    def call():
        if wl.kind == "gqa":
            kv.kvattn_decode_gqa(g.q, desc, g.bt, g.seq_lens, wl.h, wl.h_kv, wl.d, wl.scale,
                                 out, lse, ws, err=g.err)
        else:
            kv.kvattn_decode_mla(g.q, desc, g.bt, g.seq_lens, wl.h, wl.d_c, wl.d_rope,
                                 wl.scale, out, lse, ws, err=g.err)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    graph.replay()
    torch.cuda.synchronize()
    assert g.err_bits() == 0
    np.testing.assert_allclose(out.cpu().numpy(), ref_out, rtol=0, atol=1e-6)
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=0, atol=1e-6)

    # new queries (every sign flipped) in the captured buffer, two replays
    wl.q = wl.q ^ np.uint16(0x8000)
    g.q.copy_(torch.from_numpy(wl.q.view(np.int16)).cuda())
    out.fill_(float("nan"))
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert g.err_bits() == 0
    ref_o, ref_l = oracle_all(oracle, wl)
    assert_parity(out.cpu().numpy(), lse.cpu().numpy(), ref_o, ref_l)
