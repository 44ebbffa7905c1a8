"""MLA absorbed decode on the GPU vs the float64 oracle."""
import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from _harness import GpuWorkload, assert_parity, oracle_all, errors

pytestmark = pytest.mark.gpu


def _check(oracle, wl, num_ctas=0, seqs=None):
    g = GpuWorkload(wl)
    out, lse = g.decode(num_ctas=num_ctas)
    ref_o, ref_l = oracle_all(oracle, wl, seqs)
    assert_parity(out, lse, ref_o, ref_l)
    assert g.err_bits() == 0
    return g, out, lse


def test_small(oracle):
    _check(oracle, inputs.make_workload("deepseek_v3_mla", lens=[70, 129]))


def test_edge_lengths(oracle):
    wl = inputs.make_workload("deepseek_v3_mla", lens=[0, 1, 63, 64, 65, 128, 200, 0])
    g, out, lse = _check(oracle, wl)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert (out[7] == 0).all() and np.isneginf(lse[7]).all()


@pytest.mark.parametrize("pairs", [1, 2, 5, 100])
def test_forced_splits(oracle, pairs):
    wl = inputs.make_workload("deepseek_v3_mla", lens=[1000, 64, 300, 2049])
    _check(oracle, wl, num_ctas=pairs)


def test_fewer_heads(oracle):
    # fewer query heads (as one tensor-parallel rank holds): padded to M = 128 inside
    wl = inputs.make_workload("deepseek_v3_mla", lens=[500, 77])
    wl.h = 16
    wl.q = np.ascontiguousarray(wl.q[:, :16])
    _check(oracle, wl)


def test_large_logits_and_needle_rescale(oracle):
    wl = inputs.make_workload("deepseek_v3_mla", lens=[900, 2000], q_scale=8.0)
    _check(oracle, wl, num_ctas=3)
    # a dominant row late in the sequence forces the running max up by far
    # more than the lazy-rescale threshold
    wl2 = inputs.make_workload("deepseek_v3_mla", lens=[900, 2000])
    inputs.plant_needle_mla(wl2, b=1, head=37, t=1900)
    g, out, _ = _check(oracle, wl2)
    row = inputs.bf16_to_f32(wl2.c_kv[wl2.cu_seqlens[1] + 1900])
    np.testing.assert_allclose(out[1, 37], row, atol=2e-2)


def test_permuted_table_equals_identity_bit_exact():
    lens = [300, 41, 1024]
    a = GpuWorkload(inputs.make_workload("deepseek_v3_mla", lens=lens, table="identity"))
    b = GpuWorkload(inputs.make_workload("deepseek_v3_mla", lens=lens, table="permuted"))
    oa, la = a.decode(num_ctas=2)
    ob, lb = b.decode(num_ctas=2)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)


def test_bad_block_id_flagged_and_finite():
    wl = inputs.make_workload("deepseek_v3_mla", lens=[200, 300])
    g = GpuWorkload(wl)
    bt = g.bt.clone()
    bt[1, 2] = wl.num_blocks + 7
    g.err.zero_()
    out, lse = g.decode(block_table=bt)
    assert g.err_bits() & kv.KVATTN_DEVERR_BLOCK_ID
    assert np.isfinite(out).all()


@pytest.mark.parametrize("batch", [1500, 5000])
def test_large_batches_reach_every_planner_path(oracle, batch):
    # More than 1,024 sequences take the planner's multi-pass prefix scan and
    # 4,096 or more its prefix array in global memory.  With more sequences
    # than CTA pairs the balanced split runs (several sequences per pair, some
    # split between pairs and merged in the kernel).  16 heads keep the oracle
    # fast; every sequence is compared.
    lens = inputs.rng_for(batch, "large-batch lens").integers(0, 131, size=batch)
    wl = inputs.make_workload("deepseek_v3_mla", lens=lens.tolist(), heads=16)
    g, out, lse = _check(oracle, wl)
    empty = np.nonzero(lens == 0)[0]
    assert len(empty) > 0
    assert (out[empty] == 0).all() and np.isneginf(lse[empty]).all()


def test_split_count_does_not_change_result_beyond_rounding():
    wl = inputs.make_workload("deepseek_v3_mla", lens=[3000, 5000, 100])
    g = GpuWorkload(wl)
    base, base_l = g.decode(num_ctas=1)
    for n in (3, 40):
        o, l = g.decode(num_ctas=n)
        assert errors(o, base.astype(np.float64))[0] < 1e-3
        np.testing.assert_allclose(l, base_l, atol=1e-4)


def test_full_size_sampled(oracle):
    # DeepSeek-V3 decode layer: batch 64, 4096 tokens each, default launch
    wl = inputs.make_workload("deepseek_v3_mla")
    g = GpuWorkload(wl)
    out, lse = g.decode()
    assert g.err_bits() == 0 and np.isfinite(out).all()
    ref_o, ref_l = oracle_all(oracle, wl, [0, 31, 63])
    assert_parity(out, lse, ref_o, ref_l)
