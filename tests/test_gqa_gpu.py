"""GQA / MQA / MHA decode on the GPU vs the float64 oracle."""
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
    assert_parity(out, lse, ref_o, ref_l, fp8=wl.kv_dtype == "fp8")
    assert g.err_bits() == 0
    return g, out, lse


def test_tiny_config(oracle):
    # batch 2, h=8, h_kv=2, d=64, lengths 37 and 100, contiguous cache
    wl = inputs.make_workload("tiny")
    assert (wl.block_table[1, :7] == np.arange(3, 10)).all()   # identity table: contiguous
    _check(oracle, wl)


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_tiny_block_sizes(oracle, bs):
    _check(oracle, inputs.make_workload("tiny", block_size=bs, table="permuted"))


def test_tiny_one_block_per_sequence(oracle):
    # config 1's contiguous cache read as one 128-token block per sequence
    wl = inputs.make_workload("tiny", block_size=128)
    assert wl.block_table.shape[1] == 1
    _check(oracle, wl)


@pytest.mark.parametrize("bs", [128, 256])
def test_large_blocks_fp8_and_split(oracle, bs):
    # many 16-token chunks per block, an FP8 cache, and a forced split
    _check(oracle, inputs.make_workload("llama3_70b_fp8", lens=[700, 2049, 1], block_size=bs))
    _check(oracle, inputs.make_workload("llama3_8b", lens=[3000, 129], block_size=bs), num_ctas=7)


@pytest.mark.parametrize("name,lens", [
    ("llama3_8b", [512, 8192, 3001, 777]),          # g = 4
    ("llama3_70b", [8192, 4099]),                  # g = 8
    ("long_gqa8", [1024, 20000]),                  # g = 8, long
    ("long_mqa", [1500, 30000, 1]),                # MQA g = 32 (two m-tiles)
])
def test_model_shapes_reduced_batch(oracle, name, lens):
    _check(oracle, inputs.make_workload(name, lens=lens))


def test_mha_g1(oracle):
    wl = inputs.make_workload("tiny", lens=[33, 70])
    wl2 = inputs.Workload(**{**wl.__dict__})
    # same tensors viewed as MHA: 2 query heads per sequence, one per KV head
    wl2.h = wl.h_kv
    wl2.q = wl.q[:, : wl.h_kv].copy()
    _check(oracle, wl2)


def test_g64_four_mtiles(oracle):
    wl = inputs.make_workload("long_mqa", lens=[700, 2049])
    wl.h = 64
    wl.q = inputs.normal_bf16(inputs.rng_for(1, "q64"), wl.B * 64 * wl.d).reshape(wl.B, 64, wl.d)
    _check(oracle, wl)


def test_edge_lengths(oracle):
    # empty sequence, single token, exact block multiples, one past a block
    wl = inputs.make_workload("llama3_70b", lens=[0, 1, 16, 17, 15, 32, 0, 48])
    g, out, lse = _check(oracle, wl)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert (out[6] == 0).all() and np.isneginf(lse[6]).all()


@pytest.mark.parametrize("num_ctas", [1, 2, 7, 64, 5000])
def test_forced_splits(oracle, num_ctas):
    wl = inputs.make_workload("llama3_8b", lens=[1000, 37, 2500, 16, 0, 700])
    _check(oracle, wl, num_ctas=num_ctas)


@pytest.mark.parametrize("batch", [1500, 5000])
def test_large_batches_reach_every_planner_path(oracle, batch):
    # More than 1,024 sequences take the planner's multi-pass prefix scan, and
    # 4,096 or more keep the prefix array in global memory instead of shared
    # memory.  Short ragged lengths (empty ones included) keep the case small
    # while the 304 default CTAs cut many units into pieces; every sequence is
    # compared with the oracle.
    lens = inputs.rng_for(batch, "large-batch lens").integers(0, 65, size=batch)
    wl = inputs.make_workload("llama3_8b", lens=lens.tolist())
    g, out, lse = _check(oracle, wl)
    empty = np.nonzero(lens == 0)[0]
    assert len(empty) > 0
    assert (out[empty] == 0).all() and np.isneginf(lse[empty]).all()


def test_split_count_does_not_change_result_beyond_rounding():
    # splits change only rounding: the probabilities enter the P.V product as
    # bf16 relative to each split's running max (2^-9 relative), far inside
    # the parity tolerance
    wl = inputs.make_workload("long_gqa8", lens=[3000, 5000, 100])
    g = GpuWorkload(wl)
    base, base_l = g.decode(num_ctas=1)
    for n in (3, 50, 1000):
        o, l = g.decode(num_ctas=n)
        assert errors(o, base.astype(np.float64))[0] < 1e-3
        np.testing.assert_allclose(l, base_l, atol=1e-4)


def test_permuted_table_equals_identity_bit_exact():
    # the block-table gather is pure index work: the same values through a
    # different placement give bit-identical results
    lens = [300, 41, 1024]
    a = GpuWorkload(inputs.make_workload("llama3_8b", lens=lens, table="identity"))
    b = GpuWorkload(inputs.make_workload("llama3_8b", lens=lens, table="permuted"))
    oa, la = a.decode(num_ctas=5)
    ob, lb = b.decode(num_ctas=5)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)


def test_large_logits_and_needle(oracle):
    wl = inputs.make_workload("llama3_70b", lens=[900, 2000], q_scale=8.0)
    _check(oracle, wl, num_ctas=9)
    wl2 = inputs.make_workload("llama3_70b", lens=[900, 2000])
    inputs.plant_needle(wl2, b=1, head=13, t=1234, strength=60.0)
    g, out, _ = _check(oracle, wl2)
    vt = inputs.bf16_to_f32(wl2.v[wl2.cu_seqlens[1] + 1234, 13 // wl2.g])
    np.testing.assert_allclose(out[1, 13], vt, atol=2e-2)


def test_poisoned_pool_never_leaks():
    # unwritten slots hold NaN; tails of last blocks must be masked
    wl = inputs.make_workload("llama3_8b", lens=[1, 15, 17, 33, 47])
    g = GpuWorkload(wl, poison=True)
    out, lse = g.decode()
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_bad_block_id_flagged_and_finite():
    import torch
    wl = inputs.make_workload("llama3_8b", lens=[200, 300])
    g = GpuWorkload(wl)
    bt = g.bt.clone()
    bt[1, 3] = wl.num_blocks + 100
    bt[0, 0] = -7
    g.err.zero_()
    out, lse = g.decode(block_table=bt)
    assert g.err_bits() & kv.KVATTN_DEVERR_BLOCK_ID
    assert np.isfinite(out).all()


def test_full_size_llama3_8b_sampled(oracle):
    # the bench workload at full size, default launch; oracle on sampled sequences
    wl = inputs.make_workload("llama3_8b")
    g = GpuWorkload(wl)
    out, lse = g.decode()
    assert g.err_bits() == 0 and np.isfinite(out).all()
    order = np.argsort(wl.seq_lens)
    seqs = [int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    ref_o, ref_l = oracle_all(oracle, wl, seqs)
    assert_parity(out, lse, ref_o, ref_l)


def test_full_size_llama3_70b_sampled(oracle):
    wl = inputs.make_workload("llama3_70b")
    g = GpuWorkload(wl)
    out, lse = g.decode()
    ref_o, ref_l = oracle_all(oracle, wl, [0, 31])
    assert_parity(out, lse, ref_o, ref_l)


@pytest.mark.parametrize("name", ["long_gqa8", "long_mqa"])
def test_full_size_long_sampled(oracle, name):
    wl = inputs.make_workload(name)
    g = GpuWorkload(wl)
    out, lse = g.decode()
    order = np.argsort(wl.seq_lens)
    ref_o, ref_l = oracle_all(oracle, wl, [int(order[0]), int(order[-1])])
    assert_parity(out, lse, ref_o, ref_l)


# ------------------------------------------------------------------ FP8-E4M3

@pytest.mark.parametrize("lens,num_ctas", [([8192, 300, 17], 0), ([1000, 1, 0, 64], 7),
                                           ([5000, 4000], 1)])
def test_fp8_reduced(oracle, lens, num_ctas):
    # per-tensor scale = amax / 448; oracle decodes the same stored codes
    _check(oracle, inputs.make_workload("llama3_70b_fp8", lens=lens), num_ctas=num_ctas)


def test_fp8_mqa_and_g4(oracle):
    wl = inputs.make_workload("long_mqa", lens=[2000, 33])
    wl.kv_dtype = "fp8"
    f = lambda a: inputs.bf16_to_f32(a)
    wl.k_scale = float(np.float32(np.abs(f(wl.k)).max()) / np.float32(448))
    wl.v_scale = float(np.float32(np.abs(f(wl.v)).max()) / np.float32(448))
    _check(oracle, wl)
    wl2 = inputs.make_workload("llama3_8b", lens=[777, 2049])
    wl2.kv_dtype = "fp8"
    wl2.k_scale = float(np.float32(np.abs(f(wl2.k)).max()) / np.float32(448))
    wl2.v_scale = float(np.float32(np.abs(f(wl2.v)).max()) / np.float32(448))
    _check(oracle, wl2, num_ctas=11)


def _fp8_scales(wl):
    f = lambda a: inputs.bf16_to_f32(a)
    wl.k_scale = float(np.float32(np.abs(f(wl.k)).max()) / np.float32(448))
    wl.v_scale = float(np.float32(np.abs(f(wl.v)).max()) / np.float32(448))


def test_fp8_large_logits_and_needle(oracle):
    # An E4M3 cache under 8x logits (peaked rows, the lazy rescale taken
    # often) and with one dominant key, whose scale is refit so that it is
    # stored without saturating.
    wl = inputs.make_workload("llama3_70b_fp8", lens=[900, 2000], q_scale=8.0)
    _check(oracle, wl, num_ctas=9)
    wl2 = inputs.make_workload("llama3_70b_fp8", lens=[900, 2000])
    inputs.plant_needle(wl2, b=1, head=13, t=1234, strength=60.0)
    _fp8_scales(wl2)
    g, out, _ = _check(oracle, wl2)
    sl = wl2.seq_slice(1)
    vc = oracle.quantize_e4m3(wl2.v[sl], wl2.v_scale)
    vt = np.array([oracle.e4m3_decode(c) for c in vc[1234, 13 // wl2.g]]) * wl2.v_scale
    np.testing.assert_allclose(out[1, 13], vt, atol=5e-2)


def test_fp8_close_to_bf16_originals(oracle):
    # secondary check: the FP8 cache against the unquantised bf16 values, 5e-2
    wl = inputs.make_workload("llama3_70b_fp8", lens=[3000, 8192])
    g = GpuWorkload(wl)
    out, _ = g.decode()
    for b in range(wl.B):
        sl = wl.seq_slice(b)
        ref, _ = oracle.gqa_decode(wl.q[b], wl.k[sl], wl.v[sl], wl.scale)
        assert np.abs(out[b] - ref).max() <= 5e-2


def test_full_size_llama3_70b_fp8_sampled(oracle):
    wl = inputs.make_workload("llama3_70b_fp8")
    g = GpuWorkload(wl)
    out, lse = g.decode()
    assert g.err_bits() == 0
    ref_o, ref_l = oracle_all(oracle, wl, [0, 17, 31])
    assert_parity(out, lse, ref_o, ref_l, fp8=True)
