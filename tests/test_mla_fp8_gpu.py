"""MLA absorbed decode over an FP8-E4M3 latent cache on the GPU vs the float64
oracle.

The cache stores e4m3(c_KV / s_c) and e4m3(k_R / s_r) with one per-tensor
scale each (amax / 448), the latent and the RoPE key quantised separately
("MLA：为什么一份 Latent 可以代替多头 KV Cache", section "MLA 与 KV Cache 量化可以叠加";
"Multi-Head Latent Attention (MLA): Mathematical Foundations, ...", section
"High-Throughput Serving Kernels: FlashMLA and SGLang").  The oracle decodes
the same stored codes exactly and attends in float64."""
import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from _harness import GpuWorkload, assert_parity, errors, mla_codes, oracle_all

pytestmark = pytest.mark.gpu

NAME = "deepseek_v3_mla_fp8"


def _check(oracle, wl, num_ctas=0, seqs=None):
    g = GpuWorkload(wl)
    out, lse = g.decode(num_ctas=num_ctas)
    ref_o, ref_l = oracle_all(oracle, wl, seqs)
    assert_parity(out, lse, ref_o, ref_l, fp8=True)
    assert g.err_bits() == 0
    return g, out, lse


def test_append_writes_the_oracles_codes(oracle):
    # every row of the pool that a token lands in holds exactly the oracle's
    # E4M3 codes of [c_KV / s_c | k_R / s_r]
    wl = inputs.make_workload(NAME, lens=[70, 129, 1])
    g = GpuWorkload(wl)
    pool = g.cache.latent.cpu().numpy().astype(np.uint8)
    for b in range(wl.B):
        sl = wl.seq_slice(b)
        codes = mla_codes(oracle, wl, sl)
        for t in range(int(wl.seq_lens[b])):
            blk = wl.block_table[b, t // wl.block_size]
            np.testing.assert_array_equal(pool[blk, t % wl.block_size], codes[t])
    assert g.err_bits() == 0


def test_small(oracle):
    _check(oracle, inputs.make_workload(NAME, lens=[70, 129]))


def test_edge_lengths(oracle):
    wl = inputs.make_workload(NAME, lens=[0, 1, 63, 64, 65, 128, 200, 0])
    g, out, lse = _check(oracle, wl)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert (out[7] == 0).all() and np.isneginf(lse[7]).all()


@pytest.mark.parametrize("pairs", [1, 2, 5, 100])
def test_forced_splits(oracle, pairs):
    wl = inputs.make_workload(NAME, lens=[1000, 64, 300, 2049])
    _check(oracle, wl, num_ctas=pairs)


def test_fewer_heads(oracle):
    _check(oracle, inputs.make_workload(NAME, lens=[500, 77], heads=16))


def test_rope_scale_far_from_latent_scale(oracle):
    # k_R sixteen times larger than c_KV: its scale is ~16x the c_KV scale, so
    # a kernel that used one scale for the whole row, or swapped them, fails
    wl = inputs.make_workload(NAME, lens=[300, 900])
    wl.k_r = inputs.bf16_bits(inputs.bf16_to_f32(wl.k_r) * np.float32(16.0))
    wl.v_scale = inputs.fp8_scale(wl.k_r)
    assert wl.v_scale > 10 * wl.k_scale
    _check(oracle, wl)


def test_large_logits_and_needle_rescale(oracle):
    wl = inputs.make_workload(NAME, lens=[900, 2000], q_scale=8.0)
    _check(oracle, wl, num_ctas=3)
    wl2 = inputs.make_workload(NAME, lens=[900, 2000])
    inputs.plant_needle_mla(wl2, b=1, head=37, t=1900)
    wl2.k_scale = inputs.fp8_scale(wl2.c_kv)
    wl2.v_scale = inputs.fp8_scale(wl2.k_r)
    _check(oracle, wl2)


def test_close_to_the_unquantised_cache(oracle):
    # secondary check: within the FP8 bound of the bf16 values the codes stand for
    wl = inputs.make_workload(NAME, lens=[777, 2048])
    g = GpuWorkload(wl)
    out, _ = g.decode()
    for b in range(wl.B):
        sl = wl.seq_slice(b)
        rows = np.concatenate([wl.c_kv[sl], wl.k_r[sl]], axis=1)
        ref, _ = oracle.mla_decode(wl.q[b], rows, wl.d_c, wl.scale)
        assert np.abs(out[b] - ref).max() <= 5e-2


def test_permuted_table_equals_identity_bit_exact():
    lens = [300, 41, 1024]
    a = GpuWorkload(inputs.make_workload(NAME, lens=lens, table="identity"))
    b = GpuWorkload(inputs.make_workload(NAME, lens=lens, table="permuted"))
    oa, la = a.decode(num_ctas=2)
    ob, lb = b.decode(num_ctas=2)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)


def test_split_count_does_not_change_result_beyond_rounding():
    wl = inputs.make_workload(NAME, lens=[3000, 5000, 100])
    g = GpuWorkload(wl)
    base, base_l = g.decode(num_ctas=1)
    for n in (3, 40):
        o, l = g.decode(num_ctas=n)
        assert errors(o, base.astype(np.float64))[0] < 1e-3
        np.testing.assert_allclose(l, base_l, atol=1e-4)


def test_large_batch(oracle):
    lens = inputs.rng_for(1500, "large-batch lens").integers(0, 131, size=1500)
    _check(oracle, inputs.make_workload(NAME, lens=lens.tolist(), heads=16))


def test_full_size_sampled(oracle):
    # DeepSeek-V3 decode layer: batch 64, 4096 tokens each, default launch
    wl = inputs.make_workload(NAME)
    g = GpuWorkload(wl)
    out, lse = g.decode()
    assert g.err_bits() == 0 and np.isfinite(out).all()
    ref_o, ref_l = oracle_all(oracle, wl, [0, 31, 63])
    assert_parity(out, lse, ref_o, ref_l, fp8=True)
