"""The tcgen05 form of the GQA decode (d_h 128; bf16 caches with 33..128 rows
per unit, FP8-E4M3 caches with 17..128) on the GPU vs the float64 oracle.

A unit's rows are the q_len new tokens x g query heads of one KV head
(single-token decode: the g heads).  With more than 32 of them the library
runs them as the M dimension of tensor-core MMAs (M = 128, rows past q_len * g
are padding); these cases cover every row count class, tiles that end inside
a page and pages that end inside a tile, split units merged by the combine,
lengths shorter than the new-token count, the lazy rescale, bad block ids and
the benchmark's full-size launch."""
import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from _harness import (GpuWorkload, assert_parity, oracle_all, oracle_multi)

pytestmark = pytest.mark.gpu


def _multi(oracle, wl, q_len, num_ctas=0, seqs=None, seed=0, qm=None):
    qm = inputs.multi_token_queries(wl, q_len, seed) if qm is None else qm
    g = GpuWorkload(wl)
    out, lse = g.decode_multi(qm, num_ctas=num_ctas)
    ref_o, ref_l = oracle_multi(oracle, wl, qm, seqs)
    assert_parity(out, lse, ref_o, ref_l, fp8=wl.kv_dtype == "fp8")
    assert g.err_bits() == 0
    return g, qm, out, lse


def _mqa(h, lens, seed=1):
    """long_mqa's cache (one KV head) read by h query heads."""
    wl = inputs.make_workload("long_mqa", lens=lens)
    wl.h = h
    wl.q = inputs.normal_bf16(inputs.rng_for(seed, f"q{h}"), wl.B * h * wl.d).reshape(wl.B, h, wl.d)
    return wl


@pytest.mark.parametrize("q_len", [5, 9, 12, 16])
def test_row_counts(oracle, q_len):
    # g = 8: 40, 72, 96 and 128 rows per KV head (72 and more were not
    # supported before this path)
    _multi(oracle, inputs.make_workload("llama3_70b", lens=[2000, 129, 7, 64, 0]), q_len)


@pytest.mark.parametrize("num_ctas", [1, 7, 300])
def test_forced_splits(oracle, num_ctas):
    # split units (partials through the combine), several units per CTA
    _multi(oracle, inputs.make_workload("llama3_70b", lens=[3000, 700, 65, 1]), 8,
           num_ctas=num_ctas)


@pytest.mark.parametrize("bs", [32, 64, 128, 256])
def test_block_sizes(oracle, bs):
    # a 64-token tile is 2 pages, 1 page, half and a quarter of one
    _multi(oracle, inputs.make_workload("llama3_70b", lens=[1000, 300, 77], block_size=bs), 8,
           num_ctas=5)


@pytest.mark.parametrize("h", [48, 64, 128])
def test_single_token_many_heads(oracle, h):
    # single-token decode with g = h (one KV head): rows = g
    wl = _mqa(h, [1500, 30000, 1, 64])
    g = GpuWorkload(wl)
    out, lse = g.decode()
    ref_o, ref_l = oracle_all(oracle, wl)
    assert_parity(out, lse, ref_o, ref_l)
    assert g.err_bits() == 0


def test_mqa_multi_token_128_rows(oracle):
    _multi(oracle, inputs.make_workload("long_mqa", lens=[9000, 40, 3]), 4)


def test_large_logits_and_needle(oracle):
    # 8x query spread (scores far above the first tile's: the lazy rescale of
    # O fires), split over CTAs; then one key that dominates a row
    wl = inputs.make_workload("llama3_70b", lens=[900, 2000], q_scale=8.0)
    qm = inputs.multi_token_queries(wl, 8)
    qm = inputs.bf16_bits(inputs.bf16_to_f32(qm) * np.float32(8.0))
    _multi(oracle, wl, 8, num_ctas=9, qm=qm)
    wl2 = inputs.make_workload("llama3_70b", lens=[900, 2000])
    qm2 = inputs.multi_token_queries(wl2, 8)
    # plant a key late in sequence 1 along the query of its last token, head 13
    b, head, t = 1, 13, 1700
    qv = inputs.bf16_to_f32(qm2[b, -1, head]).astype(np.float64)
    kvh = head // wl2.g
    wl2.k[wl2.cu_seqlens[b] + t, kvh] = inputs.bf16_bits((60.0 * qv / np.linalg.norm(qv)).astype(np.float32))
    g, _, out, _ = _multi(oracle, wl2, 8, qm=qm2)
    vt = inputs.bf16_to_f32(wl2.v[wl2.cu_seqlens[b] + t, kvh])
    np.testing.assert_allclose(out[b, -1, head], vt, atol=2e-2)


def test_bad_block_id_flagged_and_finite():
    wl = inputs.make_workload("llama3_70b", lens=[200, 300])
    g = GpuWorkload(wl)
    bt = g.bt.clone()
    bt[1, 3] = wl.num_blocks + 100
    bt[0, 0] = -7
    g.bt = bt
    g.err.zero_()
    out, lse = g.decode_multi(inputs.multi_token_queries(wl, 8))
    assert g.err_bits() & kv.KVATTN_DEVERR_BLOCK_ID
    assert np.isfinite(out).all()


def test_full_size_sampled(oracle):
    # the benchmark's multi-token launch: Llama-3-70B, 32 x 8192, 8 new tokens
    # (64 rows per KV head), default CTAs; three sampled sequences
    wl = inputs.make_workload("llama3_70b")
    _multi(oracle, wl, 8, seqs=[0, 13, 31])


# ---- FP8-E4M3 cache: kind::f8f6f4 MMAs over 128-token tiles, query and
# probabilities as two E4M3 terms each, against the oracle's decode of the
# stored codes


@pytest.mark.parametrize("q_len", [3, 4, 8, 12, 16])
def test_fp8_row_counts(oracle, q_len):
    # g = 8: 24, 32, 64, 96 and 128 rows (four, four, two, one, one copies)
    _multi(oracle, inputs.make_workload("llama3_70b_fp8", lens=[2000, 129, 7, 64, 0]), q_len)


@pytest.mark.parametrize("num_ctas", [1, 7, 300])
def test_fp8_forced_splits(oracle, num_ctas):
    _multi(oracle, inputs.make_workload("llama3_70b_fp8", lens=[3000, 700, 65, 1]), 8,
           num_ctas=num_ctas)


@pytest.mark.parametrize("bs", [16, 32, 48, 64, 128, 256])
def test_fp8_block_sizes(oracle, bs):
    # an E4M3 tile is 128 tokens: 8 pages, 4, 2 and 2/3 of a page, 2, 1, half
    # of one
    _multi(oracle, inputs.make_workload("llama3_70b_fp8", lens=[1000, 300, 77], block_size=bs), 8,
           num_ctas=5)


def test_fp8_large_logits(oracle):
    wl = inputs.make_workload("llama3_70b_fp8", lens=[900, 2000])
    qm = inputs.multi_token_queries(wl, 8)
    qm = inputs.bf16_bits(inputs.bf16_to_f32(qm) * np.float32(8.0))
    _multi(oracle, wl, 8, num_ctas=9, qm=qm)


def test_fp8_single_token_mqa(oracle):
    # long_mqa's FP8 twin read by 32 query heads per KV head, single token
    wl = inputs.make_workload("long_mqa", lens=[1500, 30000, 1, 64])
    wl.kv_dtype = "fp8"
    wl.k_scale = inputs.fp8_scale(wl.k)
    wl.v_scale = inputs.fp8_scale(wl.v)
    g = GpuWorkload(wl)
    out, lse = g.decode()
    ref_o, ref_l = oracle_all(oracle, wl)
    assert_parity(out, lse, ref_o, ref_l, fp8=True)


def test_fp8_full_size_sampled(oracle):
    wl = inputs.make_workload("llama3_70b_fp8")
    _multi(oracle, wl, 8, seqs=[0, 13, 31])
