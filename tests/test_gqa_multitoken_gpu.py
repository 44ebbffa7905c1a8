"""Multi-token GQA decode (q_len new tokens per sequence, causal among them) on
the GPU vs the float64 oracle."""
import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from _harness import TOL_ABS_BF16, GpuWorkload, assert_parity, oracle_multi

pytestmark = pytest.mark.gpu


def _check(oracle, wl, q_len, num_ctas=0, seqs=None, seed=0):
    qm = inputs.multi_token_queries(wl, q_len, seed)
    g = GpuWorkload(wl)
    out, lse = g.decode_multi(qm, num_ctas=num_ctas)
    ref_o, ref_l = oracle_multi(oracle, wl, qm, seqs)
    assert_parity(out, lse, ref_o, ref_l, fp8=wl.kv_dtype == "fp8")
    assert g.err_bits() == 0
    return g, qm, out, lse


@pytest.mark.parametrize("q_len", [2, 4, 16])
def test_tiny(oracle, q_len):
    # g = 4: 8, 16 and 64 rows per KV head (one, one and four m-tiles)
    _check(oracle, inputs.make_workload("tiny", table="permuted"), q_len)


@pytest.mark.parametrize("name,lens,q_len", [
    ("llama3_8b", [512, 3001, 777, 17], 4),        # g = 4: 16 rows
    ("llama3_8b", [2049, 100], 8),                 # 32 rows: two m-tiles
    ("llama3_70b", [4099, 1000], 8),               # g = 8: 64 rows
    ("llama3_70b_fp8", [4099, 300], 4),            # FP8 cache, 32 rows
    ("llama3_70b_fp8", [8192, 4099, 300, 17], 8),  # FP8 cache, 64 rows: the benched shape
    ("long_mqa", [9000, 40], 2),                   # MQA g = 32: 64 rows
])
def test_model_shapes(oracle, name, lens, q_len):
    _check(oracle, inputs.make_workload(name, lens=lens), q_len)


@pytest.mark.parametrize("num_ctas", [1, 7, 300])
def test_forced_splits(oracle, num_ctas):
    # partial outputs of split units go through the combine with the
    # (sequence, token, head) row map
    _check(oracle, inputs.make_workload("llama3_8b", lens=[3000, 129, 64, 1000]), 4,
           num_ctas=num_ctas)


@pytest.mark.parametrize("num_ctas", [7, 300])
def test_fp8_64_rows_forced_splits(oracle, num_ctas):
    # FP8 cache at 64 rows per KV head (g = 8, 8 new tokens), units split over
    # CTAs and merged by the combine
    _check(oracle, inputs.make_workload("llama3_70b_fp8", lens=[5000, 1500, 9]), 8,
           num_ctas=num_ctas)


def test_fp8_64_rows_full_size_sampled(oracle):
    # the benchmark's FP8 multi-token launch (batch 32 x 8192, default CTAs);
    # the oracle checks three sampled sequences, every row of each
    wl = inputs.make_workload("llama3_70b_fp8")
    _check(oracle, wl, 8, seqs=[0, 13, 31])


def test_short_sequences(oracle):
    # lengths around q_len: a sequence shorter than q_len leaves its first new
    # tokens with nothing to see (out 0, lse -inf); empty sequences stay empty
    wl = inputs.make_workload("tiny", lens=[1, 3, 4, 0, 5])
    g, qm, out, lse = _check(oracle, wl, 4)
    assert (out[0, :3] == 0).all() and np.isneginf(lse[0, :3]).all()
    assert (out[3] == 0).all() and np.isneginf(lse[3]).all()


def test_q_len_one_equals_single_token_decode():
    wl = inputs.make_workload("llama3_8b", lens=[700, 33, 2000])
    g = GpuWorkload(wl)
    o1, l1 = g.decode()
    om, lm = g.decode_multi(wl.q[:, None])
    np.testing.assert_array_equal(om[:, 0], o1)
    np.testing.assert_array_equal(lm[:, 0], l1)


def test_last_token_equals_single_token_decode_of_it():
    # the last new token sees the whole sequence, like a single-token decode
    # with its query.  The log-sum-exp (fp32 sums of the unrounded scores)
    # must agree to fp32 rounding: one token more or less would move it by
    # far more.  The outputs differ by the bf16 rounding of P, which depends
    # on where the two launches split a sequence.
    wl = inputs.make_workload("llama3_70b", lens=[1500, 64])
    qm = inputs.multi_token_queries(wl, 8)
    g = GpuWorkload(wl)
    om, lm = g.decode_multi(qm)
    wl.q = np.ascontiguousarray(qm[:, -1])
    g1 = GpuWorkload(wl)
    o1, l1 = g1.decode()
    assert np.abs(lm[:, -1] - l1).max() < 1e-4
    assert np.abs(om[:, -1] - o1).max() < TOL_ABS_BF16


def test_rejects_too_many_rows():
    wl = inputs.make_workload("llama3_70b", lens=[100])   # g = 8
    g = GpuWorkload(wl)
    with pytest.raises(kv.KvattnError) as e:
        g.decode_multi(inputs.multi_token_queries(wl, 17))   # 136 rows > 128
    assert e.value.status == kv.KVATTN_ERR_UNSUPPORTED
    wl8 = inputs.make_workload("llama3_70b_fp8", lens=[100])
    g8 = GpuWorkload(wl8)
    with pytest.raises(kv.KvattnError) as e:
        g8.decode_multi(inputs.multi_token_queries(wl8, 17))   # FP8: 136 rows > 128
    assert e.value.status == kv.KVATTN_ERR_UNSUPPORTED
