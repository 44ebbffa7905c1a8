"""kvattn_append on the GPU vs the oracle's slot placement: bit-exact."""
import numpy as np
import pytest

import kv_cache_decode_paged_gb300 as kv
from kv_cache_decode_paged_gb300 import inputs
from _harness import GpuWorkload, dev_bits

pytestmark = pytest.mark.gpu


def _pool_bits(t):
    a = t.cpu().numpy()
    return a.view(np.uint16) if a.dtype == np.int16 else a


@pytest.mark.parametrize("bs", [16, 32, 64])
def test_append_gqa_bf16_bit_exact(oracle, bs):
    wl = inputs.make_workload("llama3_8b", lens=[37, 100, 1, 64, 17], block_size=bs)
    g = GpuWorkload(wl)
    seq_idx, pos = wl.append_indices()
    for name, src in (("k", wl.k), ("v", wl.v)):
        exp = oracle.expected_gqa_pool(src, seq_idx, pos, wl.block_table, wl.num_blocks, bs,
                                       fill=inputs.BF16_NAN)
        got = _pool_bits(getattr(g.cache, name))
        np.testing.assert_array_equal(got, exp, err_msg=name)
    assert g.err_bits() == 0


def test_append_gqa_fp8_bit_exact(oracle):
    wl = inputs.make_workload("llama3_70b_fp8", lens=[50, 129, 16])
    g = GpuWorkload(wl)
    seq_idx, pos = wl.append_indices()
    for name, src, sc in (("k", wl.k, wl.k_scale), ("v", wl.v, wl.v_scale)):
        codes = oracle.quantize_e4m3(src, sc)
        exp = oracle.expected_gqa_pool(codes, seq_idx, pos, wl.block_table, wl.num_blocks, 16,
                                       fill=inputs.E4M3_NAN)
        got = _pool_bits(getattr(g.cache, name))
        np.testing.assert_array_equal(got, exp, err_msg=name)
    assert g.err_bits() == 0


def test_append_fp8_saturates_and_rounds_like_the_format(oracle):
    # values beyond 448 * scale saturate; ties round to even -- same decision
    # as the oracle's format-definition encoder, element for element
    import torch
    vals = np.array([0.0, -0.0, 1.0625, 1.1875, 448.0, 449.0, 500.0, -1e4, 2.0 ** -10,
                     3 * 2.0 ** -10, 0.3, -7.77, 100.0, 240.0, 241.0, 232.0], dtype=np.float32)
    bits = inputs.bf16_bits(vals)
    wl = inputs.make_workload("llama3_70b_fp8", lens=[1])
    d = wl.d
    k = np.tile(bits, d // len(bits))[None, None, :].repeat(wl.h_kv, axis=1)
    cache = kv.PagedCache.allocate_gqa(4, 16, wl.h_kv, d, dtype=kv.KVATTN_FP8_E4M3,
                                       k_scale=1.0, v_scale=1.0, fill_bits=inputs.E4M3_NAN)
    bt = torch.tensor([[2]], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kt = dev_bits(np.ascontiguousarray(k))
    kv.kvattn_append(cache.descriptor(), kt, kt, torch.tensor([0], dtype=torch.int32, device="cuda"),
                     torch.tensor([5], dtype=torch.int32, device="cuda"), bt, err=err)
    got = cache.k.cpu().numpy()[2, :, 5, :]
    exp = oracle.quantize_e4m3(k[0], 1.0)
    np.testing.assert_array_equal(got, exp)
    assert int(err.item()) == 0


def test_append_mla_bit_exact(oracle):
    wl = inputs.make_workload("deepseek_v3_mla", lens=[65, 3, 128, 64])
    g = GpuWorkload(wl)
    seq_idx, pos = wl.append_indices()
    rows = np.concatenate([wl.c_kv, wl.k_r], axis=1)
    exp = oracle.expected_mla_pool(rows, seq_idx, pos, wl.block_table, wl.num_blocks, 64,
                                   fill=inputs.BF16_NAN)
    np.testing.assert_array_equal(_pool_bits(g.cache.latent), exp)
    assert g.err_bits() == 0


def test_append_bad_positions_flagged_not_written(oracle):
    import torch
    wl = inputs.make_workload("tiny", lens=[20, 5])
    g = GpuWorkload(wl)
    before_k = _pool_bits(g.cache.k).copy()
    bad_bt = g.bt.clone()
    bad_bt[1, 0] = wl.num_blocks + 5          # block id outside the pool
    seq_idx = torch.tensor([0, 1, 2, 0], dtype=torch.int32, device="cuda")
    pos = torch.tensor([10_000, 0, 0, -1], dtype=torch.int32, device="cuda")
    k = g.k_tok[:4].clone()
    g.err.zero_()
    kv.kvattn_append(g.cache.descriptor(), k, k, seq_idx, pos, bad_bt, err=g.err)
    torch.cuda.synchronize()
    bits = g.err_bits()
    assert bits & kv.KVATTN_DEVERR_POSITION
    assert bits & kv.KVATTN_DEVERR_BLOCK_ID
    np.testing.assert_array_equal(_pool_bits(g.cache.k), before_k)
