"""The seeded synthetic workloads (kv_cache_decode_paged_gb300/inputs.py).

Both the CUDA path and the oracle read what this module makes, so its recipe
is checked on its own: shapes of the pages' models, the length mixes, block
tables that are permutations of a pool with spare blocks, bf16 rounding to
nearest even, per-tensor FP8 scales, and reproducible, independent streams.
"""
import math

import numpy as np
import pytest
import torch

from kv_cache_decode_paged_gb300 import inputs


@pytest.mark.parametrize("name,h,h_kv,d,bs", [
    ("tiny", 8, 2, 64, 16),
    ("llama3_8b", 32, 8, 128, 16),
    ("llama3_70b", 64, 8, 128, 16),
    ("llama3_70b_fp8", 64, 8, 128, 16),
    ("long_gqa8", 64, 8, 128, 16),
    ("long_mqa", 32, 1, 128, 16),
])
def test_gqa_shapes(name, h, h_kv, d, bs):
    wl = inputs.make_workload(name, lens=[17, 40, 0])
    assert (wl.kind, wl.h, wl.h_kv, wl.d, wl.block_size) == ("gqa", h, h_kv, d, bs)
    assert wl.q.shape == (3, h, d) and wl.q.dtype == np.uint16
    assert wl.k.shape == (57, h_kv, d) and wl.v.shape == (57, h_kv, d)
    assert wl.scale == pytest.approx(1.0 / math.sqrt(d))
    assert wl.kv_dtype == ("fp8" if name.endswith("fp8") else "bf16")


def test_mla_shapes_and_scale():
    wl = inputs.make_workload("deepseek_v3_mla", lens=[70, 129])
    assert (wl.kind, wl.h, wl.d_c, wl.d_rope, wl.d, wl.block_size) == ("mla", 128, 512, 64, 576, 64)
    assert wl.q.shape == (2, 128, 576)
    assert wl.c_kv.shape == (199, 512) and wl.k_r.shape == (199, 64)
    assert wl.scale == pytest.approx(1.0 / math.sqrt(192.0))   # not 1/sqrt(576)


def test_length_recipes_at_full_batch():
    r = inputs.WORKLOADS
    assert list(inputs.draw_lengths(r["tiny"]["lens"], 2, 0)) == [37, 100]
    assert (inputs.draw_lengths(r["llama3_70b"]["lens"], 32, 0) == 8192).all()
    assert (inputs.draw_lengths(r["deepseek_v3_mla"]["lens"], 64, 0) == 4096).all()
    u = inputs.draw_lengths(r["llama3_8b"]["lens"], 64, 0)
    assert u.dtype == np.int32 and u.min() >= 512 and u.max() <= 8192 and len(set(u)) > 32
    lg = inputs.draw_lengths(r["long_gqa8"]["lens"], 16, 0)
    assert lg.min() >= 1024 and lg.max() <= 131072
    # log-uniform: the logs spread over the range rather than crowding at the top
    logs = np.log(lg)
    assert logs.max() - logs.min() > 0.5 * (math.log(131072) - math.log(1024))
    # both long workloads share the same lengths (same seed, same stream)
    assert (inputs.draw_lengths(r["long_mqa"]["lens"], 16, 0) == lg).all()


@pytest.mark.parametrize("how", ["permuted", "identity"])
def test_block_table(how):
    lens = np.array([0, 1, 15, 16, 17, 300, 33], dtype=np.int32)
    bs = 16
    table, num_blocks = inputs.make_block_table(lens, bs, how, seed=0)
    need = -(-lens.astype(np.int64) // bs)
    assert table.shape == (len(lens), need.max())
    used = []
    for b, n in enumerate(need):
        row = table[b]
        assert (row[n:] == -1).all()
        assert (row[:n] >= 0).all() and (row[:n] < num_blocks).all()
        used.extend(row[:n].tolist())
    assert len(used) == len(set(used)) == need.sum()   # no block serves two positions
    if how == "identity":
        assert num_blocks == need.sum() and used == list(range(need.sum()))
    else:
        assert num_blocks == need.sum() + math.ceil(0.02 * need.sum()) + 1   # spare blocks
        assert used != sorted(used)


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        (rng.standard_normal(1000) * 1e30).astype(np.float32),
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -0.0], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (inputs.bf16_bits(x) == ref).all()
    assert (inputs.bf16_to_f32(ref) == torch.from_numpy(ref.view(np.int16)).view(
        torch.bfloat16).float().numpy()).all()


def test_streams_are_seeded_and_independent():
    a = inputs.make_workload("llama3_8b", lens=[100, 50])
    b = inputs.make_workload("llama3_8b", lens=[100, 50])
    c = inputs.make_workload("llama3_8b", lens=[100, 50], seed=1)
    assert (a.q == b.q).all() and (a.k == b.k).all() and (a.v == b.v).all()
    assert (a.block_table == b.block_table).all()
    assert not (a.q == c.q).all()
    assert not (a.k[:50] == a.v[:50]).all()          # K and V come from separate streams
    # one array's shape does not reshuffle another's values
    d = inputs.make_workload("llama3_8b", lens=[100, 50, 7])
    assert (d.q[:2] == a.q).all()


def test_value_spreads():
    wl = inputs.make_workload("llama3_8b", lens=[4096])
    k = inputs.bf16_to_f32(wl.k).astype(np.float64)
    assert abs(k.mean()) < 0.01 and abs(k.std() - 1.0) < 0.01
    m = inputs.make_workload("deepseek_v3_mla", lens=[64])
    q = inputs.bf16_to_f32(m.q).astype(np.float64)
    assert abs(q.std() - 1.0 / 24.0) < 0.02 / 24.0     # N(0, 1/576)


def test_fp8_per_tensor_scales():
    wl = inputs.make_workload("llama3_70b_fp8", lens=[300, 17])
    for bits, scale in ((wl.k, wl.k_scale), (wl.v, wl.v_scale)):
        amax = np.float32(np.abs(inputs.bf16_to_f32(bits)).max())
        assert scale == float(amax / np.float32(448.0))


def test_append_indices_place_every_token():
    wl = inputs.make_workload("tiny", lens=[5, 0, 3])
    seq_idx, pos = wl.append_indices()
    assert list(seq_idx) == [0, 0, 0, 0, 0, 2, 2, 2]
    assert list(pos) == [0, 1, 2, 3, 4, 0, 1, 2]
