"""The C ABI without a GPU: the library loads, exports what include/kvattn.h
declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import kv_cache_decode_paged_gb300 as kv

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kvattn.h")


def _declared():
    src = open(HEADER, encoding="utf-8").read()
    return re.findall(r"KVATTN_API\s+[\w\s\*]+?\b(kvattn_\w+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    return kv.load_library()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 10
    assert sorted(names) == sorted(kv.EXPORTED)
    for n in names:
        assert getattr(lib, n) is not None


def test_abi_version(lib):
    assert kv.kvattn_abi_version() == 3


def test_struct_layout():
    # int32 x2, int64, int32 x5, float x2, int32, 3 pointers
    assert ctypes.sizeof(kv.kvattn_cache) == 72
    assert kv.kvattn_cache.k.offset == 48 and kv.kvattn_cache.latent.offset == 64


def test_status_strings():
    for s in range(5):
        assert kv.kvattn_status_string(s)
    assert kv.kvattn_status_string(99) == "unknown status"


def test_page_and_cell_bytes_match_page_figures():
    c = kv.kvattn_cache(kv.KVATTN_GQA, kv.KVATTN_BF16, 10, 16, 8, 128, 0, 0, 1.0, 1.0, 0)
    assert kv.kvattn_page_bytes(c) == 65536            # vLLM page, Llama-3-8B
    c.h_kv = 1
    assert kv.kvattn_page_bytes(c) == 8192             # per-rank page at TP=8
    assert kv.kvattn_cell_bytes(kv.KVATTN_GQA, 32, 8, 128, 0, 0, 2) == 131072
    assert kv.kvattn_cell_bytes(kv.KVATTN_GQA, 80, 8, 128, 0, 0, 2) == 327680
    assert kv.kvattn_cell_bytes(kv.KVATTN_MLA, 61, 1, 0, 512, 64, 2) == 70272
    assert kv.kvattn_cell_bytes(kv.KVATTN_MLA, 1, 1, 0, 512, 64, 2) == 1152
    m = kv.kvattn_cache(kv.KVATTN_MLA, kv.KVATTN_BF16, 10, 64, 1, 0, 512, 64, 1.0, 1.0, 0)
    assert kv.kvattn_page_bytes(m) == 64 * 576 * 2
    assert kv.kvattn_cell_bytes(kv.KVATTN_GQA, 0, 8, 128, 0, 0, 2) == -1


def test_workspace_bytes_explicit_ctas():
    a = kv.kvattn_decode_workspace_bytes(kv.KVATTN_GQA, 64, 32, 8, 128, 304)
    b = kv.kvattn_decode_workspace_bytes(kv.KVATTN_GQA, 64, 32, 8, 128, 608)
    assert 0 < a < b
    # partial slots (units + CTAs) x rows x dv floats dominate
    assert a >= (64 * 8 + 304) * 4 * 128 * 4
    assert kv.kvattn_decode_workspace_bytes(kv.KVATTN_GQA, 4, 6, 4, 128, 10) == 0   # h % h_kv
    assert kv.kvattn_decode_workspace_bytes(kv.KVATTN_MLA, 64, 128, 1, 512, 152) > 64 * 128 * 512 * 4


FAKE = 0x10000  # aligned, never dereferenced: every call below is rejected first


def _gqa_call(lib, cache, **kw):
    args = dict(q=FAKE, bt=FAKE, sl=FAKE, batch=2, maxb=4, h=8, h_kv=2, d=128, scale=0.1,
                out=FAKE, lse=FAKE, ws=FAKE, wsb=1 << 20, ctas=4)
    args.update(kw)
    return lib.kvattn_decode_gqa(args["q"], ctypes.byref(cache), args["bt"], args["sl"],
                                 args["batch"], args["maxb"], args["h"], args["h_kv"], args["d"],
                                 args["scale"], args["out"], args["lse"], args["ws"], args["wsb"],
                                 args["ctas"], None, None)


def _gqa_cache(**kw):
    c = kv.kvattn_cache(kv.KVATTN_GQA, kv.KVATTN_BF16, 100, 16, 2, 128, 0, 0, 1.0, 1.0, 0,
                        FAKE, FAKE, None)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,cache_kw,status", [
    (dict(h=6, h_kv=4), dict(h_kv=4), kv.KVATTN_ERR_INVALID_ARG),       # h % h_kv != 0
    (dict(h_kv=4), {}, kv.KVATTN_ERR_INVALID_ARG),                      # descriptor mismatch
    (dict(q=0), {}, kv.KVATTN_ERR_INVALID_ARG),                         # null q
    (dict(q=FAKE + 2), {}, kv.KVATTN_ERR_INVALID_ARG),                  # misaligned q
    (dict(scale=0.0), {}, kv.KVATTN_ERR_INVALID_ARG),
    (dict(maxb=0), {}, kv.KVATTN_ERR_INVALID_ARG),
    (dict(d=96), dict(d_h=96), kv.KVATTN_ERR_UNSUPPORTED),              # head dim not built
    (dict(h=130, h_kv=1), dict(h_kv=1), kv.KVATTN_ERR_UNSUPPORTED),     # g > 128
    (dict(h=130, h_kv=1), dict(h_kv=1, dtype=kv.KVATTN_FP8_E4M3),
     kv.KVATTN_ERR_UNSUPPORTED),                                        # FP8: g > 128
    (dict(h=80, h_kv=1, d=64), dict(h_kv=1, d_h=64), kv.KVATTN_ERR_UNSUPPORTED),  # d 64: g > 64
    ({}, dict(block_size=8), kv.KVATTN_ERR_UNSUPPORTED),
    ({}, dict(block_size=40), kv.KVATTN_ERR_UNSUPPORTED),             # not whole 16-token chunks
    ({}, dict(block_size=512), kv.KVATTN_ERR_UNSUPPORTED),            # more than 16 chunks
    ({}, dict(dtype=7), kv.KVATTN_ERR_UNSUPPORTED),
    ({}, dict(dtype=kv.KVATTN_FP8_E4M3, k_scale=0.0), kv.KVATTN_ERR_INVALID_ARG),
    ({}, dict(kind=kv.KVATTN_MLA), kv.KVATTN_ERR_INVALID_ARG),
    ({}, dict(reserved=1), kv.KVATTN_ERR_INVALID_ARG),
    (dict(ctas=70000), {}, kv.KVATTN_ERR_INVALID_ARG),
])
def test_gqa_host_validation(lib, kw, cache_kw, status):
    assert _gqa_call(lib, _gqa_cache(**cache_kw), **kw) == status


def test_gqa_empty_batch_is_ok_without_launch(lib):
    assert _gqa_call(lib, _gqa_cache(), batch=0) == kv.KVATTN_OK


def _noalloc_call(lib, cache, **kw):
    args = dict(q=FAKE, bt=FAKE, sl=FAKE, batch=2, maxb=4, h=8, h_kv=2, d=128, scale=0.1,
                out=FAKE, lse=FAKE, ctas=4)
    args.update(kw)
    return lib.kvattn_decode_gqa_noalloc(args["q"], ctypes.byref(cache), args["bt"], args["sl"],
                                         args["batch"], args["maxb"], args["h"], args["h_kv"],
                                         args["d"], args["scale"], args["out"], args["lse"],
                                         args["ctas"], None, None)


@pytest.mark.parametrize("kw,cache_kw", [
    (dict(h=6, h_kv=4), dict(h_kv=4)),
    (dict(q=0), {}),
    (dict(d=96), dict(d_h=96)),
    ({}, dict(block_size=40)),
    # argument errors whose (hypothetical) workspace would also exceed the
    # built-in scratch: the argument error is what the caller hears about
    (dict(ctas=70000), {}),
    (dict(batch=100000, ctas=70000), {}),
])
def test_noalloc_reports_argument_errors_like_the_workspace_entry(lib, kw, cache_kw):
    # no device is needed to reach these answers: the checks run first
    want = _gqa_call(lib, _gqa_cache(**cache_kw), **kw)
    assert want in (kv.KVATTN_ERR_INVALID_ARG, kv.KVATTN_ERR_UNSUPPORTED)
    assert _noalloc_call(lib, _gqa_cache(**cache_kw), **kw) == want


def test_noalloc_empty_batch_is_ok_without_launch(lib):
    assert _noalloc_call(lib, _gqa_cache(), batch=0) == kv.KVATTN_OK


def test_gqa_multi_host_validation(lib):
    c = _gqa_cache()   # h_kv = 2, d_h = 128

    def call(q_len=4, h=8, batch=2):
        return lib.kvattn_decode_gqa_multi(FAKE, ctypes.byref(c), FAKE, FAKE, batch, 4, q_len, h,
                                           2, 128, 0.1, FAKE, FAKE, FAKE, 1 << 20, 4, None, None)

    assert call(q_len=0) == kv.KVATTN_ERR_INVALID_ARG
    assert call(q_len=-3) == kv.KVATTN_ERR_INVALID_ARG
    assert call(h=32, q_len=9) == kv.KVATTN_ERR_UNSUPPORTED     # 16 heads x 9 tokens > 128 rows
    assert call(h=7) == kv.KVATTN_ERR_INVALID_ARG                # h % h_kv != 0
    assert call(batch=0) == kv.KVATTN_OK                         # nothing to do, nothing launched


def test_mla_host_validation(lib):
    c = kv.kvattn_cache(kv.KVATTN_MLA, kv.KVATTN_BF16, 100, 64, 1, 0, 512, 64, 1.0, 1.0, 0,
                        None, None, FAKE)
    call = lambda **kw: lib.kvattn_decode_mla(
        kw.get("q", FAKE), ctypes.byref(c), FAKE, FAKE, kw.get("batch", 2), 4, kw.get("h", 128),
        kw.get("d_c", 512), kw.get("d_rope", 64), 0.07, FAKE, FAKE, FAKE, 1 << 20, 4, None, None)
    assert call(d_c=256) == kv.KVATTN_ERR_INVALID_ARG          # mismatch with descriptor
    assert call(h=129) == kv.KVATTN_ERR_UNSUPPORTED
    assert call(q=0) == kv.KVATTN_ERR_INVALID_ARG
    assert call(batch=0) == kv.KVATTN_OK
    c.block_size = 16
    assert call() == kv.KVATTN_ERR_UNSUPPORTED
    c.block_size = 64
    c.dtype = kv.KVATTN_FP8_E4M3          # E4M3 latent: both per-tensor scales must be > 0
    c.k_scale = 0.0
    assert call() == kv.KVATTN_ERR_INVALID_ARG
    c.k_scale, c.v_scale = 0.01, -1.0
    assert call() == kv.KVATTN_ERR_INVALID_ARG
    c.dtype = 7
    assert call() == kv.KVATTN_ERR_UNSUPPORTED


def test_append_and_combine_validation(lib):
    c = _gqa_cache()
    assert lib.kvattn_append(ctypes.byref(c), FAKE, FAKE, 0, FAKE, FAKE, FAKE, 2, 4, None, None) == 0
    assert lib.kvattn_append(ctypes.byref(c), None, FAKE, 5, FAKE, FAKE, FAKE, 2, 4, None, None) == 1
    assert lib.kvattn_append(None, FAKE, FAKE, 5, FAKE, FAKE, FAKE, 2, 4, None, None) == 1
    c.kind = 9
    assert lib.kvattn_append(ctypes.byref(c), FAKE, FAKE, 5, FAKE, FAKE, FAKE, 2, 4, None, None) == 1
    assert lib.kvattn_combine(FAKE, FAKE, FAKE, FAKE, 3, 4, 6, FAKE, FAKE, None) == 1   # dv % 4
    assert lib.kvattn_combine(FAKE, FAKE, FAKE, FAKE, 0, 4, 8, FAKE, FAKE, None) == 0
    assert lib.kvattn_combine(FAKE, FAKE, FAKE, FAKE, 3, 4, 516, FAKE, FAKE, None) == 2  # dv > 512


def test_projection_host_validation(lib):
    # kvattn_mla_absorb_q(q_nope, q_rope, w_uk, batch, h, d_hc, d_c, d_rope, q_abs, err, stream)
    absorb = lambda **kw: lib.kvattn_mla_absorb_q(
        kw.get("q", FAKE), FAKE, FAKE, kw.get("batch", 64), kw.get("h", 128),
        kw.get("d_hc", 128), kw.get("d_c", 512), kw.get("d_rope", 64), kw.get("out", FAKE),
        None, None)
    assert absorb(batch=0) == kv.KVATTN_OK
    assert absorb(batch=-1) == kv.KVATTN_ERR_INVALID_ARG
    assert absorb(q=None) == kv.KVATTN_ERR_INVALID_ARG
    assert absorb(out=FAKE + 8) == kv.KVATTN_ERR_INVALID_ARG     # misaligned
    assert absorb(d_hc=64) == kv.KVATTN_ERR_UNSUPPORTED
    assert absorb(d_c=384) == kv.KVATTN_ERR_UNSUPPORTED          # not whole 256-column tiles
    assert absorb(d_rope=60) == kv.KVATTN_ERR_UNSUPPORTED
    assert absorb(batch=128 * 65535 + 1) == kv.KVATTN_ERR_UNSUPPORTED
    # kvattn_mla_up_v(u, w_uv, batch, h, d_c, d_v, v, err, stream)
    up = lambda **kw: lib.kvattn_mla_up_v(
        kw.get("u", FAKE), FAKE, kw.get("batch", 64), kw.get("h", 128), kw.get("d_c", 512),
        kw.get("d_v", 128), FAKE, None, None)
    assert up(batch=0) == kv.KVATTN_OK
    assert up(h=0) == kv.KVATTN_ERR_INVALID_ARG
    assert up(u=None) == kv.KVATTN_ERR_INVALID_ARG
    assert up(d_v=64) == kv.KVATTN_ERR_UNSUPPORTED
    assert up(d_c=200) == kv.KVATTN_ERR_UNSUPPORTED
