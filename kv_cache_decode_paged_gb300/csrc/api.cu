// api.cu -- the C ABI: argument validation and dispatch.  Every check here runs
// on the host before anything is enqueued.
#include <limits.h>

#include "common.cuh"
#include "internal.h"

using namespace kv;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(int dtype) {
  return dtype == KVATTN_BF16 ? 2 : dtype == KVATTN_FP8_E4M3 ? 1 : 0;
}

}  // namespace

extern "C" const char* kvattn_status_string(int status) {
  switch (status) {
    case KVATTN_OK: return "ok";
    case KVATTN_ERR_INVALID_ARG: return "invalid argument";
    case KVATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVATTN_ERR_CUDA: return "CUDA error";
    case KVATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

extern "C" int kvattn_abi_version(void) { return KVATTN_ABI_VERSION; }

extern "C" int64_t kvattn_page_bytes(const kvattn_cache* c) {
  if (!c || c->block_size <= 0) return -1;
  const int eb = elem_bytes(c->dtype);
  if (!eb) return -1;
  if (c->kind == KVATTN_GQA) {
    if (c->h_kv <= 0 || c->d_h <= 0) return -1;
    return int64_t(2) * c->h_kv * c->block_size * c->d_h * eb;
  }
  if (c->kind == KVATTN_MLA) {
    if (c->d_c <= 0 || c->d_rope < 0) return -1;
    return int64_t(c->block_size) * (c->d_c + c->d_rope) * eb;
  }
  return -1;
}

extern "C" int64_t kvattn_cell_bytes(int kind, int num_layers, int h_kv, int d_h, int d_c,
                                     int d_rope, int eb) {
  if (num_layers <= 0 || eb <= 0) return -1;
  if (kind == KVATTN_GQA) {
    if (h_kv <= 0 || d_h <= 0) return -1;
    return int64_t(2) * num_layers * h_kv * d_h * eb;
  }
  if (kind == KVATTN_MLA) {
    if (d_c <= 0 || d_rope < 0) return -1;
    return int64_t(num_layers) * (d_c + d_rope) * eb;
  }
  return -1;
}

extern "C" int kvattn_default_num_ctas(int kind, int dtype, int h, int h_kv, int d_h) {
  if (kind == KVATTN_GQA) return gqa_default_ctas(dtype, h, h_kv, d_h);
  if (kind == KVATTN_MLA) return mla_default_ctas(h);
  return -1;
}

extern "C" size_t kvattn_decode_workspace_bytes(int kind, int batch, int h, int h_kv, int dv,
                                                int num_ctas) {
  if (batch < 0 || h <= 0 || dv <= 0) return 0;
  int units, rows;
  if (kind == KVATTN_GQA) {
    if (h_kv <= 0 || h % h_kv) return 0;
    units = batch * h_kv;
    rows = h / h_kv;
  } else if (kind == KVATTN_MLA) {
    units = batch;
    rows = h;
  } else {
    return 0;
  }
  int G = num_ctas;
  if (G <= 0) {
    if (kind == KVATTN_GQA) {
      // enough for either cache dtype's default launch
      const int gb = gqa_default_ctas(KVATTN_BF16, h, h_kv, dv);
      const int gf = dv == 128 ? gqa_default_ctas(KVATTN_FP8_E4M3, h, h_kv, dv) : -1;
      G = gb > gf ? gb : gf;
    } else {
      G = mla_default_ctas(h);
    }
    if (G <= 0) return 0;
  }
  return ws_layout(batch, units, G, rows, dv).total;
}

namespace kv {

// Host validation of a GQA decode call, in the order the checks are made;
// KVATTN_OK with *nothing = true for an empty batch (nothing to enqueue).
kvattn_status check_gqa_args(const void* q, const kvattn_cache* cache, const int32_t* block_table,
                             const int32_t* seq_lens, int batch, int max_blocks_per_seq, int q_len,
                             int h, int h_kv, int d_h, float scale, const float* out,
                             const float* lse, int num_ctas, bool* nothing) {
  *nothing = false;
  if (!cache || cache->kind != KVATTN_GQA) return KVATTN_ERR_INVALID_ARG;
  if (batch < 0 || max_blocks_per_seq <= 0 || h <= 0 || h_kv <= 0 || d_h <= 0 || num_ctas < 0 ||
      q_len <= 0)
    return KVATTN_ERR_INVALID_ARG;
  if (h % h_kv != 0) return KVATTN_ERR_INVALID_ARG;  // "num_heads % num_kv_heads == 0"
  if (cache->h_kv != h_kv || cache->d_h != d_h || cache->reserved != 0) return KVATTN_ERR_INVALID_ARG;
  if (cache->num_blocks <= 0 || cache->block_size <= 0) return KVATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || scale == INFINITY) return KVATTN_ERR_INVALID_ARG;
  if (batch == 0) {
    *nothing = true;
    return KVATTN_OK;
  }
  if (!q || !block_table || !seq_lens || !out || !lse || !cache->k || !cache->v)
    return KVATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(cache->k, 16) ||
      !aligned(cache->v, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return KVATTN_ERR_INVALID_ARG;
  if (cache->dtype != KVATTN_BF16 && cache->dtype != KVATTN_FP8_E4M3) return KVATTN_ERR_UNSUPPORTED;
  if (cache->dtype == KVATTN_FP8_E4M3 && !(cache->k_scale > 0.f && cache->v_scale > 0.f))
    return KVATTN_ERR_INVALID_ARG;
  const int g = h / h_kv;
  // rows per KV head: four 16-row m-tiles, or one 128-row tcgen05 tile (d_h 128)
  if (int64_t(g) * q_len > (d_h == 128 ? 128 : 64)) return KVATTN_ERR_UNSUPPORTED;
  if (d_h != 64 && d_h != 128) return KVATTN_ERR_UNSUPPORTED;
  if (cache->dtype == KVATTN_FP8_E4M3 && d_h != 128) return KVATTN_ERR_UNSUPPORTED;
  // whole 16-token TMA chunks per block, at most 16 of them
  if (cache->block_size % 16 != 0 || cache->block_size > 256) return KVATTN_ERR_UNSUPPORTED;
  if (cache->num_blocks * int64_t(h_kv) >= INT_MAX) return KVATTN_ERR_UNSUPPORTED;
  if (int64_t(batch) * h_kv >= INT_MAX / 2 || int64_t(batch) * q_len * h >= INT_MAX)
    return KVATTN_ERR_UNSUPPORTED;
  if (num_ctas > 65535) return KVATTN_ERR_INVALID_ARG;
  return KVATTN_OK;
}

}  // namespace kv

extern "C" kvattn_status kvattn_decode_gqa_multi(const void* q, const kvattn_cache* cache,
                                                 const int32_t* block_table,
                                                 const int32_t* seq_lens, int batch,
                                                 int max_blocks_per_seq, int q_len, int h,
                                                 int h_kv, int d_h, float scale, float* out,
                                                 float* lse, void* workspace,
                                                 size_t workspace_bytes, int num_ctas,
                                                 int32_t* err, void* stream) {
  bool nothing = false;
  const kvattn_status st = check_gqa_args(q, cache, block_table, seq_lens, batch,
                                          max_blocks_per_seq, q_len, h, h_kv, d_h, scale, out,
                                          lse, num_ctas, &nothing);
  if (st != KVATTN_OK || nothing) return st;
  GqaArgs a;
  a.q = q;
  a.cache = cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.B = batch;
  a.max_blocks = max_blocks_per_seq;
  a.h = h;
  a.h_kv = h_kv;
  a.d = d_h;
  a.qlen = q_len;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.ws_bytes = workspace_bytes;
  a.G = num_ctas;
  a.err = err;
  a.stream = static_cast<cudaStream_t>(stream);
  return run_decode_gqa(a);
}

extern "C" kvattn_status kvattn_decode_gqa(const void* q, const kvattn_cache* cache,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           int batch, int max_blocks_per_seq, int h, int h_kv,
                                           int d_h, float scale, float* out, float* lse,
                                           void* workspace, size_t workspace_bytes, int num_ctas,
                                           int32_t* err, void* stream) {
  return kvattn_decode_gqa_multi(q, cache, block_table, seq_lens, batch, max_blocks_per_seq, 1, h,
                                 h_kv, d_h, scale, out, lse, workspace, workspace_bytes, num_ctas,
                                 err, stream);
}

extern "C" kvattn_status kvattn_decode_mla(const void* q_absorbed, const kvattn_cache* cache,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           int batch, int max_blocks_per_seq, int h, int d_c,
                                           int d_rope, float scale, float* out, float* lse,
                                           void* workspace, size_t workspace_bytes, int num_ctas,
                                           int32_t* err, void* stream) {
  if (!cache || cache->kind != KVATTN_MLA) return KVATTN_ERR_INVALID_ARG;
  if (batch < 0 || max_blocks_per_seq <= 0 || h <= 0 || num_ctas < 0) return KVATTN_ERR_INVALID_ARG;
  if (cache->d_c != d_c || cache->d_rope != d_rope || cache->reserved != 0) return KVATTN_ERR_INVALID_ARG;
  if (cache->num_blocks <= 0 || cache->block_size <= 0) return KVATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || scale == INFINITY) return KVATTN_ERR_INVALID_ARG;
  if (batch == 0) return KVATTN_OK;
  if (!q_absorbed || !block_table || !seq_lens || !out || !lse || !cache->latent)
    return KVATTN_ERR_INVALID_ARG;
  if (!aligned(q_absorbed, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(cache->latent, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return KVATTN_ERR_INVALID_ARG;
  if (cache->dtype != KVATTN_BF16 && cache->dtype != KVATTN_FP8_E4M3) return KVATTN_ERR_UNSUPPORTED;
  if (cache->dtype == KVATTN_FP8_E4M3 && !(cache->k_scale > 0.f && cache->v_scale > 0.f))
    return KVATTN_ERR_INVALID_ARG;
  if (d_c != 512 || d_rope != 64 || h > 128) return KVATTN_ERR_UNSUPPORTED;
  if (cache->block_size != 64) return KVATTN_ERR_UNSUPPORTED;
  if (cache->num_blocks >= INT_MAX / 64) return KVATTN_ERR_UNSUPPORTED;
  if (num_ctas > 65535) return KVATTN_ERR_INVALID_ARG;
  MlaArgs a;
  a.q = q_absorbed;
  a.cache = cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.B = batch;
  a.max_blocks = max_blocks_per_seq;
  a.h = h;
  a.d_c = d_c;
  a.d_rope = d_rope;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.ws_bytes = workspace_bytes;
  a.G = num_ctas;
  a.err = err;
  a.stream = static_cast<cudaStream_t>(stream);
  return run_decode_mla(a);
}

extern "C" kvattn_status kvattn_mla_absorb_q(const void* q_nope, const void* q_rope,
                                            const void* w_uk, int batch, int h, int d_hc, int d_c,
                                            int d_rope, void* q_absorbed, int32_t* err,
                                            void* stream) {
  if (batch < 0 || h <= 0 || d_hc <= 0 || d_c <= 0 || d_rope < 0) return KVATTN_ERR_INVALID_ARG;
  if (batch == 0) return KVATTN_OK;
  if (!q_nope || !w_uk || !q_absorbed || (d_rope > 0 && !q_rope)) return KVATTN_ERR_INVALID_ARG;
  if (!aligned(q_nope, 16) || !aligned(w_uk, 16) || !aligned(q_absorbed, 16) ||
      (d_rope > 0 && !aligned(q_rope, 16)))
    return KVATTN_ERR_INVALID_ARG;
  // one K = 128 tile, 256-column N tiles, q^R copied in 16-byte pieces
  if (d_hc != 128 || d_c % 256 || d_rope % 8 || d_c + d_rope > 4096) return KVATTN_ERR_UNSUPPORTED;
  if ((int64_t(batch) + 127) / 128 > 65535 || h > 65535) return KVATTN_ERR_UNSUPPORTED;
  AbsorbArgs a;
  a.q_nope = q_nope;
  a.q_rope = q_rope;
  a.w_uk = w_uk;
  a.B = batch;
  a.h = h;
  a.d_hc = d_hc;
  a.d_c = d_c;
  a.d_rope = d_rope;
  a.q_abs = q_absorbed;
  a.err = err;
  a.stream = static_cast<cudaStream_t>(stream);
  return run_mla_absorb_q(a);
}

extern "C" kvattn_status kvattn_mla_up_v(const float* u_tilde, const void* w_uv, int batch, int h,
                                        int d_c, int d_v, float* v, int32_t* err, void* stream) {
  if (batch < 0 || h <= 0 || d_c <= 0 || d_v <= 0) return KVATTN_ERR_INVALID_ARG;
  if (batch == 0) return KVATTN_OK;
  if (!u_tilde || !w_uv || !v) return KVATTN_ERR_INVALID_ARG;
  if (!aligned(u_tilde, 16) || !aligned(w_uv, 16) || !aligned(v, 16)) return KVATTN_ERR_INVALID_ARG;
  // N = d_v = 128 in one MMA, K = d_c in chunks of 128
  if (d_v != 128 || d_c % 128 || d_c > 65536) return KVATTN_ERR_UNSUPPORTED;
  if ((int64_t(batch) + 127) / 128 > 65535 || h > 65535) return KVATTN_ERR_UNSUPPORTED;
  UpArgs a;
  a.u = u_tilde;
  a.w_uv = w_uv;
  a.B = batch;
  a.h = h;
  a.d_c = d_c;
  a.d_v = d_v;
  a.v = v;
  a.err = err;
  a.stream = static_cast<cudaStream_t>(stream);
  return run_mla_up_v(a);
}

extern "C" kvattn_status kvattn_mla_prefill(const void* q_nope, const void* q_rope,
                                            const kvattn_cache* cache, const int32_t* block_table,
                                            const int32_t* seq_lens, int batch,
                                            int max_blocks_per_seq, int q_len, int h, int d_hc,
                                            int d_v, const void* w_uk, const void* w_uv,
                                            float scale, float* out, float* lse, int32_t* err,
                                            void* stream) {
  if (!cache || cache->kind != KVATTN_MLA) return KVATTN_ERR_INVALID_ARG;
  if (batch < 0 || max_blocks_per_seq <= 0 || q_len <= 0 || h <= 0 || d_hc <= 0 || d_v <= 0)
    return KVATTN_ERR_INVALID_ARG;
  if (cache->num_blocks <= 0 || cache->block_size <= 0 || cache->reserved != 0)
    return KVATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || scale == INFINITY) return KVATTN_ERR_INVALID_ARG;
  if (batch == 0) return KVATTN_OK;
  if (!q_nope || !q_rope || !block_table || !seq_lens || !w_uk || !w_uv || !out || !lse ||
      !cache->latent)
    return KVATTN_ERR_INVALID_ARG;
  if (!aligned(q_nope, 16) || !aligned(q_rope, 16) || !aligned(w_uk, 16) || !aligned(w_uv, 16) ||
      !aligned(out, 16) || !aligned(lse, 4) || !aligned(cache->latent, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return KVATTN_ERR_INVALID_ARG;
  if (cache->dtype != KVATTN_BF16) return KVATTN_ERR_UNSUPPORTED;
  if (cache->d_c != 512 || cache->d_rope != 64 || cache->block_size != 64)
    return KVATTN_ERR_UNSUPPORTED;
  if (d_hc != 128 || d_v != 128) return KVATTN_ERR_UNSUPPORTED;
  if (h > 65535 || batch > 65535 || cache->num_blocks >= INT_MAX / 64 ||
      int64_t(max_blocks_per_seq) * 64 >= INT_MAX ||
      int64_t(batch) * q_len * h >= INT_MAX / 128)
    return KVATTN_ERR_UNSUPPORTED;
  PrefillArgs a;
  a.q_nope = q_nope;
  a.q_rope = q_rope;
  a.cache = cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.B = batch;
  a.max_blocks = max_blocks_per_seq;
  a.q_len = q_len;
  a.h = h;
  a.w_uk = w_uk;
  a.w_uv = w_uv;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.err = err;
  a.stream = static_cast<cudaStream_t>(stream);
  return run_mla_prefill(a);
}

extern "C" kvattn_status kvattn_combine(const float* part_out, const float* part_lse,
                                        const int32_t* split_first, const int32_t* split_count,
                                        int n_units, int rows_per_unit, int dv, float* out,
                                        float* lse, void* stream) {
  if (n_units < 0 || rows_per_unit <= 0 || dv <= 0 || dv % 4) return KVATTN_ERR_INVALID_ARG;
  if (n_units == 0) return KVATTN_OK;
  if (dv > 512) return KVATTN_ERR_UNSUPPORTED;  // row widths of the decode paths: 64, 128, 512
  if (!part_out || !part_lse || !split_first || !split_count || !out || !lse)
    return KVATTN_ERR_INVALID_ARG;
  if (!aligned(part_out, 16) || !aligned(out, 16)) return KVATTN_ERR_INVALID_ARG;
  if (int64_t(rows_per_unit) * (dv / 4) >= INT_MAX ||
      int64_t(n_units) * rows_per_unit >= INT_MAX)  // one block per (unit, row)
    return KVATTN_ERR_UNSUPPORTED;
  return launch_combine(part_out, part_lse, split_first, split_count, n_units, rows_per_unit, dv,
                        out, lse, false, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KVATTN_OK
             : KVATTN_ERR_CUDA;
}
