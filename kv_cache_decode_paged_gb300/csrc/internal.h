// internal.h -- host-side plumbing shared by the translation units of libkvattn.
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvattn.h"

namespace kv {

// A decode splits the flattened page list of all units -- GQA unit = (sequence,
// KV head), MLA unit = sequence; pages ordered (b, kvh, page) -- into G equal
// contiguous ranges, one per CTA.  The plan kernel writes, into the caller's
// workspace:
//   cum[B+1]         prefix sums over sequences of pages per unit
//   cta_start[G+1]   (b, kvh, page) where CTA c's range starts
//   split_first[U]   first partial slot of unit u (slot = u + c for CTA c)
//   split_count[U]   how many CTAs touched unit u (0, 1 or more)
//   arrive[2(U+U+G)] zeroed: arrival counters of the in-kernel merge (MLA),
//                    for its two column parts (merge.cuh): per part, U unit
//                    counters, then U+G slot counters
// and the decode kernel writes partial outputs (and their lse, one copy per
// column part) for units it did not finish.  GQA merges them with the combine
// kernel; MLA merges them inside the decode kernel.
struct WsLayout {
  size_t cum, cta, split_first, split_count, arrive, part_lse, part_out, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(int B, int units, int G, int rows, int dv) {
  WsLayout L;
  size_t off = 0;
  L.cum = off;
  off = align256(off + size_t(B + 1) * 8);
  L.cta = off;
  off = align256(off + size_t(G + 1) * 16);
  L.split_first = off;
  off = align256(off + size_t(units) * 4);
  L.split_count = off;
  off = align256(off + size_t(units) * 4);
  L.arrive = off;
  off = align256(off + size_t(2 * (units + units + G)) * 4);
  L.part_lse = off;
  off = align256(off + size_t(units + G) * 2 * rows * 4);
  L.part_out = off;
  off = align256(off + size_t(units + G) * rows * size_t(dv) * 4);
  L.total = off;
  return L;
}

struct PlanArgs {
  const int32_t* seq_lens;
  int B;
  int units_per_seq;   // h_kv for GQA, 1 for MLA
  int block_size;
  int max_blocks;
  int G;
  // >= 0: give every unit its own CTA (no split, no combine) when there are at
  // most G units and the longest is at most this many pages longer than the
  // balanced share ceil(T / G); < 0: always balance by splitting
  int whole_unit_slack;
  int64_t* cum;
  int4* cta_start;
  int32_t* split_first;
  int32_t* split_count;
  // In-kernel merge only (null otherwise): 2 * (units + units + G) arrival
  // counters, zeroed here; the rows of units with no token are final at once
  // and written here (out = 0, lse = -inf).
  int32_t* arrive;
  float* out;      // [units][rows][dv]
  float* lse;      // [units][rows]
  int rows, dv;
  int32_t* err;
};

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s);

// Launch with programmatic stream serialisation: the kernel may start while the
// previous kernel of the stream finishes and must call pdl_wait() before it
// reads that kernel's results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// Merge split units' partials.  few_splits picks one warp per (unit, row)
// (units split a handful of ways); otherwise a block per (unit, row) spreads
// the splits over its warps.  A unit's rows are qlen tokens x g heads of one
// of hkv KV heads of a sequence; the final rows are [sequence][token][hkv * g]
// (g = 0: g = rows, hkv = qlen = 1, unit-major rows).
cudaError_t launch_combine(const float* part_out, const float* part_lse, const int32_t* first,
                           const int32_t* count, int n_units, int rows, int dv, float* out,
                           float* lse, bool skip_single, cudaStream_t s, bool few_splits = false,
                           int g = 0, int hkv = 1, int qlen = 1);

// Number of SMs of the current device (cached per device), or -1.
int device_sm_count();

// cuTensorMapEncodeTiled through the runtime's driver entry point (so the
// library does not link libcuda directly).  Returns false on failure.
bool encode_tensor_map_3d(void* map, CUtensorMapDataType dtype, const void* base,
                          const uint64_t dims[3], const uint64_t strides_bytes[2],
                          const uint32_t box[3], CUtensorMapSwizzle swizzle);

// The same for a 4-D tensor.
bool encode_tensor_map_4d(void* map, CUtensorMapDataType dtype, const void* base,
                          const uint64_t dims[4], const uint64_t strides_bytes[3],
                          const uint32_t box[4], CUtensorMapSwizzle swizzle);

struct GqaArgs {
  const void* q;
  const kvattn_cache* cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int B, max_blocks, h, h_kv, d;
  int qlen;   // new tokens per sequence (1: plain decode)
  float scale;
  float* out;
  float* lse;
  void* workspace;
  size_t ws_bytes;
  int G;
  int32_t* err;
  cudaStream_t stream;
};
kvattn_status run_decode_gqa(const GqaArgs& a);
// Kernel parameters of the GQA decode kernels (decode_gqa.cu, decode_gqa_tc.cu).
struct GqaParams {
  const uint16_t* q;
  const int32_t* bt;
  const int32_t* seq_lens;
  const int64_t* cum;
  const int4* cta_start;
  float* out;
  float* lse;
  float* part_out;
  float* part_lse;
  int B, h, hkv, g, bs, max_blocks;
  int qlen;   // new tokens per sequence (1: plain decode)
  int rows;   // rows per unit: qlen * g, ordered (token j, head in group)
  int64_t num_blocks;
  float qk_scale_log2;  // softmax scale * log2(e), times k_scale for FP8
  float v_mult;         // 1, or v_scale for FP8
  int32_t* err;
};
// The tcgen05 form for units of many rows (decode_gqa_tc.cu): bf16 cache,
// d_h 128, 32 < rows <= 128.  gqa_tc_ctas: its default grid (one CTA per SM).
bool gqa_tc_applies(int dtype, int rows, int d);
int gqa_tc_ctas();
kvattn_status launch_gqa_tc(const GqaArgs& a, const GqaParams& prm, int G);
// Host validation of a GQA decode call (api.cu); KVATTN_OK with *nothing set
// for an empty batch.
kvattn_status check_gqa_args(const void* q, const kvattn_cache* cache, const int32_t* block_table,
                             const int32_t* seq_lens, int batch, int max_blocks_per_seq, int q_len,
                             int h, int h_kv, int d_h, float scale, const float* out,
                             const float* lse, int num_ctas, bool* nothing);
int gqa_default_ctas(int dtype, int h, int h_kv, int d);

struct MlaArgs {
  const void* q;
  const kvattn_cache* cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int B, max_blocks, h, d_c, d_rope;
  float scale;
  float* out;
  float* lse;
  void* workspace;
  size_t ws_bytes;
  int G;
  int32_t* err;
  cudaStream_t stream;
};
kvattn_status run_decode_mla(const MlaArgs& a);
int mla_default_ctas(int h);

// Explicit-form MLA prefill over the paged latent (prefill_mla.cu).
struct PrefillArgs {
  const void* q_nope;   // [B][q_len][h][128] bf16
  const void* q_rope;   // [B][q_len][h][64] bf16
  const kvattn_cache* cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int B, max_blocks, q_len, h;
  const void* w_uk;     // [h][128][512] bf16
  const void* w_uv;     // [h][128][512] bf16
  float scale;
  float* out;           // [B][q_len][h][128] f32
  float* lse;           // [B][q_len][h] f32
  int32_t* err;
  cudaStream_t stream;
};
kvattn_status run_mla_prefill(const PrefillArgs& a);

// Per-head projections around MLA decode (absorb.cu).
struct AbsorbArgs {
  const void* q_nope;   // [B][h][d_hc] bf16
  const void* q_rope;   // [B][h][d_rope] bf16
  const void* w_uk;     // [h][d_hc][d_c] bf16
  int B, h, d_hc, d_c, d_rope;
  void* q_abs;          // [B][h][d_c + d_rope] bf16
  int32_t* err;
  cudaStream_t stream;
};
kvattn_status run_mla_absorb_q(const AbsorbArgs& a);

struct UpArgs {
  const float* u;       // [B][h][d_c] f32
  const void* w_uv;     // [h][d_v][d_c] bf16
  int B, h, d_c, d_v;
  float* v;             // [B][h][d_v] f32
  int32_t* err;
  cudaStream_t stream;
};
kvattn_status run_mla_up_v(const UpArgs& a);

}  // namespace kv
