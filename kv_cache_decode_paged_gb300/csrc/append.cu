// append.cu -- paged cache writer.
//
// The writer, the block table and the decode kernels agree on one layout
// ("MLA：为什么一份 Latent 可以代替多头 KV Cache", section "Paged KV Cache 的
// Block 里放什么"): token t of sequence b goes to block
// block_table[b][t / block_size], slot t % block_size.
//   GQA pools: [num_blocks][h_kv][block_size][d_h], K and V separately.
//   MLA pool:  [num_blocks][block_size][d_c + d_rope], rows [c_KV | k_R].
// One thread moves one 16-byte chunk of bf16 input (8 elements); FP8 pools
// store e4m3(x / scale) with x / scale in binary32, round to nearest even,
// saturating to +-448 (cvt.rn.satfinite.e4m3x2.f32).
#include "common.cuh"
#include "internal.h"

namespace kv {

struct AppendArgs {
  const uint16_t* src0;  // K or c_KV
  const uint16_t* src1;  // V or k_R
  int64_t n_tokens;
  const int32_t* seq_idx;
  const int32_t* pos;
  const int32_t* bt;
  int batch, max_blocks, bs;
  int64_t num_blocks;
  int h_kv, d;           // GQA: heads, head dim.  MLA: h_kv = 1, d = d_c
  int d_rope;            // MLA only
  float inv_k, inv_v;    // unused for bf16
  float k_scale, v_scale;
  void* dst0;            // K pool or latent pool
  void* dst1;            // V pool
  int32_t* err;
};

// Resolve (seq, pos) to a block id, or -1 after flagging the error.
__device__ __forceinline__ int64_t resolve_block(const AppendArgs& a, int64_t n) {
  const int b = a.seq_idx[n];
  const int t = a.pos[n];
  if (b < 0 || b >= a.batch || t < 0 || t / a.bs >= a.max_blocks) {
    report(a.err, KVATTN_DEVERR_POSITION);
    return -1;
  }
  const int64_t blk = a.bt[int64_t(b) * a.max_blocks + t / a.bs];
  if (blk < 0 || blk >= a.num_blocks) {
    report(a.err, KVATTN_DEVERR_BLOCK_ID);
    return -1;
  }
  return blk;
}


__device__ __forceinline__ uint2 quantize8(uint4 x, float scale) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16);
    const float hi = __uint_as_float(w[i] & 0xffff0000u);
    q[i] = e4m3x2(__fdiv_rn(lo, scale), __fdiv_rn(hi, scale));
  }
  return make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
}

template <bool FP8>
__global__ void __launch_bounds__(256) append_gqa_kernel(AppendArgs a) {
  const int chunks = a.d / 8;  // 16-byte chunks of one bf16 head vector
  const int64_t total = a.n_tokens * a.h_kv * chunks;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int c = int(i % chunks);
    const int64_t vec = i / chunks;
    const int kvh = int(vec % a.h_kv);
    const int64_t n = vec / a.h_kv;
    const int64_t blk = resolve_block(a, n);
    if (blk < 0) continue;
    const int t = a.pos[n];
    const int64_t dst_elem = ((blk * a.h_kv + kvh) * a.bs + t % a.bs) * int64_t(a.d) + c * 8;
    const uint4 kx = reinterpret_cast<const uint4*>(a.src0 + vec * a.d)[c];
    const uint4 vx = reinterpret_cast<const uint4*>(a.src1 + vec * a.d)[c];
    if (FP8) {
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.dst0) + dst_elem) = quantize8(kx, a.k_scale);
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.dst1) + dst_elem) = quantize8(vx, a.v_scale);
    } else {
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dst0) + dst_elem) = kx;
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dst1) + dst_elem) = vx;
    }
  }
}

// MLA rows [c_KV | k_R]; an FP8 pool quantises c_KV with k_scale and k_R with
// v_scale (one per-tensor scale each: "MLA 与 KV Cache 量化可以叠加" quantises the
// latent and the RoPE key separately).
template <bool FP8>
__global__ void __launch_bounds__(256) append_mla_kernel(AppendArgs a) {
  const int cc = a.d / 8, cr = a.d_rope / 8, width = a.d + a.d_rope;
  const int chunks = cc + cr;
  const int64_t total = a.n_tokens * chunks;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int c = int(i % chunks);
    const int64_t n = i / chunks;
    const int64_t blk = resolve_block(a, n);
    if (blk < 0) continue;
    const int t = a.pos[n];
    const int64_t row0 = (blk * a.bs + t % a.bs) * int64_t(width);
    const uint4 x = c < cc ? reinterpret_cast<const uint4*>(a.src0 + n * a.d)[c]
                           : reinterpret_cast<const uint4*>(a.src1 + n * a.d_rope)[c - cc];
    if (FP8)
      reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.dst0) + row0)[c] =
          quantize8(x, c < cc ? a.k_scale : a.v_scale);
    else
      reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dst0) + row0)[c] = x;
  }
}

}  // namespace kv

using namespace kv;

extern "C" kvattn_status kvattn_append(const kvattn_cache* cache, const void* k_or_ckv,
                                       const void* v_or_kr, int64_t n_tokens,
                                       const int32_t* seq_idx, const int32_t* pos,
                                       const int32_t* block_table, int batch,
                                       int max_blocks_per_seq, int32_t* err, void* stream) {
  if (!cache || n_tokens < 0 || batch < 0 || max_blocks_per_seq <= 0) return KVATTN_ERR_INVALID_ARG;
  if (cache->block_size <= 0 || cache->num_blocks <= 0) return KVATTN_ERR_INVALID_ARG;
  if (n_tokens == 0) return KVATTN_OK;
  if (!k_or_ckv || !v_or_kr || !seq_idx || !pos || !block_table) return KVATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_or_ckv) | reinterpret_cast<uintptr_t>(v_or_kr)) & 15)
    return KVATTN_ERR_INVALID_ARG;
  AppendArgs a{};
  a.src0 = static_cast<const uint16_t*>(k_or_ckv);
  a.src1 = static_cast<const uint16_t*>(v_or_kr);
  a.n_tokens = n_tokens;
  a.seq_idx = seq_idx;
  a.pos = pos;
  a.bt = block_table;
  a.batch = batch;
  a.max_blocks = max_blocks_per_seq;
  a.bs = cache->block_size;
  a.num_blocks = cache->num_blocks;
  a.err = err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int threads = 256;
  int64_t work;
  if (cache->kind == KVATTN_GQA) {
    if (cache->h_kv <= 0 || cache->d_h <= 0 || cache->d_h % 8 || !cache->k || !cache->v)
      return KVATTN_ERR_INVALID_ARG;
    if (cache->dtype != KVATTN_BF16 && cache->dtype != KVATTN_FP8_E4M3) return KVATTN_ERR_UNSUPPORTED;
    const size_t align = cache->dtype == KVATTN_BF16 ? 16 : 8;
    if ((reinterpret_cast<uintptr_t>(cache->k) | reinterpret_cast<uintptr_t>(cache->v)) % align)
      return KVATTN_ERR_INVALID_ARG;
    if (cache->dtype == KVATTN_FP8_E4M3 && !(cache->k_scale > 0.f && cache->v_scale > 0.f))
      return KVATTN_ERR_INVALID_ARG;
    a.h_kv = cache->h_kv;
    a.d = cache->d_h;
    a.k_scale = cache->k_scale;
    a.v_scale = cache->v_scale;
    a.dst0 = cache->k;
    a.dst1 = cache->v;
    work = n_tokens * a.h_kv * (a.d / 8);
    const int64_t blocks64 = (work + threads - 1) / threads;
    const int blocks = int(blocks64 < (1 << 20) ? blocks64 : (1 << 20));
    if (cache->dtype == KVATTN_FP8_E4M3)
      append_gqa_kernel<true><<<blocks, threads, 0, s>>>(a);
    else
      append_gqa_kernel<false><<<blocks, threads, 0, s>>>(a);
  } else if (cache->kind == KVATTN_MLA) {
    if (cache->dtype != KVATTN_BF16 && cache->dtype != KVATTN_FP8_E4M3) return KVATTN_ERR_UNSUPPORTED;
    if (cache->d_c <= 0 || cache->d_rope < 0 || cache->d_c % 8 || cache->d_rope % 8 || !cache->latent)
      return KVATTN_ERR_INVALID_ARG;
    const bool fp8 = cache->dtype == KVATTN_FP8_E4M3;
    if (reinterpret_cast<uintptr_t>(cache->latent) & (fp8 ? 7 : 15)) return KVATTN_ERR_INVALID_ARG;
    if (fp8 && !(cache->k_scale > 0.f && cache->v_scale > 0.f)) return KVATTN_ERR_INVALID_ARG;
    a.h_kv = 1;
    a.d = cache->d_c;
    a.d_rope = cache->d_rope;
    a.k_scale = cache->k_scale;
    a.v_scale = cache->v_scale;
    a.dst0 = cache->latent;
    work = n_tokens * ((a.d + a.d_rope) / 8);
    const int64_t blocks64 = (work + threads - 1) / threads;
    const int blocks = int(blocks64 < (1 << 20) ? blocks64 : (1 << 20));
    if (fp8)
      append_mla_kernel<true><<<blocks, threads, 0, s>>>(a);
    else
      append_mla_kernel<false><<<blocks, threads, 0, s>>>(a);
  } else {
    return KVATTN_ERR_INVALID_ARG;
  }
  return cudaGetLastError() == cudaSuccess ? KVATTN_OK : KVATTN_ERR_CUDA;
}
