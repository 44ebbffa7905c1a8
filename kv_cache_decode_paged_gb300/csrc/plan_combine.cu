// plan_combine.cu -- split-KV planner, log-sum-exp combine, device helpers.
//
// Variable-length batches are split so every CTA streams the same number of
// pages: short sequences do not waste CTAs and long ones do not straggle
// ("MLA：为什么一份 Latent 可以代替多头 KV Cache", section "FlashMLA 解决的不是
// 模型公式本身": tile scheduler metadata and split info, then a stable merge of
// each split's local max, normaliser and output).
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace kv {

// One CTA.  cum[] over sequences, then each CTA's start, then each unit's split
// slots.  With T pages in total and G' = min(G, T) working CTAs, CTA c < G'
// owns flattened pages [floor(c*T/G'), floor((c+1)*T/G')) -- at least one --
// and page p belongs to CTA ((p+1)*G' - 1) / T.  The slot of (unit u, CTA c) is u + c,
// unique because walking the page list increases u or c (or both) at every
// segment boundary.
// Whole-unit mode (see PlanArgs::whole_unit_slack): CTA c owns unit c, split
// counts are 1 (0 for empty units) and no partial slot is used.  It wins when
// the split would save little: a CTA that crosses a unit boundary drains its
// pipeline, and every split unit costs a combine pass over its partials.
// cum[] is also kept in shared memory when it fits (B < kPlanSmemSeqs), so the
// searches below do not chase global memory.
constexpr int kPlanSmemSeqs = 4096;  // 32 KB, inside the default dynamic limit

// In-kernel merge set-up: zero the arrival counters, and write the rows of
// units of sequences with no token (no CTA visits them): out = 0, lse = -inf.
__device__ void merge_setup(const PlanArgs& a, const int64_t* cum) {
  if (!a.arrive) return;
  const int64_t U = a.units_per_seq, units = int64_t(a.B) * U;
  for (int64_t i = threadIdx.x; i < 2 * (units + units + a.G); i += blockDim.x) a.arrive[i] = 0;
  const int v4 = a.dv >> 2;
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    if (cum[b + 1] != cum[b]) continue;   // empty sequences are rare: one thread each
    const int64_t row0 = int64_t(b) * U * a.rows, nrows = U * a.rows;
    float4* o = reinterpret_cast<float4*>(a.out + row0 * a.dv);
    for (int64_t i = 0; i < nrows * v4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = 0; i < nrows; ++i) a.lse[row0 + i] = -INFINITY;
  }
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanArgs a) {
  __shared__ int64_t warp_tot[32];
  __shared__ int64_t carry_s;
  __shared__ unsigned long long maxn_s;
  extern __shared__ int64_t cum_s[];  // [B + 1] when B < kPlanSmemSeqs
  // Launched with programmatic serialisation: wait for whatever kernel wrote
  // seq_lens, then let the decode kernel that follows get scheduled.
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  const bool smem_cum = a.B < kPlanSmemSeqs;
  if (tid == 0) {
    carry_s = 0;
    maxn_s = 0;
    a.cum[0] = 0;
    if (smem_cum) cum_s[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int i = base + tid;
    int64_t n = 0;
    if (i < a.B) {
      int s = a.seq_lens[i];
      if (s < 0) {
        report(a.err, KVATTN_DEVERR_SEQ_LEN);
        s = 0;
      }
      n = (int64_t(s) + a.block_size - 1) / a.block_size;
      if (n > a.max_blocks) {
        report(a.err, KVATTN_DEVERR_SEQ_LEN);
        n = a.max_blocks;
      }
      atomicMax(&maxn_s, static_cast<unsigned long long>(n));
    }
    int64_t x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int64_t w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < nw) warp_tot[lane] = w;
    }
    __syncthreads();
    const int64_t carry = carry_s;
    if (i < a.B) {
      const int64_t v = carry + (wid > 0 ? warp_tot[wid - 1] : 0) + x;
      a.cum[i + 1] = v;
      if (smem_cum) cum_s[i + 1] = v;
    }
    __syncthreads();
    if (tid == 0) carry_s = carry + warp_tot[nw - 1];
    __syncthreads();
  }
  __syncthreads();
  const int64_t* cum = smem_cum ? cum_s : a.cum;
  const int64_t U = a.units_per_seq;
  const int64_t T = U * cum[a.B];
  // With more CTAs than pages, only the first T CTAs get work (one page or
  // more each); the rest get empty ranges.  Every CTA between the first and
  // the last one touching a unit then owns part of that unit, so the unit's
  // partial slots u + c0 .. u + c1 are all written.
  const int64_t G = T < a.G ? T : a.G;
  const int64_t units = int64_t(a.B) * U;
  const bool whole = a.whole_unit_slack >= 0 && T > 0 && units <= a.G &&
                     int64_t(maxn_s) <= (T + G - 1) / G + a.whole_unit_slack;
  if (whole) {
    for (int c = tid; c <= a.G; c += blockDim.x)
      a.cta_start[c] = c < units ? make_int4(int(c / U), int(c % U), 0, 0) : make_int4(a.B, 0, 0, 0);
    for (int64_t u = tid; u < units; u += blockDim.x) {
      const int64_t b = u / U;
      a.split_first[u] = int32_t(2 * u);
      a.split_count[u] = cum[b + 1] > cum[b] ? 1 : 0;
    }
    merge_setup(a, cum);
    return;
  }
  for (int c = tid; c <= a.G; c += blockDim.x) {
    const int64_t p = c <= G ? (int64_t(c) * T) / (G > 0 ? G : 1) : T;
    int4 st = make_int4(a.B, 0, 0, 0);
    if (p < T) {
      int lo = 0, hi = a.B - 1;  // largest b with U*cum[b] <= p
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (U * cum[mid] <= p)
          lo = mid;
        else
          hi = mid - 1;
      }
      const int64_t r = p - U * cum[lo];
      const int64_t n = cum[lo + 1] - cum[lo];
      st = make_int4(lo, int(r / n), int(r % n), 0);
    }
    a.cta_start[c] = st;
  }
  for (int64_t u = tid; u < units; u += blockDim.x) {
    const int64_t b = u / U, kvh = u % U;
    const int64_t n = cum[b + 1] - cum[b];
    if (n == 0) {
      a.split_first[u] = 0;
      a.split_count[u] = 0;
      continue;
    }
    const int64_t u0 = U * cum[b] + kvh * n, u1 = u0 + n;
    const int64_t c0 = ((u0 + 1) * G - 1) / T;
    const int64_t c1 = (u1 * G - 1) / T;
    a.split_first[u] = int32_t(u + c0);
    a.split_count[u] = int32_t(c1 - c0 + 1);
  }
  merge_setup(a, cum);
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t s) {
  const size_t smem = a.B < kPlanSmemSeqs ? size_t(a.B + 1) * sizeof(int64_t) : 0;
  return launch_pdl(plan_kernel, dim3(1), dim3(1024), smem, s, a);
}

// Merge the partial results of every split unit:
//   M = max_w lse_w,  o = sum_w e^(lse_w - M) o_w / sum_w e^(lse_w - M),
//   lse = M + log sum_w e^(lse_w - M).
// One block per (unit, row).  Warp i takes splits i, i+8, ... and keeps a
// running (max, normaliser, weighted sum) over them -- the online form of the
// same merge, so each split's lse and output row are loaded together in one
// pass -- and lane l the float4 columns l, l+32, ...; the eight warp states
// meet in shared memory.  A unit can have hundreds of splits (a long sequence
// over many CTAs), so the splits, not only the columns, are spread over warps.
// skip_single leaves units with one split alone (the decode kernel already
// wrote their rows).
constexpr int kCombineThreads = 256;

// Where row r of unit u goes.  Units are (sequence, KV head) pairs with hkv
// per sequence; a unit's rows are (new token j, head in group): q_len tokens x
// g heads.  The final rows are laid out [sequence][token][hkv * g heads], so
// with q_len = 1 (or hkv = 1, g = rows) this is simply u * rows + r.
struct RowMap {
  int g, hkv, qlen;
  __device__ __forceinline__ int64_t operator()(int u, int r) const {
    const int b = u / hkv, kvh = u - b * hkv, j = r / g, i = r - j * g;
    return (int64_t(b) * qlen + j) * (int64_t(hkv) * g) + int64_t(kvh) * g + i;
  }
};
constexpr int kCombineWarps = kCombineThreads / 32;
constexpr int kCombineMaxCols = 4;   // float4 columns per lane: dv <= 512

// COLS float4 columns per lane (dv <= 128 COLS); each warp loads BATCH splits
// (its splits w, w + 8, ...) before merging them, so that a row split many
// ways waits for a few batches of loads rather than one load per split.
#ifndef KV_COMBINE_BATCH
#define KV_COMBINE_BATCH 8
#endif
template <int COLS, int BATCH>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse,
                   const int32_t* __restrict__ first, const int32_t* __restrict__ count,
                   int rows, int dv, float* __restrict__ out, float* __restrict__ lse,
                   int skip_single, RowMap map) {
  // skip_single is set only behind this library's decode kernels, whose split
  // counts were written before the decode started (its own dependency wait
  // precedes its trigger): then they are read before waiting for the decode,
  // and units with one split leave at once.  Otherwise (the public call, after
  // arbitrary kernels) everything is read after the wait.
  if (!skip_single) pdl_wait();
  __shared__ float s_m[kCombineWarps], s_l[kCombineWarps];
  __shared__ float4 s_acc[kCombineWarps][kCombineMaxCols * 32];
  const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
  const int u = blockIdx.x / rows, r = blockIdx.x % rows;
  const int cnt = count[u];
  if (cnt == 1 && skip_single) return;
  const int f = first[u];
  if (skip_single) pdl_wait();  // the partials come from the decode kernel
  const int v4 = dv >> 2;
  const float* lrow = part_lse + size_t(f) * rows + r;  // split w at lrow[w * rows]
  const float4* prow = reinterpret_cast<const float4*>(part_out + (size_t(f) * rows + r) * dv);
  const size_t wstride = size_t(rows) * v4;             // float4s between splits
  float m = -INFINITY, l = 0.f;                         // log2 units
  float4 acc[COLS];
#pragma unroll
  for (int j = 0; j < COLS; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int w0 = wi; w0 < cnt; w0 += kCombineWarps * BATCH) {
    float lw[BATCH];
    float4 v[BATCH][COLS];
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      const int w = w0 + kCombineWarps * k;
      lw[k] = w < cnt ? lrow[size_t(w) * rows] * kLog2e : -INFINITY;
#pragma unroll
      for (int j = 0; j < COLS; ++j)
        v[k][j] = (w < cnt && lane + 32 * j < v4) ? prow[size_t(w) * wstride + lane + 32 * j]
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      if (lw[k] == -INFINITY) continue;  // past the end, or a split with no valid token
      const float mn = fmaxf(m, lw[k]);
      const float a = exp2_approx(m - mn), e = exp2_approx(lw[k] - mn);  // a = 0 while m = -inf
      l = l * a + e;
#pragma unroll
      for (int j = 0; j < COLS; ++j) {
        acc[j].x = acc[j].x * a + e * v[k][j].x;
        acc[j].y = acc[j].y * a + e * v[k][j].y;
        acc[j].z = acc[j].z * a + e * v[k][j].z;
        acc[j].w = acc[j].w * a + e * v[k][j].w;
      }
      m = mn;
    }
  }
  if (lane == 0) {
    s_m[wi] = m;
    s_l[wi] = l;
  }
#pragma unroll
  for (int j = 0; j < COLS; ++j)
    if (lane + 32 * j < v4) s_acc[wi][lane + 32 * j] = acc[j];
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kCombineWarps; ++i) M = fmaxf(M, s_m[i]);
  const int64_t orow_i = map(u, r);
  float4* orow = reinterpret_cast<float4*>(out + orow_i * dv);
  if (M == -INFINITY) {  // no split saw a valid token for this row
    for (int c = tid; c < v4; c += kCombineThreads) orow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0) lse[orow_i] = -INFINITY;
    return;
  }
  float sc[kCombineWarps];
  float L = 0.f;
#pragma unroll
  for (int i = 0; i < kCombineWarps; ++i) {
    sc[i] = s_m[i] == -INFINITY ? 0.f : exp2_approx(s_m[i] - M);
    L += s_l[i] * sc[i];
  }
  const float inv = 1.f / L;
  for (int c = tid; c < v4; c += kCombineThreads) {
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kCombineWarps; ++i) {
      const float4 q = s_acc[i][c];
      t.x += sc[i] * q.x;
      t.y += sc[i] * q.y;
      t.z += sc[i] * q.z;
      t.w += sc[i] * q.w;
    }
    orow[c] = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
  }
  if (tid == 0) lse[orow_i] = (M + log2_approx(L)) * kLn2;
}

// The same merge with one warp per (unit, row) and eight rows per block, for
// decodes whose units have few splits each (a handful of loads per warp):
// a quarter as many blocks as rows, so they start in one wave.  dv <= 128.
__global__ void __launch_bounds__(kCombineThreads)
    combine_rows_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse,
                        const int32_t* __restrict__ first, const int32_t* __restrict__ count,
                        int64_t n_items, int rows, int dv, float* __restrict__ out,
                        float* __restrict__ lse, int skip_single, RowMap map) {
  const int lane = threadIdx.x & 31;
  const int64_t item = int64_t(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
  // as in combine_kernel: behind a decode kernel the split counts are read
  // before waiting for it
  if (!skip_single) pdl_wait();
  if (item >= n_items) return;
  const int u = int(item / rows), r = int(item % rows);
  const int cnt = count[u];
  if (cnt == 1 && skip_single) return;
  const int f = first[u];
  if (skip_single) pdl_wait();  // the partials come from the decode kernel
  const int v4 = dv >> 2;
  const bool col = lane < v4;
  const float* lrow = part_lse + size_t(f) * rows + r;
  const float4* prow = reinterpret_cast<const float4*>(part_out + (size_t(f) * rows + r) * dv);
  const size_t wstride = size_t(rows) * v4;
  float m = -INFINITY, l = 0.f;                 // log2 units
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int w = 0; w < cnt; ++w) {
    const float lw = lrow[size_t(w) * rows] * kLog2e;
    const float4 v = col ? prow[size_t(w) * wstride + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (lw == -INFINITY) continue;  // a split with no valid token for this row
    const float mn = fmaxf(m, lw);
    const float a = exp2_approx(m - mn), e = exp2_approx(lw - mn);
    l = l * a + e;
    acc.x = acc.x * a + e * v.x;
    acc.y = acc.y * a + e * v.y;
    acc.z = acc.z * a + e * v.z;
    acc.w = acc.w * a + e * v.w;
    m = mn;
  }
  const int64_t orow_i = map(u, r);
  float4* orow = reinterpret_cast<float4*>(out + orow_i * dv);
  const float inv = m == -INFINITY ? 0.f : 1.f / l;   // no valid token: zeros, lse -inf
  if (col) orow[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lane == 0) lse[orow_i] = m == -INFINITY ? -INFINITY : (m + log2_approx(l)) * kLn2;
}

cudaError_t launch_combine(const float* part_out, const float* part_lse, const int32_t* first,
                           const int32_t* count, int n_units, int rows, int dv, float* out,
                           float* lse, bool skip_single, cudaStream_t s, bool few_splits,
                           int g, int hkv, int qlen) {
  if (n_units <= 0 || rows <= 0) return cudaSuccess;
  RowMap map{g > 0 ? g : rows, hkv > 0 ? hkv : 1, qlen > 0 ? qlen : 1};
  if (int64_t(map.g) * map.qlen != rows) return cudaErrorInvalidValue;
  if (dv > 4 * 32 * kCombineMaxCols) return cudaErrorInvalidValue;
  const int64_t items = int64_t(n_units) * rows;
  if (few_splits && dv <= 128) {
    const int64_t blocks = (items + kCombineWarps - 1) / kCombineWarps;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    return launch_pdl(combine_rows_kernel, dim3(unsigned(blocks)), dim3(kCombineThreads), 0, s,
                      part_out, part_lse, first, count, items, rows, dv, out, lse,
                      skip_single ? 1 : 0, map);
  }
  if (items > 0x7fffffff) return cudaErrorInvalidValue;
  using CombineFn = void (*)(const float*, const float*, const int32_t*, const int32_t*, int, int,
                             float*, float*, int, RowMap);
  const CombineFn k = dv <= 128 ? CombineFn(&combine_kernel<1, KV_COMBINE_BATCH>)
                    : dv <= 256 ? CombineFn(&combine_kernel<2, 4>)
                                : CombineFn(&combine_kernel<4, 2>);
  return launch_pdl(k, dim3(unsigned(items)), dim3(kCombineThreads), 0, s, part_out, part_lse, first,
                    count, rows, dv, out, lse, skip_single ? 1 : 0, map);
}

// ---- device queries -----------------------------------------------------------

int device_sm_count() {
  static int cache[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::call_once(flags[dev], [dev] {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = -1;
    cache[dev] = n;
  });
  return cache[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_tensor_map_4d(void* map, CUtensorMapDataType dtype, const void* base,
                          const uint64_t dims[4], const uint64_t strides_bytes[3],
                          const uint32_t box[4], CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gstr[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(reinterpret_cast<CUtensorMap*>(map), dtype, 4, const_cast<void*>(base), gdim,
                  gstr, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tensor_map_3d(void* map, CUtensorMapDataType dtype, const void* base,
                          const uint64_t dims[3], const uint64_t strides_bytes[2],
                          const uint32_t box[3], CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t gstr[2] = {strides_bytes[0], strides_bytes[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(reinterpret_cast<CUtensorMap*>(map), dtype, 3, const_cast<void*>(base), gdim,
                  gstr, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace kv
