// decode_mla.cu -- MLA absorbed ("MQA mode") decode over a paged latent cache.
//
// For each sequence and query head i (h <= 128), with cached rows
// row_t = [c_KV (512) | k_R (64)]:
//   s_t = scale * q~_i . row_t,  p = softmax(s),  u~_i = sum_t p_t c_t  (512 wide)
// ("Multi-Head Latent Attention (MLA): Mathematical Foundations, ...", sections
// "Attention Logit Matrix Absorption" and "Value Output Matrix Absorption";
// "MLA：为什么一份 Latent 可以代替多头 KV Cache", "第一次矩阵吸收" / "第二次矩阵吸收").
//
// One latent row serves all 128 heads, so this is a dense contraction at about
// 242 FLOP/byte -- at the GB300 ridge.  It runs on tcgen05 with M = 128 heads.
// Two facts shape the kernel: O[128 x 512] in fp32 needs all 512 TMEM columns
// of an SM, and Q[128 x 576] in bf16 needs 147 KB of shared memory.  So a
// cluster of two CTAs (two SMs) shares each tile of 64 tokens:
//   * the score contraction is split by K: rank 0 holds Q[:, 0:288], rank 1
//     Q[:, 288:576]; each computes a partial S[128 x 64] and the two partials are
//     exchanged through distributed shared memory and added;
//   * both ranks then compute the same softmax, and each accumulates half of
//     the output, O[:, 256r : 256r + 256] += P . C[:, 256r : 256r + 256], in its
//     own TMEM (P is written to TMEM as bf16 and used as the A operand).
// Each rank loads the five 64-column boxes of every row it needs (dims
// 256r .. 256r + 319), so box 4 (dims 256..319) is read by both.
//
// Warps: 0 = TMA producer, 1 = MMA issuer (+ TMEM allocation), 2..5 = softmax,
// exchange, correction and epilogue (thread = head row).
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "walk.cuh"

namespace kv {

namespace mla {
constexpr int ROWW = 576;              // latent row width (d_c + d_rope)
constexpr int DC = 512;
constexpr int BS = 64;                 // tokens per page = tokens per tile
constexpr int NBOX = 5;                // 64-column boxes per rank
constexpr int QBOX_BYTES = 128 * 128;  // [128 heads x 64 dims] bf16
constexpr int KBOX_BYTES = BS * 128;   // [64 tokens x 64 dims] bf16
constexpr int Q_BYTES = NBOX * QBOX_BYTES;         // 80 KB
constexpr int STAGE_BYTES = NBOX * KBOX_BYTES;     // 40 KB
constexpr int NSTAGE = 2;
constexpr int XROW = 64 * 4;                       // one row of a partial score tile
constexpr int XSLOT = 128 * XROW;                  // 32 KB
constexpr int NXSLOT = 2;
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + Q_BYTES;
constexpr int OFF_X = OFF_KV + NSTAGE * STAGE_BYTES;
constexpr int OFF_BAR = OFF_X + NXSLOT * XSLOT;
constexpr int NBARS = 32;
constexpr int SMEM = 1024 + OFF_BAR + NBARS * 8 + 16;
constexpr int THREADS = 192;
constexpr int KSTEPS = 18;             // 288 / 16 score k-steps per rank
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;           // S slots at columns 0 and 64 (P aliases them)
constexpr uint32_t TM_O = 256;         // O half: columns 256..511
constexpr float RESCALE_THRESHOLD = 8.f;  // log2 units: rescale O only when the max grows by 2^8
}  // namespace mla

struct MlaParams {
  const int32_t* bt;
  const int32_t* seq_lens;
  const int64_t* cum;
  const int4* cta_start;   // per pair
  float* out;
  float* lse;
  float* part_out;
  float* part_lse;
  int B, h, max_blocks;
  int64_t num_blocks;
  float scale_log2;
  int32_t* err;
};

// Barrier indices
enum : int {
  kQFull = 0, kQEmpty, kOFree,
  kKVFull0, kKVFull1, kKVEmpty0, kKVEmpty1,
  kSFull0, kSFull1, kPFull0, kPFull1, kPVDone0, kPVDone1,
  kXFull0, kXFull1, kXEmpty0, kXEmpty1,
  kAbort = 31
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(mla::THREADS, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmL, const MlaParams p) {
  using namespace mla;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int4 st = p.cta_start[pair], en = p.cta_start[pair + 1];
  if (!pos_less(st, en)) return;  // both ranks of the pair take the same exit

  if (threadIdx.x == 0) {
    mbar_init(&bars[kQFull], 1);
    mbar_init(&bars[kQEmpty], 1);
    mbar_init(&bars[kOFree], 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kKVFull0 + i], 1);
      mbar_init(&bars[kKVEmpty0 + i], 1);
      mbar_init(&bars[kSFull0 + i], 1);
      mbar_init(&bars[kPFull0 + i], 128);
      mbar_init(&bars[kPVDone0 + i], 1);
      mbar_init(&bars[kXFull0 + i], 128);   // arrivals from the peer's 128 threads
      mbar_init(&bars[kXEmpty0 + i], 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  // Both CTAs of the cluster start together; this makes each one's barriers
  // visible to the other before any remote arrive.
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmL);
      const uint64_t pol = policy_evict_first();
      Walker w{p.cum, 1, st, en};
      Seg sg;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      while (ok && w.next(sg)) {
        if (seg > 0 && !mbar_wait(&bars[kQEmpty], (seg - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[kQFull], Q_BYTES);
        for (int i = 0; i < NBOX; ++i)
          tma_load_3d_nohint(smem + OFF_Q + i * QBOX_BYTES, &tmQ, 64 * (4 * int(rank) + i), 0,
                             sg.b, &bars[kQFull]);
        const int32_t* row = p.bt + int64_t(sg.b) * p.max_blocks;
        for (int j = sg.j0; j < sg.j1 && ok; ++j, ++it) {
          const int s = it % NSTAGE;
          if (!mbar_wait(&bars[kKVEmpty0 + s], ((it / NSTAGE) & 1) ^ 1)) { ok = false; break; }
          const int blk = row[j];
          int page = int(p.num_blocks);  // out of range: zero fill
          if (blk < 0 || int64_t(blk) >= p.num_blocks)
            report(p.err, KVATTN_DEVERR_BLOCK_ID);
          else
            page = blk;
          mbar_arrive_expect_tx(&bars[kKVFull0 + s], STAGE_BYTES);
          for (int i = 0; i < NBOX; ++i)
            tma_load_3d(smem + OFF_KV + s * STAGE_BYTES + i * KBOX_BYTES, &tmL,
                        64 * (4 * int(rank) + i), 0, page, &bars[kKVFull0 + s], pol);
          if (*abort_flag) ok = false;
        }
        ++seg;
      }
      if (!ok) {
        report(p.err, KVATTN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 64, false);
      const uint32_t id_o = idesc_bf16(128, 256, true);
      const uint32_t q_base = smem_u32(smem + OFF_Q);
      const uint32_t kv_base = smem_u32(smem + OFF_KV);
      const int j_first = 2 * int(rank);  // first of this rank's 18 score k-steps
      Walker w{p.cum, 1, st, en};
      Seg sg;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      // issue S(t) = Q_r . K_r(t)^T into S slot t % 2
      auto issue_s = [&](uint32_t t) -> bool {
        const int s = t % NSTAGE;
        if (!mbar_wait(&bars[kKVFull0 + s], (t / NSTAGE) & 1)) return false;
        tc_fence_after();
        const uint32_t d = tmem + TM_S + 64 * (t & 1);
#pragma unroll 1
        for (int k = 0; k < KSTEPS; ++k) {
          const int j = j_first + k;
          const uint64_t a = sdesc_sw128(q_base + (j >> 2) * QBOX_BYTES + (j & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(kv_base + s * STAGE_BYTES + (j >> 2) * KBOX_BYTES +
                                             (j & 3) * 32, 16, 1024);
          umma_ss(d, a, b, id_s, k > 0);
        }
        umma_commit(&bars[kSFull0 + (t & 1)]);
        return true;
      };
      while (ok && w.next(sg)) {
        if (!mbar_wait(&bars[kQFull], seg & 1)) { ok = false; break; }
        const uint32_t n = uint32_t(sg.j1 - sg.j0);
        const uint32_t it0 = it;
        if (!issue_s(it0)) { ok = false; break; }
        for (uint32_t k = 0; k < n && ok; ++k) {
          const uint32_t t = it0 + k;
          if (k + 1 < n) {
            if (!issue_s(t + 1)) { ok = false; break; }
          } else {
            umma_commit(&bars[kQEmpty]);  // all score MMAs of this segment issued
          }
          if (k == 0 && seg > 0 && !mbar_wait(&bars[kOFree], (seg - 1) & 1)) { ok = false; break; }
          if (!mbar_wait(&bars[kPFull0 + (t & 1)], (t >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const int s = t % NSTAGE;
          const uint32_t pa = tmem + TM_S + 64 * (t & 1);
#pragma unroll
          for (int kk = 0; kk < BS / 16; ++kk) {
            const uint64_t b = sdesc_sw128(kv_base + s * STAGE_BYTES + kk * 2048, KBOX_BYTES, 1024);
            umma_ts(tmem + TM_O, pa + 8 * kk, b, id_o, (k > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bars[kKVEmpty0 + s]);
          umma_commit(&bars[kPVDone0 + (t & 1)]);
        }
        it += n;
        ++seg;
        if (*abort_flag) ok = false;
      }
      if (!ok) {
        report(p.err, KVATTN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else {
    // ------------------------------------- softmax / exchange / epilogue warps
    const int r = 32 * (warp & 3) + lane;          // head row = TMEM lane
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const int tid = threadIdx.x - 64;              // 0..127
    uint8_t* xbuf = smem + OFF_X;
    const uint32_t xrow_local = smem_u32(xbuf) + r * XROW;
    const uint32_t xrow_peer = map_peer(xrow_local, peer);
    const uint32_t xfull_peer0 = map_peer(smem_u32(&bars[kXFull0]), peer);
    const uint32_t xempty_peer0 = map_peer(smem_u32(&bars[kXEmpty0]), peer);
    Walker w{p.cum, 1, st, en};
    Seg sg;
    uint32_t it = 0;
    bool ok = true;
    while (ok && w.next(sg)) {
      int len = p.seq_lens[sg.b];
      len = max(0, min(len, sg.n * BS));
      const uint32_t n = uint32_t(sg.j1 - sg.j0);
      float m_ref = -INFINITY, l = 0.f;
      for (uint32_t k = 0; k < n && ok; ++k) {
        const uint32_t t = it + k;
        const int slot = t & 1;
        if (!mbar_wait(&bars[kSFull0 + slot], (t >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        uint32_t sa[32], sb[32];
        tmem_ld32(tmem + lane_off + TM_S + 64 * slot, sa);
        tmem_ld32(tmem + lane_off + TM_S + 64 * slot + 32, sb);
        tmem_ld_wait();
        // send my partial scores to the peer (XOR-swizzled 16-byte chunks)
        if (!mbar_wait(&bars[kXEmpty0 + slot], ((t >> 1) & 1) ^ 1)) { ok = false; break; }
        const uint32_t xs = uint32_t(slot) * XSLOT;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t* src = c < 8 ? &sa[4 * c] : &sb[4 * (c - 8)];
          st_cluster_v4(xrow_peer + xs + ((c ^ (r & 15)) << 4), __uint_as_float(src[0]),
                        __uint_as_float(src[1]), __uint_as_float(src[2]), __uint_as_float(src[3]));
        }
        mbar_arrive_remote(xfull_peer0 + 8 * slot);
        if (!mbar_wait_cluster(&bars[kXFull0 + slot], (t >> 1) & 1)) { ok = false; break; }
        float sc[64];
        const float4* xr = reinterpret_cast<const float4*>(xbuf + xs + r * XROW);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 v = xr[c ^ (r & 15)];
          const uint32_t* src = c < 8 ? &sa[4 * c] : &sb[4 * (c - 8)];
          sc[4 * c + 0] = __uint_as_float(src[0]) + v.x;
          sc[4 * c + 1] = __uint_as_float(src[1]) + v.y;
          sc[4 * c + 2] = __uint_as_float(src[2]) + v.z;
          sc[4 * c + 3] = __uint_as_float(src[3]) + v.w;
        }
        mbar_arrive_remote(xempty_peer0 + 8 * slot);  // done reading what the peer sent

        const int valid = len - (sg.j0 + int(k)) * BS;
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          sc[j] = j < valid ? sc[j] * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, sc[j]);
        }
        if (k == 0) {
          m_ref = mx;
        } else if (mx > m_ref + RESCALE_THRESHOLD) {
          // the running max grew a lot: rescale O (after the previous P.V landed) and l
          if (!mbar_wait(&bars[kPVDone0 + ((t - 1) & 1)], ((t - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const float alpha = exp2_approx(m_ref - mx);
          m_ref = mx;
          l *= alpha;
#pragma unroll 1
          for (int cb = 0; cb < 256; cb += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + TM_O + cb, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(tmem + lane_off + TM_O + cb, o);
          }
          tmem_st_wait();
        }
        uint32_t pk[32];
        float lsum = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float p0 = exp2_approx(sc[2 * j] - m_ref), p1 = exp2_approx(sc[2 * j + 1] - m_ref);
          lsum += p0 + p1;
          pk[j] = pack_bf16(p0, p1);
        }
        l += lsum;
        tmem_st32(tmem + lane_off + TM_S + 64 * slot, pk);
        tmem_st_wait();
        if (valid < BS) {
          // Zero the latent rows past the end of the sequence in the four boxes
          // the P.V product reads: P is 0 there, but 0 * NaN would be NaN.
          uint8_t* stg = smem + OFF_KV + (t % NSTAGE) * STAGE_BYTES;
          const int nrow = BS - max(valid, 0);
          for (int idx = tid; idx < nrow * 4 * 8; idx += 128) {
            const int row = max(valid, 0) + idx / 32, rem = idx % 32;
            *reinterpret_cast<uint4*>(stg + (rem >> 3) * KBOX_BYTES + row * 128 + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        tc_fence_before();
        mbar_arrive(&bars[kPFull0 + slot]);
      }
      if (!ok) break;
      // epilogue: O / l for this segment's rows
      const uint32_t last = it + n - 1;
      if (!mbar_wait(&bars[kPVDone0 + (last & 1)], (last >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const bool row_ok = r < p.h;
      float* dst;
      float* dl;
      if (sg.full) {
        dst = p.out + (int64_t(sg.b) * p.h + r) * DC + 256 * rank;
        dl = p.lse + int64_t(sg.b) * p.h + r;
      } else {
        const int64_t slot_idx = int64_t(sg.b) + pair;
        dst = p.part_out + (slot_idx * p.h + r) * DC + 256 * rank;
        dl = p.part_lse + slot_idx * p.h + r;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int cb = 0; cb < 256; cb += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + TM_O + cb, o);
        tmem_ld_wait();
        if (row_ok) {
          float4* d4 = reinterpret_cast<float4*>(dst + cb);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            d4[j] = make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                                __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
        }
      }
      if (row_ok && rank == 0) *dl = (l > 0.f) ? (m_ref + log2_approx(l)) * kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(&bars[kOFree]);
      it += n;
      if (*abort_flag) ok = false;
    }
    if (!ok) {
      report(p.err, KVATTN_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
    // Drain: the peer's last two "done reading" arrivals target this CTA's
    // barriers; wait for them so this CTA's shared memory outlives every access.
    for (uint32_t t = it > 2 ? it - 2 : 0; t < it; ++t)
      mbar_wait_cluster(&bars[kXEmpty0 + (t & 1)], (t >> 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

static int mla_pairs_for_device() {
  static int cache[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::call_once(flags[dev], [dev] {
    int result = -1;
    if (cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mla::SMEM) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * 1024, 1, 1);
      cfg.blockDim = dim3(mla::THREADS, 1, 1);
      cfg.dynamicSmemBytes = mla::SMEM;
      cfg.attrs = nullptr;  // the kernel fixes its cluster shape at compile time
      cfg.numAttrs = 0;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, mla_decode_kernel, &cfg) == cudaSuccess &&
          clusters > 0)
        result = clusters;
    }
    cache[dev] = result;
  });
  return cache[dev];
}

int mla_default_ctas(int h) {
  (void)h;
  return mla_pairs_for_device();
}

kvattn_status run_decode_mla(const MlaArgs& a) {
  const kvattn_cache* cc = a.cache;
  const int pairs_max = mla_pairs_for_device();
  if (pairs_max <= 0) return KVATTN_ERR_CUDA;
  const int G = a.G > 0 ? a.G : pairs_max;
  const WsLayout L = ws_layout(a.B, a.B, G, a.h, mla::DC);
  if (!a.workspace || a.ws_bytes < L.total || (reinterpret_cast<uintptr_t>(a.workspace) & 255))
    return KVATTN_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  PlanArgs pa;
  pa.seq_lens = a.seq_lens;
  pa.B = a.B;
  pa.units_per_seq = 1;
  pa.block_size = cc->block_size;
  pa.max_blocks = a.max_blocks;
  pa.G = G;
  pa.cum = reinterpret_cast<int64_t*>(ws + L.cum);
  pa.cta_start = reinterpret_cast<int4*>(ws + L.cta);
  pa.split_first = reinterpret_cast<int32_t*>(ws + L.split_first);
  pa.split_count = reinterpret_cast<int32_t*>(ws + L.split_count);
  pa.err = a.err;
  if (launch_plan(pa, a.stream) != cudaSuccess) return KVATTN_ERR_CUDA;

  alignas(64) CUtensorMap tmQ, tmL;
  {
    const uint64_t dims[3] = {uint64_t(mla::ROWW), uint64_t(a.h), uint64_t(a.B)};
    const uint64_t strides[2] = {uint64_t(mla::ROWW) * 2, uint64_t(mla::ROWW) * 2 * a.h};
    const uint32_t box[3] = {64u, 128u, 1u};
    if (!encode_tensor_map_3d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return KVATTN_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {uint64_t(mla::ROWW), uint64_t(mla::BS), uint64_t(cc->num_blocks)};
    const uint64_t strides[2] = {uint64_t(mla::ROWW) * 2, uint64_t(mla::ROWW) * 2 * mla::BS};
    const uint32_t box[3] = {64u, uint32_t(mla::BS), 1u};
    if (!encode_tensor_map_3d(&tmL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cc->latent, dims, strides,
                              box, CU_TENSOR_MAP_SWIZZLE_128B))
      return KVATTN_ERR_CUDA;
  }
  MlaParams prm;
  prm.bt = a.block_table;
  prm.seq_lens = a.seq_lens;
  prm.cum = pa.cum;
  prm.cta_start = pa.cta_start;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.part_out = reinterpret_cast<float*>(ws + L.part_out);
  prm.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  prm.B = a.B;
  prm.h = a.h;
  prm.max_blocks = a.max_blocks;
  prm.num_blocks = cc->num_blocks;
  prm.scale_log2 = a.scale * kLog2e;
  prm.err = a.err;
  mla_decode_kernel<<<2 * G, mla::THREADS, mla::SMEM, a.stream>>>(tmQ, tmL, prm);
  if (cudaGetLastError() != cudaSuccess) return KVATTN_ERR_CUDA;
  if (launch_combine(prm.part_out, prm.part_lse, pa.split_first, pa.split_count, a.B, a.h,
                     mla::DC, a.out, a.lse, true, a.stream) != cudaSuccess)
    return KVATTN_ERR_CUDA;
  return KVATTN_OK;
}

}  // namespace kv
