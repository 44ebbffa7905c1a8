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
// O[128 x 512] in fp32 would fill all 512 TMEM columns of an SM and Q[128 x 576]
// would take 147 KB of shared memory, so a cluster of two CTAs (two SMs) shares
// each tile of 64 latent rows:
//   * the score contraction is split by K: rank 0 holds Q[:, 0:288], rank 1
//     Q[:, 288:576] in shared memory; each computes a partial S[128 x 64],
//     scales it to log2 units, rounds it to f16 and pushes it to the other
//     rank with one bulk copy; both ranks add the same two f16 partials, so
//     their softmax inputs are bit-identical;
//   * both ranks then compute the same softmax, write P to TMEM as bf16 and
//     accumulate their half O[:, 256r : 256r + 256] += P . C[:, 256r : +256].
// Rank 0 loads latent dims 0..287 of each row, rank 1 dims 256..575 (dims
// 256..287 by both); the 32-dim pieces use 64-byte swizzled half boxes.
//
// Measured on GB300: a K=16 MMA with M = 128 costs about the same for N = 32,
// 64 or 128 (~80 cycles), and distributed shared memory sustains only ~20
// bytes per clock per SM for bulk pushes (~10 for per-thread stores) with ~1000
// cycles of round-trip latency.  Hence tiles of 64 rows, score MMAs from
// shared memory, a half-size (f16) exchange moved by the bulk-copy engine, and
// tile t+1's exchange issued right after P(t) so its latency overlaps P.V(t)
// and S(t+2) on the tensor pipe.
//
// Warps: 0 = TMA producer (3-stage ring), 1 = MMA issuer and TMEM owner,
// 2..9 = softmax group: two threads per head row, 32 of the tile's 64 tokens
// each (the pair combines its row max through shared memory).
#include <cuda_fp16.h>
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
constexpr int QF_BYTES = 128 * 128;    // full Q box [128 heads x 64 dims]
constexpr int QH_BYTES = 128 * 64;     // half Q box [128 heads x 32 dims]
constexpr int KF_BYTES = BS * 128;     // full latent box [64 rows x 64 dims]
constexpr int KH_BYTES = BS * 64;      // half latent box [64 rows x 32 dims]
constexpr int OFF_QF = 0;              // 4 full Q boxes
constexpr int OFF_QH = 4 * QF_BYTES;   // 1 half Q box
constexpr int Q_BYTES = 4 * QF_BYTES + QH_BYTES;        // 72 KB
constexpr int STAGE_BYTES = 5 * KF_BYTES;               // 40 KB (rank 0 uses 36 KB)
constexpr int NSTAGE = 3;
constexpr int OFF_KV = 73728;          // 1024-aligned
constexpr int XROW = BS * 2;           // one row of a partial score tile, f16 (128 B)
constexpr int XBYTES = 128 * XROW;     // 16 KB
constexpr int OFF_X = OFF_KV + NSTAGE * STAGE_BYTES;   // receive buffer (written by the peer)
constexpr int OFF_XS = OFF_X + XBYTES;                 // send staging
constexpr int OFF_MX = OFF_XS + XBYTES;   // row-max exchange between the two halves of a row
constexpr int OFF_BAR = OFF_MX + 2 * 128 * 4;
constexpr int NBARS = 24;
constexpr int SMEM = 1024 + OFF_BAR + NBARS * 8 + 16;
constexpr int NSW = 256;               // softmax group: two threads per head row
constexpr int THREADS = 64 + NSW;
constexpr int KSTEPS = 18;             // 288 score dims per rank / 16
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;           // two S/P slots at columns 0 and 64
constexpr uint32_t TM_O = 256;         // O half: columns 256..511
constexpr float RESCALE_THRESHOLD = 8.f;  // log2 units: rescale O only when the max grows by 2^8
static_assert(OFF_KV >= Q_BYTES && OFF_KV % 1024 == 0, "layout");
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
  kQFull = 0, kQEmpty = 1, kOFree = 2,
  kSFull0 = 3,      // 2: S(t) landed in slot t % 2
  kPFull0 = 5,      // 2: P(t) written to slot t % 2
  kPVDone0 = 7,     // 2: P.V of tile t finished (by t % 2)
  kXFull = 9,       // the peer's partial of the next tile is in the exchange buffer (tx bytes)
  kXEmpty = 10,     // the peer has read this CTA's partial of the last sent tile
  kKVFull0 = 11,    // 3
  kKVEmpty0 = 14,   // 3
  kAbort = 20
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(mla::THREADS, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmQF,
                      const __grid_constant__ CUtensorMap tmQH,
                      const __grid_constant__ CUtensorMap tmLF,
                      const __grid_constant__ CUtensorMap tmLH, const MlaParams p) {
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
    mbar_init(&bars[kOFree], NSW);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kSFull0 + i], 1);
      mbar_init(&bars[kPFull0 + i], NSW);
      mbar_init(&bars[kPVDone0 + i], 1);
    }
    mbar_init(&bars[kXFull], 1);     // one local expect_tx arrival + the peer's bytes
    mbar_init(&bars[kXEmpty], 1);    // one arrival from the peer's softmax group
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&bars[kKVFull0 + i], 1);
      mbar_init(&bars[kKVEmpty0 + i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    mbar_arrive_expect_tx(&bars[kXFull], XBYTES);  // phase 0: the peer's tile 0
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  // Both CTAs of the cluster start together; this makes each one's barriers
  // visible to the other before any remote access.
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // this rank's latent / query columns: full boxes and the 32-wide half box
  const int fx0 = rank == 0 ? 0 : 256;     // first full latent box (PV dims)
  const int qx0 = rank == 0 ? 0 : 320;     // first full Q box
  const int hx = rank == 0 ? 256 : 288;    // half box (Q; latent for rank 0)
  const uint32_t stage_tx = rank == 0 ? uint32_t(4 * KF_BYTES + KH_BYTES) : uint32_t(5 * KF_BYTES);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQF);
      tma_prefetch_desc(&tmQH);
      tma_prefetch_desc(&tmLF);
      tma_prefetch_desc(&tmLH);
      const uint64_t pol = policy_evict_first();
      Walker w{p.cum, 1, st, en};
      Seg sg;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      while (ok && w.next(sg)) {
        if (seg > 0 && !mbar_wait(&bars[kQEmpty], (seg - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[kQFull], Q_BYTES);
        for (int i = 0; i < 4; ++i)
          tma_load_3d_nohint(smem + OFF_QF + i * QF_BYTES, &tmQF, qx0 + 64 * i, 0, sg.b,
                             &bars[kQFull]);
        tma_load_3d_nohint(smem + OFF_QH, &tmQH, hx, 0, sg.b, &bars[kQFull]);
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
          uint8_t* stg = smem + OFF_KV + s * STAGE_BYTES;
          mbar_arrive_expect_tx(&bars[kKVFull0 + s], stage_tx);
          for (int i = 0; i < 4; ++i)
            tma_load_3d(stg + i * KF_BYTES, &tmLF, fx0 + 64 * i, 0, page, &bars[kKVFull0 + s], pol);
          if (rank == 0)
            tma_load_3d(stg + 4 * KF_BYTES, &tmLH, 256, 0, page, &bars[kKVFull0 + s], pol);
          else
            tma_load_3d(stg + 4 * KF_BYTES, &tmLF, 512, 0, page, &bars[kKVFull0 + s], pol);
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
      const uint32_t id_s = idesc_bf16(128, BS, false);
      const uint32_t id_o = idesc_bf16(128, 256, true);
      const uint32_t qf = smem_u32(smem + OFF_QF), qh = smem_u32(smem + OFF_QH);
      const uint32_t kv_base = smem_u32(smem + OFF_KV);
      Walker w{p.cum, 1, st, en};
      Seg sg;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      // S(t) = Q_r . K_r(t)^T into S slot t % 2 (18 MMAs, K = 16 each)
      auto issue_s = [&](uint32_t t) -> bool {
        const int s = t % NSTAGE;
        if (!mbar_wait(&bars[kKVFull0 + s], (t / NSTAGE) & 1)) return false;
        tc_fence_after();
        const uint32_t d = tmem + TM_S + BS * (t & 1);
        const uint32_t kb = kv_base + s * STAGE_BYTES;
#pragma unroll 1
        for (int j = 0; j < KSTEPS; ++j) {
          uint64_t a, b;
          if (rank == 0) {
            if (j < 16) {
              a = sdesc_sw128(qf + (j >> 2) * QF_BYTES + (j & 3) * 32, 16, 1024);
              b = sdesc_sw128(kb + (j >> 2) * KF_BYTES + (j & 3) * 32, 16, 1024);
            } else {
              a = sdesc_sw64(qh + (j - 16) * 32, 512);
              b = sdesc_sw64(kb + 4 * KF_BYTES + (j - 16) * 32, 512);
            }
          } else {
            if (j < 2) {
              a = sdesc_sw64(qh + j * 32, 512);
              b = sdesc_sw128(kb + (2 + j) * 32, 16, 1024);
            } else {
              const int m = j - 2;
              a = sdesc_sw128(qf + (m >> 2) * QF_BYTES + (m & 3) * 32, 16, 1024);
              b = sdesc_sw128(kb + ((m >> 2) + 1) * KF_BYTES + (m & 3) * 32, 16, 1024);
            }
          }
          umma_ss(d, a, b, id_s, j > 0);
        }
        umma_commit(&bars[kSFull0 + (t & 1)]);
        return true;
      };
      while (ok && w.next(sg)) {
        const uint32_t n = uint32_t(sg.j1 - sg.j0);
        if (!mbar_wait(&bars[kQFull], seg & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t it0 = it;
        if (!issue_s(it0)) { ok = false; break; }
        if (n > 1 && !issue_s(it0 + 1)) { ok = false; break; }
        if (n <= 2) umma_commit(&bars[kQEmpty]);  // every score MMA of this segment is issued
        for (uint32_t k = 0; k < n && ok; ++k) {
          const uint32_t t = it0 + k;
          if (k == 0 && seg > 0 && !mbar_wait(&bars[kOFree], (seg - 1) & 1)) { ok = false; break; }
          if (!mbar_wait(&bars[kPFull0 + (t & 1)], (t >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const int s = t % NSTAGE;
          const uint32_t pa = tmem + TM_S + BS * (t & 1);
#pragma unroll
          for (int kk = 0; kk < BS / 16; ++kk) {
            const uint64_t b = sdesc_sw128(kv_base + s * STAGE_BYTES + kk * 2048, KF_BYTES, 1024);
            umma_ts(tmem + TM_O, pa + 8 * kk, b, id_o, (k > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bars[kKVEmpty0 + s]);
          umma_commit(&bars[kPVDone0 + (t & 1)]);
          // S(t+2) reuses P(t)'s slot; MMAs run in issue order, so it lands after
          // P.V(t) has read P(t)
          if (k + 2 < n) {
            if (!issue_s(t + 2)) { ok = false; break; }
            if (k + 3 == n) umma_commit(&bars[kQEmpty]);
          }
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
    const int hh = (warp - 2) >> 2;                // which 32 tokens (and 128 O columns)
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const int tid = threadIdx.x - 64;              // 0..255
    uint8_t* xbuf = smem + OFF_X;
    uint8_t* xstage = smem + OFF_XS;
    float* mx_s = reinterpret_cast<float*>(smem + OFF_MX);   // [2][128]
    const uint32_t xbuf_peer = map_peer(smem_u32(xbuf), peer);
    const uint32_t xfull_peer = map_peer(smem_u32(&bars[kXFull]), peer);
    const uint32_t xempty_peer = map_peer(smem_u32(&bars[kXEmpty]), peer);
    Walker w{p.cum, 1, st, en};
    Seg sg;
    uint32_t it = 0;
    bool ok = true;
    // Every wait result is made warp-uniform: the warp-collective TMEM
    // instructions that follow must be executed by all 32 lanes or none.
    auto wait_all = [](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity) ? 1 : 0) != 0;
    };
    auto wait_all_cluster = [](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity) ? 1 : 0) != 0;
    };
    // This thread's 32 partial scores of tile t, in log2 units, as f16 pairs.
    auto own_partial = [&](uint32_t t, uint32_t (&h)[16]) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + TM_S + BS * (t & 1) + 32 * hh, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j)
        h[j] = pack_f16(__uint_as_float(v[2 * j]) * p.scale_log2,
                        __uint_as_float(v[2 * j + 1]) * p.scale_log2);
    };
    // Push this rank's partial of tile t to the peer: stage it locally (row r,
    // 16-byte chunks XOR-swizzled by r), then one bulk copy after the peer has
    // released the previous tile (which also means the previous copy has
    // finished reading the staging buffer).  `good` is the caller's state; the
    // result is uniform over the group (the named barrier ANDs it).
    auto send = [&](uint32_t t, bool good, uint32_t (&h)[16]) -> bool {
      good = good && wait_all(&bars[kSFull0 + (t & 1)], (t >> 1) & 1);
      if (good) {
        tc_fence_after();
        own_partial(t, h);
        good = wait_all_cluster(&bars[kXEmpty], (t & 1) ^ 1);
        if (good) {
          uint4* srow = reinterpret_cast<uint4*>(xstage + r * XROW);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            srow[(4 * hh + c) ^ (r & 7)] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
      }
      good = named_bar_and(2, NSW, good);
      if (good && tid == 0) bulk_copy_to_peer(xbuf_peer, xstage, XBYTES, xfull_peer);
      return good;
    };

    uint32_t hcur[16], hnext[16];
    while (ok && w.next(sg)) {
      const int len = max(0, min(p.seq_lens[sg.b], sg.n * BS));
      const uint32_t n = uint32_t(sg.j1 - sg.j0);
      float m_ref = -INFINITY, l = 0.f;   // l: this thread's half of the row sum
      if (!send(it, true, hcur)) { ok = false; break; }
      for (uint32_t k = 0; k < n && ok; ++k) {
        const uint32_t t = it + k;
        const int slot = t & 1;
        // A failed (bounded) wait below does not leave the loop at once: the
        // warp skips its work and the group agrees to stop at the next barrier.
        bool good = wait_all_cluster(&bars[kXFull], t & 1);
        float sc[32];
        float mx = -INFINITY;
        const int valid = len - (sg.j0 + int(k)) * BS - 32 * hh;
        if (good) {
          if (tid == 0) mbar_arrive_expect_tx(&bars[kXFull], XBYTES);  // next tile's bytes
          const uint4* xr = reinterpret_cast<const uint4*>(xbuf + r * XROW);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 v = xr[(4 * hh + c) ^ (r & 7)];
            const uint32_t pv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              // both ranks add the same two f16 partials: bit-identical scores
              const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&hcur[4 * c + q]));
              const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&pv[q]));
              sc[8 * c + 2 * q] = a.x + b.x;
              sc[8 * c + 2 * q + 1] = a.y + b.y;
            }
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            sc[j] = j < valid ? sc[j] : -INFINITY;
            mx = fmaxf(mx, sc[j]);
          }
          mx_s[hh * 128 + r] = mx;
        }
        // the row max over both halves of the tile
        good = named_bar_and(3, NSW, good);
        // Every thread has read the peer's partial (before the barrier): release
        // the exchange buffer.  One thread that has issued no bulk copy does it,
        // so its cluster-scope release does not wait for an outgoing copy.
        if (good && tid == 32) mbar_arrive_remote(xempty_peer);
        if (good) {
          mx = fmaxf(mx, mx_s[(hh ^ 1) * 128 + r]);
          if (k == 0) {
            m_ref = mx;
          } else if (__any_sync(0xffffffffu, mx > m_ref + RESCALE_THRESHOLD)) {
            // Some row's running max grew a lot: rescale this thread's half of
            // O (after the previous P.V landed) and l.  Both warps of a row pair
            // see the same maxima, so they take this branch together; TMEM
            // accesses are warp-collective, rows that keep their max scale by 1.
            good = wait_all(&bars[kPVDone0 + ((t - 1) & 1)], ((t - 1) >> 1) & 1);
            if (good) {
              tc_fence_after();
              const float m_new = mx > m_ref + RESCALE_THRESHOLD ? mx : m_ref;
              const float alpha = exp2_approx(m_ref - m_new);
              m_ref = m_new;
              l *= alpha;
#pragma unroll 1
              for (int cb = 0; cb < 128; cb += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + TM_O + 128 * hh + cb, o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                tmem_st32(tmem + lane_off + TM_O + 128 * hh + cb, o);
              }
              tmem_st_wait();
            }
          }
          if (good) {
            uint32_t pk[16];
            float lsum = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float p0 = exp2_approx(sc[2 * j] - m_ref), p1 = exp2_approx(sc[2 * j + 1] - m_ref);
              lsum += p0 + p1;
              pk[j] = pack_bf16(p0, p1);
            }
            l += lsum;
            tmem_st16(tmem + lane_off + TM_S + BS * slot + 16 * hh, pk);
            tmem_st_wait();
            const int vt = len - (sg.j0 + int(k)) * BS;   // valid rows of the whole tile
            if (vt < BS) {
              // Zero the latent rows past the end of the sequence in the four
              // boxes the P.V product reads: P is 0 there, but 0 * NaN is NaN.
              uint8_t* stg = smem + OFF_KV + (t % NSTAGE) * STAGE_BYTES;
              const int v0 = max(vt, 0);
              for (int idx = tid; idx < (BS - v0) * 4 * 8; idx += NSW) {
                const int row = v0 + idx / 32, rem = idx % 32;
                *reinterpret_cast<uint4*>(stg + (rem >> 3) * KF_BYTES + row * 128 + (rem & 7) * 16) =
                    make_uint4(0, 0, 0, 0);
              }
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tc_fence_before();
            mbar_arrive(&bars[kPFull0 + slot]);
          }
        }
        if (k + 1 < n) {
          ok = send(t + 1, good, hnext);
#pragma unroll
          for (int j = 0; j < 16; ++j) hcur[j] = hnext[j];
        } else {
          ok = named_bar_and(2, NSW, good);
        }
      }
      if (!ok) break;
      // ---- epilogue: O / l for this segment's rows (each thread: 128 columns)
      const uint32_t last = it + n - 1;
      // group-uniform, like every failure decision of this group
      if (!named_bar_and(2, NSW, wait_all(&bars[kPVDone0 + (last & 1)], (last >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      mx_s[hh * 128 + r] = l;
      named_bar_sync(3, NSW);
      const float lrow = l + mx_s[(hh ^ 1) * 128 + r];
      const bool row_ok = r < p.h;
      float* dst;
      float* dl;
      if (sg.full) {
        dst = p.out + (int64_t(sg.b) * p.h + r) * DC + 256 * rank + 128 * hh;
        dl = p.lse + int64_t(sg.b) * p.h + r;
      } else {
        const int64_t slot_idx = int64_t(sg.b) + pair;
        dst = p.part_out + (slot_idx * p.h + r) * DC + 256 * rank + 128 * hh;
        dl = p.part_lse + slot_idx * p.h + r;
      }
      const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
#pragma unroll 1
      for (int cb = 0; cb < 128; cb += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_off + TM_O + 128 * hh + cb, o);
        tmem_ld_wait();
        if (row_ok) {
          float4* d4 = reinterpret_cast<float4*>(dst + cb);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            d4[j] = make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                                __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
        }
      }
      if (row_ok && rank == 0 && hh == 0)
        *dl = (lrow > 0.f) ? (m_ref + log2_approx(lrow)) * kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(&bars[kOFree]);
      it += n;
      // the row-sum slots are rewritten next segment only after this barrier
      ok = named_bar_and(2, NSW, *abort_flag == 0);
    }
    if (!ok) {
      report(p.err, KVATTN_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
    // Drain: the peer's last "done reading" arrival targets this CTA's barrier;
    // wait for it so this CTA's shared memory outlives every remote access.
    if (it > 0) mbar_wait_cluster(&bars[kXEmpty], (it - 1) & 1);
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

  alignas(64) CUtensorMap tmQF, tmQH, tmLF, tmLH;
  {
    const uint64_t dims[3] = {uint64_t(mla::ROWW), uint64_t(a.h), uint64_t(a.B)};
    const uint64_t strides[2] = {uint64_t(mla::ROWW) * 2, uint64_t(mla::ROWW) * 2 * a.h};
    const uint32_t boxf[3] = {64u, 128u, 1u}, boxh[3] = {32u, 128u, 1u};
    if (!encode_tensor_map_3d(&tmQF, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, dims, strides, boxf,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_3d(&tmQH, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, dims, strides, boxh,
                              CU_TENSOR_MAP_SWIZZLE_64B))
      return KVATTN_ERR_CUDA;
  }
  {
    const uint64_t dims[3] = {uint64_t(mla::ROWW), uint64_t(mla::BS), uint64_t(cc->num_blocks)};
    const uint64_t strides[2] = {uint64_t(mla::ROWW) * 2, uint64_t(mla::ROWW) * 2 * mla::BS};
    const uint32_t boxf[3] = {64u, uint32_t(mla::BS), 1u}, boxh[3] = {32u, uint32_t(mla::BS), 1u};
    if (!encode_tensor_map_3d(&tmLF, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cc->latent, dims, strides,
                              boxf, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_3d(&tmLH, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cc->latent, dims, strides,
                              boxh, CU_TENSOR_MAP_SWIZZLE_64B))
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
  mla_decode_kernel<<<2 * G, mla::THREADS, mla::SMEM, a.stream>>>(tmQF, tmQH, tmLF, tmLH, prm);
  if (cudaGetLastError() != cudaSuccess) return KVATTN_ERR_CUDA;
  if (launch_combine(prm.part_out, prm.part_lse, pa.split_first, pa.split_count, a.B, a.h,
                     mla::DC, a.out, a.lse, true, a.stream) != cudaSuccess)
    return KVATTN_ERR_CUDA;
  return KVATTN_OK;
}

}  // namespace kv
