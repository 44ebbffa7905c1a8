// decode_gqa_tc.cu -- GQA decode on tcgen05 for units of many rows.
//
// The same computation as decode_gqa.cu ("MHA → MQA → GQA → MLA", the grouped
// attention of one KV head; "MLA：为什么一份 Latent 可以代替多头 KV Cache",
// section "Prefill 为什么未必使用与 Decode 相同的吸收方式", several new tokens
// verified per pass, causal among themselves): for each unit (sequence b, KV
// head), its rows r = (new token j, head i of the group), r = j * g + i, attend
// to the cached positions [0, s_b - (q_len - 1 - j)).
//
// When a unit has more than 32 rows the mma.sync kernel runs every 16-row
// m-tile of a chunk through its own warps, and its fixed-latency MMA chains
// cap it at 190-250 TFLOP/s whatever the bytes.  Here the unit's rows are the
// M dimension of tcgen05 MMAs (M = 128; rows past q_len * g are padding that
// no thread writes out), over tiles of TT tokens (64 for bf16 caches, 128 for
// E4M3):
//   S = Q K^T   M = 128 rows, N = TT tokens, K = 128 dims
//   O += P V    M = 128 rows, N = 128 dims, K = TT tokens, P from TMEM
// with S, P and O in tensor memory.  Thread r of the four softmax warps owns
// TMEM lane r, i.e. row r, so the online softmax (lazy rescale of O when a
// row's max grows by more than 2^8) needs no exchange between threads.
//
// A tile is TT / 16 chunks of 16 tokens; a chunk of bf16 K (or V) arrives as
// two TMA boxes [16 tokens x 64 dims] (128-byte swizzle) at row 16c of the
// tile's two 64-dim halves, which makes each half one swizzled [64 x 64]
// operand (E4M3: one box [16 tokens x 128 codes] into a [128 x 128] one).  Chunks past the CTA's range are loaded from an out-of-range page
// (zero fill); cached rows past the sequence's length are zeroed in shared
// memory by the softmax warps before P.V reads them (P is 0 there, but 0 * NaN
// would be NaN).  The planner, the partial slots and the combine are those of
// the mma.sync kernel.
//   warps 0, 6-8  TMA producers: warp 0 loads the unit's Q per segment (a 4-D
//              box [q_len][g][64 dims], twice) and arms each tile's barrier;
//              producer warp pc issues the boxes of chunks pc, pc + 4, ... of
//              each tile (one warp issuing all 16 boxes of a bf16 tile
//              serialises them at ~120 cycles apiece, ~1 us per tile: the HBM
//              needs one per ~0.7 us)
//   warps 1, 14  TMEM owner (1) and S issuers: even tiles from warp 1, odd
//              ones from warp 14 (one thread issuing every tile's MMAs at
//              ~110 cycles apiece set the pace), into S slot t % 2 (bf16) or
//              the one S slot (E4M3)
//   warp 9     P.V issuer (one thread issuing both MMA chains, ~100 cycles
//              per tcgen05.mma, set a period of ~1 us per tile)
//   warps 2-5, 10-13  softmax and epilogue, two threads per row
#include <cuda_fp16.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"
#include "walk.cuh"

// Test builds only (-DKV_TEST_DROP_CHUNK=n, with a short KV_WAIT_NS): CTA 0's
// first producer warp issues none of its loads of tile n, as copies that never
// land would, so that the tile's barrier never completes, the bounded waits on
// it run out and the abort path (error bit, stop, drain, exit) runs on the
// GPU.  The library is built without it.
#ifdef KV_TEST_DROP_CHUNK
#define KV_TEST_DROPS_TILE(t, w) (blockIdx.x == 0 && (w) == 0 && (t) == uint32_t(KV_TEST_DROP_CHUNK))
#else
#define KV_TEST_DROPS_TILE(t, w) false
#endif

namespace kv {

namespace gtc {
constexpr int D = 128;
constexpr int NSTAGE_MAX = 8;
constexpr int QHALF = 128 * 128;        // [128 rows x 128 B]: Q's dims 0-63 / 64-127 (bf16), or
                                        // its hi / lo E4M3 term (128 codes)
constexpr int OFF_Q = 0;
constexpr int OFF_ST = 2 * QHALF;
constexpr int XB_BYTES = 2 * 3 * 32 * 32 * 4;      // [hh][copy - 1][row][32 columns], 4 copies
constexpr int NBARS = 40;
// Per cache format.  bf16: a tile is 64 tokens and a stage holds K dims 0-63,
// K dims 64-127, V dims 0-63, V dims 64-127 (32 KB).  E4M3: a tile is 128
// tokens (a 64-token tile of codes is 16 KB, and the softmax's fixed cost per
// tile, not the bytes, then set the pace) and a stage holds K codes, V codes
// (32 KB).
template <bool FP8>
struct Lay {
  static constexpr int TT = FP8 ? 128 : 64;                   // tokens per tile
  static constexpr int HALF = TT * 128;                       // [TT tokens x 128 B]
  static constexpr int STAGE = FP8 ? 2 * HALF : 4 * HALF;
  static constexpr int NSTAGE = 5;
  static constexpr int V_OFF = FP8 ? HALF : 2 * HALF;        // V within a stage
  static constexpr int NS = FP8 ? 1 : 2;                      // S slots of TT columns
  static constexpr int PCOLS = TT / 2;                        // columns of a P slot
  static constexpr int OFF_ML = OFF_ST + NSTAGE * STAGE;      // the epilogue's row max / sum exchange
  static constexpr int OFF_QF = OFF_ML + 4 * 128 * 4;         // E4M3: each row's 2^-e
  static constexpr int OFF_XB = OFF_QF + 128 * 4;             // the epilogue's merge of the row copies
  static constexpr int OFF_BAR = OFF_XB + XB_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + NBARS * 8 + 16;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(NSTAGE <= NSTAGE_MAX, "barrier slots");
};
constexpr int THREADS = 480;
constexpr int PV_WARP = 9;
constexpr int S2_WARP = 14;             // the second S issuer (odd tiles)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;            // S slots: two of 64 columns (bf16), one of 128 (E4M3)
constexpr uint32_t TM_P = 128;          // two P slots of TT / 2 columns (bf16 pairs, E4M3 quads
                                        // of the two terms)
constexpr int NP = 2;                   // P slots: the softmax of tile t waits for P.V(t - 2)
constexpr uint32_t TM_O = 256;          // O of each tile's first half of tokens, then of its second
constexpr float RESCALE = 8.f;          // log2 units
static_assert(Lay<false>::NS * Lay<false>::TT <= 128 && Lay<true>::NS * Lay<true>::TT <= 128, "S");
static_assert(NP * Lay<false>::PCOLS <= 128 && NP * Lay<true>::PCOLS <= 128, "P");
}  // namespace gtc

enum : int {
  gQFull = 0, gQEmpty = 1, gOFree = 2,
  gSFull0 = 3,    // 2: S(t) is in its slot, by the parity of t
  gSRead0 = 5,    // 2: the softmax warps have read S(t), by the parity of t
  gPFull0 = 7,    // NP: P(t) is in P slot t % NP (and the tile's tail rows zeroed)
  gPVDone0 = 10,  // NP: P.V(t) has completed (P slot t % NP free)
  gDrain = 13,
  gFull0 = 14,                              // NSTAGE: the tile's K and V landed
  gEmpty0 = gFull0 + gtc::NSTAGE_MAX,       // NSTAGE: P.V finished with the stage
  gAbort = gEmpty0 + gtc::NSTAGE_MAX,       // an int flag in this slot
  gDrain2 = gAbort + 1,                     // the P.V issuer's last MMAs completed
  gDrain3 = gDrain2 + 1,                    // the second S issuer's last MMAs completed
  gNumBars = gDrain3 + 1,
  gQBuilt = gQFull                          // E4M3: the softmax warps built Q's terms (no TMA)
};
static_assert(gNumBars <= gtc::NBARS, "barrier slots");

// Two E4M3 terms of a float pair: hi = e4m3(x), lo = e4m3(x - hi), each a
// 16-bit code pair (first value in the low byte).  x is first rounded to f16
// (both callers pass values below 2^9, and E4M3 keeps 4 significant bits per
// term, so the f16 rounding is far below the terms' own); then hi is exact in
// f16 and so is x - hi, which one f16x2 subtraction gives for both values.
KV_DEVI void e4m3_two_terms_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const uint32_t xf = pack_f16(x0, x1);
  uint16_t h, l;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(h) : "r"(xf));
  const uint32_t hf = e4m3x2_to_f16x2(h);
  uint32_t rf;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(rf) : "r"(xf), "r"(hf));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l) : "r"(rf));
  hi = h;
  lo = l;
}

// E4M3 cache: MMA row m (copy of unit row r) of the query as two E4M3 terms
// (dims 64 hh .. 64 hh + 63 from this thread; both threads of a row find the
// same scale),
// x 2^e with e chosen so that the row's largest magnitude lands in [128, 256):
// hi codes at q + m * 128, lo codes at q + QHALF + m * 128, in the 128-byte
// swizzled K-major layout; 2^-e to qf[m].  Rows past the unit's are zero.
KV_DEVI void build_q_terms(const GqaParams& p, const Seg& sg, int r, bool row_ok, uint8_t* q,
                           int m, int hh, float* qf) {
  int64_t qi = 0;
  if (row_ok) {
    if (p.qlen > 1) {
      const int j = r / p.g, i = r - j * p.g;
      qi = (int64_t(sg.b) * p.qlen + j) * p.h + sg.kvh * p.g + i;
    } else {
      qi = int64_t(sg.b) * p.h + sg.kvh * p.g + r;
    }
  }
  const uint4* src = reinterpret_cast<const uint4*>(p.q + qi * gtc::D);
  auto lo16 = [](uint32_t w) { return __uint_as_float(w << 16); };
  auto hi16 = [](uint32_t w) { return __uint_as_float(w & 0xffff0000u); };
  // pass 1: the row's largest magnitude (eight loads in flight at a time)
  float mx = 0.f;
#pragma unroll 1
  for (int g0 = 0; g0 < 16; g0 += 8) {
    uint4 x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = row_ok ? __ldg(src + g0 + i) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) mx = fmaxf(mx, fmaxf(fabsf(lo16(w[k])), fabsf(hi16(w[k]))));
    }
  }
  const int e = mx > 0.f ? min(max(7 - (int((__float_as_uint(mx) >> 23) & 255) - 127), -120), 120) : 0;
  const float sc = __uint_as_float(uint32_t(127 + e) << 23);
  if (hh == 0) qf[m] = __uint_as_float(uint32_t(127 - e) << 23);
  // pass 2: this thread's 64 dims, 16 (one 16-byte piece of codes per term)
  // at a time
#pragma unroll 1
  for (int c = 4 * hh; c < 4 * hh + 4; ++c) {
    const uint4 x0 = row_ok ? __ldg(src + 2 * c) : make_uint4(0, 0, 0, 0);
    const uint4 x1 = row_ok ? __ldg(src + 2 * c + 1) : make_uint4(0, 0, 0, 0);
    const uint32_t wv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t h0, l0, h1, l1;
      e4m3_two_terms_pair(lo16(wv[2 * k]) * sc, hi16(wv[2 * k]) * sc, h0, l0);
      e4m3_two_terms_pair(lo16(wv[2 * k + 1]) * sc, hi16(wv[2 * k + 1]) * sc, h1, l1);
      hw[k] = h0 | (h1 << 16);
      lw[k] = l0 | (l1 << 16);
    }
    const int off = m * 128 + ((c ^ (m & 7)) << 4);
    *reinterpret_cast<uint4*>(q + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(q + gtc::QHALF + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

// DUP copies of the unit's rows fill the MMA's 128 rows (rows <= 128 / DUP):
// copy c sits at rows [c * 128 / DUP, (c + 1) * 128 / DUP).  Their scores are
// equal; each copy's threads take a different part of the tile's tokens.
//
// E4M3 cache (FP8): the MMAs are kind::f8f6f4 (K = 32, both operands E4M3).
// The cached codes are used as stored; the query and the probabilities enter
// as two E4M3 terms each, hi = e4m3(x) and lo = e4m3(x - hi).  The softmax
// warps of the first token half build each row's query terms from bf16 at a
// segment's start, scaled by 2^e that brings the row's largest magnitude into
// [128, 256); the scores are multiplied back by 2^-e and k_scale, O by
// v_scale.
template <bool MQ, int DUP, bool FP8>
__global__ void __launch_bounds__(gtc::THREADS, 1)
    gqa_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const GqaParams p) {
  using namespace gtc;
  using L = Lay<FP8>;
  constexpr int TT = L::TT, HALF = L::HALF, STAGE = L::STAGE, NSTAGE = L::NSTAGE, V_OFF = L::V_OFF;
  constexpr int NS = L::NS, PCOLS = L::PCOLS;
  constexpr int CPT = TT / 16;   // 16-token chunks per tile
  constexpr int OFF_ML = L::OFF_ML, OFF_QF = L::OFF_QF, OFF_XB = L::OFF_XB, OFF_BAR = L::OFF_BAR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + gAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(&bars[gQFull], FP8 ? 8 : 1);   // TMA (bf16), or the eight builder warps (E4M3)
    mbar_init(&bars[gQEmpty], 2);            // both S issuers

    mbar_init(&bars[gOFree], 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[gSFull0 + i], 1);
      mbar_init(&bars[gSRead0 + i], 8);
    }
    for (int i = 0; i < NP; ++i) {
      mbar_init(&bars[gPFull0 + i], 8);
      mbar_init(&bars[gPVDone0 + i], 1);
    }
    mbar_init(&bars[gDrain], 1);
    mbar_init(&bars[gDrain2], 1);
    mbar_init(&bars[gDrain3], 1);
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&bars[gFull0 + i], 1);
      mbar_init(&bars[gEmpty0 + i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  __syncwarp();
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Launched right behind the planner: wait for its plan, and let the combine
  // that follows get scheduled while this grid runs.
  pdl_wait();
  pdl_launch_dependents();
  const int4 st = p.cta_start[c], en = p.cta_start[c + 1];
  const uint32_t tmem = *tmem_slot;
  const int cpp = p.bs >> 4;  // 16-token chunks per page

  if (pos_less(st, en)) {
    if (warp == 0 || (warp >= 6 && warp < PV_WARP)) {
      // ------------------------------------------------------------- producers
      const int pc = warp == 0 ? 0 : warp - 5;   // the chunk of each tile this warp loads
      const uint64_t pol = policy_evict_first();
      const int oob_page = int(p.num_blocks * p.hkv);  // past the end: zero fill
      Walker w{p.cum, p.hkv, st, en};
      Seg sg;
      uint32_t t = 0, seg = 0;
      bool ok = true;
      while (ok && w.next(sg)) {
        if (!FP8 && warp == 0 && lane == 0) {
          if (seg > 0 && !mbar_wait(&bars[gQEmpty], (seg - 1) & 1)) {
            ok = false;
          } else {
            // rows j * g + i: the box [q_len][g][64 dims] at head kvh * g, once
            // per copy
            mbar_arrive_expect_tx(&bars[gQFull], uint32_t(2 * DUP * 128 * p.rows));
            for (int cp = 0; cp < DUP; ++cp) {
              uint8_t* qd = smem + OFF_Q + cp * (128 / DUP) * 128;
              tma_load_4d(qd, &tmQ, 0, sg.kvh * p.g, 0, sg.b, &bars[gQFull]);
              tma_load_4d(qd + QHALF, &tmQ, 64, sg.kvh * p.g, 0, sg.b, &bars[gQFull]);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++seg;
        const int32_t* row = p.bt + int64_t(sg.b) * p.max_blocks;
        const int nch = (sg.j1 - sg.j0) * cpp;
        for (int pb = sg.j0; pb < sg.j1 && ok; pb += 32) {
          // block ids of pages pb .. pb + 31, one per lane
          int page = oob_page;
          if (pb + lane < sg.j1) {
            const int blk = row[pb + lane];
            if (blk < 0 || int64_t(blk) >= p.num_blocks)
              report(p.err, KVATTN_DEVERR_BLOCK_ID);
            else
              page = blk * p.hkv + sg.kvh;
          }
          // tiles of CPT chunks; a tile never straddles two groups of 32 pages
          const int c0 = (pb - sg.j0) * cpp;
          const int c1 = min(pb + 32 - sg.j0, sg.j1 - sg.j0) * cpp;
          for (int cc = c0; cc < c1 && ok; cc += CPT) {
            const int s = int(t % NSTAGE);
            int lok = 1;
            if (lane == 0) {
              lok = mbar_wait(&bars[gEmpty0 + s], ((t / NSTAGE) & 1) ^ 1) ? 1 : 0;
              // one arrival, and the tile's bytes from all four warps' loads
              if (lok && warp == 0) mbar_arrive_expect_tx(&bars[gFull0 + s], uint32_t(STAGE));
            }
            lok = __shfl_sync(0xffffffffu, lok, 0);
            if (!lok) {
              ok = false;
              break;
            }
#pragma unroll
            for (int qc = 0; qc < CPT / 4; ++qc) {
              const int ci = cc + pc + 4 * qc;                           // this warp's chunk
              const int src = min(max(ci / cpp - (pb - sg.j0), 0), 31);  // lane holding its page
              const int pg_l = __shfl_sync(0xffffffffu, page, src);
              if (lane == 0 && !KV_TEST_DROPS_TILE(t, warp)) {
                const int pg = ci < nch ? pg_l : oob_page;
                const int sub = ci % cpp;
                uint8_t* dst = smem + OFF_ST + s * STAGE + (pc + 4 * qc) * (16 * 128);
                if constexpr (FP8) {   // one box of 128 codes per row for K and for V
                  tma_load_3d(dst, &tmK, 0, sub * 16, pg, &bars[gFull0 + s], pol);
                  tma_load_3d(dst + V_OFF, &tmV, 0, sub * 16, pg, &bars[gFull0 + s], pol);
                } else {
                  tma_load_3d(dst, &tmK, 0, sub * 16, pg, &bars[gFull0 + s], pol);
                  tma_load_3d(dst + HALF, &tmK, 64, sub * 16, pg, &bars[gFull0 + s], pol);
                  tma_load_3d(dst + V_OFF, &tmV, 0, sub * 16, pg, &bars[gFull0 + s], pol);
                  tma_load_3d(dst + V_OFF + HALF, &tmV, 64, sub * 16, pg, &bars[gFull0 + s], pol);
                }
              }
            }
            ++t;   // issued: the exit drain waits for it
            ok = __shfl_sync(0xffffffffu, lane == 0 ? (*abort_flag == 0) : true, 0);
          }
        }
      }
      if (lane == 0) {
        if (!ok) {
          report(p.err, KVATTN_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        // every load issued lands before the CTA exits
        if (!FP8 && warp == 0 && seg > 0) mbar_wait(&bars[gQFull], (seg - 1) & 1, KV_DRAIN_WAIT_NS);
        for (uint32_t k = t > uint32_t(NSTAGE) ? t - NSTAGE : 0u; k < t; ++k)
          mbar_wait(&bars[gFull0 + k % NSTAGE], (k / NSTAGE) & 1, KV_DRAIN_WAIT_NS);
      }
    } else if (warp == 1 || warp == PV_WARP || warp == S2_WARP) {
      // ---------------------------------------------- MMA issuers: S, and P.V
      if (lane == 0) {
        const uint32_t st0 = smem_u32(smem + OFF_ST);
        Walker w{p.cum, p.hkv, st, en};
        Seg sg;
        uint32_t t = 0, seg = 0;
        bool ok = true;
        if (warp != PV_WARP) {
          const uint32_t sp = warp == 1 ? 0u : 1u;   // the tiles t with t % 2 == sp
          const uint32_t id_s = FP8 ? idesc_e4m3(128, TT, false) : idesc_bf16(128, TT, false);
          const uint64_t qa0 = sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
          while (ok && w.next(sg)) {
            const int ntile = ((sg.j1 - sg.j0) * cpp + CPT - 1) / CPT;
            if (!mbar_wait(&bars[gQFull], seg & 1)) {
              ok = false;
              break;
            }
            for (int k = 0; k < ntile && ok; ++k, ++t) {
              if ((t & 1) != sp) continue;
              // the tile's K and V, and its S slot: the softmax has read S(t - NS).
              // The barriers go by tile parity whatever the slots: an issuer
              // sees every completion of the barrier it waits on, so its
              // parity cannot alias (with one slot, a single barrier would
              // complete twice between this issuer's waits).
              const uint32_t tr = t - NS;
              if ((t >= uint32_t(NS) && !mbar_wait(&bars[gSRead0 + (tr & 1)], (tr >> 1) & 1)) ||
                  !mbar_wait(&bars[gFull0 + t % NSTAGE], (t / NSTAGE) & 1)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t kd = sdesc_sw128(st0 + (t % NSTAGE) * STAGE, 16, 1024);
              const uint32_t sd = tmem + TM_S + TT * (t % NS);
              if constexpr (FP8) {
                // 32 codes per MMA: the hi term of Q, then the lo term
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                  umma_ss_f8(sd, qa0 + uint64_t((kk * 32) >> 4), kd + uint64_t((kk * 32) >> 4), id_s,
                             kk > 0 ? 1u : 0u);
                  umma_ss_f8(sd, qa0 + uint64_t((QHALF + kk * 32) >> 4),
                             kd + uint64_t((kk * 32) >> 4), id_s, 1u);
                }
              } else {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                  const uint32_t off = (kk >> 2) * HALF + (kk & 3) * 32;     // K: half, 16 dims
                  const uint32_t qoff = (kk >> 2) * QHALF + (kk & 3) * 32;   // Q: same dims
                  umma_ss(sd, qa0 + uint64_t(qoff >> 4),
                          kd + uint64_t(off >> 4), id_s, kk > 0 ? 1u : 0u);
                }
              }
              umma_commit(&bars[gSFull0 + (t & 1)]);
              if (*abort_flag) ok = false;
            }
            // every S of this issuer in the segment is issued (the barrier
            // completes when both issuers' score MMAs have)
            if (ok) umma_commit(&bars[gQEmpty]);
            ++seg;
          }
        } else {
          const uint32_t id_o = FP8 ? idesc_e4m3(128, D, true) : idesc_bf16(128, D, true);
          while (ok && w.next(sg)) {
            const int ntile = ((sg.j1 - sg.j0) * cpp + CPT - 1) / CPT;
            for (int k = 0; k < ntile && ok; ++k, ++t) {
              // O (+)= P(t) V(t): the first tile of a segment overwrites O, once
              // the previous segment's epilogue has read it
              if ((k == 0 && seg > 0 && !mbar_wait(&bars[gOFree], (seg - 1) & 1)) ||
                  !mbar_wait(&bars[gPFull0 + t % NP], (t / NP) & 1)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t vd = sdesc_sw128(st0 + (t % NSTAGE) * STAGE + V_OFF, HALF, 1024);
              // the tile's first half of tokens into O_0, its second into O_1
              // (the two softmax halves)
              if constexpr (FP8) {
                // 32 tokens per MMA, for the hi and the lo term of P (P slot
                // columns: hi half 0, hi half 1, lo half 0, lo half 1, TT / 8
                // each)
#pragma unroll
                for (int kk = 0; kk < TT / 16; ++kk) {
                  const int ks = kk % (TT / 64), h2 = (kk / (TT / 64)) & 1, term = kk / (TT / 32);
                  umma_ts_f8(tmem + TM_O + 128 * h2,
                             tmem + TM_P + PCOLS * (t % NP) + (TT / 4) * term + (TT / 8) * h2 + 8 * ks,
                             vd + uint64_t(((h2 * (TT / 2) + ks * 32) * 128) >> 4), id_o,
                             (k == 0 && term == 0 && ks == 0) ? 0u : 1u);
                }
              } else {
#pragma unroll
                for (int kk = 0; kk < TT / 16; ++kk)
                  umma_ts(tmem + TM_O + 128 * (kk >> 1), tmem + TM_P + PCOLS * (t % NP) + 8 * kk,
                          vd + uint64_t((kk * 16 * 128) >> 4), id_o,
                          (k == 0 && (kk & 1) == 0) ? 0u : 1u);
              }
              umma_commit(&bars[gEmpty0 + t % NSTAGE]);
              umma_commit(&bars[gPVDone0 + t % NP]);
              if (*abort_flag) ok = false;
            }
            ++seg;
          }
        }
        if (!ok) {
          report(p.err, KVATTN_DEVERR_TIMEOUT);
          *abort_flag = 1;
        }
        // no MMA of this thread may still write TMEM when it is released
        uint64_t* drain = &bars[warp == 1 ? gDrain : warp == PV_WARP ? gDrain2 : gDrain3];
        umma_commit(drain);
        mbar_wait(drain, 0, KV_DRAIN_WAIT_NS);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------- softmax / epilogue
      // Threads by MMA row (TMEM lane) m and token half hh: warps 2-5 take the
      // tile's first TT / 2 tokens (hh = 0), warps 10-13 the rest (hh = 1).  Row m
      // is copy c = m / RP of unit row r = m % RP, and of its half the thread
      // takes the TP tokens of part c.  Each (lane, half) keeps its own
      // running max, sum and share of O_hh (O_hh += P[:, half] V[half, :]), so
      // the threads never wait for each other inside a segment; the epilogue
      // merges the 2 DUP states of each row.  (With one thread per row the
      // softmax, one warp per SM sub-partition with nothing to hide its
      // latencies, set the kernel's pace at ~1 us per 64-token tile; TMEM lane
      // quadrant q is readable only from sub-partition q, so spare MMA rows
      // spread the work only by holding copies.)
      constexpr int RP = 128 / DUP;                         // rows per copy
      constexpr int TP = TT / 2 / DUP;                      // tokens per thread and tile
      const int m = 32 * (warp & 3) + lane;                 // MMA row = TMEM lane
      const int cpy = m / RP, r = m % RP;
      const int hh = warp >= 10 ? 1 : 0;
      const int part = (TT / 2) * hh + TP * cpy;            // first token of this thread's part
      const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
      const int tid = hh * 128 + m;                         // 0..255
      const uint32_t tm_oh = TM_O + 128 * hh;               // this half's O
      const bool row_ok = r < p.rows;
      // causal limit among the new tokens: row r's token is r / g
      const int back = MQ ? p.qlen - 1 - min(r, p.rows - 1) / p.g : 0;
      float* ml_s = reinterpret_cast<float*>(smem + OFF_ML);   // [hh][m or l][128 lanes]
      float* qf_s = reinterpret_cast<float*>(smem + OFF_QF);   // E4M3: [128 lanes] 2^-e
      float4* xb = reinterpret_cast<float4*>(smem + OFF_XB);   // [hh][copy - 1][RP][8]
      static_assert(2 * (DUP - 1) * RP * 8 * 16 <= XB_BYTES, "merge buffer");
      // every wait result is warp-uniform: the TMEM instructions that follow
      // are warp-collective
      auto wait_all = [](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity) ? 1 : 0) != 0;
      };
      {
        // zero this row's columns of this half in both P slots (both terms for
        // E4M3): each tile then writes only its own part
        const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int sl = 0; sl < NP; ++sl) {
          if constexpr (FP8) {
#pragma unroll
            for (int term = 0; term < 2; ++term)
              tmem_st16(tmem + lane_off + TM_P + PCOLS * sl + (TT / 4) * term + (TT / 8) * hh, z);
          } else {
            tmem_st16(tmem + lane_off + TM_P + PCOLS * sl + 16 * hh, z);
          }
        }
        tmem_st_wait();
      }
      Walker w{p.cum, p.hkv, st, en};
      Seg sg;
      uint32_t t = 0, seg = 0;
      bool good = true;
      while (w.next(sg)) {
        int len = p.seq_lens[sg.b];
        len = max(0, min(len, sg.n * p.bs));
        const int lim = row_ok ? len - back : 0;            // this row sees tokens [0, lim)
        const int tok_beg = sg.j0 * p.bs, tok_end = sg.j1 * p.bs;
        const int ntile = ((sg.j1 - sg.j0) * cpp + CPT - 1) / CPT;
        float m_ref = -INFINITY, l = 0.f;
        float qk = p.qk_scale_log2;   // raw score -> log2 units (E4M3: times this row's 2^-e)
        if constexpr (FP8) {
          // This row's query as two E4M3 terms (this thread: the half hh of
          // its dims), once the previous segment's score MMAs (which read
          // them) have completed.
          good = seg == 0 || wait_all(&bars[gQEmpty], (seg - 1) & 1);
          if (good) {
            build_q_terms(p, sg, r, row_ok, smem + OFF_Q, m, hh, qf_s);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[gQBuilt]);
          }
          good = good && wait_all(&bars[gQBuilt], seg & 1);
          if (good) qk *= qf_s[m];
        }
        for (int k = 0; k < ntile && good; ++k, ++t) {
          good = wait_all(&bars[gSFull0 + (t & 1)], (t >> 1) & 1);
          if (!good) break;
          tc_fence_after();
          uint32_t sv[TP];
          const uint32_t sa = tmem + lane_off + TM_S + TT * (t % NS) + part;
          if constexpr (TP == 64) {
            tmem_ld32(sa, *reinterpret_cast<uint32_t(*)[32]>(sv));
            tmem_ld32(sa + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
          } else if constexpr (TP == 32) {
            tmem_ld32(sa, sv);
          } else if constexpr (TP == 16) {
            tmem_ld16(sa, sv);
          } else {
            tmem_ld8(sa, sv);
          }
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[gSRead0 + (t & 1)]);
          const int t0 = tok_beg + TT * k + part;           // this thread's first token
          const int nv = min(lim, tok_end) - t0;            // tokens n < nv are seen
          float mx = -INFINITY;
#pragma unroll
          for (int n = 0; n < TP; ++n)
            if (n < nv) mx = fmaxf(mx, __uint_as_float(sv[n]));
          mx *= qk;
          const bool grow = mx > m_ref + RESCALE;
          if (__any_sync(0xffffffffu, grow)) {
            const float m_new = grow ? mx : m_ref;
            const float alpha = grow ? exp2_approx(m_ref - m_new) : 1.f;   // 0 while m_ref = -inf
            if (k > 0) {
              // O_hh holds this segment's earlier tiles: rescale this row once
              // P.V(t - 1) has landed
              good = wait_all(&bars[gPVDone0 + (t - 1) % NP], ((t - 1) / NP) & 1);
              if (!good) break;
              tc_fence_after();
#pragma unroll 1
              for (int cb = 0; cb < D; cb += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_off + tm_oh + cb, o);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                tmem_st32(tmem + lane_off + tm_oh + cb, o);
              }
              tmem_st_wait();
            }
            l = k > 0 ? l * alpha : 0.f;
            m_ref = m_new;
          }
          // the P slot was last read by P.V(t - NP)
          good = t < uint32_t(NP) || wait_all(&bars[gPVDone0 + t % NP], ((t - NP) / NP) & 1);
          if (!good) break;
          tc_fence_after();
          float ls = 0.f;
          if constexpr (FP8) {
            // two E4M3 terms, four codes per TMEM column: this copy's part of
            // the half's TT / 2 tokens (the half has TT / 8 columns per term)
            constexpr int HC = TT / 8, MC = TP / 4;   // columns of the half, of this part
            uint32_t ph[MC], pl[MC];
#pragma unroll
            for (int j = 0; j < TP / 2; ++j) {
              const float a0 = 2 * j < nv ? exp2_approx(fmaf(__uint_as_float(sv[2 * j]), qk, -m_ref)) : 0.f;
              const float a1 = 2 * j + 1 < nv ? exp2_approx(fmaf(__uint_as_float(sv[2 * j + 1]), qk, -m_ref)) : 0.f;
              ls += a0 + a1;
              uint32_t h2, l2;
              e4m3_two_terms_pair(a0, a1, h2, l2);
              if (j & 1) {
                ph[j >> 1] |= h2 << 16;
                pl[j >> 1] |= l2 << 16;
              } else {
                ph[j >> 1] = h2;
                pl[j >> 1] = l2;
              }
            }
            // only this part's columns: the rest of the row stays zero from
            // the start of the kernel (no other thread writes this row)
            const uint32_t pa = tmem + lane_off + TM_P + PCOLS * (t % NP) + HC * hh + MC * cpy;
            if constexpr (MC == 16) {
              tmem_st16(pa, ph);
              tmem_st16(pa + 2 * HC, pl);
            } else if constexpr (MC == 8) {
              tmem_st8(pa, ph);
              tmem_st8(pa + 2 * HC, pl);
            } else {
              static_assert(MC == 4, "P store");
              tmem_st4(pa, ph);
              tmem_st4(pa + 2 * HC, pl);
            }
          } else {
            uint32_t pv[TP / 2];
#pragma unroll
            for (int j = 0; j < TP / 2; ++j) {
              const float a0 = 2 * j < nv ? exp2_approx(fmaf(__uint_as_float(sv[2 * j]), qk, -m_ref)) : 0.f;
              const float a1 = 2 * j + 1 < nv ? exp2_approx(fmaf(__uint_as_float(sv[2 * j + 1]), qk, -m_ref)) : 0.f;
              ls += a0 + a1;
              pv[j] = pack_bf16(a0, a1);
            }
            // this half's 32 tokens are 16 bf16 pairs; this thread stores its
            // copy's part (the other copies' rows hold the other parts, and
            // these columns of this row stay zero from the start)
            const uint32_t pa = tmem + lane_off + TM_P + PCOLS * (t % NP) + 16 * hh + (TP / 2) * cpy;
            if constexpr (TP / 2 == 16) {
              tmem_st16(pa, pv);
            } else if constexpr (TP / 2 == 8) {
              tmem_st8(pa, pv);
            } else {
              static_assert(TP / 2 == 4, "P store");
              tmem_st4(pa, pv);
            }
          }
          l += ls;
          tmem_st_wait();
          const int vt = len - (tok_beg + TT * k);   // cached rows of the tile that hold tokens
          if (vt < TT) {
            // Zero the V rows past the sequence's end (stale or never-written
            // slots of its last page); rows past the CTA's range came from
            // the out-of-range page and are zero already.
            uint8_t* vb = smem + OFF_ST + (t % NSTAGE) * STAGE + V_OFF;
            const int v0 = max(vt, 0);
            constexpr int PIECES = FP8 ? 8 : 16;   // 16-byte pieces of a row (both bf16 halves)
            for (int idx = tid; idx < (TT - v0) * PIECES; idx += 256) {
              const int row = v0 + idx / PIECES, piece = idx % PIECES;
              *reinterpret_cast<uint4*>(vb + (piece >> 3) * HALF + row * 128 + (piece & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[gPFull0 + t % NP]);
        }
        // ---- epilogue: merge the 2 DUP states of each row.  Every softmax
        // warp arrives here once per segment, failed or not, and they decide
        // together.
        const uint32_t last = t - 1;
        good = good && wait_all(&bars[gPVDone0 + last % NP], (last / NP) & 1);
        ml_s[(hh * 2) * 128 + m] = m_ref;
        ml_s[(hh * 2 + 1) * 128 + m] = l;
        if (!named_bar_and(1, 256, good)) {
          good = false;
          break;
        }
        tc_fence_after();
        float M = -INFINITY;
#pragma unroll
        for (int c2 = 0; c2 < DUP; ++c2)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) M = fmaxf(M, ml_s[(h2 * 2) * 128 + c2 * RP + r]);
        float L = 0.f;
#pragma unroll
        for (int c2 = 0; c2 < DUP; ++c2)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const float mm = ml_s[(h2 * 2) * 128 + c2 * RP + r];
            if (mm != -INFINITY) L += ml_s[(h2 * 2 + 1) * 128 + c2 * RP + r] * exp2_approx(mm - M);
          }
        const float inv = L > 0.f ? p.v_mult / L : 0.f;
        // this lane's two states: (copy, half 0) in O_0 and (copy, half 1) in O_1
        const float m0 = ml_s[m], m1 = ml_s[256 + m];
        const float f0 = m0 == -INFINITY ? 0.f : exp2_approx(m0 - M) * inv;
        const float f1 = m1 == -INFINITY ? 0.f : exp2_approx(m1 - M) * inv;
        float* dst = nullptr;
        float* dl = nullptr;
        if (sg.full) {
          int64_t orow;
          if constexpr (MQ) {
            const int rr = min(r, p.rows - 1), j = rr / p.g, i = rr - j * p.g;
            orow = (int64_t(sg.b) * p.qlen + j) * p.h + sg.kvh * p.g + i;
          } else {
            orow = int64_t(sg.b) * p.h + sg.kvh * p.g + min(r, p.rows - 1);
          }
          dst = p.out + orow * D;
          dl = p.lse + orow;
        } else {
          // row r of this CTA's partial slot for the unit (slot u + c)
          const int64_t slot = int64_t(sg.b) * p.hkv + sg.kvh + c;
          dst = p.part_out + (slot * p.rows + min(r, p.rows - 1)) * D;
          dl = p.part_lse + slot * p.rows + min(r, p.rows - 1);
        }
        // this thread's columns: 64 hh .. 64 hh + 63 of the merged row, 32 at
        // a time; copies other than 0 hand their share to copy 0 through
        // shared memory (16-byte pieces swizzled by row)
#pragma unroll 1
        for (int cb = 64 * hh; cb < 64 * hh + 64; cb += 32) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tmem + lane_off + TM_O + cb, o0);
          tmem_ld32(tmem + lane_off + TM_O + 128 + cb, o1);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] = __uint_as_float(o0[j]) * f0 + __uint_as_float(o1[j]) * f1;
          if constexpr (DUP > 1) {
            float4* xr = xb + ((hh * (DUP - 1) + (cpy > 0 ? cpy - 1 : 0)) * RP + r) * 8;
            if (cpy > 0) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                xr[j ^ (r & 7)] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
            named_bar_sync(2, 256);
            if (cpy == 0) {
#pragma unroll
              for (int c2 = 1; c2 < DUP; ++c2) {
                const float4* xs = xb + ((hh * (DUP - 1) + c2 - 1) * RP + r) * 8;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const float4 a = xs[j ^ (r & 7)];
                  v[4 * j] += a.x;
                  v[4 * j + 1] += a.y;
                  v[4 * j + 2] += a.z;
                  v[4 * j + 3] += a.w;
                }
              }
            }
            named_bar_sync(2, 256);   // the buffer is rewritten by the next round
          }
          if (cpy == 0 && row_ok) {
            float4* d4 = reinterpret_cast<float4*>(dst + cb);
#pragma unroll
            for (int j = 0; j < 8; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
        }
        if (cpy == 0 && row_ok && hh == 0)
          *dl = L > 0.f ? (M + log2_approx(L)) * kLn2 : -INFINITY;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[gOFree]);
        ++seg;
      }
      if (!good) {
        report(p.err, KVATTN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  }
  // every warp is done with TMEM and with its waits
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

// Up to 32 rows the mma.sync kernel measured faster (Llama-3-70B shapes, 4 new
// tokens: 175 against 196 us per call); from 64 rows on this one (8 new
// tokens: 200 against 277 us).
#ifndef KV_GQA_TC_MIN_ROWS
#define KV_GQA_TC_MIN_ROWS 33
#endif
#ifndef KV_GQA_TC_MIN_ROWS_FP8
#define KV_GQA_TC_MIN_ROWS_FP8 17
#endif
bool gqa_tc_applies(int dtype, int rows, int d) {
  if (d != gtc::D || rows > 128) return false;
  if (dtype == KVATTN_BF16) return rows >= KV_GQA_TC_MIN_ROWS;
  return dtype == KVATTN_FP8_E4M3 && rows >= KV_GQA_TC_MIN_ROWS_FP8;
}

int gqa_tc_ctas() {
  static int cache[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::call_once(flags[dev], [dev] {
    using gtc::Lay;
    const void* ks[6] = {(const void*)gqa_tc_kernel<true, 1, false>, (const void*)gqa_tc_kernel<true, 2, false>,
                         (const void*)gqa_tc_kernel<true, 4, false>, (const void*)gqa_tc_kernel<false, 1, false>,
                         (const void*)gqa_tc_kernel<false, 2, false>, (const void*)gqa_tc_kernel<false, 4, false>};
    const void* k8[6] = {(const void*)gqa_tc_kernel<true, 1, true>, (const void*)gqa_tc_kernel<true, 2, true>,
                         (const void*)gqa_tc_kernel<true, 4, true>, (const void*)gqa_tc_kernel<false, 1, true>,
                         (const void*)gqa_tc_kernel<false, 2, true>, (const void*)gqa_tc_kernel<false, 4, true>};
    for (const void* k : ks)
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<false>::SMEM);
    for (const void* k : k8)
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<true>::SMEM);
    // both forms hold one CTA per SM (shared memory and 448 threads)
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_tc_kernel<false, 1, false>,
                                                      gtc::THREADS, Lay<false>::SMEM) != cudaSuccess)
      n = 0;
    const int sms = device_sm_count();
    cache[dev] = (n > 0 && sms > 0) ? n * sms : -1;
  });
  return cache[dev];
}

template <bool FP8>
static cudaError_t launch_tc(const GqaArgs& a, const GqaParams& prm, int G, const CUtensorMap& tmQ,
                             const CUtensorMap& tmK, const CUtensorMap& tmV) {
  using namespace gtc;
  constexpr int SM = Lay<FP8>::SMEM;
  const dim3 grid(G), block(THREADS);
  // rows <= 32: four copies of the rows in the MMA's 128, <= 64: two, else one
  if (prm.qlen > 1)
    return prm.rows <= 32   ? launch_pdl(gqa_tc_kernel<true, 4, FP8>, grid, block, SM, a.stream, tmQ, tmK, tmV, prm)
           : prm.rows <= 64 ? launch_pdl(gqa_tc_kernel<true, 2, FP8>, grid, block, SM, a.stream, tmQ, tmK, tmV, prm)
                            : launch_pdl(gqa_tc_kernel<true, 1, FP8>, grid, block, SM, a.stream, tmQ, tmK, tmV, prm);
  return prm.rows <= 32   ? launch_pdl(gqa_tc_kernel<false, 4, FP8>, grid, block, SM, a.stream, tmQ, tmK, tmV, prm)
         : prm.rows <= 64 ? launch_pdl(gqa_tc_kernel<false, 2, FP8>, grid, block, SM, a.stream, tmQ, tmK, tmV, prm)
                          : launch_pdl(gqa_tc_kernel<false, 1, FP8>, grid, block, SM, a.stream, tmQ, tmK, tmV, prm);
}

kvattn_status launch_gqa_tc(const GqaArgs& a, const GqaParams& prm, int G) {
  using namespace gtc;
  if (gqa_tc_ctas() <= 0) return KVATTN_ERR_CUDA;   // also sets the shared-memory attribute
  const kvattn_cache* cc = a.cache;
  const bool fp8 = cc->dtype == KVATTN_FP8_E4M3;
  alignas(64) CUtensorMap tmQ, tmK, tmV;
  // q [B][q_len][h][d] as (d, h, q_len, B); a box is one unit's rows (the
  // E4M3 form builds its query terms without it)
  const uint64_t qdims[4] = {uint64_t(D), uint64_t(prm.h), uint64_t(prm.qlen), uint64_t(prm.B)};
  const uint64_t qstr[3] = {uint64_t(D) * 2, uint64_t(prm.h) * D * 2,
                            uint64_t(prm.qlen) * prm.h * D * 2};
  const uint32_t qbox[4] = {64u, uint32_t(prm.g), uint32_t(prm.qlen), 1u};
  // K and V pools as (d, block_size, blocks x KV heads); boxes of 16 tokens x
  // 128 bytes (64 bf16 dims or 128 E4M3 codes)
  const uint64_t eb = fp8 ? 1 : 2;
  const uint64_t dims[3] = {uint64_t(D), uint64_t(cc->block_size),
                            uint64_t(cc->num_blocks) * uint64_t(cc->h_kv)};
  const uint64_t strides[2] = {uint64_t(D) * eb, uint64_t(D) * eb * uint64_t(cc->block_size)};
  const uint32_t box[3] = {uint32_t(128 / eb), 16u, 1u};
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_tensor_map_4d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, qdims, qstr, qbox,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_3d(&tmK, dt, cc->k, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_3d(&tmV, dt, cc->v, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return KVATTN_ERR_CUDA;
  const cudaError_t e = fp8 ? launch_tc<true>(a, prm, G, tmQ, tmK, tmV)
                            : launch_tc<false>(a, prm, G, tmQ, tmK, tmV);
  return e == cudaSuccess ? KVATTN_OK : KVATTN_ERR_CUDA;
}

}  // namespace kv
