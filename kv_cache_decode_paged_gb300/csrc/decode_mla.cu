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
// each tile of 64 latent rows, split by latent dimension:
//   rank r owns dims D_r = [256r, 256r + 256) U [512 + 32r, 544 + 32r),
// i.e. half of c_KV and half of k_R.  It loads only those 288 dims of Q and of
// every row (no byte is loaded twice), computes the partial score
// S_r = Q[:, D_r] . row[:, D_r]^T  (M = 128 heads, N = 64 rows, K = 288), and
// its half of the output O[:, 256r : 256r + 256] += P . c[:, 256r : 256r + 256]
// (the c_KV part of D_r is exactly the value columns it needs).
// The two partial scores meet through distributed shared memory: each rank
// rounds its raw partial to f16 and pushes it into the peer's receive slot
// with bulk copies; both ranks add the same two f16 partials, so their softmax
// inputs and P are bit-identical.
//
// Measured on GB300 (unrolled issue, one SM): a K = 16 MMA with M = 128 takes
// ~48 cycles at N = 64, ~67 at N = 128 and ~131 at N = 256, with A in shared
// memory or in tensor memory alike; with the P.V chain of another tile issued
// beside it a tile's 22 MMAs occupy the tensor core ~1,300 cycles.  A bulk
// copy into the peer's shared memory lands ~0.6 us after issue, and loads from
// the peer's shared memory or release-ordered remote arrives cost about as
// much, so partials are pushed, never pulled; per-thread asynchronous remote
// stores (st.async) measured slower than staging plus one bulk copy per warp.
// Two staging and two receive slots let the exchange of tile t+1 start while
// tile t is still in the peer's receive slot.  The first 192 c_KV dims of this
// rank's Q sit in TMEM (score K steps 2..13 read A from TMEM), the other 64
// and the 32 rope dims in shared memory; that leaves room for four value
// stages.  A tile's value stage lives from its load until its P.V completes
// (load ~0.9 us, score MMAs, exchange, softmax, P.V: ~4.4 us in a timeline
// trace), which with four stages sets the period of ~1.1 us per tile.
//   warp 0      TMA producer: per sequence the shared-memory part of Q; per
//               tile 4 value boxes (4-stage ring) and one rope box (2-slot
//               ring, freed once S is computed)
//   warp 1      TMEM owner and S issuer: S(t) into one of two S slots
//   warp 14     P.V issuer: P.V(t) with P from the P slot
//   warps 10-13 senders: per sequence Q[:, 256r : 256r + 192] into TMEM; per
//               tile S(t) partial -> f16 -> staging slot -> bulk copy to the
//               peer (one thread per head row)
//   warps 2-9   softmax: peer partial + own partial, online softmax with lazy
//               rescaling, P(t) -> TMEM, epilogue (two threads per head row,
//               32 of the tile's 64 rows each)
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "merge.cuh"
#include "tcgen05.cuh"
#include "walk.cuh"

// Test builds only (-DKV_TEST_DROP_CHUNK=n, with a short KV_WAIT_NS): the
// producer of CTA 0 (rank 0 of pair 0) arms tile n's barrier but issues none
// of its loads, as copies that never land would, so that the waits on that
// tile (and through the exchange, the peer's) run out and both ranks take the
// abort path on the GPU.  The library is built without it.
#ifdef KV_TEST_DROP_CHUNK
#define KV_TEST_DROPS_MLA_TILE(it) (blockIdx.x == 0 && (it) == uint32_t(KV_TEST_DROP_CHUNK))
#else
#define KV_TEST_DROPS_MLA_TILE(it) false
#endif

namespace kv {

namespace mla {
// Shared by both cache formats.
constexpr int ROWW = 576;              // latent row width (d_c + d_rope)
constexpr int DC = 512;
constexpr int BS = 64;                 // tokens per page = tokens per tile
constexpr int NROPE = 2;               // rope ring
constexpr int XROW = BS * 2;           // a row of a partial tile, f16
constexpr int XBYTES = 128 * XROW;     // 16 KB
#ifndef KV_MLA_NX
#define KV_MLA_NX 1
#endif
constexpr int NX = KV_MLA_NX;          // exchange ring depth (staging and receive slots)
static_assert(NX >= 1 && NX <= 2, "two barrier slots per exchange ring");
constexpr int NBARS = 48;
constexpr int NSTAGE_MAX = 10;         // barrier slots reserved per value stage ring
constexpr int NSW = 256;               // softmax warps: two threads per head row
constexpr int NSEND = 128;             // sender warps: one thread per head row
constexpr int SW0 = 64, SEND0 = 64 + NSW;
constexpr int PV_WARP = (SEND0 + NSEND) / 32;   // the P.V issuer
constexpr int THREADS = 64 + NSW + NSEND + 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;           // two S slots of 64 columns
constexpr uint32_t TM_Q = 128;         // the TMEM part of this rank's Q
constexpr uint32_t TM_P = 224;         // one P slot of 32 columns
constexpr uint32_t TM_O = 256;         // O half: columns 256..511
constexpr float RESCALE_THRESHOLD = 8.f;  // log2 units: rescale O only when the max grows by 2^8

#ifndef KV_MLA_NQT
#define KV_MLA_NQT 12
#endif
#ifndef KV_MLA_NSTAGE
#define KV_MLA_NSTAGE 5
#endif
#ifndef KV_MLA_NSTAGE_FP8
#define KV_MLA_NSTAGE_FP8 7
#endif

// Per cache format.  A value stage holds this rank's 256 c_KV dims of one page
// as boxes of 128-byte rows: bf16 four boxes of 64 dims, E4M3 two boxes of 128.
template <bool FP8>
struct Geo;
template <>
struct Geo<false> {
  static constexpr int NVB = 4;                        // value boxes per stage
  static constexpr int BOX_DIMS = 64;
  static constexpr int VF_BYTES = BS * 128;            // one box: [64 rows x 64 dims]
  static constexpr int RH_BYTES = BS * 64;             // rope box [64 rows x this rank's 32 dims]
  static constexpr int QF_BYTES = 128 * 128;           // Q box [128 heads x 64 dims], 128-byte swizzle
  static constexpr int QH_BYTES = 128 * 64;            // Q box [128 heads x 32 rope dims], 64-byte swizzle
  static constexpr int NQT = KV_MLA_NQT;               // score K steps with Q in TMEM
  static constexpr int NQF = 4 - NQT / 4;              // Q boxes in shared memory
  static constexpr int Q_BYTES = NQF * QF_BYTES + QH_BYTES;   // 24 KB
  static constexpr int NSTAGE = KV_MLA_NSTAGE;         // value ring
  static_assert(TM_Q + 8 * NQT <= TM_P && NQT % 4 == 0 && NQT <= 16, "Q columns in TMEM");
};
// E4M3: the query and the probabilities enter the MMAs as two E4M3 terms each
// (hi = e4m3(x), lo = e4m3(x - hi)); the hi term of Q sits in TMEM (72
// columns: 288 codes, four per column), the lo term in shared memory.  The
// rope box carries all 64 rope dims (64-byte rows); each rank multiplies its
// own 32 of them.
template <>
struct Geo<true> {
  static constexpr int NVB = 2;
  static constexpr int BOX_DIMS = 128;
  static constexpr int VF_BYTES = BS * 128;            // one box: [64 rows x 128 codes]
  static constexpr int RH_BYTES = BS * 64;             // rope box [64 rows x 64 codes]
  static constexpr int QF_BYTES = 128 * 128;           // lo term, [128 heads x 128 codes]
  static constexpr int QH_BYTES = 128 * 64;            // lo term, rope [128 heads x 64 B rows]
  static constexpr int NQF = 2;
  static constexpr int Q_BYTES = NQF * QF_BYTES + QH_BYTES;   // 40 KB
  static constexpr int NSTAGE = KV_MLA_NSTAGE_FP8;
  static_assert(TM_Q + 72 <= TM_P, "Q hi columns in TMEM");
};

// Shared-memory layout per cache format.
template <bool FP8>
struct Lay {
  using G = Geo<FP8>;
  static constexpr int VSTAGE = G::NVB * G::VF_BYTES;
  // The value ring is laid out box-major: box i of stage s sits at
  // OFF_V + i * VBOX + s * VF_BYTES.
  static constexpr int VBOX = G::NSTAGE * G::VF_BYTES;
  static constexpr int OFF_QF = 0;
  static constexpr int OFF_QH = G::NQF * G::QF_BYTES;
  static constexpr int OFF_V = G::Q_BYTES;
  static constexpr int OFF_R = OFF_V + G::NSTAGE * VSTAGE;
  static constexpr int OFF_X = OFF_R + NROPE * G::RH_BYTES;   // receive slots (the peer writes)
  static constexpr int OFF_XS = OFF_X + NX * XBYTES;          // send staging slots
  static constexpr int OFF_MX = OFF_XS + NX * XBYTES;         // row max / row sum exchange
  static constexpr int OFF_QSC = OFF_MX + 2 * 128 * 4;        // E4M3: per-row partial scale
  static constexpr int OFF_BAR = OFF_QSC + 128 * 4;
  static constexpr int SMEM = 1024 + OFF_BAR + NBARS * 8 + 16;
  static_assert(OFF_V % 1024 == 0 && OFF_R % 1024 == 0 && OFF_X % 1024 == 0 &&
                    OFF_XS % 1024 == 0 && OFF_QH % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(G::NSTAGE <= NSTAGE_MAX, "barrier slots per stage");
  // The last epilogue stages O (128 KB) in idle shared memory: the value ring
  // (bf16), or Q and the value ring (E4M3, whose ring is smaller)
  static constexpr int OFF_EPI = FP8 ? 0 : OFF_V;
  static_assert(OFF_EPI + (NSW / 32) * 4 * 32 * 128 <= OFF_R, "epilogue staging fits");
  static_assert(merge_scratch_floats(128) * 4 <= G::NSTAGE * VSTAGE,
                "merge scratch fits the value ring");
};
}  // namespace mla

struct MlaParams {
  const uint16_t* q;       // absorbed queries, [B][h][576] bf16
  const int32_t* bt;
  const int32_t* seq_lens;
  const int64_t* cum;
  const int4* cta_start;   // per pair
  float* out;
  float* lse;
  float* part_out;
  float* part_lse;              // [slots][2][h]: one copy per rank
  const int32_t* split_first;  // per sequence: first partial slot and number of splits
  const int32_t* split_count;
  int32_t* arrive;             // merge counters, per rank: [B] units, then [B + G] slots
  int B, h, max_blocks, G;
  int64_t num_blocks;
  float scale_log2;
  float c_scale;           // E4M3 cache: value of a c_KV code unit (1 for bf16)
  float r_ratio;           // E4M3 cache: k_R scale / c_KV scale (1 for bf16)
  int32_t* err;
  uint32_t zero;           // always 0: a mask the compiler cannot fold (see the receive-slot release)
};

// E4M3 query of one head row for one rank of the pair: the rank's 256 c_KV
// dims and 32 rope dims (the rope scaled by r_ratio, so that one accumulator
// adds both parts in c_KV code units), times 2^e, split into two E4M3 terms
// hi = e4m3(x) and lo = e4m3(x - hi).  2^e brings the row's largest magnitude
// into [128, 256), inside E4M3's normal range with room below for lo.  The hi
// codes go to TMEM (columns TM_Q .. TM_Q + 71, four codes per column: c_KV dims
// first, rope last), the lo codes to shared memory in the layouts the MMAs
// read (c_KV: two 128-code atoms with 128-byte rows and swizzle; rope: 64-byte
// rows with 64-byte swizzle, this rank's codes at bytes 32r .. 32r+31).
// A partial score times 2^-e is in c_KV code units.  The exponent is computed
// by q_row_exp, which the softmax warps call too (same inputs, same e).
KV_DEVI uint4 q_load8(const uint16_t* qrow, bool live, int dim0, int i) {
  return live ? __ldg(reinterpret_cast<const uint4*>(qrow + dim0) + i) : make_uint4(0, 0, 0, 0);
}
KV_DEVI float bf16_half(uint32_t w, int hi) {
  return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16));
}
// The row is read 12 loads at a time (all in flight together): one load per
// round trip to L2 made this the longest step of a sequence's start.
KV_DEVI int q_row_exp(const uint16_t* qrow, bool live, uint32_t rank, float r_ratio) {
  const int c0 = 256 * int(rank), r0 = 512 + 32 * int(rank);
  float mx = 0.f;
#pragma unroll 1
  for (int g = 0; g < 3; ++g) {
    uint4 x[12];
#pragma unroll
    for (int i = 0; i < 12; ++i) {
      const int idx = 12 * g + i;
      x[i] = idx < 32 ? q_load8(qrow, live, c0, idx) : q_load8(qrow, live, r0, idx - 32);
    }
#pragma unroll
    for (int i = 0; i < 12; ++i) {
      const float f = 12 * g + i < 32 ? 1.f : r_ratio;
      const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mx = fmaxf(mx, fmaxf(fabsf(bf16_half(w[k], 0) * f), fabsf(bf16_half(w[k], 1) * f)));
    }
  }
  return mx > 0.f ? min(max(7 - (int((__float_as_uint(mx) >> 23) & 255) - 127), -120), 120) : 0;
}
// Two E4M3 terms of a float pair: hi = e4m3(x), lo = e4m3(x - hi), each a
// 16-bit code pair (first value in the low byte).  x is first rounded to f16
// (the query is scaled below 2^8 and P stays below 2^9, and E4M3 keeps 4
// significant bits per term, so the f16 rounding is far below the terms'
// own); then hi is exact in f16 and so is x - hi, which one f16x2
// subtraction gives for both values.
KV_DEVI void e4m3_two_terms(float x0, float x1, uint32_t& hi, uint32_t& lo) {
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
KV_DEVI void build_q_e4m3(const uint16_t* qrow, bool live, uint32_t rank, float r_ratio, int e,
                          uint32_t tq, uint8_t* lo_c, uint8_t* lo_r, int r) {
  const int c0 = 256 * int(rank), r0 = 512 + 32 * int(rank);
  const float sc = __uint_as_float(uint32_t(127 + e) << 23);
#pragma unroll 1
  for (int g = 0; g < 3; ++g) {     // 96 dims (12 loads in flight) at a time
  uint4 xs[12];
#pragma unroll
  for (int i = 0; i < 12; ++i) {
    const int k = 3 * g + i / 4;
    xs[i] = k < 8 ? q_load8(qrow, live, c0 + 32 * k, i % 4) : q_load8(qrow, live, r0, i % 4);
  }
#pragma unroll
  for (int kk = 0; kk < 3; ++kk) {  // 32 dims at a time: c_KV 0..7, rope 8
    const int k = 3 * g + kk;
    const float f = k < 8 ? sc : sc * r_ratio;
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = xs[4 * kk + i];
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        // codes 8i + 2j .. 8i + 2j + 3 (two pairs) into word 2i + j / 2
        uint32_t hw = 0, lw = 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          uint32_t h, l;
          e4m3_two_terms(bf16_half(w[j + t], 0) * f, bf16_half(w[j + t], 1) * f, h, l);
          hw |= h << (16 * t);
          lw |= l << (16 * t);
        }
        hi[2 * i + j / 2] = hw;
        lo[2 * i + j / 2] = lw;
      }
    }
    tmem_st8(tq + 8 * k, hi);
    if (k < 8) {
      uint8_t* row = lo_c + (k >> 2) * (128 * 128) + r * 128;
      const int pc = 2 * (k & 3);
      *reinterpret_cast<uint4*>(row + ((pc ^ (r & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4*>(row + (((pc + 1) ^ (r & 7)) << 4)) =
          make_uint4(lo[4], lo[5], lo[6], lo[7]);
    } else {
      uint8_t* row = lo_r + r * 64;
      const int pc = 2 * int(rank), sw = (r >> 1) & 3;
      *reinterpret_cast<uint4*>(row + ((pc ^ sw) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4*>(row + (((pc + 1) ^ sw) << 4)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    }
  }
  }
}

// Barrier indices
enum : int {
  kQFull = 0, kQEmpty = 1, kOFree = 2,
  kSFull0 = 3,      // 2: S(t) landed in S slot t % 2
  kSRead0 = 5,      // 2: the senders and the softmax warps have read S slot t % 2
  kPFull0 = 7,      // 2: P(t) written to the P slot (barrier t % 2)
  kPVDone0 = 9,     // 2: P.V of tile t finished (barrier t % 2)
  kXFull0 = 11,     // 2: the peer's partial of tile t is in receive slot t % 2 (tx bytes)
  kXEmpty0 = 13,    // 2: the peer has read this rank's partial of tile t (slot t % 2)
  kXSent0 = 15,     // 2: the peer has received the copy from staging slot t % 2
  kQTmem = 17,      // the sender warps have written this sequence's Q columns to TMEM
  kMmaDrain = 18,   // 2: each MMA issuer's last operations completed (exit path)
  kKVFull0 = 20,                          // NSTAGE: value boxes (and rope box) landed
  kKVEmpty0 = kKVFull0 + mla::NSTAGE_MAX,     // NSTAGE: P.V finished with the value stage
  kRopeEmpty0 = kKVEmpty0 + mla::NSTAGE_MAX,  // 2: S finished with the rope slot
  kAbort = kRopeEmpty0 + 2,               // an int flag in this slot
  kMergeFlags = kAbort + 1,               // 2 slots: 3 ints for the in-kernel merge
  kNumBars = kMergeFlags + 2
};
static_assert(kNumBars <= mla::NBARS, "barrier slots");

// One f16 pair of partial scores (raw dot products, unscaled): the senders
// and the softmax warps round the same fp32 values the same way, and both
// ranks add the same two f16 pairs (f16 addition is commutative), so their
// softmax inputs are bit-identical.
KV_DEVI uint32_t partial_pair(uint32_t a, uint32_t b) {
  return pack_f16(__uint_as_float(a), __uint_as_float(b));
}
KV_DEVI uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hadd2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
KV_DEVI uint32_t hmax2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hmax2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <bool FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(mla::THREADS, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmQF,
                      const __grid_constant__ CUtensorMap tmQH,
                      const __grid_constant__ CUtensorMap tmLF,
                      const __grid_constant__ CUtensorMap tmLH,
                      const __grid_constant__ CUtensorMap tmO, const MlaParams p) {
  using namespace mla;
  using G = Geo<FP8>;
  using L = Lay<FP8>;
  constexpr int NSTAGE = G::NSTAGE, VF_BYTES = G::VF_BYTES, RH_BYTES = G::RH_BYTES;
  constexpr int QF_BYTES = G::QF_BYTES, NQF = G::NQF, Q_BYTES = G::Q_BYTES;
  constexpr int VSTAGE = L::VSTAGE, VBOX = L::VBOX, OFF_QF = L::OFF_QF, OFF_QH = L::OFF_QH;
  constexpr int OFF_V = L::OFF_V, OFF_R = L::OFF_R, OFF_X = L::OFF_X, OFF_XS = L::OFF_XS;
  constexpr int OFF_MX = L::OFF_MX, OFF_BAR = L::OFF_BAR, OFF_QSC = L::OFF_QSC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kAbort);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  // Set-up that needs nothing from the planner runs before waiting for it:
  // barriers, descriptors, tensor memory and the cluster handshake.
  if (threadIdx.x == 0) {
    mbar_init(&bars[kQFull], 1);
    mbar_init(&bars[kQEmpty], 1);
    mbar_init(&bars[kOFree], NSW);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kSFull0 + i], 1);
      mbar_init(&bars[kSRead0 + i], (NSW + NSEND) / 32);  // one arrival per reading warp
      mbar_init(&bars[kPFull0 + i], NSW / 32);  // one arrival per softmax warp
      mbar_init(&bars[kPVDone0 + i], 1);
      mbar_init(&bars[kRopeEmpty0 + i], 1);
    }
    for (int i = 0; i < NX; ++i) {
      mbar_init(&bars[kXFull0 + i], 1);           // one local expect_tx arrival + the peer's bytes
      mbar_init(&bars[kXEmpty0 + i], NSW / 32);   // one arrival per softmax warp of the peer
      mbar_init(&bars[kXSent0 + i], 1);           // one arrival from the peer
    }
    mbar_init(&bars[kQTmem], NSEND / 32);
    mbar_init(&bars[kMmaDrain], 1);
    mbar_init(&bars[kMmaDrain + 1], 1);
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&bars[kKVFull0 + i], 1);
      mbar_init(&bars[kKVEmpty0 + i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    if (!FP8) {   // the E4M3 form builds Q from global memory without TMA
      tma_prefetch_desc(&tmQF);
      tma_prefetch_desc(&tmQH);
    }
    tma_prefetch_desc(&tmLF);
    tma_prefetch_desc(&tmLH);
    for (int i = 0; i < NX; ++i) mbar_arrive_expect_tx(&bars[kXFull0 + i], XBYTES);  // tiles 0, 1
  }
  __syncwarp();  // warp 0 reconverges before the warp-aligned instructions below
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  // Both CTAs of the cluster start together; this makes each one's barriers
  // visible to the other before any remote access.
  cluster_sync_all();
  tc_fence_after();
  // Launched right behind the planner: wait for its plan, and let whatever
  // follows get scheduled while this grid runs.
  pdl_wait();
  pdl_launch_dependents();
  const int4 st = p.cta_start[pair], en = p.cta_start[pair + 1];
  if (!pos_less(st, en)) {   // both ranks of the pair take the same exit
    if (warp == 1) tmem_dealloc(*tmem_slot, TMEM_COLS);
    return;
  }
  const uint32_t tmem = *tmem_slot;
  const int vx0 = 256 * int(rank);       // first value dim of this rank
  // first rope dim this rank loads: its own 32 (bf16), or all 64 (E4M3)
  const int rx = FP8 ? 512 : 512 + 32 * int(rank);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // The whole warp walks the segments; lane 0 waits and issues, and the
    // block ids are read 32 at a time, one per lane, before the waits that
    // precede their tiles (a block id read right after a stage frees would
    // add an L2 round trip to every stage's lifetime, and at a sequence's
    // start one round trip per tile).
    const uint64_t pol = policy_evict_first();
    Walker w{p.cum, 1, st, en};
    Seg sg;
    uint32_t it = 0, seg = 0;
    bool ok = true;
    while (ok && w.next(sg)) {
      if constexpr (!FP8) {
        // bf16: the shared-memory part of Q is loaded as it is (the E4M3
        // form is built by the sender warps)
        if (lane == 0) {
          if (seg > 0 && !mbar_wait(&bars[kQEmpty], (seg - 1) & 1)) {
            ok = false;
          } else {
            mbar_arrive_expect_tx(&bars[kQFull], Q_BYTES);
            for (int i = 0; i < NQF; ++i)
              tma_load_3d_nohint(smem + OFF_QF + i * QF_BYTES, &tmQF, vx0 + 16 * G::NQT + 64 * i, 0,
                                 sg.b, &bars[kQFull]);
            tma_load_3d_nohint(smem + OFF_QH, &tmQH, rx, 0, sg.b, &bars[kQFull]);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      const int32_t* row = p.bt + int64_t(sg.b) * p.max_blocks;
      for (int jb = sg.j0; jb < sg.j1 && ok; jb += 32) {
        int page = int(p.num_blocks);  // out of range: zero fill
        if (jb + lane < sg.j1) {
          const int blk = row[jb + lane];
          if (blk < 0 || int64_t(blk) >= p.num_blocks)
            report(p.err, KVATTN_DEVERR_BLOCK_ID);
          else
            page = blk;
        }
        const int cnt = min(32, sg.j1 - jb);
        for (int i = 0; i < cnt && ok; ++i) {
          const int pg = __shfl_sync(0xffffffffu, page, i);
          int issued = 0;
          if (lane == 0) {
            const int s = it % NSTAGE, q = it & 1;
            if (!mbar_wait(&bars[kKVEmpty0 + s], ((it / NSTAGE) & 1) ^ 1) ||
                !mbar_wait(&bars[kRopeEmpty0 + q], ((it >> 1) & 1) ^ 1)) {
              ok = false;
            } else {
              uint8_t* stg = smem + OFF_V + s * VF_BYTES;
              mbar_arrive_expect_tx(&bars[kKVFull0 + s], uint32_t(VSTAGE + RH_BYTES));
              if (!KV_TEST_DROPS_MLA_TILE(it)) {
                for (int b = 0; b < G::NVB; ++b)
                  tma_load_3d(stg + b * VBOX, &tmLF, vx0 + G::BOX_DIMS * b, 0, pg,
                              &bars[kKVFull0 + s], pol);
                tma_load_3d(smem + OFF_R + q * RH_BYTES, &tmLH, rx, 0, pg, &bars[kKVFull0 + s], pol);
              }
              issued = 1;
              if (*abort_flag) ok = false;
            }
          }
          // it counts the tiles issued (the exit drain waits for their loads)
          it += uint32_t(__shfl_sync(0xffffffffu, issued, 0));
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      }
      ++seg;
    }
    if (lane == 0) {
      if (!ok) {
        report(p.err, KVATTN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // Every load this thread issued lands before the CTA can exit (on the
      // normal path the consumers have waited for all of them already).
      if (!FP8 && seg > 0) mbar_wait(&bars[kQFull], (seg - 1) & 1, KV_DRAIN_WAIT_NS);
      for (uint32_t k = it > uint32_t(NSTAGE) ? it - NSTAGE : 0; k < it; ++k)
        mbar_wait(&bars[kKVFull0 + k % NSTAGE], (k / NSTAGE) & 1, KV_DRAIN_WAIT_NS);
    }
  } else if (warp == 1 || warp == PV_WARP) {
    // ------------------------------------------ MMA issuers: S (warp 1), P.V
    // Two threads feed the tensor core: one tcgen05.mma takes about as long to
    // issue as to run at these shapes, so a single issuer would set the pace.
    // Their operands and accumulators are disjoint (S slots vs P slots and O).
    if (lane == 0) {
      const uint32_t v_base = smem_u32(smem + OFF_V), r_base = smem_u32(smem + OFF_R);
      Walker w{p.cum, 1, st, en};
      Seg sg;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      if (warp == 1) {
        const uint32_t id_s = FP8 ? idesc_e4m3(128, BS, false) : idesc_bf16(128, BS, false);
        const uint32_t qf = smem_u32(smem + OFF_QF), qh = smem_u32(smem + OFF_QH);
        // Descriptors are built once; a K step only moves the start address,
        // whose field is the low bits of the descriptor (address / 16, no carry
        // below 256 KB).  The issue loop is unrolled: with the address
        // arithmetic in the loop the issue, not the tensor core, set the pace.
        const uint64_t qa0 = sdesc_sw128(qf, 16, 1024), qh0 = sdesc_sw64(qh, 512);
        // E4M3: the rope box and the lo term's rope region have 64-byte rows;
        // this rank's 32 rope codes are bytes 32r .. 32r+31 of each.
        const uint64_t rope_k = FP8 ? uint64_t(2 * rank) : 0;
        // S(t) = Q[:, D_r] . row(t)[:, D_r]^T into S slot t % 2, MMAs [J0, J1)
        // of 18.  MMAs 0 and 1 cover the rope dims, so that the small rope
        // ring can be refilled as soon as they are done.
        //   bf16 (K = 16): MMA j >= 2 covers c_KV dims 16m .. 16m+15 of this
        //     rank, m = j - 2, with Q from TMEM for m < NQT, else from shared
        //     memory.
        //   E4M3 (K = 32): the rope dims and then each 32 c_KV dims m = 0..7
        //     take two MMAs, the hi term of Q (TMEM) and the lo term (shared
        //     memory), accumulating into the same S.
        auto issue_s = [&](uint32_t t, auto j0c, auto j1c) {
          constexpr int J0 = decltype(j0c)::value, J1 = decltype(j1c)::value;
          const uint32_t d = tmem + TM_S + BS * (t & 1);
          const uint64_t vb0 = sdesc_sw128(v_base + (t % NSTAGE) * VF_BYTES, 16, 1024);
          const uint64_t rb0 = sdesc_sw64(r_base + (t & 1) * RH_BYTES, 512) + rope_k;
#pragma unroll
          for (int j = J0; j < J1; ++j) {
            if constexpr (FP8) {
              if (j < 2) {
                if (j == 0)
                  umma_ts_f8(d, tmem + TM_Q + 64, rb0, id_s, 0u);
                else
                  umma_ss_f8(d, qh0 + rope_k, rb0, id_s, 1u);
              } else {
                const int m = (j - 2) >> 1;   // c_KV dims 32m .. 32m+31 of this rank
                const uint64_t b = vb0 + uint64_t(((m >> 2) * VBOX + (m & 3) * 32) >> 4);
                if (((j - 2) & 1) == 0)
                  umma_ts_f8(d, tmem + TM_Q + 8 * m, b, id_s, 1u);
                else
                  umma_ss_f8(d, qa0 + uint64_t(((m >> 2) * QF_BYTES + (m & 3) * 32) >> 4), b, id_s,
                             1u);
              }
            } else {
              if (j < 2) {        // rope dims of this rank
                umma_ss(d, qh0 + uint64_t((j * 32) >> 4), rb0 + uint64_t((j * 32) >> 4), id_s,
                        j > 0);
              } else {
                const int m = j - 2;  // c_KV dims 16m .. 16m+15 of this rank
                const uint64_t b = vb0 + uint64_t(((m >> 2) * VBOX + (m & 3) * 32) >> 4);
                if (m < G::NQT)
                  umma_ts(d, tmem + TM_Q + 8 * m, b, id_s, 1u);
                else
                  umma_ss(d,
                          qa0 + uint64_t((((m - G::NQT) >> 2) * QF_BYTES + (m & 3) * 32) >> 4),
                          b, id_s, 1u);
              }
            }
          }
        };
        using C0 = std::integral_constant<int, 0>;
        using C2 = std::integral_constant<int, 2>;
        using C18 = std::integral_constant<int, 18>;
        while (ok && w.next(sg)) {
          const uint32_t end = it + uint32_t(sg.j1 - sg.j0);
          if ((!FP8 && !mbar_wait(&bars[kQFull], seg & 1)) || !mbar_wait(&bars[kQTmem], seg & 1)) {
            ok = false;
            break;
          }
          for (uint32_t t = it; t < end; ++t) {
            // the tile's rows, and its S slot: both readers are done with S(t-2)
            if ((t >= 2 && !mbar_wait(&bars[kSRead0 + (t & 1)], ((t - 2) >> 1) & 1)) ||
                !mbar_wait(&bars[kKVFull0 + t % NSTAGE], (t / NSTAGE) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(t, C0{}, C2{});
            umma_commit(&bars[kRopeEmpty0 + (t & 1)]);
            issue_s(t, C2{}, C18{});
            umma_commit(&bars[kSFull0 + (t & 1)]);
          }
          if (!ok) break;
          umma_commit(&bars[kQEmpty]);  // every score MMA of this sequence is issued
          it = end;
          ++seg;
          if (*abort_flag) ok = false;
        }
      } else {
        const uint32_t id_o = FP8 ? idesc_e4m3(128, 256, true) : idesc_bf16(128, 256, true);
        while (ok && w.next(sg)) {
          const uint32_t end = it + uint32_t(sg.j1 - sg.j0);
          for (uint32_t t = it; t < end; ++t) {
            // P(t), and for the first tile of a later sequence the previous
            // epilogue must be done with O
            if ((t == it && seg > 0 && !mbar_wait(&bars[kOFree], (seg - 1) & 1)) ||
                !mbar_wait(&bars[kPFull0 + (t & 1)], (t >> 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // O[:, 256r:+256] (+)= P(t) . c(t)[:, 256r:+256]  (4 MMAs, A = P from TMEM)
            //   bf16: 16 tokens per MMA.  E4M3: 32 tokens per MMA, for the hi
            //   and the lo term of P (columns TM_P and TM_P + 16).
            const uint64_t vb0 = sdesc_sw128(v_base + (t % NSTAGE) * VF_BYTES, VBOX, 1024);
            const uint32_t pa = tmem + TM_P;
            if constexpr (FP8) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ts_f8(tmem + TM_O, pa + 16 * (kk >> 1) + 8 * (kk & 1),
                           vb0 + uint64_t(((kk & 1) * 32 * 128) >> 4), id_o,
                           (t > it || kk > 0) ? 1u : 0u);
            } else {
#pragma unroll
              for (int kk = 0; kk < BS / 16; ++kk)
                umma_ts(tmem + TM_O, pa + 8 * kk, vb0 + uint64_t((kk * 2048) >> 4), id_o,
                        (t > it || kk > 0) ? 1u : 0u);
            }
            umma_commit(&bars[kKVEmpty0 + (t % NSTAGE)]);
            umma_commit(&bars[kPVDone0 + (t & 1)]);
          }
          if (!ok) break;
          it = end;
          ++seg;
          if (*abort_flag) ok = false;
        }
      }
      if (!ok) {
        report(p.err, KVATTN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // no MMA of this thread may still write TMEM when it is released
      umma_commit(&bars[kMmaDrain + (warp == 1 ? 0 : 1)]);
      mbar_wait(&bars[kMmaDrain + (warp == 1 ? 0 : 1)], 0, KV_DRAIN_WAIT_NS);
    }
  } else if (warp >= SEND0 / 32) {   // (warps SEND0/32 .. PV_WARP-1)
    // ---------------------------------------------------------------- senders
    const int r = 32 * (warp & 3) + lane;          // head row = TMEM lane
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const uint32_t xbuf_peer = map_peer(smem_u32(smem + OFF_X), peer);
    const uint32_t xfull_peer = map_peer(smem_u32(&bars[kXFull0]), peer);
    auto wait_all = [](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity) ? 1 : 0) != 0;
    };
    Walker w{p.cum, 1, st, en};
    Seg sg;
    uint32_t u = 0, seg = 0;
    bool ok = true;
    float part_scale = 1.f;   // partial score -> raw score units (E4M3: c_scale * 2^-e)
    while (ok && w.next(sg)) {
      // This sequence's Q[:, 256r : 256r + 16 NQT] into TMEM (bf16), or both
      // E4M3 terms of its Q (hi into TMEM, lo into shared memory), once the
      // previous sequence's score MMAs (which read it) have completed.  Rows
      // past h are 0.
      bool qgood = seg == 0 || wait_all(&bars[kQEmpty], (seg - 1) & 1);
      if (qgood) {
        tc_fence_after();
        if constexpr (FP8) {
          const uint16_t* qrow = p.q + (int64_t(sg.b) * p.h + r) * ROWW;
          const int e = q_row_exp(qrow, r < p.h, rank, p.r_ratio);
          part_scale = p.c_scale * __uint_as_float(uint32_t(127 - e) << 23);
          // for the softmax warps, which read it after this sequence's Q barrier
          reinterpret_cast<float*>(smem + OFF_QSC)[r] = part_scale;
          build_q_e4m3(qrow, r < p.h, rank, p.r_ratio, e, tmem + lane_off + TM_Q, smem + OFF_QF,
                       smem + OFF_QH, r);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        } else {
          const uint4* src =
              reinterpret_cast<const uint4*>(p.q + (int64_t(sg.b) * p.h + r) * ROWW + 256 * rank);
#pragma unroll
          for (int half = 0; half < G::NQT / 4; ++half) {
            uint32_t qv[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 x = r < p.h ? __ldg(src + 8 * half + i) : make_uint4(0, 0, 0, 0);
              qv[4 * i] = x.x;
              qv[4 * i + 1] = x.y;
              qv[4 * i + 2] = x.z;
              qv[4 * i + 3] = x.w;
            }
            tmem_st32(tmem + lane_off + TM_Q + 32 * half, qv);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kQTmem]);
      }
      ++seg;
      for (int k = sg.j0; k < sg.j1; ++k, ++u) {
        const uint32_t slot = u & 1;   // S slot
        bool good = qgood && wait_all(&bars[kSFull0 + slot], (u >> 1) & 1);
        uint32_t hx[32];
        if (good) {
          tc_fence_after();
          uint32_t v0[32], v1[32];
          tmem_ld32(tmem + lane_off + TM_S + BS * slot, v0);
          tmem_ld32(tmem + lane_off + TM_S + BS * slot + 32, v1);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kSRead0 + slot]);
          if constexpr (FP8) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              v0[j] = __float_as_uint(__uint_as_float(v0[j]) * part_scale);
              v1[j] = __float_as_uint(__uint_as_float(v1[j]) * part_scale);
            }
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            hx[j] = partial_pair(v0[2 * j], v0[2 * j + 1]);
            hx[16 + j] = partial_pair(v1[2 * j], v1[2 * j + 1]);
          }
        }
        // the abort flag is read by every lane but decided for the warp
        good = good && !__any_sync(0xffffffffu, *abort_flag != 0);
        if (!good) { ok = false; break; }
        // Two staging slots and two receive slots: partial u goes through
        // staging slot u % 2 into the peer's receive slot u % 2.  The staging
        // slot is free once the peer has received the copy of partial u - 2,
        // the receive slot once the peer has read partial u - 2 out of it (both
        // signals say that reads have finished, so waits at CTA scope suffice),
        // so the round trip of one exchange overlaps the next.  Each warp stages
        // and pushes its own 32 rows (4 KB): no barrier across the sender warps;
        // the peer's barrier counts the bytes of all four.
        const uint32_t xs = u % NX;
        if (u >= uint32_t(NX) && !wait_all(&bars[kXSent0 + xs], ((u - NX) / NX) & 1)) { ok = false; break; }
        uint8_t* sbuf = smem + OFF_XS + xs * XBYTES;
        uint4* srow = reinterpret_cast<uint4*>(sbuf + r * XROW);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          srow[c ^ (r & 7)] = make_uint4(hx[4 * c], hx[4 * c + 1], hx[4 * c + 2], hx[4 * c + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (u >= uint32_t(NX) && !wait_all(&bars[kXEmpty0 + xs], ((u - NX) / NX) & 1)) { ok = false; break; }
        __syncwarp();
        if (lane == 0) {
          const uint32_t off = uint32_t(32 * (warp & 3)) * XROW;
          bulk_copy_to_peer(xbuf_peer + xs * XBYTES + off, sbuf + off, 32 * XROW,
                            xfull_peer + xs * 8u);
        }
      }
    }
    if (!ok) {
      report(p.err, KVATTN_DEVERR_TIMEOUT);
      *abort_flag = 1;
    }
    // Drain: the peer's last arrivals on this CTA's barriers (received / read)
    // for the last partials pushed
    for (uint32_t k = u > uint32_t(NX) ? u - NX : 0; k < u; ++k) {
      mbar_wait_cluster(&bars[kXSent0 + k % NX], (k / NX) & 1, KV_DRAIN_WAIT_NS);
      mbar_wait_cluster(&bars[kXEmpty0 + k % NX], (k / NX) & 1, KV_DRAIN_WAIT_NS);
    }
  } else {
    // ------------------------------------------ softmax / epilogue warps (2..9)
    const int r = 32 * (warp & 3) + lane;          // head row = TMEM lane
    const int hh = (warp - 2) >> 2;                // which 32 rows of the tile (and 128 O columns)
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const int tid = threadIdx.x - SW0;             // 0..255
    const uint8_t* xbuf = smem + OFF_X;
    float* mx_s = reinterpret_cast<float*>(smem + OFF_MX);   // [2][128]
    const uint32_t xempty_peer = map_peer(smem_u32(&bars[kXEmpty0]), peer);
    const uint32_t xsent_peer = map_peer(smem_u32(&bars[kXSent0]), peer);
    Walker w{p.cum, 1, st, en};
    Seg sg;
    uint32_t it = 0, received = 0, sgi = 0;
    bool ok = true;
    int nseg = 0, seg_unit[2] = {0, 0}, seg_slot[2] = {0, 0};   // this CTA's partials
    // Every wait result is made warp-uniform: the warp-collective TMEM
    // instructions that follow must be executed by all 32 lanes or none.
    auto wait_all = [](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity) ? 1 : 0) != 0;
    };
    while (ok && w.next(sg)) {
      const int len = max(0, min(p.seq_lens[sg.b], sg.n * BS));
      const uint32_t n = uint32_t(sg.j1 - sg.j0);
      float m_ref = -INFINITY, l = 0.f;   // l: this thread's half of the row sum
      bool good = true;
      // E4M3: this rank's partial scores come out of the MMAs in c_KV code
      // units times 2^e; the sender of this row wrote the factor back to
      // score units before arriving on the sequence's Q barrier
      float part_scale = 1.f;
      if constexpr (FP8) {
        good = wait_all(&bars[kQTmem], sgi & 1);
        part_scale = reinterpret_cast<const float*>(smem + OFF_QSC)[r];
      }
      ++sgi;
      // This rank's own partial of tile t (f16 pairs of this thread's 32
      // tokens), read out of S slot t % 2, which is then released.  The next
      // tile's partial is read in the middle of this tile's step, as soon as
      // the exchange has delivered this tile's peer partial: the score MMAs
      // of tile t + 2 wait for that slot, and with it the senders and the
      // exchange of tile t + 2, which the softmax of tile t + 2 waits for.
      uint32_t own[16];
      auto read_own = [&](uint32_t t) {
        const uint32_t slot = t & 1;
        if (!wait_all(&bars[kSFull0 + slot], (t >> 1) & 1)) return false;
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + TM_S + BS * slot + 32 * hh, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kSRead0 + slot]);
        if constexpr (FP8) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * part_scale);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) own[j] = partial_pair(v[2 * j], v[2 * j + 1]);
        return true;
      };
      if (n > 0) good = good && read_own(it);
      for (uint32_t k = 0; k < n; ++k) {
        const uint32_t t = it + k;
        const uint32_t slot = t & 1;
        // The peer's bulk copy writes this CTA's shared memory and completes on
        // this CTA's barrier: observing the phase makes the bytes visible.
        const uint32_t xs = t % NX;
        good = good && wait_all(&bars[kXFull0 + xs], (t / NX) & 1);
        received += good ? 1u : 0u;
        if (good && tid == 0) {
          // the bulk copy has landed, so it has read the peer's staging slot
          mbar_arrive_remote_relaxed(xsent_peer + xs * 8u);
          // arm for tile t + NX: the peer pushes it into this slot only after
          // the slot is released below, after every thread saw this phase
          mbar_arrive_expect_tx(&bars[kXFull0 + xs], XBYTES);
        }
        // hs: f16 pairs of full raw scores, tokens 32hh + 2j and + 2j + 1
        uint32_t hs[16];
        float mx = -INFINITY;
        if (good) {
          const int valid = len - (sg.j0 + int(k)) * BS - 32 * hh;
          const uint4* xr = reinterpret_cast<const uint4*>(xbuf + xs * XBYTES + r * XROW);
          uint4 pv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) pv[c] = xr[(4 * hh + c) ^ (r & 7)];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            hs[4 * c] = hadd2_u32(own[4 * c], pv[c].x);
            hs[4 * c + 1] = hadd2_u32(own[4 * c + 1], pv[c].y);
            hs[4 * c + 2] = hadd2_u32(own[4 * c + 2], pv[c].z);
            hs[4 * c + 3] = hadd2_u32(own[4 * c + 3], pv[c].w);
          }
          // Once every lane's loads have returned, the warp releases its share
          // of the receive slot, so that the peer can push the next partial
          // while this tile's softmax goes on.  The arrive is relaxed (a
          // release-ordered remote arrive costs about a microsecond), so it is
          // ordered after the loads by data: its address adds a value derived
          // from every lane's four loaded words, masked by p.zero (0 at run
          // time, unknown to the compiler), so it cannot issue before they
          // have returned.
          const uint32_t dep = __reduce_or_sync(0xffffffffu, pv[0].x ^ pv[1].y ^ pv[2].z ^ pv[3].w);
          if (lane == 0) mbar_arrive_remote_relaxed(xempty_peer + xs * 8u + (dep & p.zero));
          if (valid < 32) {   // tokens past the end of the sequence score -inf
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (2 * j >= valid) hs[j] = (hs[j] & 0xffff0000u) | 0xfc00u;
              if (2 * j + 1 >= valid) hs[j] = (hs[j] & 0x0000ffffu) | 0xfc000000u;
            }
          }
          uint32_t hm = hs[0];
#pragma unroll
          for (int j = 1; j < 16; ++j) hm = hmax2_u32(hm, hs[j]);
          const float2 m2 = __half22float2(*reinterpret_cast<const __half2*>(&hm));
          mx = fmaxf(m2.x, m2.y) * p.scale_log2;   // log2 units (scale > 0 keeps the order)
        }
        if (k + 1 < n) good = good && read_own(t + 1);
        // One barrier per tile in the common case: every thread has read the
        // receive slot, and no row's max has outgrown its reference by the
        // threshold.  Otherwise the two halves of each row exchange maxima.
        const bool slow = named_bar_or(3, NSW, !good || mx > m_ref + RESCALE_THRESHOLD);
        if (slow) {
          mx_s[hh * 128 + r] = mx;
          good = named_bar_and(3, NSW, good);
          if (!good) break;
          mx = fmaxf(mx, mx_s[(hh ^ 1) * 128 + r]);
          const bool grow = mx > m_ref + RESCALE_THRESHOLD;
          if (__any_sync(0xffffffffu, grow)) {
            // Both warps of a row pair see the same maxima, so they take this
            // branch together; rows that keep their reference scale by 1.
            const float m_new = grow ? mx : m_ref;
            const float alpha = grow ? exp2_approx(m_ref - m_new) : 1.f;
            if (k > 0) {
              // O holds earlier tiles: rescale this thread's half after the
              // previous P.V has landed
              good = wait_all(&bars[kPVDone0 + ((t - 1) & 1)], ((t - 1) >> 1) & 1);
              if (good) {
                tc_fence_after();
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
            l = k > 0 ? l * alpha : 0.f;
            m_ref = m_new;
          }
        }
        // the P slot was last read by P.V(t - 1)
        good = good && (t < 1 || wait_all(&bars[kPVDone0 + ((t - 1) & 1)], ((t - 1) >> 1) & 1));
        if (good) {
          tc_fence_after();
          uint32_t pk[16];
          float lsum = 0.f;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hs[j]));
            const float p0 = exp2_approx(fmaf(f.x, p.scale_log2, -m_ref));
            const float p1 = exp2_approx(fmaf(f.y, p.scale_log2, -m_ref));
            lsum += p0 + p1;
            if constexpr (FP8) {
              // two E4M3 terms; p <= 2^8 (the lazy-rescale threshold) stays
              // inside E4M3's range.  Word j / 2 of each term holds tokens
              // 32hh + 4(j / 2) .. + 3.
              uint32_t h2, l2;
              e4m3_two_terms(p0, p1, h2, l2);
              if (j & 1) {
                pk[j >> 1] |= h2 << 16;
                pk[8 + (j >> 1)] |= l2 << 16;
              } else {
                pk[j >> 1] = h2;
                pk[8 + (j >> 1)] = l2;
              }
            } else {
              pk[j] = pack_bf16(p0, p1);
            }
          }
          l += lsum;
          if constexpr (FP8) {
            tmem_st8(tmem + lane_off + TM_P + 8 * hh, pk);            // hi term
            tmem_st8(tmem + lane_off + TM_P + 16 + 8 * hh, pk + 8);   // lo term
          } else {
            tmem_st16(tmem + lane_off + TM_P + 16 * hh, pk);
          }
          tmem_st_wait();
          const int vt = len - (sg.j0 + int(k)) * BS;   // valid rows of the whole tile
          if (vt < BS) {
            // Zero the latent rows past the end of the sequence in the value
            // boxes that P.V reads: P is 0 there, but 0 * NaN is NaN.
            uint8_t* stg = smem + OFF_V + (t % NSTAGE) * VF_BYTES;
            const int v0 = max(vt, 0);
            constexpr int PIECES = G::NVB * 8;   // 16-byte pieces of a row, all boxes
            for (int idx = tid; idx < (BS - v0) * PIECES; idx += NSW) {
              const int row = v0 + idx / PIECES, rem = idx % PIECES;
              *reinterpret_cast<uint4*>(stg + (rem >> 3) * VBOX + row * 128 + (rem & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          }
          tc_fence_before();
          __syncwarp();  // good is warp-uniform: the whole warp is here
          if (lane == 0) mbar_arrive(&bars[kPFull0 + slot]);
        }
      }
      // ---- epilogue: O / l for this segment's rows (each thread: 128 columns)
      const uint32_t last = it + n - 1;
      // group-uniform, like every failure decision of this group
      if (!named_bar_and(2, NSW, good && wait_all(&bars[kPVDone0 + (last & 1)], (last >> 1) & 1))) {
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
        dl = p.part_lse + (slot_idx * 2 + rank) * p.h + r;   // each rank merges with its own copy
        if (nseg < 2) {   // only the first and the last segment of a range can be parts
          seg_unit[nseg] = sg.b;
          seg_slot[nseg] = int(slot_idx);
          ++nseg;
        }
      }
      // E4M3: O is in c_KV code units; c_scale turns it into values
      const float inv = lrow > 0.f ? p.c_scale / lrow : 0.f;
      Walker wn = w;
      Seg sn;
      if (sg.full && !wn.next(sn)) {
        // The CTA's last segment, final rows: the value ring (and Q) are idle
        // (every load was consumed by a P.V that has completed, after every
        // score MMA), so each warp stages its 32 rows x 128 columns there
        // (L::OFF_EPI) in four 128-byte swizzled boxes and one lane
        // stores them with TMA (whole lines, instead of one 16-byte piece of
        // 32 rows per store instruction).  Rows past h fall outside the
        // tensor and are clipped.
        uint8_t* ob = smem + L::OFF_EPI + (warp - 2) * (4 * 32 * 128);
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + TM_O + 128 * hh + 32 * cb, o);
          tmem_ld_wait();
          uint8_t* brow = ob + cb * (32 * 128) + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(brow + ((j ^ (lane & 7)) << 4)) =
                make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                            __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
#pragma unroll 1
          for (int cb = 0; cb < 4; ++cb)
            tma_store_3d(&tmO, ob + cb * (32 * 128), 256 * int(rank) + 128 * hh + 32 * cb,
                         32 * (warp & 3), sg.b);
          bulk_commit();
          bulk_wait_read();   // the staging is reused; the stores themselves finish on their own
        }
        __syncwarp();
      } else {
        // Each lane writes its own row: 32-byte stores where the row is 32-byte
        // aligned (the workspace always is), halving the store transactions of
        // these scattered rows.
        const bool v8 = (reinterpret_cast<uintptr_t>(dst) & 31) == 0;
#pragma unroll 1
        for (int cb = 0; cb < 128; cb += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + TM_O + 128 * hh + cb, o);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * inv);
          if (row_ok && v8) {
#pragma unroll
            for (int j = 0; j < 4; ++j) st_global_v8(dst + cb + 8 * j, o + 8 * j);
          } else if (row_ok) {
            float4* d4 = reinterpret_cast<float4*>(dst + cb);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              d4[j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                  __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
          }
        }
      }
      if (row_ok && (rank == 0 || !sg.full) && hh == 0)
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
      // The peer may have pushed up to NX partials that were not consumed (it
      // pushes into a receive slot only after this rank released it); they
      // land before this CTA's shared memory goes away.
      uint32_t total = 0;
      Walker w2{p.cum, 1, st, en};
      Seg s2;
      while (w2.next(s2)) total += uint32_t(s2.j1 - s2.j0);
      for (uint32_t k = received; k < total && k < received + NX; ++k)
        mbar_wait_cluster(&bars[kXFull0 + k % NX], (k / NX) & 1, KV_DRAIN_WAIT_NS);
    } else {
      // Publish this rank's halves of the partials it wrote and merge the
      // groups and sequences they complete (merge.cuh): each rank merges its
      // own 256 output columns, so no combine pass is launched.  The value
      // ring is idle by now (every load consumed, every P.V and TMA store
      // complete) and holds the merge's scratch.
      MergeArgs m;
      m.part_out = p.part_out + 256 * rank;
      m.part_lse = p.part_lse + int(rank) * p.h;
      m.split_first = p.split_first;
      m.split_count = p.split_count;
      m.arrive_unit = p.arrive + int64_t(rank) * (2 * p.B + p.G);
      m.arrive_slot = m.arrive_unit + p.B;
      m.out = p.out + 256 * rank;
      m.lse = p.lse;
      m.rows = p.h;
      m.dv = 256;
      m.ld = DC;
      m.lse_stride = 2 * p.h;
      m.write_lse = rank == 0;
      finish_splits<NSW>(m, nseg, seg_unit, seg_slot, reinterpret_cast<int*>(&bars[kMergeFlags]),
                         reinterpret_cast<float*>(smem + OFF_V), tid, 2);
    }
  }
  // Role code diverges within warps (single-lane producers and issuers); the
  // CTA barrier and the cluster barrier below are warp-aligned, so every warp
  // reconverges first.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  // Neither CTA leaves while the other may still address its shared memory.
  cluster_sync_all();
}

// ---------------------------------------------------------------- host side

static int mla_pairs_for_device() {
  static int cache[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::call_once(flags[dev], [dev] {
    int result = -1;
    if (cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mla::Lay<false>::SMEM) == cudaSuccess &&
        cudaFuncSetAttribute(mla_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             mla::Lay<true>::SMEM) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * 1024, 1, 1);
      cfg.blockDim = dim3(mla::THREADS, 1, 1);
      cfg.dynamicSmemBytes = std::max(mla::Lay<false>::SMEM, mla::Lay<true>::SMEM);
      cfg.attrs = nullptr;  // the kernel fixes its cluster shape at compile time
      cfg.numAttrs = 0;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, mla_decode_kernel<false>, &cfg) == cudaSuccess &&
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
  const bool fp8 = cc->dtype == KVATTN_FP8_E4M3;
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
  // A pair that crosses a sequence boundary drains its pipeline (epilogue,
  // Q reload: about as long as 7 tiles) and a split sequence costs a merge of
  // 256 KB partials; below this many extra tiles one pair per sequence is
  // faster.
  pa.whole_unit_slack = 12;
  pa.cum = reinterpret_cast<int64_t*>(ws + L.cum);
  pa.cta_start = reinterpret_cast<int4*>(ws + L.cta);
  pa.split_first = reinterpret_cast<int32_t*>(ws + L.split_first);
  pa.split_count = reinterpret_cast<int32_t*>(ws + L.split_count);
  pa.arrive = reinterpret_cast<int32_t*>(ws + L.arrive);
  pa.out = a.out;
  pa.lse = a.lse;
  pa.rows = a.h;
  pa.dv = mla::DC;
  pa.err = a.err;
  if (launch_plan(pa, a.stream) != cudaSuccess) return KVATTN_ERR_CUDA;

  alignas(64) CUtensorMap tmQF = {}, tmQH = {}, tmLF, tmLH, tmO;
  if (!fp8) {
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
    // latent rows of 576 elements; value boxes of 128-byte rows (64 bf16 or
    // 128 E4M3 dims), rope boxes of 64-byte rows (this rank's 32 bf16 dims,
    // or all 64 E4M3 dims)
    const uint64_t eb = fp8 ? 1 : 2;
    const uint64_t dims[3] = {uint64_t(mla::ROWW), uint64_t(mla::BS), uint64_t(cc->num_blocks)};
    const uint64_t strides[2] = {uint64_t(mla::ROWW) * eb, uint64_t(mla::ROWW) * eb * mla::BS};
    const uint32_t boxf[3] = {fp8 ? 128u : 64u, uint32_t(mla::BS), 1u};
    const uint32_t boxh[3] = {fp8 ? 64u : 32u, uint32_t(mla::BS), 1u};
    const CUtensorMapDataType dt =
        fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!encode_tensor_map_3d(&tmLF, dt, cc->latent, dims, strides, boxf,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_3d(&tmLH, dt, cc->latent, dims, strides, boxh,
                              CU_TENSOR_MAP_SWIZZLE_64B))
      return KVATTN_ERR_CUDA;
  }
  {
    // final outputs as [B][h][512] fp32, stored in 32 x 32 boxes (128-byte swizzle)
    const uint64_t so[2] = {uint64_t(mla::DC) * 4, uint64_t(mla::DC) * 4 * a.h};
    const uint32_t box[3] = {32u, 32u, 1u};
    const uint64_t dims_o[3] = {uint64_t(mla::DC), uint64_t(a.h), uint64_t(a.B)};
    if (!encode_tensor_map_3d(&tmO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.out, dims_o, so, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return KVATTN_ERR_CUDA;
  }
  MlaParams prm;
  prm.q = static_cast<const uint16_t*>(a.q);
  prm.bt = a.block_table;
  prm.seq_lens = a.seq_lens;
  prm.cum = pa.cum;
  prm.cta_start = pa.cta_start;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.part_out = reinterpret_cast<float*>(ws + L.part_out);
  prm.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  prm.split_first = pa.split_first;
  prm.split_count = pa.split_count;
  prm.arrive = pa.arrive;
  prm.G = G;
  prm.B = a.B;
  prm.h = a.h;
  prm.max_blocks = a.max_blocks;
  prm.num_blocks = cc->num_blocks;
  prm.scale_log2 = a.scale * kLog2e;
  prm.c_scale = fp8 ? cc->k_scale : 1.f;
  prm.r_ratio = fp8 ? cc->v_scale / cc->k_scale : 1.f;
  prm.err = a.err;
  prm.zero = 0u;
  // the kernel fixes its cluster shape (a CTA pair) at compile time
  const cudaError_t e =
      fp8 ? launch_pdl(mla_decode_kernel<true>, dim3(2 * G), dim3(mla::THREADS),
                       mla::Lay<true>::SMEM, a.stream, tmQF, tmQH, tmLF, tmLH, tmO, prm)
          : launch_pdl(mla_decode_kernel<false>, dim3(2 * G), dim3(mla::THREADS),
                       mla::Lay<false>::SMEM, a.stream, tmQF, tmQH, tmLF, tmLH, tmO, prm);
  return e == cudaSuccess ? KVATTN_OK : KVATTN_ERR_CUDA;
}

}  // namespace kv
