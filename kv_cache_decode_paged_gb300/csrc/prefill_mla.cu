// prefill_mla.cu -- explicit-form ("MHA mode") MLA prefill over the paged latent.
//
// A chunk of q_len new tokens per sequence, causal among them, attends over the
// sequence's cached latent rows with per-head keys and values expanded from
// the latent (the new tokens are already appended: token j sits at position
// s_b - q_len + j):
//   k_t,i = [W_UK,i c_t | k_R,t] (192 wide),  v_t,i = W_UV,i c_t (128 wide),
//   out_j,i = sum_{t <= s_b - q_len + j} softmax_t(scale * [q^C_j,i | q^R_j,i] . k_t,i) v_t,i
// ("MLA：为什么一份 Latent 可以代替多头 KV Cache", sections "MHA Mode" and
// "Prefill 为什么未必使用与 Decode 相同的吸收方式": prefill expands k and v per
// head, decode absorbs; "Multi-Head Latent Attention (MLA): Mathematical
// Foundations, ...", sections "Low-Rank Joint Key-Value Compression" and
// "The Decoupled RoPE Solution").
//
// One CTA per (128 new tokens, head, sequence).  Per tile of 128 cached rows it
// expands K^C = C W_UK,i^T and V = C W_UV,i^T on the tensor cores (M = 128 rows,
// N = 128, K = 512 streamed in 64-dim chunks of latent and weights through a
// two-slot TMA ring) into TMEM, and the expanded tile never leaves the SM: the
// compute warps round it to bf16 into shared memory, where it is the B operand
// of S = Q [K^C | k_R]^T (K = 192) and of O += P V.  The softmax is online with
// a lazy rescale of O (only when a row's max grows by more than 2^8).  The
// expansion of tile t+1 is issued while the softmax of tile t runs.
//   warps 0-3  compute: thread r owns row r (TMEM lane r): drains the expanded
//              tile (row r = cached row r of the tile), softmax of query row r,
//              epilogue
//   warp 4     TMA producer: Q once, per tile the rope box and the 8 chunks
//   warp 5     MMA issuer
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

// Test builds only (-DKV_TEST_DROP_CHUNK=n, with a short KV_WAIT_NS): the
// producer of the CTA of (query tile 0, head 0, sequence 0) arms chunk n's
// barrier but issues none of its loads, as copies that never land would, so
// that the waits on it run out and the abort path runs on the GPU.  The
// library is built without it.
#ifdef KV_TEST_DROP_CHUNK
#define KV_TEST_DROPS_PREFILL_CHUNK(g) \
  (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (g) == uint32_t(KV_TEST_DROP_CHUNK))
#else
#define KV_TEST_DROPS_PREFILL_CHUNK(g) false
#endif

namespace kv {

namespace pf {
constexpr int BS = 64;                 // latent page (tokens)
constexpr int TILE = 128;              // cached rows per tile = two pages
constexpr int QT = 128;                // new tokens per CTA
constexpr int DHC = 128, DR = 64, DV = 128, DC = 512;
constexpr int BOX = 128 * 128;         // [128 rows x 64 bf16 dims], 128-byte swizzle: 16 KB
constexpr int OFF_Q = 0;               // Q: q^C dims 0..63, 64..127, q^R: three boxes
constexpr int NCH = 2;                 // chunk ring: latent chunk, W_UK chunk, W_UV chunk
constexpr int CH_BYTES = 3 * BOX;
constexpr int OFF_CH = OFF_Q + 3 * BOX;
constexpr int OFF_KR = OFF_CH + NCH * CH_BYTES;   // k_R of the tile
constexpr int OFF_K = OFF_KR + BOX;    // expanded K^C, two boxes
constexpr int OFF_V = OFF_K + 2 * BOX; // expanded V, two boxes
constexpr int OFF_BAR = OFF_V + 2 * BOX;
constexpr int NBARS = 24;
constexpr int SMEM = 1024 + OFF_BAR + NBARS * 8 + 16;
constexpr int THREADS = 192;
constexpr uint32_t TM_EK = 0;          // K^C accumulator, then S
constexpr uint32_t TM_EV = 128;        // V accumulator
constexpr uint32_t TM_P = 256;         // P, 64 columns of bf16 pairs
constexpr uint32_t TM_O = 384;         // O
constexpr float RESCALE_THRESHOLD = 8.f;
static_assert(SMEM <= 232448, "shared memory");
}  // namespace pf

enum : int {
  pQ = 0, pKR = 1, pKREmpty = 2, pChFull0 = 3, pChEmpty0 = 5, pEFull = 7, pEDrained = 8,
  pSFull = 9, pSRead = 10, pPFull = 11, pPVDone = 12, pDrain = 13, pAbort = 14, pNum = 15
};
static_assert(pNum <= pf::NBARS, "barrier slots");

struct PrefillParams {
  const int32_t* bt;
  const int32_t* seq_lens;
  float* out;
  float* lse;
  int q_len, h, max_blocks;
  int64_t num_blocks;
  float scale_log2;
  int32_t* err;
};

__global__ void __launch_bounds__(pf::THREADS, 1)
    mla_prefill_kernel(const __grid_constant__ CUtensorMap tmQC,
                       const __grid_constant__ CUtensorMap tmQR,
                       const __grid_constant__ CUtensorMap tmL,
                       const __grid_constant__ CUtensorMap tmWK,
                       const __grid_constant__ CUtensorMap tmWV, const PrefillParams p) {
  using namespace pf;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + pAbort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, head = blockIdx.y, b = blockIdx.z;

  if (threadIdx.x == 0) {
    mbar_init(&bars[pQ], 1);
    mbar_init(&bars[pKR], 1);
    mbar_init(&bars[pKREmpty], 1);
    for (int i = 0; i < NCH; ++i) {
      mbar_init(&bars[pChFull0 + i], 1);
      mbar_init(&bars[pChEmpty0 + i], 1);
    }
    mbar_init(&bars[pEFull], 1);
    mbar_init(&bars[pEDrained], 4);   // one arrival per compute warp
    mbar_init(&bars[pSFull], 1);
    mbar_init(&bars[pSRead], 4);
    mbar_init(&bars[pPFull], 4);
    mbar_init(&bars[pPVDone], 1);
    mbar_init(&bars[pDrain], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // This CTA's new tokens j in [j0, j1) sit at positions s - q_len + j; the
  // cached rows any of them sees are [0, pos_max] (tiles of 128 rows).
  int s = p.seq_lens[b];
  if (s < 0 || s > p.max_blocks * BS) {
    report(p.err, KVATTN_DEVERR_SEQ_LEN);
    s = max(0, min(s, p.max_blocks * BS));
  }
  const int j0 = QT * qt, j1 = min(p.q_len, j0 + QT);
  const int pos_max = s - p.q_len + j1 - 1;
  const int n_kt = pos_max >= 0 ? (pos_max + TILE) / TILE : 0;
  const int npages = (s + BS - 1) / BS;

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && n_kt > 0) {
      const int32_t* row = p.bt + int64_t(b) * p.max_blocks;
      auto page_of = [&](int pg) {
        if (pg >= npages) return int(p.num_blocks);   // past the sequence: zero fill
        const int blk = row[pg];
        if (blk < 0 || int64_t(blk) >= p.num_blocks) {
          report(p.err, KVATTN_DEVERR_BLOCK_ID);
          return int(p.num_blocks);
        }
        return blk;
      };
      mbar_arrive_expect_tx(&bars[pQ], 3 * BOX);
      tma_load_4d(smem + OFF_Q, &tmQC, 0, head, j0, b, &bars[pQ]);
      tma_load_4d(smem + OFF_Q + BOX, &tmQC, 64, head, j0, b, &bars[pQ]);
      tma_load_4d(smem + OFF_Q + 2 * BOX, &tmQR, 0, head, j0, b, &bars[pQ]);
      bool ok = true;
      uint32_t g = 0;   // chunk counter over all tiles
      int nkr = 0;      // rope loads issued
      for (int kt = 0; kt < n_kt && ok; ++kt) {
        const int pg0 = page_of(2 * kt), pg1 = page_of(2 * kt + 1);
        for (int ch = 0; ch < DC / 64; ++ch, ++g) {
          if (ch == NCH) {
            // the rope rows of the tile, once S(kt - 1) is done with the buffer
            // (after the first chunks, so that they are not held back by it)
            if (kt > 0 && !mbar_wait(&bars[pKREmpty], (kt - 1) & 1)) { ok = false; break; }
            mbar_arrive_expect_tx(&bars[pKR], BOX);
            tma_load_3d_nohint(smem + OFF_KR, &tmL, DC, 0, pg0, &bars[pKR]);
            tma_load_3d_nohint(smem + OFF_KR + BOX / 2, &tmL, DC, 0, pg1, &bars[pKR]);
            ++nkr;
          }
          const int slot = int(g % NCH);
          if (g >= uint32_t(NCH) && !mbar_wait(&bars[pChEmpty0 + slot], ((g - NCH) / NCH) & 1)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + OFF_CH + slot * CH_BYTES;
          mbar_arrive_expect_tx(&bars[pChFull0 + slot], CH_BYTES);
          if (!KV_TEST_DROPS_PREFILL_CHUNK(g)) {
            tma_load_3d_nohint(dst, &tmL, 64 * ch, 0, pg0, &bars[pChFull0 + slot]);
            tma_load_3d_nohint(dst + BOX / 2, &tmL, 64 * ch, 0, pg1, &bars[pChFull0 + slot]);
            tma_load_3d_nohint(dst + BOX, &tmWK, 64 * ch, 0, head, &bars[pChFull0 + slot]);
            tma_load_3d_nohint(dst + 2 * BOX, &tmWV, 64 * ch, 0, head, &bars[pChFull0 + slot]);
          }
        }
        if (*abort_flag) ok = false;
      }
      if (!ok) {
        report(p.err, KVATTN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // every load issued lands before the CTA can exit
      mbar_wait(&bars[pQ], 0, KV_DRAIN_WAIT_NS);
      if (nkr > 0) mbar_wait(&bars[pKR], (nkr - 1) & 1, KV_DRAIN_WAIT_NS);
      for (uint32_t k = g > uint32_t(NCH) ? g - NCH : 0; k < g; ++k)
        mbar_wait(&bars[pChFull0 + k % NCH], (k / NCH) & 1, KV_DRAIN_WAIT_NS);
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_kt > 0) {
      const uint32_t id_e = idesc_bf16(128, 128, false);   // expansion and S: B K-major
      const uint32_t id_o = idesc_bf16(128, 128, true);    // P.V: B (V) MN-major
      const uint32_t ch_base = smem_u32(smem + OFF_CH);
      bool ok = true;
      uint32_t g = 0;
      // expansion of tile kt: E_K = C W_UK^T, E_V = C W_UV^T over 8 chunks of 64 dims
      auto expand = [&](int kt) {
        for (int ch = 0; ch < DC / 64 && ok; ++ch, ++g) {
          const int slot = int(g % NCH);
          if (!mbar_wait(&bars[pChFull0 + slot], (g / NCH) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t base = ch_base + slot * CH_BYTES;
          const uint64_t a0 = sdesc_sw128(base, 16, 1024);
          const uint64_t k0 = sdesc_sw128(base + BOX, 16, 1024);
          const uint64_t v0 = sdesc_sw128(base + 2 * BOX, 16, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k) {   // K = 16 dims per MMA, 32 bytes of a 128-byte row
            umma_ss(tmem + TM_EK, a0 + uint64_t(2 * k), k0 + uint64_t(2 * k), id_e,
                    (ch > 0 || k > 0) ? 1u : 0u);
            umma_ss(tmem + TM_EV, a0 + uint64_t(2 * k), v0 + uint64_t(2 * k), id_e,
                    (ch > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&bars[pChEmpty0 + slot]);
        }
        umma_commit(&bars[pEFull]);
        (void)kt;
      };
      if (!mbar_wait(&bars[pQ], 0)) ok = false;
      if (ok) expand(0);
      const uint64_t q0 = sdesc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
      const uint64_t kc0 = sdesc_sw128(smem_u32(smem + OFF_K), 16, 1024);
      const uint64_t kr0 = sdesc_sw128(smem_u32(smem + OFF_KR), 16, 1024);
      const uint64_t vv0 = sdesc_sw128(smem_u32(smem + OFF_V), BOX, 1024);
      for (int kt = 0; kt < n_kt && ok; ++kt) {
        // S = Q [K^C | k_R]^T once the tile is in shared memory
        if (!mbar_wait(&bars[pEDrained], kt & 1) || !mbar_wait(&bars[pKR], kt & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < (DHC + DR) / 16; ++k) {
          const int box = k >> 2;                       // q^C 0..63, 64..127, q^R
          const uint64_t a = q0 + uint64_t((box * BOX + (k & 3) * 32) >> 4);
          const uint64_t bb = box < 2 ? kc0 + uint64_t((box * BOX + (k & 3) * 32) >> 4)
                                      : kr0 + uint64_t(((k & 3) * 32) >> 4);
          umma_ss(tmem + TM_EK, a, bb, id_e, k > 0 ? 1u : 0u);
        }
        umma_commit(&bars[pSFull]);
        umma_commit(&bars[pKREmpty]);
        // the next tile's expansion runs while the softmax of this one does
        if (kt + 1 < n_kt) {
          if (!mbar_wait(&bars[pSRead], kt & 1)) { ok = false; break; }
          tc_fence_after();
          expand(kt + 1);
          if (!ok) break;
        }
        // O += P V
        if (!mbar_wait(&bars[pPFull], kt & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)
          umma_ts(tmem + TM_O, tmem + TM_P + 8 * kk, vv0 + uint64_t((kk * 2048) >> 4), id_o,
                  (kt > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars[pPVDone]);
        if (*abort_flag) ok = false;
      }
      if (!ok) {
        report(p.err, KVATTN_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(&bars[pDrain]);
      mbar_wait(&bars[pDrain], 0, KV_DRAIN_WAIT_NS);
    }
  } else {
    // ---------------------------------------------------------------- compute
    const int r = 32 * warp + lane;
    const uint32_t lane_off = uint32_t(32 * warp) << 16;
    const int j = j0 + r;                               // query row r: new token j
    const bool qvalid = j < j1;
    const int qpos = s - p.q_len + j;                   // its position
    auto wait_all = [](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity) ? 1 : 0) != 0;
    };
    float m_ref = -INFINITY, l = 0.f;
    bool good = true;
    for (int kt = 0; kt < n_kt && good; ++kt) {
      // 1. the expanded tile to shared memory as bf16 (row r = cached row 128 kt + r;
      //    rows past the sequence are zero: their latent slots may hold anything)
      good = wait_all(&bars[pEFull], kt & 1) &&
             (kt == 0 || wait_all(&bars[pPVDone], (kt - 1) & 1));
      if (!good) break;
      tc_fence_after();
      const bool rvalid = TILE * kt + r < s;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {            // K^C, then V
        uint8_t* dst = smem + (part == 0 ? OFF_K : OFF_V);
#pragma unroll 1
        for (int cb = 0; cb < 128; cb += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + (part == 0 ? TM_EK : TM_EV) + cb, v);
          tmem_ld_wait();
          uint8_t* rowp = dst + (cb >> 6) * BOX + r * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {                 // 16-byte pieces of 8 dims
            const int piece = ((cb & 63) >> 3) + c;
            uint4 w = make_uint4(0, 0, 0, 0);
            if (rvalid)
              w = make_uint4(pack_bf16(__uint_as_float(v[8 * c]), __uint_as_float(v[8 * c + 1])),
                             pack_bf16(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                             pack_bf16(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                             pack_bf16(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
            *reinterpret_cast<uint4*>(rowp + ((piece ^ (r & 7)) << 4)) = w;
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[pEDrained]);
      // 2. S row r, causal mask, online softmax
      good = wait_all(&bars[pSFull], kt & 1);
      if (!good) break;
      tc_fence_after();
      float sv[128];
#pragma unroll
      for (int cb = 0; cb < 128; cb += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + TM_EK + cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = TILE * kt + cb + i;            // cached row of the column
          sv[cb + i] = (qvalid && t <= qpos) ? __uint_as_float(v[i]) * p.scale_log2 : -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[pSRead]);
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) mx = fmaxf(mx, sv[i]);
      const bool grow = mx > m_ref + RESCALE_THRESHOLD;
      if (__any_sync(0xffffffffu, grow)) {
        // rows whose max outgrew the reference rescale O (after P.V(kt - 1), which
        // was waited for above); the others scale by 1
        const float m_new = grow ? mx : m_ref;
        const float alpha = grow ? exp2_approx(m_ref - m_new) : 1.f;
        if (kt > 0) {
#pragma unroll 1
          for (int cb = 0; cb < DV; cb += 32) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + TM_O + cb, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tmem + lane_off + TM_O + cb, o);
          }
          tmem_st_wait();
        }
        l = kt > 0 ? l * alpha : 0.f;
        m_ref = m_new;
      }
      // P = 2^(s - m_ref) as bf16 pairs (0 for masked columns and empty rows)
#pragma unroll
      for (int cb = 0; cb < 128; cb += 64) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = m_ref == -INFINITY ? 0.f : exp2_approx(sv[cb + 2 * i] - m_ref);
          const float p1 = m_ref == -INFINITY ? 0.f : exp2_approx(sv[cb + 2 * i + 1] - m_ref);
          l += p0 + p1;
          pk[i] = pack_bf16(p0, p1);
        }
        tmem_st32(tmem + lane_off + TM_P + (cb >> 1), pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[pPFull]);
    }
    // 3. epilogue: out row j = O / l, lse (natural log).  The TMEM loads are
    //    warp-collective: every lane of the warp executes them, and only lanes
    //    with a new token store.
    if (good && n_kt > 0) good = wait_all(&bars[pPVDone], (n_kt - 1) & 1);
    if (!good) {
      report(p.err, KVATTN_DEVERR_TIMEOUT);
      *abort_flag = 1;
    } else {
      float* dst = p.out + ((int64_t(b) * p.q_len + j) * p.h + head) * DV;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (n_kt > 0) {
        tc_fence_after();
#pragma unroll 1
        for (int cb = 0; cb < DV; cb += 32) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + TM_O + cb, o);
          tmem_ld_wait();
          if (qvalid) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + cb + i) =
                  make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                              __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
          }
        }
      } else if (qvalid) {
        for (int c = 0; c < DV; c += 4)
          *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (qvalid)
        p.lse[(int64_t(b) * p.q_len + j) * p.h + head] =
            l > 0.f ? (m_ref + log2_approx(l)) * kLn2 : -INFINITY;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side

kvattn_status run_mla_prefill(const PrefillArgs& a) {
  static std::once_flag once;
  static cudaError_t attr_status = cudaSuccess;
  std::call_once(once, [] {
    attr_status = cudaFuncSetAttribute(mla_prefill_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, pf::SMEM);
  });
  if (attr_status != cudaSuccess) return KVATTN_ERR_CUDA;
  const kvattn_cache* cc = a.cache;
  alignas(64) CUtensorMap tmQC, tmQR, tmL, tmWK, tmWV;
  {
    // q^C [B][q_len][h][128]: boxes of 64 dims x 1 head x 128 tokens
    const uint64_t dims[4] = {uint64_t(pf::DHC), uint64_t(a.h), uint64_t(a.q_len), uint64_t(a.B)};
    const uint64_t st[3] = {uint64_t(pf::DHC) * 2, uint64_t(pf::DHC) * 2 * a.h,
                            uint64_t(pf::DHC) * 2 * a.h * a.q_len};
    const uint32_t box[4] = {64u, 1u, uint32_t(pf::QT), 1u};
    if (!encode_tensor_map_4d(&tmQC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q_nope, dims, st, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return KVATTN_ERR_CUDA;
  }
  {
    const uint64_t dims[4] = {uint64_t(pf::DR), uint64_t(a.h), uint64_t(a.q_len), uint64_t(a.B)};
    const uint64_t st[3] = {uint64_t(pf::DR) * 2, uint64_t(pf::DR) * 2 * a.h,
                            uint64_t(pf::DR) * 2 * a.h * a.q_len};
    const uint32_t box[4] = {64u, 1u, uint32_t(pf::QT), 1u};
    if (!encode_tensor_map_4d(&tmQR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q_rope, dims, st, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return KVATTN_ERR_CUDA;
  }
  {
    // latent pool [num_blocks][64][576]: boxes of 64 dims x 64 rows
    const uint64_t dims[3] = {uint64_t(pf::DC + pf::DR), uint64_t(pf::BS), uint64_t(cc->num_blocks)};
    const uint64_t st[2] = {uint64_t(pf::DC + pf::DR) * 2, uint64_t(pf::DC + pf::DR) * 2 * pf::BS};
    const uint32_t box[3] = {64u, uint32_t(pf::BS), 1u};
    if (!encode_tensor_map_3d(&tmL, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cc->latent, dims, st, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return KVATTN_ERR_CUDA;
  }
  {
    // W_UK, W_UV [h][128][512]: boxes of 64 latent dims x 128 rows of one head
    const uint64_t dims[3] = {uint64_t(pf::DC), uint64_t(pf::DHC), uint64_t(a.h)};
    const uint64_t st[2] = {uint64_t(pf::DC) * 2, uint64_t(pf::DC) * 2 * pf::DHC};
    const uint32_t box[3] = {64u, uint32_t(pf::DHC), 1u};
    if (!encode_tensor_map_3d(&tmWK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_uk, dims, st, box,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_3d(&tmWV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_uv, dims, st, box,
                              CU_TENSOR_MAP_SWIZZLE_128B))
      return KVATTN_ERR_CUDA;
  }
  PrefillParams prm;
  prm.bt = a.block_table;
  prm.seq_lens = a.seq_lens;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.q_len = a.q_len;
  prm.h = a.h;
  prm.max_blocks = a.max_blocks;
  prm.num_blocks = cc->num_blocks;
  prm.scale_log2 = a.scale * kLog2e;
  prm.err = a.err;
  const dim3 grid((a.q_len + pf::QT - 1) / pf::QT, a.h, a.B);
  mla_prefill_kernel<<<grid, pf::THREADS, pf::SMEM, a.stream>>>(tmQC, tmQR, tmL, tmWK, tmWV, prm);
  return cudaGetLastError() == cudaSuccess ? KVATTN_OK : KVATTN_ERR_CUDA;
}

}  // namespace kv
