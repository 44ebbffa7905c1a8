// decode_gqa.cu -- single-token GQA / MQA / MHA decode over a paged cache.
//
// o_i = softmax_t(scale * q_i . K_t) V over the s_b cached tokens, query head i
// reading KV head i / g ("MHA -> MQA -> GQA -> MLA", mlinterviewnotes §3.5: one
// code path, a different integer; "The KV cache size formula", §2.1).
//
// The kernel is HBM-bound (intensity 2g/b FLOP/byte, far left of the GB300
// ridge), so the design is about streaming K/V at full bandwidth and touching
// each byte once:
//  * Warp 0 (producer) walks the CTA's page range and issues TMA tile loads of
//    16-token K and V chunks ([16 tokens x d] each, 128-byte swizzled) into an
//    mbarrier ring of NSTAGE stages.  Block ids come from the block table 32 at
//    a time; an id outside the pool is flagged and loaded out of bounds, which
//    TMA zero-fills, so the kernel never dereferences it.
//  * Warps 1..4 (consumers) take chunks round-robin ("streams").  Each keeps
//    its own online-softmax state for 16 query heads of the group and runs
//    S = Q K^T and O += P V on the tensor cores with mma.sync m16n8k16 (Q and
//    P in registers, K/V through ldmatrix), so one K/V read serves all g heads.
//    For g > 16 (MT m-tiles) MT warps share each chunk.
//  * At the end of a unit's segment the streams merge through shared memory;
//    a segment that covers the whole unit writes the final row, otherwise a
//    normalised partial and its lse go to the workspace for the combine.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "walk.cuh"

// Test builds only (-DKV_TEST_DROP_CHUNK=n, with a short KV_WAIT_NS): CTA 0's
// producer neither signals nor loads chunk n of its walk, as a copy that never
// lands would, so that the consumer's bounded wait on that stage runs out and
// the abort path (error bit, stop, drain, exit) runs on the GPU.  The library
// is built without it.
#ifdef KV_TEST_DROP_CHUNK
#define KV_TEST_DROPS_CHUNK(ic) (blockIdx.x == 0 && (ic) == uint32_t(KV_TEST_DROP_CHUNK))
#else
#define KV_TEST_DROPS_CHUNK(ic) false
#endif

namespace kv {


template <int D, int MT, bool FP8>
struct GqaCfg {
  static constexpr int EB = FP8 ? 1 : 2;
  static constexpr int ROWB = D * EB;               // bytes of one token's vector
  static constexpr int NBOX = ROWB / 128;           // 128-byte wide TMA boxes per row
  static constexpr int BOX_ELEMS = 128 / EB;
  static constexpr int BOX_BYTES = 16 * 128;
  static constexpr int TILE_BYTES = 16 * ROWB;      // K (or V) of one 16-token chunk
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int NSTAGE = 65536 / STAGE_BYTES;
  static constexpr int GROUP = NSTAGE / 2 < 16 ? NSTAGE / 2 : 16;  // producer lanes per issue round
  static constexpr int NC = 4;                      // consumer warps
  static constexpr int NSTREAM = NC / MT;
  static constexpr int THREADS = 32 * (NC + 1);
  static constexpr int OPAD = D + 8;                // padded row of the merge buffer
  static constexpr int SMEM_STAGES = NSTAGE * STAGE_BYTES;
  static constexpr int SMEM_OBUF = NC * 16 * OPAD * 4;
  static constexpr int SMEM_STATS = NC * 16 * 2 * 4;
  static constexpr int SMEM_BARS = 2 * NSTAGE * 8 + 16;
  static constexpr int SMEM = 1024 + SMEM_STAGES + SMEM_OBUF + SMEM_STATS + SMEM_BARS;
  static_assert(ROWB % 128 == 0, "rows must be whole 128-byte boxes");
  static_assert(NC % MT == 0, "m-tiles must divide the consumer warps");
};

// Rescale O only when a row's running max grows by more than 2^8.
constexpr float kRescaleLog2 = 8.f;

// (e4m3x2_to_f16x2, common.cuh: the hardware conversion of a packed byte
// pair, exact for every E4M3 value, subnormals and NaN included)
// codes 0,1 and 2,3 of w
KV_DEVI uint32_t e4m3_b01(uint32_t w) { return e4m3x2_to_f16x2(uint16_t(w & 0xffffu)); }
KV_DEVI uint32_t e4m3_b23(uint32_t w) { return e4m3x2_to_f16x2(uint16_t(w >> 16)); }
// codes 0,2 and 1,3 of w (one byte permutation serves both)
KV_DEVI void e4m3_b02_b13(uint32_t w, uint32_t& b02, uint32_t& b13) {
  const uint32_t y = __byte_perm(w, 0u, 0x3120);
  b02 = e4m3x2_to_f16x2(uint16_t(y & 0xffffu));
  b13 = e4m3x2_to_f16x2(uint16_t(y >> 16));
}

// Byte offset of (token r, 16-byte chunk c) inside a 128B-swizzled tile.
template <int BOX_BYTES>
KV_DEVI uint32_t swz(int r, int c) {
  return (c >> 3) * BOX_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Row r of unit (b, kvh) is query token j = r / g (at position s_b - qlen + j)
// and head kvh * g + r % g; its index among the [B][qlen][h] q, out and lse rows.
// MQ = false is the single-token form (qlen = 1, r < g).
template <bool MQ>
KV_DEVI int64_t unit_row(const GqaParams& p, int b, int kvh, int r) {
  if constexpr (!MQ) return int64_t(b) * p.h + kvh * p.g + r;
  const int j = r / p.g, i = r - j * p.g;
  return (int64_t(b) * p.qlen + j) * p.h + kvh * p.g + i;
}

// MQ: several new tokens per sequence (qlen > 1), causal among themselves.
// The single-token instantiation carries none of the causal-limit work.
template <int D, int MT, bool FP8, bool MQ>
__global__ void __launch_bounds__(GqaCfg<D, MT, FP8>::THREADS)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const GqaParams p) {
  using C = GqaCfg<D, MT, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* obuf = reinterpret_cast<float*>(smem + C::SMEM_STAGES);
  float* ms = obuf + C::NC * 16 * C::OPAD;
  float* ls = ms + C::NC * 16;
  uint64_t* full = reinterpret_cast<uint64_t*>(ls + C::NC * 16);
  uint64_t* empty = full + C::NSTAGE;
  int* abort_flag = reinterpret_cast<int*>(empty + C::NSTAGE);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  // Launched right behind the planner: wait for its plan, and let the combine
  // that follows get scheduled while this grid runs.
  pdl_wait();
  pdl_launch_dependents();
  const int4 st = p.cta_start[c], en = p.cta_start[c + 1];
  if (!pos_less(st, en)) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], MT);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  const int cpp = p.bs >> 4;  // 16-token chunks per page

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const uint64_t pol = policy_evict_first();
    const int64_t oob_page = p.num_blocks * p.hkv;  // past the end: zero fill
    Walker w{p.cum, p.hkv, st, en};
    Seg sg;
    uint32_t it = 0;
    bool ok = true;
    while (ok && w.next(sg)) {
      const int32_t* row = p.bt + int64_t(sg.b) * p.max_blocks;
      for (int jb = sg.j0; jb < sg.j1 && ok; jb += 32) {
        int page = int(oob_page);
        const int j = jb + lane;
        if (j < sg.j1) {
          const int blk = row[j];
          if (blk < 0 || int64_t(blk) >= p.num_blocks)
            report(p.err, KVATTN_DEVERR_BLOCK_ID);
          else
            page = blk * p.hkv + sg.kvh;
        }
        const int cnt = min(32, sg.j1 - jb);
        const int nchunk = cnt * cpp;
        // Chunks go out C::GROUP at a time, one lane each: a wait on an mbarrier
        // and a TMA issue cost a few hundred cycles apiece, which one lane
        // issuing chunk by chunk could not hide (it would set the stream rate).
        // The chunks of a group use distinct stages, last filled at least one
        // group earlier, so their waits do not depend on each other.
        for (int c0 = 0; c0 < nchunk && ok; c0 += C::GROUP) {
          const int cl = c0 + lane;
          const int pg = __shfl_sync(0xffffffffu, page, min(cl / cpp, 31));
          bool lok = true, issued = false;
          const uint32_t ic = it + uint32_t(cl);
          if (lane < C::GROUP && cl < nchunk) {
            const int s = ic % C::NSTAGE;
            const int sub = cl % cpp;
            if (!mbar_wait(&empty[s], ((ic / C::NSTAGE) & 1) ^ 1)) {
              lok = false;
            } else if (!KV_TEST_DROPS_CHUNK(ic)) {
              issued = true;
              mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
              uint8_t* dst = stages + s * C::STAGE_BYTES;
#pragma unroll
              for (int bx = 0; bx < C::NBOX; ++bx) {
                tma_load_3d(dst + bx * C::BOX_BYTES, &tmK, bx * C::BOX_ELEMS, sub * 16, pg,
                            &full[s], pol);
                tma_load_3d(dst + C::TILE_BYTES + bx * C::BOX_BYTES, &tmV, bx * C::BOX_ELEMS,
                            sub * 16, pg, &full[s], pol);
              }
            }
          }
          lok = lok && *reinterpret_cast<volatile int*>(abort_flag) == 0;
          ok = __all_sync(0xffffffffu, lok) != 0;
          if (!ok) {
            if (lane == 0) {
              report(p.err, KVATTN_DEVERR_TIMEOUT);
              *reinterpret_cast<volatile int*>(abort_flag) = 1;
            }
            // Drain before exiting: wait (bounded) for the last copy issued
            // into each stage, which may still be landing in this CTA's shared
            // memory.  Chunks before this group were all issued, and the last
            // NSTAGE - GROUP of them hold stages that no chunk of this group
            // touched; each of this group's lanes covers the stage of its own
            // chunk: that chunk if it issued it, else the one NSTAGE before.
            const uint32_t base = it + uint32_t(c0);
            const uint32_t span = uint32_t(C::NSTAGE - C::GROUP);
            if (lane == 0)
              for (uint32_t k = base > span ? base - span : 0u; k < base; ++k)
                mbar_wait(&full[k % C::NSTAGE], (k / C::NSTAGE) & 1, KV_DRAIN_WAIT_NS);
            if (lane < C::GROUP) {
              if (issued)
                mbar_wait(&full[ic % C::NSTAGE], (ic / C::NSTAGE) & 1, KV_DRAIN_WAIT_NS);
              else if (ic >= uint32_t(C::NSTAGE))
                mbar_wait(&full[(ic - C::NSTAGE) % C::NSTAGE], ((ic - C::NSTAGE) / C::NSTAGE) & 1,
                          KV_DRAIN_WAIT_NS);
            }
            __syncwarp();
          }
        }
        it += uint32_t(nchunk);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int stream = cw / MT, mt = cw % MT;
  const int r0 = lane >> 2, tig = lane & 3;
  const int lrow = lane & 7, lmat = lane >> 3;
  const int ctid = threadIdx.x - 32;
  constexpr int NKS = D / 16;  // k-steps of S = Q K^T
  constexpr int NNT = D / 8;   // n-tiles of O

  Walker w{p.cum, p.hkv, st, en};
  Seg sg;
  uint32_t it = 0;
  bool ok = true;
  while (w.next(sg)) {
    const int hl0 = 16 * mt + r0, hl1 = hl0 + 8;
    // Causal limit among the new tokens: row hl's token sees the first
    // len - (qlen - 1 - j) cached tokens (all of them when qlen = 1).
    const int back0 = MQ ? p.qlen - 1 - min(hl0, p.rows - 1) / p.g : 0;
    const int back1 = MQ ? p.qlen - 1 - min(hl1, p.rows - 1) / p.g : 0;
    uint32_t qa[NKS][4];
    {
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(
          p.q + unit_row<MQ>(p, sg.b, sg.kvh, min(hl0, p.rows - 1)) * D);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(
          p.q + unit_row<MQ>(p, sg.b, sg.kvh, min(hl1, p.rows - 1)) * D);
      const bool v0 = hl0 < p.rows, v1 = hl1 < p.rows;
      if constexpr (!FP8) {
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
          qa[ks][0] = v0 ? q0[ks * 8 + tig] : 0u;
          qa[ks][1] = v1 ? q1[ks * 8 + tig] : 0u;
          qa[ks][2] = v0 ? q0[ks * 8 + 4 + tig] : 0u;
          qa[ks][3] = v1 ? q1[ks * 8 + 4 + tig] : 0u;
        }
      } else {
        // f16 q with the summation index permuted to match how the K bytes
        // arrive (see the FP8 S loop): k-step c, logical k = 2t, 2t+1 are dims
        // 16c + 4t + {0,1}; logical k = 2t+8, 2t+9 are dims 16c + 4t + {2,3}.
        auto f16pair = [](uint32_t u) {
          return pack_f16(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
        };
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
          const uint2 x0 = v0 ? *reinterpret_cast<const uint2*>(q0 + ks * 8 + 2 * tig) : make_uint2(0, 0);
          const uint2 x1 = v1 ? *reinterpret_cast<const uint2*>(q1 + ks * 8 + 2 * tig) : make_uint2(0, 0);
          qa[ks][0] = f16pair(x0.x);
          qa[ks][1] = f16pair(x1.x);
          qa[ks][2] = f16pair(x0.y);
          qa[ks][3] = f16pair(x1.y);
        }
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[NNT][4];
#pragma unroll
    for (int i = 0; i < NNT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    int len = p.seq_lens[sg.b];
    len = max(0, min(len, sg.n * p.bs));
    const int nchunks = (sg.j1 - sg.j0) * cpp;
    for (int k = stream; k < nchunks && ok; k += C::NSTREAM) {
      const uint32_t itk = it + k;
      const int s = itk % C::NSTAGE;
      // warp-uniform result: the mma.sync / ldmatrix below need all 32 lanes
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (itk / C::NSTAGE) & 1) ? 1 : 0)) {
        report(p.err, KVATTN_DEVERR_TIMEOUT);
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
        ok = false;
        break;
      }
      const int valid = len - (sg.j0 * cpp + k) * 16;
      if (valid > 0) {
        const uint32_t kb = smem_u32(stages + s * C::STAGE_BYTES);
        const uint32_t vb = kb + C::TILE_BYTES;
        // S^T tile: 16 heads x 16 tokens, two n-tiles of 8 tokens.  The
        // multi-token form runs every chunk through every consumer warp, so
        // the latency of a chain of dependent MMAs sets its pace: it splits
        // each n-tile's sum over K into two chains (acc2 takes every other
        // K step) and adds them at the end.
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if constexpr (!FP8) {
#pragma unroll
          for (int ks = 0; ks < NKS; ++ks) {
            const int tok = (lmat >> 1) * 8 + lrow;
            const int ch = 2 * ks + (lmat & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kb + swz<C::BOX_BYTES>(tok, ch), b0, b1, b2, b3);
            float(&a)[2][4] = MQ && (ks & 1) ? acc2 : acc;
            mma_bf16(a[0], qa[ks], b0, b1);
            mma_bf16(a[1], qa[ks], b2, b3);
          }
        } else {
          // K rows are 128 bytes = 8 chunks of 16 dims.  A b16 ldmatrix of
          // (8 tokens x one chunk) gives each thread 4 consecutive codes of
          // token t/4: dims 16c + 4t .. +3, widened to two f16 pairs.
#pragma unroll
          for (int cp = 0; cp < NKS / 2; ++cp) {
            const int tok = (lmat & 1) * 8 + lrow;
            const int ch = 2 * cp + (lmat >> 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kb + swz<C::BOX_BYTES>(tok, ch), r0, r1, r2, r3);
            float(&a)[2][4] = MQ ? acc2 : acc;
            mma_f16(acc[0], qa[2 * cp], e4m3_b01(r0), e4m3_b23(r0));
            mma_f16(acc[1], qa[2 * cp], e4m3_b01(r1), e4m3_b23(r1));
            mma_f16(a[0], qa[2 * cp + 1], e4m3_b01(r2), e4m3_b23(r2));
            mma_f16(a[1], qa[2 * cp + 1], e4m3_b01(r3), e4m3_b23(r3));
          }
        }
        if constexpr (MQ) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][i] += acc2[nt][i];
        }
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tok = nt * 8 + 2 * tig + (i & 1);
            sc[nt][i] = tok < valid - (i < 2 ? back0 : back1) ? acc[nt][i] * p.qk_scale_log2
                                                              : -INFINITY;
          }
        float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
        float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // Lazy rescaling: O and l keep their reference max until a row's
        // chunk max exceeds it by kRescaleLog2; P then stays below 2^8.  The
        // first chunk always takes this branch (the reference starts at -inf).
        const bool grow0 = mx0 > m0 + kRescaleLog2, grow1 = mx1 > m1 + kRescaleLog2;
        if (__any_sync(0xffffffffu, grow0 || grow1)) {
          const float mn0 = grow0 ? mx0 : m0, mn1 = grow1 ? mx1 : m1;
          const float c0 = grow0 ? exp2_approx(m0 - mn0) : 1.f;
          const float c1 = grow1 ? exp2_approx(m1 - mn1) : 1.f;
          m0 = mn0;
          m1 = mn1;
          l0 *= c0;
          l1 *= c1;
#pragma unroll
          for (int i = 0; i < NNT; ++i) {
            o[i][0] *= c0;
            o[i][1] *= c0;
            o[i][2] *= c1;
            o[i][3] *= c1;
          }
        }
        // a row that has seen no token yet (possible only for an early new
        // token in a later part of its sequence) keeps m = -inf: its scores
        // here are all -inf too, and must give p = 0, not exp2(NaN)
        const float mu0 = MQ && m0 == -INFINITY ? 0.f : m0;
        const float mu1 = MQ && m1 == -INFINITY ? 0.f : m1;
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          pr[nt][0] = exp2_approx(sc[nt][0] - mu0);
          pr[nt][1] = exp2_approx(sc[nt][1] - mu0);
          pr[nt][2] = exp2_approx(sc[nt][2] - mu1);
          pr[nt][3] = exp2_approx(sc[nt][3] - mu1);
        }
        l0 += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        l1 += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
        uint32_t pa[4];
        if constexpr (!FP8) {
          pa[0] = pack_bf16(pr[0][0], pr[0][1]);
          pa[1] = pack_bf16(pr[0][2], pr[0][3]);
          pa[2] = pack_bf16(pr[1][0], pr[1][1]);
          pa[3] = pack_bf16(pr[1][2], pr[1][3]);
        } else {
          pa[0] = pack_f16(pr[0][0], pr[0][1]);
          pa[1] = pack_f16(pr[0][2], pr[0][3]);
          pa[2] = pack_f16(pr[1][0], pr[1][1]);
          pa[3] = pack_f16(pr[1][2], pr[1][3]);
        }
        // Zero V rows past the end of the sequence: P is 0 there, but the pool
        // may hold NaN in unwritten slots and 0 * NaN is NaN.
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (valid < 16) {
          const int t0 = 2 * tig;
          mlo = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
          mhi = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
        }
        if constexpr (!FP8) {
#pragma unroll
          for (int dn = 0; dn < D / 16; ++dn) {
            const int tok = (lmat & 1) * 8 + lrow;
            const int ch = 2 * dn + (lmat >> 1);
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(vb + swz<C::BOX_BYTES>(tok, ch), v0, v1, v2, v3);
            mma_bf16(o[2 * dn], pa, v0 & mlo, v1 & mhi);
            mma_bf16(o[2 * dn + 1], pa, v2 & mlo, v3 & mhi);
          }
        } else {
          // A transposing b16 ldmatrix of (8 tokens x one 16-dim chunk) gives
          // each thread dims 16c + 2t', +1 of tokens 2t and 2t+1 (t' = lane/4).
          // Even and odd dims become two n-tiles: n-tile 2c holds dims
          // 16c + 2n, n-tile 2c+1 holds dims 16c + 2n + 1.
#pragma unroll
          for (int cp = 0; cp < D / 32; ++cp) {
            const int tok = (lmat & 1) * 8 + lrow;
            const int ch = 2 * cp + (lmat >> 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(vb + swz<C::BOX_BYTES>(tok, ch), r0, r1, r2, r3);
            const int c0 = 2 * cp, c1 = 2 * cp + 1;
            uint32_t a02, a13, b02, b13, x02, x13, y02, y13;
            e4m3_b02_b13(r0, a02, a13);
            e4m3_b02_b13(r1, b02, b13);
            e4m3_b02_b13(r2, x02, x13);
            e4m3_b02_b13(r3, y02, y13);
            mma_f16(o[2 * c0], pa, a02 & mlo, b02 & mhi);
            mma_f16(o[2 * c0 + 1], pa, a13 & mlo, b13 & mhi);
            mma_f16(o[2 * c1], pa, x02 & mlo, y02 & mhi);
            mma_f16(o[2 * c1 + 1], pa, x13 & mlo, y13 & mhi);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    it += nchunks;

    // ---- merge the streams of this segment and write it out
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (tig == 0) {
      ms[cw * 16 + r0] = m0;
      ms[cw * 16 + r0 + 8] = m1;
      ls[cw * 16 + r0] = l0;
      ls[cw * 16 + r0 + 8] = l1;
    }
    named_bar_sync(1, C::NC * 32);
    float f0 = 0.f, f1 = 0.f;
    {
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int sidx = 0; sidx < C::NSTREAM; ++sidx) {
        M0 = fmaxf(M0, ms[(sidx * MT + mt) * 16 + r0]);
        M1 = fmaxf(M1, ms[(sidx * MT + mt) * 16 + r0 + 8]);
      }
      float L0 = 0.f, L1 = 0.f;
#pragma unroll
      for (int sidx = 0; sidx < C::NSTREAM; ++sidx) {
        const float a0 = ms[(sidx * MT + mt) * 16 + r0], a1 = ms[(sidx * MT + mt) * 16 + r0 + 8];
        if (a0 != -INFINITY) L0 += ls[(sidx * MT + mt) * 16 + r0] * exp2_approx(a0 - M0);
        if (a1 != -INFINITY) L1 += ls[(sidx * MT + mt) * 16 + r0 + 8] * exp2_approx(a1 - M1);
      }
      if (m0 != -INFINITY && L0 > 0.f) f0 = exp2_approx(m0 - M0) / L0;
      if (m1 != -INFINITY && L1 > 0.f) f1 = exp2_approx(m1 - M1) / L1;
    }
    float* ob = obuf + cw * 16 * C::OPAD;
#pragma unroll
    for (int i = 0; i < NNT; ++i) {
      if constexpr (!FP8) {
        const int col = i * 8 + 2 * tig;
        *reinterpret_cast<float2*>(ob + r0 * C::OPAD + col) = make_float2(o[i][0] * f0, o[i][1] * f0);
        *reinterpret_cast<float2*>(ob + (r0 + 8) * C::OPAD + col) =
            make_float2(o[i][2] * f1, o[i][3] * f1);
      } else {
        // n-tile 2c + e holds dims 16c + 2n + e; this thread has n = 2t, 2t+1
        const int col = (i >> 1) * 16 + 4 * tig + (i & 1);
        ob[r0 * C::OPAD + col] = o[i][0] * f0;
        ob[r0 * C::OPAD + col + 2] = o[i][1] * f0;
        ob[(r0 + 8) * C::OPAD + col] = o[i][2] * f1;
        ob[(r0 + 8) * C::OPAD + col + 2] = o[i][3] * f1;
      }
    }
    named_bar_sync(1, C::NC * 32);
    {
      // Row hl goes to its [B][qlen][h] row when the segment is the whole
      // unit, else to row hl of this CTA's partial slot (slot u + c).
      const int64_t slot = int64_t(sg.b) * p.hkv + sg.kvh + c;
      auto out_row = [&](int hl) {
        return sg.full ? unit_row<MQ>(p, sg.b, sg.kvh, hl) : slot * p.rows + hl;
      };
      float* dst_o = sg.full ? p.out : p.part_out;
      float* dst_l = sg.full ? p.lse : p.part_lse;
      constexpr int V4 = D / 4;
      for (int idx = ctid; idx < MT * 16 * V4; idx += C::NC * 32) {
        const int mt2 = idx / (16 * V4);
        const int rem = idx - mt2 * 16 * V4;
        const int row = rem / V4, c4 = rem - row * V4;
        const int hl = 16 * mt2 + row;
        if (hl >= p.rows) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int sidx = 0; sidx < C::NSTREAM; ++sidx) {
          const float4 v = *reinterpret_cast<const float4*>(
              obuf + ((sidx * MT + mt2) * 16 + row) * C::OPAD + c4 * 4);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        if (FP8) {
          acc.x *= p.v_mult;
          acc.y *= p.v_mult;
          acc.z *= p.v_mult;
          acc.w *= p.v_mult;
        }
        reinterpret_cast<float4*>(dst_o + out_row(hl) * D)[c4] = acc;
      }
      if (ctid < MT * 16) {
        const int mt2 = ctid >> 4, row = ctid & 15;
        const int hl = 16 * mt2 + row;
        if (hl < p.rows) {
          float M = -INFINITY, L = 0.f;
          for (int sidx = 0; sidx < C::NSTREAM; ++sidx) M = fmaxf(M, ms[(sidx * MT + mt2) * 16 + row]);
          for (int sidx = 0; sidx < C::NSTREAM; ++sidx) {
            const float a = ms[(sidx * MT + mt2) * 16 + row];
            if (a != -INFINITY) L += ls[(sidx * MT + mt2) * 16 + row] * exp2_approx(a - M);
          }
          dst_l[out_row(hl)] = (M == -INFINITY || !(L > 0.f)) ? -INFINITY : (M + log2_approx(L)) * kLn2;
        }
      }
    }
    named_bar_sync(1, C::NC * 32);
    // every consumer warp reads the flag after the same barrier, so they stop together
    if (*reinterpret_cast<volatile int*>(abort_flag)) break;
  }
}

// ---------------------------------------------------------------- host side

template <int D, int MT, bool FP8>
static int occupancy_ctas() {
  using C = GqaCfg<D, MT, FP8>;
  static int cache[64];
  static std::once_flag flags[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::call_once(flags[dev], [dev] {
    int n = 0;
    // both forms share the configuration; the attribute is set on each
    cudaFuncSetAttribute(gqa_decode_kernel<D, MT, FP8, true>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    cudaFuncSetAttribute(gqa_decode_kernel<D, MT, FP8, false>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_decode_kernel<D, MT, FP8, false>,
                                                      C::THREADS, C::SMEM) != cudaSuccess)
      n = 0;
    int sms = device_sm_count();
    cache[dev] = (n > 0 && sms > 0) ? n * sms : -1;
  });
  return cache[dev];
}

template <int D, int MT, bool FP8, bool MQ>
static kvattn_status launch_variant(const GqaArgs& a, const GqaParams& prm, int G) {
  using C = GqaCfg<D, MT, FP8>;
  if (occupancy_ctas<D, MT, FP8>() <= 0) return KVATTN_ERR_CUDA;  // also sets the smem attribute
  const kvattn_cache* cc = a.cache;
  alignas(64) CUtensorMap tmK, tmV;
  const uint64_t dims[3] = {uint64_t(D), uint64_t(cc->block_size),
                            uint64_t(cc->num_blocks) * uint64_t(cc->h_kv)};
  const uint64_t strides[2] = {uint64_t(C::ROWB), uint64_t(C::ROWB) * uint64_t(cc->block_size)};
  const uint32_t box[3] = {uint32_t(C::BOX_ELEMS), 16u, 1u};
  const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_tensor_map_3d(&tmK, dt, cc->k, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_3d(&tmV, dt, cc->v, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return KVATTN_ERR_CUDA;
  return launch_pdl(gqa_decode_kernel<D, MT, FP8, MQ>, dim3(G), dim3(C::THREADS), C::SMEM, a.stream,
                    tmK, tmV, prm) == cudaSuccess
             ? KVATTN_OK
             : KVATTN_ERR_CUDA;
}

// m-tiles of 16 rows: a unit's rows are q_len tokens x g heads (<= 64)
template <int D, bool FP8, bool MQ>
static kvattn_status dispatch_rows(const GqaArgs& a, const GqaParams& prm, int G) {
  const int rows = prm.rows;
  if (rows <= 16) return launch_variant<D, 1, FP8, MQ>(a, prm, G);
  if (rows <= 32) return launch_variant<D, 2, FP8, MQ>(a, prm, G);
  return launch_variant<D, 4, FP8, MQ>(a, prm, G);
}

template <int D, bool FP8>
static kvattn_status dispatch_mt(const GqaArgs& a, const GqaParams& prm, int G) {
  return prm.qlen > 1 ? dispatch_rows<D, FP8, true>(a, prm, G)
                      : dispatch_rows<D, FP8, false>(a, prm, G);
}

template <int D, bool FP8>
static int default_ctas_mt(int g) {
  return g <= 16 ? occupancy_ctas<D, 1, FP8>() : g <= 32 ? occupancy_ctas<D, 2, FP8>()
                                                          : occupancy_ctas<D, 4, FP8>();
}

int gqa_default_ctas(int dtype, int h, int h_kv, int d) {
  if (h_kv <= 0 || h % h_kv) return -1;
  const int g = h / h_kv;
  if (gqa_tc_applies(dtype, g, d)) return gqa_tc_ctas();
  if (dtype == KVATTN_FP8_E4M3) return d == 128 ? default_ctas_mt<128, true>(g) : -1;
  if (d == 64) return default_ctas_mt<64, false>(g);
  if (d == 128) return default_ctas_mt<128, false>(g);
  return -1;
}

kvattn_status run_decode_gqa(const GqaArgs& a) {
  const kvattn_cache* cc = a.cache;
  const bool fp8 = cc->dtype == KVATTN_FP8_E4M3;
  const int qlen = a.qlen > 0 ? a.qlen : 1;
  int G = a.G > 0 ? a.G : gqa_default_ctas(cc->dtype, a.h * qlen, a.h_kv, a.d);
  if (G <= 0) return KVATTN_ERR_CUDA;
  const int units = a.B * a.h_kv;
  const int g = a.h / a.h_kv;
  const int rows = qlen * g;
  const WsLayout L = ws_layout(a.B, units, G, rows, a.d);
  if (!a.workspace || a.ws_bytes < L.total || (reinterpret_cast<uintptr_t>(a.workspace) & 255))
    return KVATTN_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  PlanArgs pa;
  pa.seq_lens = a.seq_lens;
  pa.B = a.B;
  pa.units_per_seq = a.h_kv;
  pa.block_size = cc->block_size;
  pa.max_blocks = a.max_blocks;
  pa.G = G;
  pa.whole_unit_slack = -1;
  pa.cum = reinterpret_cast<int64_t*>(ws + L.cum);
  pa.cta_start = reinterpret_cast<int4*>(ws + L.cta);
  pa.split_first = reinterpret_cast<int32_t*>(ws + L.split_first);
  pa.split_count = reinterpret_cast<int32_t*>(ws + L.split_count);
  pa.arrive = nullptr;   // merged by the combine kernel
  pa.out = nullptr;
  pa.lse = nullptr;
  pa.rows = rows;
  pa.dv = a.d;
  pa.err = a.err;
  if (launch_plan(pa, a.stream) != cudaSuccess) return KVATTN_ERR_CUDA;

  GqaParams prm;
  prm.q = static_cast<const uint16_t*>(a.q);
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
  prm.hkv = a.h_kv;
  prm.g = g;
  prm.qlen = qlen;
  prm.rows = rows;
  prm.bs = cc->block_size;
  prm.max_blocks = a.max_blocks;
  prm.num_blocks = cc->num_blocks;
  // FP8 codes are widened exactly; the per-tensor scales enter here
  prm.qk_scale_log2 = a.scale * kLog2e * (fp8 ? cc->k_scale : 1.f);
  prm.v_mult = fp8 ? cc->v_scale : 1.f;
  prm.err = a.err;
  kvattn_status st;
  if (gqa_tc_applies(cc->dtype, rows, a.d))
    st = launch_gqa_tc(a, prm, G);
  else if (fp8)
    st = dispatch_mt<128, true>(a, prm, G);
  else if (a.d == 64)
    st = dispatch_mt<64, false>(a, prm, G);
  else
    st = dispatch_mt<128, false>(a, prm, G);
  if (st != KVATTN_OK) return st;
  // With at most a few CTAs per unit on average (G + units <= 4 units), each
  // split unit's merge is a handful of loads: one warp per row suffices.
  const bool few = int64_t(G) + units <= 4 * int64_t(units);
  if (launch_combine(prm.part_out, prm.part_lse, pa.split_first, pa.split_count, units, rows, a.d,
                     a.out, a.lse, true, a.stream, few, g, a.h_kv, qlen) != cudaSuccess)
    return KVATTN_ERR_CUDA;
  return KVATTN_OK;
}

}  // namespace kv
