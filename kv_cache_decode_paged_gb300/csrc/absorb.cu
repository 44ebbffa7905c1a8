// absorb.cu -- the per-head projections around MLA absorbed decode, on tcgen05.
//
// Query side ("MLA：为什么一份 Latent 可以代替多头 KV Cache" and "Multi-Head
// Latent Attention (MLA) ...", section on the absorbed query): head i's
// absorbed query is q~_i = W_UK,i^T q^C_i, followed by the head's RoPE query
// q^R_i; the decode kernel takes [q~_i | q^R_i] as one bf16 row.
// Value side (same pages, the deferred value projection): the decode returns
// the probability-weighted latent sum u~_i; head i's value is W_UV,i u~_i,
// which W_O then maps to the model width (a plain GEMM over all heads, not
// built here).
//
// Both are a batch of small GEMMs, one per head, over the decode batch:
//   absorb:  Q~_i [B x d_c] = Q^C_i [B x d_hc] . W_UK,i [d_hc x d_c]
//   up-proj: V_i  [B x d_v] = U~_i  [B x d_c]  . W_UV,i^T [d_c x d_v]
// The weights dominate the bytes (W_UK and W_UV are 16 MiB each for 128 heads
// at d_c = 512, d_hc = d_v = 128), so each kernel streams every weight byte
// once and keeps the batch rows of one head in a single M = 128 tile.  The
// contraction runs on the tensor cores: one elected thread issues
// tcgen05.mma from shared memory into a TMEM accumulator, eight warps read the
// accumulator back (one TMEM lane = one batch row per thread; warps w and
// w + 4 share a 32-lane quarter and split its columns).
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

// Test builds only (-DKV_TEST_DROP_CHUNK=n, with a short KV_WAIT_NS): the CTA
// of head 0 and batch tile 0 arms a barrier but issues none of its loads (the
// query absorption: part 1 of W_UK; the up-projection: chunk n of W_UV), as
// copies that never land would, so that the waits on it run out and the
// abort path runs on the GPU.  The library is built without it.
#ifdef KV_TEST_DROP_CHUNK
#define KV_TEST_DROPS_ABSORB_PART(part) \
  (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (part) == 1)
#define KV_TEST_DROPS_UPV_CHUNK(c) (blockIdx.x == 0 && blockIdx.y == 0 && (c) == KV_TEST_DROP_CHUNK)
#else
#define KV_TEST_DROPS_ABSORB_PART(part) false
#define KV_TEST_DROPS_UPV_CHUNK(c) false
#endif

namespace kv {

namespace absorb {
constexpr int M = 128;              // batch rows per tile (TMEM lanes)
constexpr int THREADS = 256;        // eight warps, two per 32-lane TMEM quarter
constexpr int NW = THREADS / 32;
constexpr int BOX = 128 * 128;      // [128 rows x 128 bytes] swizzled box, 16 KB

// Query absorption: A = q^C [M x 128] K-major (2 boxes of 64 dims); B = W_UK
// rows [128 (K = d_hc) x 256 latent columns] MN-major (4 boxes of 64
// columns) per part of 256 columns.  A CTA takes one head (all of d_c, two
// parts at a time: two W slots, two TMEM accumulators of 256 columns), so
// every W_UK byte is read once and 128 heads fill one wave of CTAs (these
// kernels run one CTA per SM).  A part's epilogue stages its output in the
// part's W slot once its MMAs are done.
constexpr int QN = 256;             // latent columns per part (MMA N)
constexpr int Q_OFF_A = 0;
constexpr int Q_OFF_W = 2 * BOX;                       // 2 slots x 4 boxes
constexpr int Q_WSLOT = 4 * BOX;                       // 64 KB
constexpr int Q_OFF_BAR = Q_OFF_W + 2 * Q_WSLOT;       // 160 KB of operands
constexpr int Q_SMEM = 1024 + Q_OFF_BAR + 128;

// Value up-projection: K = d_c in chunks of 128 (two 64-wide boxes each).
// B = W_UV rows [128 (N = d_v) x 128 (K)] K-major, brought by TMA into a
// ring of four chunk slots (all of W_UV,i at d_c = 512, loaded up front);
// A = u~ rows rounded to bf16 by the CTA's threads into two stages.
constexpr int VK = 128;             // K per chunk
constexpr int V_BSLOTS = 4;
constexpr int V_OFF_A = 0;                             // 2 stages x 2 boxes
constexpr int V_OFF_B = 4 * BOX;                       // 4 slots x 2 boxes
constexpr int V_OFF_BAR = V_OFF_B + 2 * V_BSLOTS * BOX;  // 192 KB of operands
constexpr int V_SMEM = 1024 + V_OFF_BAR + 128;
constexpr int V_ROWS = M / NW;      // A rows per warp (16)
}  // namespace absorb

struct AbsorbParams {
  const uint16_t* q_rope;   // [B][h][d_rope] bf16
  uint16_t* q_abs;          // [B][h][d_c + d_rope] bf16
  int B, h, d_c, d_rope;
  int32_t* err;
};

struct UpParams {
  const float* u;           // [B][h][d_c] f32
  float* v;                 // [B][h][d_v] f32
  int B, h, d_c, d_v;
  int32_t* err;
};

// Shared-memory writes of the generic proxy become visible to the tensor core
// (async proxy) after this fence and a barrier.
KV_DEVI void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- absorb

// grid (h, 1, ceil(B / 128)).  CTA (i, 0, m) computes batch rows 128m ..
// 128m+127 of head i (rows past B are zero-filled by TMA and not stored), all
// d_c latent columns, and copies q^R behind them.
__global__ void __launch_bounds__(absorb::THREADS)
    mla_absorb_q_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmO, const AbsorbParams p) {
  using namespace absorb;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  // afull (q^C landed), wfull[2] (a W slot landed), mdone[2] (a part's MMAs done), drain
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Q_OFF_BAR);
  uint64_t* afull = bars;
  uint64_t* wfull = bars + 1;
  uint64_t* mdone = bars + 3;
  uint64_t* drain = bars + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, b0 = blockIdx.z * M;
  const int nparts = p.d_c / QN;

  if (tid == 0) {
    for (int s = 0; s < 6; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmO);
  }
  if (warp == 0) tmem_alloc(tmem_slot, 2 * QN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // inputs may come from the kernel before this one in the stream
  pdl_wait();
  pdl_launch_dependents();

  const int quarter = warp & 3, colh = warp >> 2;
  const int rows_here = p.B - (b0 + 32 * quarter);     // real rows of this warp's boxes
  bool ok = true;
  // q^R goes behind the absorbed part: warp w copies batch rows w, w + 8, ...,
  // lane l the 4-byte pieces l, l + 32, ... of each (whole rows per
  // instruction).  The first 32 pieces of every row (all of a 64-wide q^R)
  // are loaded here, so that they arrive while the weights stream in.
  const int nrow = min(M, p.B - b0), nw4 = p.d_rope / 2;
  auto rope_src = [&](int rr, int e) {
    return __ldg(reinterpret_cast<const uint32_t*>(p.q_rope + (size_t(b0 + rr) * p.h + i) * p.d_rope) + e);
  };
  auto rope_dst = [&](int rr) {
    return reinterpret_cast<uint32_t*>(p.q_abs + (size_t(b0 + rr) * p.h + i) * (p.d_c + p.d_rope) + p.d_c);
  };
  uint32_t rope[M / NW];
#pragma unroll
  for (int t = 0; t < M / NW; ++t) {
    const int rr = warp + NW * t;
    rope[t] = rr < nrow && lane < nw4 ? rope_src(rr, lane) : 0u;
  }
  // Parts in pairs: slot / accumulator e of pair g holds part 2g + e.
  for (int g = 0; 2 * g < nparts; ++g) {
    const int np = min(2, nparts - 2 * g);
    // Warp 0 loads and multiplies: the whole warp waits on each barrier and
    // lane 0 issues.  (A lone issuing lane whose warp-mates spin on a barrier
    // only it can complete is starved by their waits.)
    if (warp == 0) {
      if (lane == 0) {
        if (g == 0) {
          mbar_arrive_expect_tx(afull, 2 * BOX);
          for (int kb = 0; kb < 2; ++kb)      // q^C dims 64kb.., rows b0.. of head i
            tma_load_3d_nohint(smem + Q_OFF_A + kb * BOX, &tmQ, 64 * kb, i, b0, afull);
        }
        for (int e = 0; e < np; ++e) {
          mbar_arrive_expect_tx(&wfull[e], 4 * BOX);
          if (!KV_TEST_DROPS_ABSORB_PART(2 * g + e))
            for (int nb = 0; nb < 4; ++nb)    // W_UK,i columns 256 (2g+e) + 64 nb.., all rows
              tma_load_3d_nohint(smem + Q_OFF_W + e * Q_WSLOT + nb * BOX, &tmW,
                                 QN * (2 * g + e) + 64 * nb, 0, i, &wfull[e]);
        }
      }
      __syncwarp();
      for (int e = 0; e < np; ++e) {
        const bool landed = mbar_wait(afull, 0) && mbar_wait(&wfull[e], g & 1);
        if (__all_sync(0xffffffffu, landed ? 1 : 0)) {
          tc_fence_after();
          if (lane == 0) {
            const uint32_t idesc = idesc_bf16(M, QN, true);
            const uint64_t a0 = sdesc_sw128(smem_u32(smem + Q_OFF_A), 16, 1024);
            const uint64_t w0 = sdesc_sw128(smem_u32(smem + Q_OFF_W + e * Q_WSLOT), BOX, 1024);
#pragma unroll
            for (int k = 0; k < 8; ++k)        // K = 128 in steps of 16
              umma_ss(tmem + QN * e, a0 + uint64_t(((k >> 2) * BOX + (k & 3) * 32) >> 4),
                      w0 + uint64_t((k * 2048) >> 4), idesc, k > 0 ? 1u : 0u);
            umma_commit(&mdone[e]);
          }
        } else {
          ok = false;
          // the loads may still land: wait once more, with the drain's limit
          mbar_wait(afull, 0, KV_DRAIN_WAIT_NS);
          mbar_wait(&wfull[e], g & 1, KV_DRAIN_WAIT_NS);
          if (lane == 0) mbar_arrive(&mdone[e]);   // release the readers; nothing is stored
        }
        __syncwarp();
      }
    }
    // Epilogue of each part of the pair.  Warp w holds TMEM lanes 32 (w % 4) ..
    // (batch rows) and the part's columns 128 (w / 4) ..; it stages them as two
    // 128-byte swizzled boxes [32 rows x 64 columns] in the part's W slot
    // (free once the part's MMAs are done) and one lane stores them with TMA
    // (whole lines; rows past B are clipped).
    for (int e = 0; e < np; ++e) {
      if (!mbar_wait(&mdone[e], g & 1)) ok = false;
      ok = __syncthreads_and(ok) != 0;
      if (!ok) break;
      tc_fence_after();
      uint8_t* stage = smem + Q_OFF_W + e * Q_WSLOT + warp * (2 * 32 * 128);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {   // 32 columns: 128 colh + 32 c ..
        uint32_t r[32];
        __syncwarp();   // tcgen05.ld is warp-collective
        tmem_ld32(tmem + (uint32_t(32 * quarter) << 16) + uint32_t(QN * e + 128 * colh + 32 * c), r);
        tmem_ld_wait();
        uint8_t* brow = stage + (c >> 1) * (32 * 128) + lane * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int chunk = (c & 1) * 4 + j;
          *reinterpret_cast<uint4*>(brow + ((chunk ^ (lane & 7)) << 4)) =
              make_uint4(pack_bf16(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1])),
                         pack_bf16(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                         pack_bf16(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                         pack_bf16(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
        }
      }
      fence_async_smem();
      __syncwarp();
      if (rows_here > 0 && lane == 0) {
        for (int bx = 0; bx < 2; ++bx)
          tma_store_3d(&tmO, stage + bx * (32 * 128), QN * (2 * g + e) + 128 * colh + 64 * bx, i,
                       b0 + 32 * quarter);
        bulk_commit();
      }
      __syncwarp();
    }
    if (!ok) break;
    // the slots are loaded again for the next pair only after their stores
    // have read them, and the accumulators rewritten after these TMEM reads
    if (lane == 0) bulk_wait_read();
    tc_fence_before();
    __syncthreads();
  }
  ok = __syncthreads_and(ok) != 0;
  if (tid == 0 && !ok) report(p.err, KVATTN_DEVERR_TIMEOUT);

  // q^R stores; pieces past the first 32 of a row (q^R wider than 64) are
  // copied here, all of a pass's loads before its stores
  if (ok) {
#pragma unroll
    for (int t = 0; t < M / NW; ++t) {
      const int rr = warp + NW * t;
      if (rr < nrow && lane < nw4) rope_dst(rr)[lane] = rope[t];
    }
    for (int e0 = 32; e0 < nw4; e0 += 32) {
      const int e = e0 + lane;
#pragma unroll
      for (int t = 0; t < M / NW; ++t) {
        const int rr = warp + NW * t;
        rope[t] = rr < nrow && e < nw4 ? rope_src(rr, e) : 0u;
      }
#pragma unroll
      for (int t = 0; t < M / NW; ++t) {
        const int rr = warp + NW * t;
        if (rr < nrow && e < nw4) rope_dst(rr)[e] = rope[t];
      }
    }
  }
  if (lane == 0) bulk_wait_read();   // shared memory stays valid until the stores read it
  if (warp == 0 && !ok) {   // no MMA may still write TMEM when it is released
    if (lane == 0) umma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, KV_DRAIN_WAIT_NS);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 2 * QN);
}

// ---------------------------------------------------------------- up-projection

// grid (h, ceil(B / 128)).  CTA (i, m) computes batch rows 128m.. of head i,
// all d_v = 128 outputs, over d_c / 128 chunks of K.  Each thread loads its
// share of a chunk of u~ (16 rows x 4 floats) in one batch, rounds it to bf16
// (nearest even) into the swizzled A stage, and loads the next chunk while
// the tensor core multiplies this one; W_UV,i streams through its own ring.
__global__ void __launch_bounds__(absorb::THREADS)
    mla_up_v_kernel(const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmV, const UpParams p) {
  using namespace absorb;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  // bfull[4] (W chunk landed), mdone[4] (MMAs of the chunk in that slot done), drain
  uint64_t* bfull = reinterpret_cast<uint64_t*>(smem + V_OFF_BAR);
  uint64_t* mdone = bfull + V_BSLOTS;
  uint64_t* drain = mdone + V_BSLOTS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.x, b0 = blockIdx.y * M;
  const int nch = p.d_c / VK;
  constexpr int DV = 128;

  if (tid == 0) {
    for (int s = 0; s < 2 * V_BSLOTS + 1; ++s) mbar_init(&bfull[s], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 0) tmem_alloc(tmem_slot, DV);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // inputs (u~, and possibly the weights) may come from the kernel before
  // this one in the stream
  pdl_wait();
  pdl_launch_dependents();
  int issued = 0;              // W chunks whose loads thread 0 has issued
  auto load_w = [&](int c) {   // chunk c into slot c % 4
    uint8_t* sb = smem + V_OFF_B + (c % V_BSLOTS) * 2 * BOX;
    mbar_arrive_expect_tx(&bfull[c % V_BSLOTS], 2 * BOX);
    if (!KV_TEST_DROPS_UPV_CHUNK(c))
      for (int kb = 0; kb < 2; ++kb)   // W_UV,i rows 0..127, columns VK c + 64 kb..
        tma_load_3d_nohint(sb + kb * BOX, &tmW, VK * c + 64 * kb, 0, i, &bfull[c % V_BSLOTS]);
    issued = c + 1;
  };
  if (tid == 0)
    for (int c = 0; c < nch && c < V_BSLOTS; ++c) load_w(c);

  // A rows of this thread: warp + 8t, t < 16; lane l holds k = 4l .. 4l+3 of
  // the chunk (one coalesced 512-byte row per warp and t).  Two register
  // buffers keep the loads of the next two chunks in flight.
  const int k = 4 * lane, kb = k >> 6, ch = (k & 63) >> 3, half = (k & 7) >> 2;
  float4 xa[V_ROWS], xb[V_ROWS];
  auto load_u = [&](int c, float4 (&x)[V_ROWS]) {
#pragma unroll
    for (int t = 0; t < V_ROWS; ++t) {
      const int b = b0 + warp + NW * t;
      x[t] = b < p.B ? __ldg(reinterpret_cast<const float4*>(
                           p.u + (size_t(b) * p.h + i) * p.d_c + VK * c + k))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  bool ok = true;
  // One chunk: round x into A stage c % 2, then the tensor core multiplies it.
  // Returns the CTA-wide verdict of its opening barrier, so that every
  // thread leaves the chunk loop at the same chunk (a failed wait of warp 0
  // reaches the others there).
  auto step = [&](int c, float4 (&x)[V_ROWS]) -> bool {
    const int s = c & 1;
    uint8_t* sa = smem + V_OFF_A + s * 2 * BOX;
    // A stage s is free once the MMAs of chunk c - 2 are done
    if (c >= 2 && !mbar_wait(&mdone[(c - 2) % V_BSLOTS], ((c - 2) / V_BSLOTS) & 1)) ok = false;
    if (!__syncthreads_and(ok)) {
      ok = false;
      return false;
    }
#pragma unroll
    for (int t = 0; t < V_ROWS; ++t) {
      const int r = warp + NW * t;
      const uint32_t off = kb * BOX + r * 128 + (((ch ^ (r & 7)) << 4) | (half << 3));
      *reinterpret_cast<uint2*>(sa + off) =
          make_uint2(pack_bf16(x[t].x, x[t].y), pack_bf16(x[t].z, x[t].w));
    }
    fence_async_smem();
    __syncthreads();
    if (c + 2 < nch) load_u(c + 2, x);
    if (warp == 0) {   // converged: the warp waits, lane 0 issues
      const int slot = c % V_BSLOTS;
      if (__all_sync(0xffffffffu, mbar_wait(&bfull[slot], (c / V_BSLOTS) & 1) ? 1 : 0)) {
        tc_fence_after();
        if (lane == 0) {
          const uint32_t idesc = idesc_bf16(M, DV, false);
          const uint64_t a0 = sdesc_sw128(smem_u32(sa), 16, 1024);
          const uint64_t w0 = sdesc_sw128(smem_u32(smem + V_OFF_B + slot * 2 * BOX), 16, 1024);
#pragma unroll
          for (int j = 0; j < VK / 16; ++j) {
            const uint64_t off = uint64_t(((j >> 2) * BOX + (j & 3) * 32) >> 4);
            umma_ss(tmem, a0 + off, w0 + off, idesc, (c > 0 || j > 0) ? 1u : 0u);
          }
          umma_commit(&mdone[slot]);
        }
        __syncwarp();
        // refill the slot of chunk c - 1 (its MMAs are the oldest in flight)
        if (c >= 1 && c - 1 + V_BSLOTS < nch) {
          if (__all_sync(0xffffffffu,
                         mbar_wait(&mdone[(c - 1) % V_BSLOTS], ((c - 1) / V_BSLOTS) & 1) ? 1 : 0)) {
            if (lane == 0) load_w(c - 1 + V_BSLOTS);
          } else {
            ok = false;
          }
        }
      } else {
        ok = false;
        if (lane == 0) mbar_arrive(&mdone[slot]);
      }
      __syncwarp();
    }
    return true;
  };
  load_u(0, xa);
  if (nch > 1) load_u(1, xb);
  for (int c = 0; c < nch; c += 2) {
    if (!step(c, xa)) break;
    if (c + 1 < nch && !step(c + 1, xb)) break;
  }
  // the last chunk's MMAs complete after every earlier one
  if (ok && !mbar_wait(&mdone[(nch - 1) % V_BSLOTS], ((nch - 1) / V_BSLOTS) & 1)) ok = false;
  ok = __syncthreads_and(ok) != 0;
  if (warp == 0 && !ok) {
    if (lane == 0) report(p.err, KVATTN_DEVERR_TIMEOUT);
    // the newest load of each slot may still be landing: wait once more,
    // with the drain's limit (lane 0 counted the loads it issued)
    const int n = __shfl_sync(0xffffffffu, issued, 0);
    for (int c = n > V_BSLOTS ? n - V_BSLOTS : 0; c < n; ++c)
      mbar_wait(&bfull[c % V_BSLOTS], (c / V_BSLOTS) & 1, KV_DRAIN_WAIT_NS);
  }
  __syncwarp();
  tc_fence_after();

  // Epilogue: warp w holds TMEM lanes 32 (w % 4) .. (batch rows) and columns
  // 64 (w / 4) ..; it stages them in the free A stages as two 128-byte
  // swizzled boxes [32 rows x 32 floats] and one lane stores them with TMA
  // (rows past B are clipped).
  const int quarter = warp & 3, colh = warp >> 2;
  const int rows_here = p.B - (b0 + 32 * quarter);
  uint8_t* stage = smem + V_OFF_A + warp * (2 * 32 * 128);
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    __syncwarp();   // tcgen05.ld is warp-collective
    tmem_ld32(tmem + (uint32_t(32 * quarter) << 16) + uint32_t(64 * colh + 32 * c), r);
    tmem_ld_wait();
    uint8_t* brow = stage + c * (32 * 128) + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<uint4*>(brow + ((j ^ (lane & 7)) << 4)) =
          make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
  }
  fence_async_smem();
  __syncwarp();
  if (ok && rows_here > 0 && lane == 0) {
    for (int c = 0; c < 2; ++c)
      tma_store_3d(&tmV, stage + c * (32 * 128), 64 * colh + 32 * c, i, b0 + 32 * quarter);
    bulk_commit();
    bulk_wait_read();
  }
  __syncwarp();
  if (warp == 0 && !ok) {   // no MMA may still write TMEM when it is released
    if (lane == 0) umma_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, KV_DRAIN_WAIT_NS);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, DV);
}

// ---------------------------------------------------------------- host side

kvattn_status run_mla_absorb_q(const AbsorbArgs& a) {
  using namespace absorb;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(mla_absorb_q_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Q_SMEM);
  });
  if (attr_err != cudaSuccess) return KVATTN_ERR_CUDA;
  alignas(64) CUtensorMap tmQ, tmW, tmO;
  // q^C [B][h][d_hc] as (dim, head, batch); W_UK [h][d_hc][d_c] as (column, row, head)
  const uint64_t qd[3] = {uint64_t(a.d_hc), uint64_t(a.h), uint64_t(a.B)};
  const uint64_t qs[2] = {uint64_t(a.d_hc) * 2, uint64_t(a.h) * a.d_hc * 2};
  const uint32_t qb[3] = {64u, 1u, uint32_t(M)};
  const uint64_t wd[3] = {uint64_t(a.d_c), uint64_t(a.d_hc), uint64_t(a.h)};
  const uint64_t ws[2] = {uint64_t(a.d_c) * 2, uint64_t(a.d_hc) * a.d_c * 2};
  const uint32_t wb[3] = {64u, uint32_t(a.d_hc), 1u};
  // q_absorbed [B][h][d_c + d_rope] as (column, head, batch), stored in
  // [32 rows x 64 columns] boxes
  const int width = a.d_c + a.d_rope;
  const uint64_t od[3] = {uint64_t(width), uint64_t(a.h), uint64_t(a.B)};
  const uint64_t os[2] = {uint64_t(width) * 2, uint64_t(a.h) * width * 2};
  const uint32_t ob[3] = {64u, 1u, 32u};
  if (!encode_tensor_map_3d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q_nope, qd, qs, qb,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_3d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_uk, wd, ws, wb,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_3d(&tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q_abs, od, os, ob,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return KVATTN_ERR_CUDA;
  AbsorbParams p;
  p.q_rope = static_cast<const uint16_t*>(a.q_rope);
  p.q_abs = static_cast<uint16_t*>(a.q_abs);
  p.B = a.B;
  p.h = a.h;
  p.d_c = a.d_c;
  p.d_rope = a.d_rope;
  p.err = a.err;
  const dim3 grid(unsigned(a.h), 1u, unsigned((a.B + M - 1) / M));
  return launch_pdl(mla_absorb_q_kernel, grid, dim3(THREADS), Q_SMEM, a.stream, tmQ, tmW, tmO, p) ==
                 cudaSuccess
             ? KVATTN_OK
             : KVATTN_ERR_CUDA;
}

kvattn_status run_mla_up_v(const UpArgs& a) {
  using namespace absorb;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(mla_up_v_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    V_SMEM);
  });
  if (attr_err != cudaSuccess) return KVATTN_ERR_CUDA;
  alignas(64) CUtensorMap tmW, tmV;
  // W_UV [h][d_v][d_c] as (column, row, head)
  const uint64_t wd[3] = {uint64_t(a.d_c), uint64_t(a.d_v), uint64_t(a.h)};
  const uint64_t ws[2] = {uint64_t(a.d_c) * 2, uint64_t(a.d_v) * a.d_c * 2};
  const uint32_t wb[3] = {64u, uint32_t(a.d_v), 1u};
  // v [B][h][d_v] f32 as (column, head, batch), stored in [32 rows x 32 floats] boxes
  const uint64_t vd[3] = {uint64_t(a.d_v), uint64_t(a.h), uint64_t(a.B)};
  const uint64_t vs[2] = {uint64_t(a.d_v) * 4, uint64_t(a.h) * a.d_v * 4};
  const uint32_t vb[3] = {32u, 1u, 32u};
  if (!encode_tensor_map_3d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_uv, wd, ws, wb,
                            CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_3d(&tmV, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.v, vd, vs, vb,
                            CU_TENSOR_MAP_SWIZZLE_128B))
    return KVATTN_ERR_CUDA;
  UpParams p;
  p.u = a.u;
  p.v = a.v;
  p.B = a.B;
  p.h = a.h;
  p.d_c = a.d_c;
  p.d_v = a.d_v;
  p.err = a.err;
  const dim3 grid(unsigned(a.h), unsigned((a.B + M - 1) / M));
  return launch_pdl(mla_up_v_kernel, grid, dim3(THREADS), V_SMEM, a.stream, tmW, tmV, p) == cudaSuccess
             ? KVATTN_OK
             : KVATTN_ERR_CUDA;
}

}  // namespace kv
