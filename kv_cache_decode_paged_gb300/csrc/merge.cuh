// merge.cuh -- split-KV partials merged by the decode kernels themselves.
//
// Used by the MLA decode.  A sequence whose pages span several CTA pairs gets
// one normalised partial output o_w and its log-sum-exp lse_w per pair; the
// final rows are their log-sum-exp combine
//   M = max_w lse_w,  o = sum_w e^(lse_w - M) o_w / sum_w e^(lse_w - M),
//   lse = M + log sum_w e^(lse_w - M)
// ("MLA：为什么一份 Latent 可以代替多头 KV Cache", section "FlashMLA 解决的不是
// 模型公式本身": each split keeps its local max, normaliser and output, and a
// stable merge reproduces the unsplit result).
//
// No separate combine pass is launched: at the end of its work every CTA
// publishes the partials it wrote (a CTA's page range is contiguous, so only
// its first and last segments can be parts of units) and counts them on global
// arrival counters that the planner zeroed.  Partials are grouped kMergeFan
// at a time; the CTA whose arrival completes a group merges it into the
// group's first slot, and the CTA that completes the last group of a unit
// merges the group results into the final rows.  So no CTA reads more than
// kMergeFan partials, or one per group, however many CTAs a long sequence
// spans.  Ordering: writers fence before their arrival; the merging CTA
// fences after observing the last one.  When no sequence is split (one pair
// per sequence) nothing is merged and nothing is launched after the decode.
#pragma once

#include "common.cuh"

namespace kv {

constexpr int kMergeFan = 8;

// A part of the unit's columns (MLA: each CTA of a pair owns half of them)
// is merged by the CTAs that wrote it, on counters of its own.
struct MergeArgs {
  float* part_out;             // slot s, row r, column c at part_out[(s * rows + r) * ld + c]
  float* part_lse;             // slot s, row r at part_lse[s * lse_stride + r]
  const int32_t* split_first;  // per unit: first slot, number of slots
  const int32_t* split_count;
  int32_t* arrive_unit;        // [units]  groups of the unit merged so far
  int32_t* arrive_slot;        // [slots]  partials of the group starting at this slot
  float* out;                  // unit u, row r, column c at out[(u * rows + r) * ld + c]
  float* lse;                  // [units][rows]; written only if write_lse
  int rows, dv, ld, lse_stride;
  bool write_lse;
};

constexpr int kMergeMaxW = 16;   // inputs whose weights are staged in shared memory
constexpr int kMergeIPT = 4;     // output float4s per thread per batch

// Shared-memory scratch merge_slots needs for `rows` rows.
__host__ __device__ constexpr int merge_scratch_floats(int rows) { return (kMergeMaxW + 2) * rows; }

// Merge n inputs, slots s0, s0 + stride, ..., into dst / dst_lse (which may
// be slot s0 itself).  Every one of the NT threads calls it; sm holds
// merge_scratch_floats(rows) floats; bar_id is a named barrier over exactly
// these threads.  The rows' weights e^(lse_w - M) / sum are computed once;
// each thread then sums kMergeIPT output float4s at a time, so that the loads
// of a whole batch are in flight together (a merge is latency-bound: it
// touches each partial once).
template <int NT>
__device__ void merge_slots(const MergeArgs& m, int s0, int stride, int n, float* dst,
                            float* dst_lse, float* sm, int tid, int bar_id) {
  const int rows = m.rows, v4 = m.dv >> 2;
  const int64_t ls = m.lse_stride;
  float* s_max = sm;
  float* s_inv = sm + rows;
  float* s_w = sm + 2 * rows;   // [kMergeMaxW][rows], used when n <= kMergeMaxW
  const bool staged = n <= kMergeMaxW;
  for (int row = tid; row < rows; row += NT) {
    float M = -INFINITY;
    for (int k = 0; k < n; ++k)
      M = fmaxf(M, __ldcg(m.part_lse + (s0 + k * stride) * ls + row));
    float den = 0.f;
    if (M != -INFINITY)
      for (int k = 0; k < n; ++k) {
        const float lw = __ldcg(m.part_lse + (s0 + k * stride) * ls + row);
        const float e = lw != -INFINITY ? exp2_approx((lw - M) * kLog2e) : 0.f;
        den += e;
        if (staged) s_w[k * rows + row] = e;
      }
    const float inv = (M != -INFINITY && den > 0.f) ? 1.f / den : 0.f;
    s_max[row] = M;
    s_inv[row] = inv;
    if (staged)
      for (int k = 0; k < n; ++k) s_w[k * rows + row] = M != -INFINITY ? s_w[k * rows + row] * inv : 0.f;
  }
  named_bar_sync(bar_id, NT);
  const int total = rows * v4;
  for (int base = tid; base < total; base += NT * kMergeIPT) {
    float4 acc[kMergeIPT];
#pragma unroll
    for (int i = 0; i < kMergeIPT; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < n; ++k) {
      const int64_t slot = s0 + k * stride;
      float4 v[kMergeIPT];
      float e[kMergeIPT];
#pragma unroll
      for (int i = 0; i < kMergeIPT; ++i) {
        const int idx = base + i * NT;
        const int row = idx / v4, c4 = idx - row * v4;
        e[i] = 0.f;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < total) {
          if (staged) {
            e[i] = s_w[k * rows + row];
          } else if (s_inv[row] > 0.f) {
            const float lw = __ldcg(m.part_lse + slot * ls + row);
            e[i] = lw != -INFINITY ? exp2_approx((lw - s_max[row]) * kLog2e) * s_inv[row] : 0.f;
          }
          if (e[i] != 0.f)   // a split with no valid token for this row adds nothing
            v[i] = __ldcg(reinterpret_cast<const float4*>(m.part_out + (slot * rows + row) * m.ld) + c4);
        }
      }
#pragma unroll
      for (int i = 0; i < kMergeIPT; ++i) {
        acc[i].x += e[i] * v[i].x;
        acc[i].y += e[i] * v[i].y;
        acc[i].z += e[i] * v[i].z;
        acc[i].w += e[i] * v[i].w;
      }
    }
#pragma unroll
    for (int i = 0; i < kMergeIPT; ++i) {
      const int idx = base + i * NT;
      if (idx < total) {
        const int row = idx / v4, c4 = idx - row * v4;
        reinterpret_cast<float4*>(dst + int64_t(row) * m.ld)[c4] = acc[i];
      }
    }
  }
  // every lse read above is done before dst_lse (possibly slot s0's) changes
  named_bar_sync(bar_id, NT);
  if (dst_lse)
    for (int row = tid; row < rows; row += NT) {
      const float inv = s_inv[row];
      dst_lse[row] = inv > 0.f ? s_max[row] - log2_approx(inv) * kLn2 : -INFINITY;
    }
}

// End of a CTA's work: publish its nseg (<= 2) partials, given as (unit,
// slot) pairs, and merge what their arrivals complete.  Every one of the NT
// threads calls it with the same arguments; flags points to 3 ints of shared
// memory, sm to merge_scratch_floats(rows) floats.
template <int NT>
__device__ void finish_splits(const MergeArgs& m, int nseg, const int* seg_unit,
                              const int* seg_slot, int* flags, float* sm, int tid, int bar_id) {
  if (nseg == 0) return;
  __threadfence();   // this CTA's partial stores, before its arrivals
  named_bar_sync(bar_id, NT);
  if (tid == 0)
    for (int i = 0; i < nseg; ++i) {
      const int u = seg_unit[i], f = m.split_first[u], cnt = m.split_count[u];
      const int j = (seg_slot[i] - f) / kMergeFan;
      const int gs = min(kMergeFan, cnt - j * kMergeFan);
      flags[i] = atomicAdd(m.arrive_slot + f + j * kMergeFan, 1) == gs - 1;
    }
  named_bar_sync(bar_id, NT);
  for (int i = 0; i < nseg; ++i) {
    if (!flags[i]) continue;   // the same for every thread
    const int u = seg_unit[i], f = m.split_first[u], cnt = m.split_count[u];
    const int j = (seg_slot[i] - f) / kMergeFan, g0 = f + j * kMergeFan;
    const int gs = min(kMergeFan, cnt - j * kMergeFan);
    const int ng = (cnt + kMergeFan - 1) / kMergeFan;
    float* out_u = m.out + int64_t(u) * m.rows * m.ld;
    float* lse_u = m.write_lse ? m.lse + int64_t(u) * m.rows : nullptr;
    __threadfence();   // the group's partials, published before their arrivals
    if (ng == 1) {
      merge_slots<NT>(m, g0, 1, gs, out_u, lse_u, sm, tid, bar_id);
      named_bar_sync(bar_id, NT);
      continue;
    }
    merge_slots<NT>(m, g0, 1, gs, m.part_out + int64_t(g0) * m.rows * m.ld,
                    m.part_lse + int64_t(g0) * m.lse_stride, sm, tid, bar_id);
    __threadfence();   // the group result, before the unit arrival
    named_bar_sync(bar_id, NT);
    if (tid == 0) flags[2] = atomicAdd(m.arrive_unit + u, 1) == ng - 1;
    named_bar_sync(bar_id, NT);
    if (flags[2]) {
      __threadfence();
      merge_slots<NT>(m, f, kMergeFan, ng, out_u, lse_u, sm, tid, bar_id);
    }
    named_bar_sync(bar_id, NT);
  }
}

}  // namespace kv
