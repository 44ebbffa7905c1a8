// noalloc.cu -- kvattn_decode_gqa_noalloc: the GQA decode with built-in scratch.
//
// kvattn_decode_gqa needs a caller-supplied workspace (the split plan and the
// per-split partial outputs).  Some callers cannot hand one over: a plugin or
// custom-op host whose interface passes only the op's inputs and outputs, a
// runtime that gives all device memory to its own pool up front, or a code
// path that must not call cudaMalloc because that may synchronise the device.
// For them this entry point uses a fixed scratch array that lives in the
// library's own device memory, so nothing is allocated per call.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds KVATTN_NOALLOC_SCRATCH_BYTES of device memory until the
// process exits.  In host code `g_scratch` only names a host-side stand-in,
// so its device address is looked up with cudaGetSymbolAddress, once per
// device, the first time this entry point runs with that device current.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) uint8_t g_scratch[KVATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_status[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

// Device address of g_scratch on the current device, or nullptr on failure.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_scratch_once[dev], [dev] {
    void* p = nullptr;
    g_scratch_status[dev] = cudaGetSymbolAddress(&p, g_scratch);
    g_scratch_ptr[dev] = (g_scratch_status[dev] == cudaSuccess) ? p : nullptr;
  });
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" kvattn_status kvattn_decode_gqa_noalloc(const void* q, const kvattn_cache* cache,
                                                   const int32_t* block_table,
                                                   const int32_t* seq_lens, int batch,
                                                   int max_blocks_per_seq, int h, int h_kv,
                                                   int d_h, float scale, float* out, float* lse,
                                                   int num_ctas, int32_t* err, void* stream) {
  // The plan and partial outputs this problem needs (0 when the arguments are
  // invalid or there is no device; the call below then reports why).  Nothing
  // in them has to start at zero: the planner writes the plan before the
  // decode reads it, and the combine reads only partial slots the decode wrote.
  const size_t need =
      batch > 0 ? kvattn_decode_workspace_bytes(KVATTN_GQA, batch, h, h_kv, d_h, num_ctas) : 0;
  if (need > size_t(KVATTN_NOALLOC_SCRATCH_BYTES)) return KVATTN_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    ws = scratch_for_current_device();
    if (!ws) return KVATTN_ERR_CUDA;
  }
  return kvattn_decode_gqa(q, cache, block_table, seq_lens, batch, max_blocks_per_seq, h, h_kv,
                           d_h, scale, out, lse, ws, ws ? size_t(KVATTN_NOALLOC_SCRATCH_BYTES) : 0,
                           num_ctas, err, stream);
}
