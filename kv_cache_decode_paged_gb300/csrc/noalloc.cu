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
// so its device address is looked up with cudaGetSymbolAddress, with the
// device current, until a lookup on that device succeeds; the address found
// is then kept for the life of the process.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

static __device__ __align__(256) uint8_t g_scratch[KVATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];   // guarded by g_scratch_mutex; null until a lookup succeeds

// Device address of g_scratch on the current device, or nullptr on failure.
// Only a successful lookup is remembered: a failed one (for example a first
// call made inside a stream capture) is tried again on the next call.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) == cudaSuccess) g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" kvattn_status kvattn_decode_gqa_noalloc(const void* q, const kvattn_cache* cache,
                                                   const int32_t* block_table,
                                                   const int32_t* seq_lens, int batch,
                                                   int max_blocks_per_seq, int h, int h_kv,
                                                   int d_h, float scale, float* out, float* lse,
                                                   int num_ctas, int32_t* err, void* stream) {
  // The arguments are checked exactly as kvattn_decode_gqa checks them, before
  // the scratch size, so an invalid call gets the same status either way.
  bool nothing = false;
  const kvattn_status st = kv::check_gqa_args(q, cache, block_table, seq_lens, batch,
                                              max_blocks_per_seq, 1, h, h_kv, d_h, scale, out, lse,
                                              num_ctas, &nothing);
  if (st != KVATTN_OK || nothing) return st;
  // The plan and partial outputs this problem needs (0 when no device answers;
  // the lookup below then fails).  Nothing in them has to start at zero: the
  // planner writes the plan before the decode reads it, and the combine reads
  // only partial slots the decode wrote.
  const size_t need = kvattn_decode_workspace_bytes(KVATTN_GQA, batch, h, h_kv, d_h, num_ctas);
  if (need > size_t(KVATTN_NOALLOC_SCRATCH_BYTES)) return KVATTN_ERR_WORKSPACE;
  void* ws = scratch_for_current_device();
  if (!ws) return KVATTN_ERR_CUDA;
  return kvattn_decode_gqa(q, cache, block_table, seq_lens, batch, max_blocks_per_seq, h, h_kv,
                           d_h, scale, out, lse, ws, size_t(KVATTN_NOALLOC_SCRATCH_BYTES),
                           num_ctas, err, stream);
}
