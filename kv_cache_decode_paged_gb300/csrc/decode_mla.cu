// decode_mla.cu -- MLA absorbed decode (placeholder until the kernel lands).
#include "common.cuh"
#include "internal.h"

namespace kv {

int mla_default_ctas(int h) {
  (void)h;
  return device_sm_count();
}

kvattn_status run_decode_mla(const MlaArgs& a) {
  (void)a;
  return KVATTN_ERR_UNSUPPORTED;
}

}  // namespace kv
