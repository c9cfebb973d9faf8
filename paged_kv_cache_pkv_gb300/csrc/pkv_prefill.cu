// pkv_prefill.cu -- tensor-core path for chunked-prefill query rows.
// (Until this kernel is enabled every query row goes through split-KV.)
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

int prefill_max_tiles(const pkv_desc&, int32_t, int32_t) { return 0; }

int launch_prefill(const LaunchCtx&, const AttendArgs&, void*, int, int) {
  return PKV_OK;
}

}  // namespace pkv
