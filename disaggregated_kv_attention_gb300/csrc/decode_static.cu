// forkkv_residual_attn_decode_static: the decode entry point for callers that
// cannot allocate device memory.
//
// Some callers own no spare device memory to lend as scratch: a serving
// engine that hands nearly all free HBM to its own KV-cache pool at start-up,
// or a plugin host that invokes an attention op without offering a workspace
// and forbids cudaMalloc on its hot path (an allocation can synchronise the
// device and can fail under memory pressure).  For them the split-KV partial
// results live in a fixed array in this library's device image instead of a
// caller buffer.  Every GPU that loads the library holds the array until the
// process exits.
#include <mutex>

#include "../../include/forkkv.h"
#include "internal.h"

namespace {

// Scratch for the per-(item, agent, head) partials (m, l, acc, acc_r) and, when
// the caller passes no rotation table, the table itself.
static __device__ __align__(256) unsigned char g_decode_scratch[FORKKV_STATIC_SCRATCH_BYTES];

// Device address of g_decode_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached, keyed by the device ordinal:
// the address belongs to the device's primary context (the one the CUDA runtime
// uses), so it goes stale if the process resets the device (cudaDeviceReset) or
// calls from another context of the same device; such a process must not call
// this entry point after the reset.
int32_t scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FORKKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_decode_scratch) != cudaSuccess || !ptr) return FORKKV_ERR_CUDA;
    addr[dev] = ptr;
  }
  *out = addr[dev];
  return FORKKV_OK;
}

}  // namespace

extern "C" int32_t forkkv_residual_attn_decode_static(const forkkv_attn_params* p, void* stream) {
  size_t need = 0;
  int32_t rc = forkkv_decode_workspace_size(p, &need);  // validates every argument
  if (rc) return rc;
  if (need > FORKKV_STATIC_SCRATCH_BYTES) return FORKKV_ERR_SCRATCH;
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc) return rc;
  forkkv_attn_params q = *p;  // the caller's workspace fields are ignored
  q.workspace = scratch;
  q.workspace_bytes = FORKKV_STATIC_SCRATCH_BYTES;
  return forkkv_residual_attn_decode(&q, stream);
}
