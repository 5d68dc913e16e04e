// Layer forward for callers that cannot allocate device memory.
//
// moe_nvfp4_forward needs a caller-provided workspace.  Some callers cannot
// provide one: code that runs inside a host runtime or plugin that owns every
// device allocation and offers no allocator to its extensions, callers whose
// allocations are forbidden while a framework is capturing a CUDA graph, and C
// callers behind a fixed signature with no workspace argument.  For them,
// moe_nvfp4_forward_noalloc runs the same forward with its workspace (the h
// rows and the per-pair FP16 partial rows) taken from g_noalloc_ws below: a
// file-scope device array of kNoAllocBytes that every GPU which loads this
// library holds until the process exits.
//
// Nothing in that workspace has to start at zero: every h row and partial row
// that a call reads was written earlier in the same call, and rows of dropped
// pairs are never read.  The array keeps the last call's contents, and all
// calls share it, so two calls whose GPU work overlaps (on different streams,
// or on one stream from different host threads without ordering) race.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// The device address of g_noalloc_ws on the current device.  The host-side
// symbol is only a stand-in; the address is looked up once per device, with
// that device current, and kept for the life of the process: a device reset
// (cudaDeviceReset, or a destroyed and re-created primary context) between
// calls is not supported, as the kept address would then be stale.
int32_t noalloc_workspace(void** out) {
  int dev = 0;
  const cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) {
    moe::cuda_error_code(de);
    return MOE_ERR_UNSUPPORTED_DEVICE;
  }
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess) return moe::cuda_error_code(e);
    if (!p) return MOE_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int32_t moe_nvfp4_forward_noalloc(const moe_nvfp4_config* cfg, int64_t M,
                                             const void* x, const void* plan,
                                             const moe_nvfp4_weights* w13,
                                             const moe_nvfp4_weights* w2,
                                             const moe_nvfp4_weights* shared13,
                                             const moe_nvfp4_weights* shared2, void* y,
                                             uint32_t* status, void* stream) {
  size_t plan_bytes = 0, ws_bytes = 0;
  if (!cfg) return MOE_ERR_INVALID_ARG;
  if (M < 0) return MOE_ERR_SHAPE;
  if (M == 0) return MOE_OK;
  // validates cfg and M and gives the workspace this call needs
  int32_t rc = moe_nvfp4_query(cfg, M, &plan_bytes, &ws_bytes);
  if (rc) return rc;
  if (ws_bytes > kNoAllocBytes) return MOE_ERR_WORKSPACE;
  void* ws = nullptr;
  rc = noalloc_workspace(&ws);
  if (rc) return rc;
  return moe_nvfp4_forward(cfg, M, x, plan, w13, w2, shared13, shared2, y, ws, kNoAllocBytes,
                           status, stream);
}
