// Host-side launcher declarations shared by the C-ABI layer (api.cu) and the
// kernel translation units.  Launchers assume validated arguments.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

struct LayerDims {
  int H, E, k, I;
  int k_eff, e_eff;  // with the shared expert folded in as slot k / expert E
  bool shared;
};

struct Weights {
  const uint8_t* q;
  const uint8_t* s;
  const float* g;
};

cudaError_t launch_quantize(const float* w, int64_t n_mats, int64_t rows, int64_t k, int layout,
                            uint8_t* q, uint8_t* s, float* g, uint32_t* status,
                            cudaStream_t stream, int num_sms);
cudaError_t launch_dequantize(const uint8_t* q, const uint8_t* s, int64_t n_mats, int64_t rows,
                              int64_t k, int layout, void* out, cudaStream_t stream, int num_sms);

// One-time set-up of a device's kernels (shared-memory limits, the router's
// cluster size), run by the C-ABI layer under its device lock the first time
// a call uses device `dev`, before any launch there.  Each returns the first
// CUDA error; the set-up is retried on the next call after a failure.
cudaError_t router_device_init(int dev);
cudaError_t prefill_device_init();
cudaError_t decode_device_init();

// Router + plan.  ids_user / w_user are outputs unless ids_given.
cudaError_t launch_plan(const LayerDims& d, int64_t M, const __half* x, const __half* w_router,
                        const float* bias, const __half* w_gate, int32_t* ids_user,
                        float* w_user, bool ids_given, const PlanView& pv, uint32_t* status,
                        cudaStream_t stream, int num_sms);

// Forward paths.  partial: FP16 [M * k_eff][H], one row per pair at its plan
// position; h: FP16 [M * k_eff][I] in plan order.
// prepared: the scale arrays hold prepared FP16 scales (MOE_SCALES_PREPARED).
cudaError_t launch_decode_forward(const LayerDims& d, int64_t M, const __half* x,
                                  const PlanView& pv, Weights w13, Weights w2, Weights s13,
                                  Weights s2, __half* y, __half* h, __half* partial,
                                  uint32_t* status, cudaStream_t stream, int num_sms,
                                  bool prepared);
cudaError_t launch_prefill_forward(const LayerDims& d, int64_t M, const __half* x,
                                   const PlanView& pv, Weights w13, Weights w2, Weights s13,
                                   Weights s2, __half* y, __half* h, __half* partial,
                                   uint32_t* status, cudaStream_t stream, int num_sms,
                                   bool prepared);
cudaError_t launch_combine(const LayerDims& d, int64_t M, const PlanView& pv,
                           const __half* partial, __half* y, cudaStream_t stream, bool pdl);

// TMA tensor map over a byte matrix of `rows` x `row_bytes`, 8-byte elements,
// box `box_bytes` x `box_rows` (tma.cu).
cudaError_t make_rows_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows,
                          uint32_t box_bytes, uint32_t box_rows);
// TMA tensor map over an FP16 matrix rows x cols, box box_cols x box_rows,
// optionally 128-byte swizzled (tma.cu).
cudaError_t make_fp16_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                          uint32_t box_cols, uint32_t box_rows, bool swizzle128);
// FP16 matrix rows x cols as 64-element K segments: box of box_segs
// consecutive segments of box_rows rows, each a 128-byte-swizzled tile (tma.cu).
cudaError_t make_fp16_segments_map(CUtensorMap* map, const void* base, uint64_t cols,
                                   uint64_t rows, uint32_t box_rows, uint32_t box_segs);
// The same with a swizzle of 0 (none), 32, 64 or 128 bytes; a swizzled box is
// exactly one swizzle span wide (box_cols * 2 == swizzle_bytes).
cudaError_t make_fp16_map_swz(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                              uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);

// Dense few-row projection (dense.cu): weight formats, launchers.
enum DenseFormat { kDenseNvfp4 = 0, kDenseNvfp4Prepared = 1, kDenseFp8 = 2 };
constexpr int kDenseMaxTokens = 32;
size_t dense_ws_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_dense(int fmt, int64_t M, int64_t N, int64_t K, const __half* x,
                         const uint8_t* q, const uint8_t* s, const float* scale, void* ws,
                         __half* y, uint32_t* status, cudaStream_t stream);
cudaError_t launch_fp8_quantize(const float* w, int64_t rows, int64_t k, int layout, uint8_t* q,
                                float* cs, uint32_t* status, cudaStream_t stream);
cudaError_t launch_prepare_scales(const uint8_t* s, int64_t n, uint16_t* out, uint32_t* status,
                                  cudaStream_t stream);
cudaError_t dense_device_init();

// Test switch of the grouped GEMMs (prefill.cu): hold back W13's raw-weight
// producer and set the bounded waits' limit (SM cycles; <= 0: the default).
cudaError_t prefill_set_wait_test(int hold_raw, long long limit_cycles, cudaStream_t stream);

// Diagnostic: M <= 16 routes through the 128-block router (router.cu).
void set_force_small_router(bool on);
// Records the CUDA error behind a MOE_ERR_CUDA return for
// moe_nvfp4_last_cuda_error (api.cu) and clears the runtime's sticky error.
int32_t cuda_error_code(cudaError_t e);

// Diagnostic per-step event records (moe_nvfp4_set_trace_events).
enum TraceStep { kTracePlan = 0, kTraceW13 = 1, kTraceW2 = 2, kTraceCombine = 3 };
void trace_mark(cudaStream_t stream, int step, bool end);
bool trace_on();

// Launch helper: programmatic dependent launch when `pdl` is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace moe
