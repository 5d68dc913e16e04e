// C ABI of the NVFP4 MoE library (declared in include/moe_nvfp4.h).
//
// Every entry point validates its arguments on the host before anything is
// enqueued and returns a negative code without launching on any failure
// ("fails closed for tensor metadata": "[Kernel][SM70] Improve Qwen3.8 no-MTP
// concurrency", sections "Scope and related PRs" and "Guarded production
// engine result").  No exception crosses the boundary.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

struct DevInfo {
  bool init = false;
  bool supported = false;
  bool kernels_ready = false;
  int num_sms = 0;
};

std::mutex g_dev_mu;
DevInfo g_dev[64];

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

// Validates the current device (compute capability 10.3), caches its SM count
// and, once per device, sets up its kernels (shared-memory limits, the
// router's cluster size).  Returns MOE_OK or an error code.
int32_t current_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED_DEVICE;
  }
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (!di.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_UNSUPPORTED_DEVICE;
    }
    di.supported = (major == 10 && minor == 3);
    di.num_sms = sms;
    di.init = true;
  }
  if (!di.supported) return MOE_ERR_UNSUPPORTED_DEVICE;
  if (!di.kernels_ready) {
    cudaError_t e = router_device_init(dev);
    if (e == cudaSuccess) e = prefill_device_init();
    if (e == cudaSuccess) e = decode_device_init();
    if (e == cudaSuccess) e = dense_device_init();
    if (e != cudaSuccess) {
      g_last_cuda_error = e;
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    di.kernels_ready = true;
  }
  *num_sms = di.num_sms;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int32_t check_cfg(const moe_nvfp4_config* cfg, LayerDims* d) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  if (cfg->reserved[0] || cfg->reserved[1] || cfg->reserved[2]) return MOE_ERR_INVALID_ARG;
  if (cfg->flags & ~(MOE_FLAG_IDS_GIVEN | MOE_FLAG_SHARED)) return MOE_ERR_INVALID_ARG;
  const int H = cfg->hidden, E = cfg->n_experts, k = cfg->top_k, I = cfg->intermediate;
  if (H < 256 || H > 4096 || H % 256) return MOE_ERR_SHAPE;
  if (E < 8 || E > 512 || E % 8) return MOE_ERR_SHAPE;
  if (k < 1 || k > 32 || k > E) return MOE_ERR_SHAPE;
  if (I < 128 || I > 4096 || I % 128) return MOE_ERR_SHAPE;
  d->H = H;
  d->E = E;
  d->k = k;
  d->I = I;
  d->shared = (cfg->flags & MOE_FLAG_SHARED) != 0;
  d->k_eff = k + (d->shared ? 1 : 0);
  d->e_eff = E + (d->shared ? 1 : 0);
  return MOE_OK;
}

constexpr int64_t kMaxTokens = int64_t(1) << 20;

size_t plan_bytes_for(const LayerDims& d, int64_t M) {
  return plan_layout(nullptr, M, d.k_eff, d.e_eff, d.E, d.H, nullptr);
}

// The plan buffer for any M <= max_tokens.  Every array grows with M except
// the split router's partial logits (splits x M rows), which are largest at
// the top of a 64-token tile count and vanish where the tensor-core router
// takes over, so the maximum is taken over those points.
size_t plan_bytes_max(const LayerDims& d, int64_t max_tokens) {
  size_t best = plan_bytes_for(d, max_tokens);
  for (int64_t t = 1; t <= 128; ++t) {
    for (int64_t m : {64 * t - 1, 64 * t}) {
      const int64_t mm = m < max_tokens ? m : max_tokens;
      if (mm > kDecodeMaxTokens) {
        const size_t b = plan_bytes_for(d, mm);
        if (b > best) best = b;
      }
    }
    if (64 * t >= max_tokens) break;
  }
  return best;
}

size_t ws_bytes_for(const LayerDims& d, int64_t M) {
  const int64_t P = M * d.k_eff;
  return align_up((size_t)P * d.I * sizeof(__half), 256) + (size_t)P * d.H * sizeof(__half);
}

// `layout`, optionally with MOE_SCALES_PREPARED.
int32_t check_weights(const moe_nvfp4_weights* w, int32_t layout) {
  if (!w || !w->q || !w->s || !w->g) return MOE_ERR_INVALID_ARG;
  if (w->reserved) return MOE_ERR_INVALID_ARG;
  if ((w->layout & ~MOE_SCALES_PREPARED) != layout) return MOE_ERR_LAYOUT;
  if (!aligned16(w->q) || !aligned16(w->s) || (reinterpret_cast<uintptr_t>(w->g) & 3u))
    return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

void* const* g_trace_events = nullptr;
int32_t g_trace_steps = 0;
// forward: M <= this runs the weight-streaming decode kernels (diagnostic
// moe_nvfp4_set_decode_max_tokens; the default is the measured crossover)
int32_t g_decode_max_tokens = kDecodeMaxTokens;

int32_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  g_last_cuda_error = e;
  cudaGetLastError();
  return MOE_ERR_CUDA;
}

}  // namespace

namespace moe {
#ifdef MOE_TIMELINE
__device__ unsigned long long g_timeline[64];
__device__ unsigned long long g_prof[32];
__device__ unsigned long long g_dbg[20480];
#endif
bool trace_on() { return g_trace_events != nullptr; }
int32_t cuda_error_code(cudaError_t e) { return cuda_status(e); }
void trace_mark(cudaStream_t stream, int step, bool end) {
  if (!g_trace_events || step >= g_trace_steps) return;
  // external: under stream capture the record becomes an event node of the
  // graph (timed at every replay), not only a cross-stream dependency
  cudaEventRecordWithFlags(static_cast<cudaEvent_t>(g_trace_events[2 * step + (end ? 1 : 0)]),
                           stream, cudaEventRecordExternal);
}
}  // namespace moe

extern "C" {

#ifdef MOE_TIMELINE
// Timeline build only (not part of the public header): reset / read the
// per-kernel globaltimer stamps.
int32_t moe_nvfp4_timeline_reset(void* stream) {
  unsigned long long h[64];
  for (int s = 0; s < 5; ++s) {
    h[4 * s] = ~0ull;
    h[4 * s + 1] = ~0ull;
    h[4 * s + 2] = 0ull;
    h[4 * s + 3] = 0ull;
  }
  // raw cells 20..63: odd cells take minima, even cells maxima
  for (int c = 20; c < 64; ++c) h[c] = (c & 1) ? ~0ull : 0ull;
  return cuda_status(cudaMemcpyToSymbolAsync(moe::g_timeline, h, sizeof(h), 0,
                                             cudaMemcpyHostToDevice,
                                             static_cast<cudaStream_t>(stream)));
}
int32_t moe_nvfp4_timeline_read(unsigned long long* out) {
  return cuda_status(cudaMemcpyFromSymbol(out, moe::g_timeline, sizeof(unsigned long long) * 64));
}
int32_t moe_nvfp4_dbg_read(unsigned long long* out) {
  return cuda_status(cudaMemcpyFromSymbol(out, moe::g_dbg, sizeof(unsigned long long) * 20480));
}
int32_t moe_nvfp4_prof_read(unsigned long long* out, int reset) {
  cudaError_t e = cudaMemcpyFromSymbol(out, moe::g_prof, sizeof(unsigned long long) * 32);
  if (e == cudaSuccess && reset) {
    unsigned long long z[32] = {};
    e = cudaMemcpyToSymbol(moe::g_prof, z, sizeof(z));
  }
  return cuda_status(e);
}
#endif

int32_t moe_nvfp4_set_trace_events(void* const* events, int32_t n_steps) {
  if (events && (n_steps < 1 || n_steps > 4)) return MOE_ERR_INVALID_ARG;
  g_trace_events = events;
  g_trace_steps = events ? n_steps : 0;
  return MOE_OK;
}

int32_t moe_nvfp4_set_wait_test(int32_t hold_raw_producer, int64_t wait_limit_cycles,
                                void* stream) {
  if (hold_raw_producer != 0 && hold_raw_producer != 1) return MOE_ERR_INVALID_ARG;
  int sms = 0;
  int32_t rc = current_device(&sms);
  if (rc) return rc;
  return cuda_status(prefill_set_wait_test(hold_raw_producer, (long long)wait_limit_cycles,
                                           static_cast<cudaStream_t>(stream)));
}

int32_t moe_nvfp4_set_decode_max_tokens(int32_t m) {
  if (m < 0 || m > kDecodeMaxTokens) return MOE_ERR_INVALID_ARG;
  g_decode_max_tokens = m;
  return MOE_OK;
}

int32_t moe_nvfp4_set_small_router(int32_t mode) {
  if (mode != 0 && mode != 1) return MOE_ERR_INVALID_ARG;
  set_force_small_router(mode == 1);
  return MOE_OK;
}

int32_t moe_nvfp4_abi_version(void) { return MOE_NVFP4_ABI_VERSION; }

const char* moe_nvfp4_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "" : cudaGetErrorName(g_last_cuda_error);
}

const char* moe_nvfp4_status_string(int32_t code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "plan or workspace buffer too small";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3";
    case MOE_ERR_CUDA: return "CUDA runtime or launch failure";
    case MOE_ERR_LAYOUT: return "weights not in the required layout";
    case (int32_t)MOE_ST_INVALID_ID: return "status: expert id out of range (pair dropped)";
    case (int32_t)MOE_ST_NONFINITE: return "status: non-finite quantiser input";
    case (int32_t)MOE_ST_TIMEOUT: return "status: device-side wait timed out";
    default: return "unknown code";
  }
}

int32_t moe_nvfp4_query(const moe_nvfp4_config* cfg, int64_t max_tokens, size_t* plan_bytes,
                        size_t* ws_bytes) {
  LayerDims d;
  int32_t rc = check_cfg(cfg, &d);
  if (rc) return rc;
  if (max_tokens < 0 || max_tokens > kMaxTokens) return MOE_ERR_SHAPE;
  if (!plan_bytes && !ws_bytes) return MOE_OK;
  int sms = 0;
  rc = current_device(&sms);
  if (rc) return rc;
  if (plan_bytes) *plan_bytes = plan_bytes_max(d, max_tokens);
  if (ws_bytes) *ws_bytes = ws_bytes_for(d, max_tokens);
  return MOE_OK;
}

int32_t moe_nvfp4_quantize(const float* w, int64_t n_mats, int64_t rows, int64_t k,
                           int32_t layout, uint8_t* q, uint8_t* s, float* g, uint32_t* status,
                           void* stream) {
  if (!w || !q || !s || !g) return MOE_ERR_INVALID_ARG;
  if (layout < MOE_LAYOUT_CANONICAL || layout > MOE_LAYOUT_FRAGMENT_W13) return MOE_ERR_LAYOUT;
  if (n_mats < 1 || n_mats > 65535 || rows < 16 || k < 64) return MOE_ERR_SHAPE;
  if (k % 64 || rows % 16) return MOE_ERR_SHAPE;
  if (layout != MOE_LAYOUT_CANONICAL && rows % 256) return MOE_ERR_SHAPE;
  if (rows * k >= (int64_t(1) << 31)) return MOE_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(q) || !aligned16(s) || !aligned16(g)) return MOE_ERR_ALIGNMENT;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_ALIGNMENT;
  int sms = 0;
  int32_t rc = current_device(&sms);
  if (rc) return rc;
  return cuda_status(launch_quantize(w, n_mats, rows, k, layout, q, s, g, status,
                                     static_cast<cudaStream_t>(stream), sms));
}

int32_t moe_nvfp4_dequantize(const uint8_t* q, const uint8_t* s, int64_t n_mats, int64_t rows,
                             int64_t k, int32_t layout, void* out, void* stream) {
  if (!q || !s || !out) return MOE_ERR_INVALID_ARG;
  if (layout < MOE_LAYOUT_CANONICAL || layout > MOE_LAYOUT_FRAGMENT_W13) return MOE_ERR_LAYOUT;
  if (n_mats < 1 || rows < 16 || k < 64 || k % 64 || rows % 16) return MOE_ERR_SHAPE;
  if (layout != MOE_LAYOUT_CANONICAL && rows % 256) return MOE_ERR_SHAPE;
  if (n_mats * rows * k >= (int64_t(1) << 40)) return MOE_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(s) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
  int sms = 0;
  int32_t rc = current_device(&sms);
  if (rc) return rc;
  return cuda_status(
      launch_dequantize(q, s, n_mats, rows, k, layout, out, static_cast<cudaStream_t>(stream), sms));
}

int32_t moe_nvfp4_plan(const moe_nvfp4_config* cfg, int64_t M, const void* x,
                       const void* w_router, const float* bias, const void* w_gate, int32_t* ids,
                       float* topk_w, void* plan, size_t plan_bytes, uint32_t* status,
                       void* stream) {
  LayerDims d;
  int32_t rc = check_cfg(cfg, &d);
  if (rc) return rc;
  if (M < 0 || M > kMaxTokens) return MOE_ERR_SHAPE;
  if (M == 0) return MOE_OK;  // nothing to route; buffers of empty tensors may be NULL
  const bool given = (cfg->flags & MOE_FLAG_IDS_GIVEN) != 0;
  if (!x || !ids || !topk_w || !plan) return MOE_ERR_INVALID_ARG;
  if (!given && !w_router) return MOE_ERR_INVALID_ARG;
  if (d.shared && !w_gate) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(ids) || !aligned16(topk_w) || !aligned16(plan))
    return MOE_ERR_ALIGNMENT;
  if ((w_router && !aligned16(w_router)) || (bias && !aligned16(bias)) ||
      (d.shared && !aligned16(w_gate)))
    return MOE_ERR_ALIGNMENT;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_ALIGNMENT;
  if (plan_bytes < plan_bytes_for(d, M)) return MOE_ERR_WORKSPACE;
  int sms = 0;
  rc = current_device(&sms);
  if (rc) return rc;
  PlanView pv;
  plan_layout(static_cast<char*>(plan), M, d.k_eff, d.e_eff, d.E, d.H, &pv);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  trace_mark(st, kTracePlan, false);
  cudaError_t e = launch_plan(d, M, static_cast<const __half*>(x),
                              static_cast<const __half*>(w_router), bias,
                              static_cast<const __half*>(w_gate), ids, topk_w, given, pv,
                              status, st, sms);
  trace_mark(st, kTracePlan, true);
  return cuda_status(e);
}

int32_t moe_nvfp4_forward(const moe_nvfp4_config* cfg, int64_t M, const void* x, const void* plan,
                          const moe_nvfp4_weights* w13, const moe_nvfp4_weights* w2,
                          const moe_nvfp4_weights* shared13, const moe_nvfp4_weights* shared2,
                          void* y, void* ws, size_t ws_bytes, uint32_t* status, void* stream) {
  LayerDims d;
  int32_t rc = check_cfg(cfg, &d);
  if (rc) return rc;
  if (M < 0 || M > kMaxTokens) return MOE_ERR_SHAPE;
  if (M == 0) return MOE_OK;  // nothing to compute; buffers of empty tensors may be NULL
  if (!x || !plan || !y || !ws) return MOE_ERR_INVALID_ARG;
  if ((rc = check_weights(w13, MOE_LAYOUT_FRAGMENT_W13))) return rc;
  if ((rc = check_weights(w2, MOE_LAYOUT_FRAGMENT))) return rc;
  if (d.shared) {
    if ((rc = check_weights(shared13, MOE_LAYOUT_FRAGMENT_W13))) return rc;
    if ((rc = check_weights(shared2, MOE_LAYOUT_FRAGMENT))) return rc;
  }
  // one scale storage for the whole layer
  const int32_t sf = w13->layout & MOE_SCALES_PREPARED;
  if ((w2->layout & MOE_SCALES_PREPARED) != sf ||
      (d.shared && ((shared13->layout & MOE_SCALES_PREPARED) != sf ||
                    (shared2->layout & MOE_SCALES_PREPARED) != sf)))
    return MOE_ERR_LAYOUT;
  const bool prepared = sf != 0;
  if (!aligned16(x) || !aligned16(plan) || !aligned16(y) || !aligned16(ws))
    return MOE_ERR_ALIGNMENT;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < ws_bytes_for(d, M)) return MOE_ERR_WORKSPACE;
  int sms = 0;
  rc = current_device(&sms);
  if (rc) return rc;
  PlanView pv;
  plan_layout(static_cast<char*>(const_cast<void*>(plan)), M, d.k_eff, d.e_eff, d.E, d.H, &pv);
  const int64_t P = M * d.k_eff;
  __half* h = static_cast<__half*>(ws);
  __half* partial = reinterpret_cast<__half*>(static_cast<char*>(ws) +
                                              align_up((size_t)P * d.I * sizeof(__half), 256));
  Weights W13{w13->q, w13->s, w13->g}, W2{w2->q, w2->s, w2->g};
  Weights S13{nullptr, nullptr, nullptr}, S2{nullptr, nullptr, nullptr};
  if (d.shared) {
    S13 = Weights{shared13->q, shared13->s, shared13->g};
    S2 = Weights{shared2->q, shared2->s, shared2->g};
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (M <= g_decode_max_tokens)
    e = launch_decode_forward(d, M, static_cast<const __half*>(x), pv, W13, W2, S13, S2,
                              static_cast<__half*>(y), h, partial, status, st, sms, prepared);
  else
    e = launch_prefill_forward(d, M, static_cast<const __half*>(x), pv, W13, W2, S13, S2,
                               static_cast<__half*>(y), h, partial, status, st, sms, prepared);
  return cuda_status(e);
}

// ---- the whole layer in one call ----

int32_t moe_nvfp4_layer(const moe_nvfp4_config* cfg, int64_t M, const void* x,
                        const void* w_router, const float* bias, const void* w_gate, int32_t* ids,
                        float* topk_w, void* plan, size_t plan_bytes, const moe_nvfp4_weights* w13,
                        const moe_nvfp4_weights* w2, const moe_nvfp4_weights* shared13,
                        const moe_nvfp4_weights* shared2, void* y, void* ws, size_t ws_bytes,
                        uint32_t* status, void* stream) {
  LayerDims d;
  int32_t rc = check_cfg(cfg, &d);
  if (rc) return rc;
  if (M < 0 || M > kMaxTokens) return MOE_ERR_SHAPE;
  if (M == 0) return MOE_OK;
  // plan then forward on the same stream; each validates everything it reads
  // before enqueuing, and the forward's checks cannot fail for reasons the
  // plan's did not (same cfg and M), except its own buffers: checked first
  if (!y || !ws) return MOE_ERR_INVALID_ARG;
  if ((rc = check_weights(w13, MOE_LAYOUT_FRAGMENT_W13))) return rc;
  if ((rc = check_weights(w2, MOE_LAYOUT_FRAGMENT))) return rc;
  if (d.shared) {
    if ((rc = check_weights(shared13, MOE_LAYOUT_FRAGMENT_W13))) return rc;
    if ((rc = check_weights(shared2, MOE_LAYOUT_FRAGMENT))) return rc;
  }
  if (!aligned16(y) || !aligned16(ws)) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < ws_bytes_for(d, M)) return MOE_ERR_WORKSPACE;
  rc = moe_nvfp4_plan(cfg, M, x, w_router, bias, w_gate, ids, topk_w, plan, plan_bytes, status,
                      stream);
  if (rc) return rc;
  return moe_nvfp4_forward(cfg, M, x, plan, w13, w2, shared13, shared2, y, ws, ws_bytes, status,
                           stream);
}

// ---- dense few-row projections, channel-FP8 weights, prepared scales ----

static int32_t check_dense_shape(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || M > kDenseMaxTokens) return MOE_ERR_SHAPE;
  if (N < 256 || N > 65536 || N % 256) return MOE_ERR_SHAPE;
  if (K < 64 || K > 65536 || K % 64) return MOE_ERR_SHAPE;
  return MOE_OK;
}

int32_t moe_nvfp4_dense_query(int64_t M, int64_t N, int64_t K, size_t* ws_bytes) {
  int32_t rc = check_dense_shape(M, N, K);
  if (rc) return rc;
  if (!ws_bytes) return MOE_ERR_INVALID_ARG;
  *ws_bytes = dense_ws_bytes(M, N, K);
  return MOE_OK;
}

static int32_t dense_common(int fmt, int64_t M, int64_t N, int64_t K, const void* x,
                            const uint8_t* q, const uint8_t* s, const float* scale, void* y,
                            void* ws, size_t ws_bytes, uint32_t* status, void* stream) {
  int32_t rc = check_dense_shape(M, N, K);
  if (rc) return rc;
  if (M == 0) return MOE_OK;
  if (!x || !q || !scale || !y || (fmt != kDenseFp8 && !s)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(y) || (s && !aligned16(s)) ||
      !aligned16(scale))
    return MOE_ERR_ALIGNMENT;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_ALIGNMENT;
  const size_t need = dense_ws_bytes(M, N, K);
  if (need > 0 && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  if (ws && !aligned16(ws)) return MOE_ERR_ALIGNMENT;
  int sms = 0;
  rc = current_device(&sms);
  if (rc) return rc;
  return cuda_status(launch_dense(fmt, M, N, K, static_cast<const __half*>(x), q, s, scale, ws,
                                  static_cast<__half*>(y), status,
                                  static_cast<cudaStream_t>(stream)));
}

int32_t moe_nvfp4_dense(int64_t M, int64_t N, int64_t K, const void* x,
                        const moe_nvfp4_weights* w, void* y, void* ws, size_t ws_bytes,
                        uint32_t* status, void* stream) {
  if (!w || w->reserved) return MOE_ERR_INVALID_ARG;
  const int base = w->layout & ~MOE_SCALES_PREPARED;
  if (base != MOE_LAYOUT_FRAGMENT || (w->layout & ~(MOE_LAYOUT_FRAGMENT | MOE_SCALES_PREPARED)))
    return MOE_ERR_LAYOUT;
  const int fmt = (w->layout & MOE_SCALES_PREPARED) ? kDenseNvfp4Prepared : kDenseNvfp4;
  return dense_common(fmt, M, N, K, x, w->q, w->s, w->g, y, ws, ws_bytes, status, stream);
}

int32_t moe_fp8_dense(int64_t M, int64_t N, int64_t K, const void* x, const uint8_t* q,
                      const float* channel_scale, void* y, void* ws, size_t ws_bytes,
                      uint32_t* status, void* stream) {
  return dense_common(kDenseFp8, M, N, K, x, q, nullptr, channel_scale, y, ws, ws_bytes, status,
                      stream);
}

int32_t moe_fp8_quantize(const float* w, int64_t rows, int64_t k, int32_t layout, uint8_t* q,
                         float* channel_scale, uint32_t* status, void* stream) {
  if (!w || !q || !channel_scale) return MOE_ERR_INVALID_ARG;
  if (layout != MOE_LAYOUT_CANONICAL && layout != MOE_LAYOUT_FP8_FRAGMENT) return MOE_ERR_LAYOUT;
  if (rows < 1 || rows > (int64_t(1) << 24) || k < 64 || k > 65536 || k % 64)
    return MOE_ERR_SHAPE;
  if (layout == MOE_LAYOUT_FP8_FRAGMENT ? rows % 256 != 0 : rows % 16 != 0) return MOE_ERR_SHAPE;
  if (!aligned16(w) || !aligned16(q) || (reinterpret_cast<uintptr_t>(channel_scale) & 3u))
    return MOE_ERR_ALIGNMENT;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_ALIGNMENT;
  int sms = 0;
  int32_t rc = current_device(&sms);
  if (rc) return rc;
  return cuda_status(launch_fp8_quantize(w, rows, k, layout, q, channel_scale, status,
                                         static_cast<cudaStream_t>(stream)));
}

int32_t moe_nvfp4_prepare_scales(const uint8_t* s, int64_t n, void* s16, uint32_t* status,
                                 void* stream) {
  if (n < 0 || n > (int64_t(1) << 40)) return MOE_ERR_SHAPE;
  if (n == 0) return MOE_OK;
  if (!s || !s16) return MOE_ERR_INVALID_ARG;
  if (!aligned16(s) || !aligned16(s16)) return MOE_ERR_ALIGNMENT;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_ALIGNMENT;
  int sms = 0;
  int32_t rc = current_device(&sms);
  if (rc) return rc;
  return cuda_status(launch_prepare_scales(s, n, static_cast<uint16_t*>(s16), status,
                                           static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
