/*
 * moe_nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4-weight mixture-of-experts
 * layer: FP16 activations, E2M1 weights with one E4M3 scale per 16 elements
 * along K and one FP32 scale per tensor, FP32 accumulation.
 *
 * The layer, as described by the page "[Kernel][SM70] Improve Qwen3.8 no-MTP
 * concurrency" (section "Scope and related PRs"): a router, expert dispatch by
 * one integer plan shared by the grouped W13 and grouped W2 GEMMs, W13 (gate
 * and up projections) fused with SwiGLU, W2 fused with the weighted top-k
 * reduction, and an optional always-on shared expert scaled by a sigmoid gate.
 * Top-10 routing over 512 experts is the workload of "[Perf][SM70] Optimize
 * Qwen3.8 Flash Next prefill", section "SM70 QSA indexer hotspot update".
 *
 * Conventions common to every entry point
 * ---------------------------------------
 * - Pointers named "device" are CUDA device pointers owned by the caller and
 *   borrowed for the duration of the call's stream work; the library keeps no
 *   reference after the work completes.  The library allocates no memory.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   All GPU work is enqueued on it; no entry point synchronises the host, so
 *   every call may be captured in a CUDA graph.
 * - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  Arguments are
 *   validated on the host before anything is enqueued: on any error nothing
 *   is launched and no output is touched (fail closed).  No C++ exception
 *   crosses the ABI.
 * - `status` (device, uint32_t, may be NULL) collects asynchronous conditions
 *   as OR-ed MOE_ST_* bits.  The library never clears it: the caller zeroes it
 *   and reads it after synchronising.
 * - FP16 tensors are passed as `const void*` to raw IEEE binary16 data.
 * - Every device pointer must be 16-byte aligned (MOE_ERR_ALIGNMENT).
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_NVFP4_ABI_VERSION 1

/* ---- return codes ---- */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)        /* NULL where required, bad flag, M < 0 */
#define MOE_ERR_SHAPE (-2)              /* unsupported sizes (see each call) */
#define MOE_ERR_ALIGNMENT (-3)          /* a device pointer not 16-byte aligned */
#define MOE_ERR_WORKSPACE (-4)          /* plan or workspace buffer too small */
#define MOE_ERR_UNSUPPORTED_DEVICE (-5) /* current device is not compute capability 10.3 */
#define MOE_ERR_CUDA (-6)               /* a CUDA runtime call or launch failed */
#define MOE_ERR_LAYOUT (-7)             /* weights not in the layout the path needs */

/* ---- asynchronous status bits (OR-ed into *status on the device) ---- */
#define MOE_ST_INVALID_ID 0x1u /* a given expert id was outside [0, n_experts): pair dropped */
#define MOE_ST_NONFINITE 0x2u  /* quantiser input held NaN or infinity */
#define MOE_ST_TIMEOUT 0x4u    /* a bounded device-side wait gave up; outputs are invalid */

/* ---- configuration flags ---- */
#define MOE_FLAG_IDS_GIVEN 0x1u /* moe_nvfp4_plan: take ids and weights from the caller */
#define MOE_FLAG_SHARED 0x2u    /* the layer has a shared expert (gate w_g + shared MLP) */

/* ---- weight layouts (moe_nvfp4_quantize `layout`, moe_nvfp4_weights.layout) ----
 *
 * A quantised matrix has `rows` rows of `k` elements; n_mats matrices are
 * stored back to back.  Scales are E4M3 ("fn": 0x7F/0xFF NaN, max 448), one
 * per 16 consecutive elements of a row.
 *
 * MOE_LAYOUT_CANONICAL (0): q is [n_mats][rows][k/2] bytes, byte i of a row
 *   holding element 2i in its low nibble and element 2i+1 in its high nibble;
 *   s is [n_mats][rows][k/16].
 *
 * MOE_LAYOUT_FRAGMENT (1): rows % 256 == 0 and k % 64 == 0.  The matrix is cut
 *   into 16-row tiles rt (grouped 16 to a 256-row group G = rt / 16, j =
 *   rt % 16) and 64-element segments ks.  Tile rt, segment ks of matrix m owns
 *   the 512-byte q block number
 *       b = ((m * rows/256 + G) * k/64 + ks) * 16 + j
 *   (at byte 512 * b of q) and the 64-byte s block b (at byte 64 * b of s), so
 *   the 16 tiles of a group are contiguous for each segment.
 *   For L = 4*g + c (g = 0..7, c = 0..3): q block bytes [16L, 16L+8) are row
 *   16*rt+g, elements [64*ks+16*c, +16) in canonical byte order, and bytes
 *   [16L+8, 16L+16) the same elements of row 16*rt+g+8; s block bytes 2L and
 *   2L+1 are the scales of those two 16-element runs.  One warp reads one
 *   block with one 16-byte load per thread and holds an MMA operand fragment.
 *
 * MOE_LAYOUT_FRAGMENT_W13 (2): for a W13 matrix (rows = 2*I: rows 0..I-1 the
 *   gate projection, rows I..2I-1 the up projection; rows % 256 == 0): the
 *   fragment layout of the row-permuted matrix whose tile 2j is gate rows
 *   [16j, 16j+16) and tile 2j+1 is up rows [I+16j, I+16j+16).
 *
 * MOE_LAYOUT_FP8_FRAGMENT (3): channel-FP8 weights (moe_fp8_quantize,
 *   moe_fp8_dense), one E4M3 code per byte, rows % 256 == 0, k % 64 == 0.
 *   Tile rt, segment ks owns the 1024-byte block number
 *       b = (G * k/64 + ks) * 16 + j      (G = rt / 16, j = rt % 16)
 *   at byte 1024 * b; for L = 4*g + c, bytes [16L, 16L+16) are row 16*rt+g,
 *   elements [64*ks+16*c, +16) in ascending order, and bytes [512+16L,
 *   512+16L+16) the same elements of row 16*rt+g+8.  The canonical FP8 layout
 *   is [rows][k], one byte per element.
 *
 * MOE_SCALES_PREPARED (0x100, OR-ed into moe_nvfp4_weights.layout): `s` holds
 *   prepared scales (moe_nvfp4_prepare_scales): each E4M3 scale byte widened
 *   to the 2-byte FP16 bit pattern of its value, in the same order, so the
 *   scale array is twice as large.  Results are bitwise equal to raw scales.
 *
 * moe_nvfp4_forward needs W13 in layout 2 and W2 in layout 1 (either may add
 * MOE_SCALES_PREPARED); moe_nvfp4_dense needs layout 1 (+ prepared).
 */
#define MOE_LAYOUT_CANONICAL 0
#define MOE_LAYOUT_FRAGMENT 1
#define MOE_LAYOUT_FRAGMENT_W13 2
#define MOE_LAYOUT_FP8_FRAGMENT 3
#define MOE_SCALES_PREPARED 0x100

typedef struct moe_nvfp4_config {
  int32_t hidden;       /* H: model width; H % 256 == 0, 256 <= H <= 4096 */
  int32_t n_experts;    /* E: routed experts; E % 8 == 0, 8 <= E <= 512 */
  int32_t top_k;        /* k: experts per token; 1 <= k <= min(E, 32) */
  int32_t intermediate; /* I: expert intermediate size; I % 128 == 0, 128 <= I <= 4096 */
  uint32_t flags;       /* MOE_FLAG_* */
  int32_t reserved[3];  /* must be zero */
} moe_nvfp4_config;

/* One NVFP4 weight tensor set (device pointers).  For the routed experts the
 * arrays hold n_experts matrices back to back and g has n_experts entries; for
 * the shared expert they hold one matrix and g one entry. */
typedef struct moe_nvfp4_weights {
  const uint8_t* q; /* packed E2M1 codes, layout as above */
  const uint8_t* s; /* E4M3 block scales, layout as above */
  const float* g;   /* FP32 per-matrix global scale */
  int32_t layout;   /* MOE_LAYOUT_* */
  int32_t reserved; /* must be zero */
} moe_nvfp4_weights;

/* ABI capability check ("[SM70][Draft] Extend Qwen3.8 DFlash2 concurrency
 * paths", section "Purpose": a new native route is admitted only after a
 * native ABI capability check): returns MOE_NVFP4_ABI_VERSION.  Callers
 * refuse to use a library whose version differs from the header they were
 * built with.  Host-only; never fails. */
int32_t moe_nvfp4_abi_version(void);

/* Static text for a return code or a single MOE_ST_* bit; never NULL ("unknown
 * code" for anything else).  The codes are the outcomes of the host-side
 * metadata gates that fail closed ("[Kernel][SM70] Improve Qwen3.8 no-MTP
 * concurrency", section "Guarded production engine result": the CPU-integer
 * metadata hardening fails closed for tensor metadata; section "Test Result":
 * an unsafe launch request is refused rather than run).  Host-only. */
const char* moe_nvfp4_status_string(int32_t code);

/* Name of the CUDA runtime error behind the calling thread's most recent
 * MOE_ERR_CUDA return (for example "cudaErrorLaunchOutOfResources"), or ""
 * if no call on this thread has returned MOE_ERR_CUDA.  Static text; never
 * NULL.  The detail of one fail-closed outcome (same passages as
 * moe_nvfp4_status_string).  Host-only. */
const char* moe_nvfp4_last_cuda_error(void);

/* Sizes, in bytes, of the plan buffer (for moe_nvfp4_plan) and of the
 * forward workspace (for moe_nvfp4_forward) for any M <= max_tokens: the
 * workspace gate of the pages ("[SM70][Draft] Extend Qwen3.8 DFlash2
 * concurrency paths", section "Test Result": routing / workspace / ABI gates;
 * "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Scope and
 * related PRs": the plan and workspace are sized and owned outside the
 * kernels, and calls with too small a buffer fail closed).
 * Returns MOE_ERR_INVALID_ARG / MOE_ERR_SHAPE for a bad cfg or max_tokens
 * outside [0, 2^20].
 * Host-only arithmetic; also checks that the current device is an sm_103
 * part (MOE_ERR_UNSUPPORTED_DEVICE otherwise) unless `plan_bytes` and
 * `ws_bytes` are both NULL, in which case only `cfg` is validated.
 *
 * The first call of any entry point on a device that checks the device also
 * sets up the library's kernels there once (shared-memory limits, the
 * router's cluster size; MOE_ERR_CUDA if that fails, retried on the next
 * call).  The set-up is serialised across host threads and enqueues no work. */
int32_t moe_nvfp4_query(const moe_nvfp4_config* cfg, int64_t max_tokens, size_t* plan_bytes,
                        size_t* ws_bytes);

/* Quantises FP32 weights to NVFP4 (the layer's load-time step; the page
 * "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Scope and
 * related PRs", names native NVFP4 weights with raw E4M3 scale storage).
 *
 *   w      device FP32 [n_mats][rows][k], row-major.
 *   q      device out, n_mats*rows*k/2 bytes in `layout`.
 *   s      device out, n_mats*rows*k/16 bytes in `layout`.
 *   g      device out, FP32 [n_mats].
 * Per matrix, with every step one correctly rounded FP32 operation:
 *   g = amax / 2688 (6 * 448; g = 1 for an all-zero matrix),
 *   s = E4M3_rne_satfinite((amax_of_16_block / g) / 6),
 *   q = E2M1_rne_satfinite(x / (value(s) * g)), a zero keeping the sign of x
 *       (x / 0 is not formed: q = +-0 when value(s) * g == 0).
 * Requires k % 64 == 0, rows % 16 == 0 (rows % 256 == 0 for layouts 1, 2),
 * 1 <= n_mats, rows * k < 2^31.  NaN or infinite input sets MOE_ST_NONFINITE
 * in *status and is quantised as zero.  Uses `g` as scratch while running. */
int32_t moe_nvfp4_quantize(const float* w, int64_t n_mats, int64_t rows, int64_t k,
                           int32_t layout, uint8_t* q, uint8_t* s, float* g, uint32_t* status,
                           void* stream);

/* Router and routing plan (steps "router" and "one integer plan" of the page
 * "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Scope and
 * related PRs").
 *
 *   M        tokens, 0 <= M <= 2^20.  M == 0 returns MOE_OK at once, launching
 *            nothing and ignoring every buffer argument (which may be NULL).
 *   x        device FP16 [M][H].
 *   w_router device FP16 [H][E] (expert index fastest).
 *   bias     device FP32 [E] or NULL: added to the logits before selection.
 *   w_gate   device FP16 [H]; required with MOE_FLAG_SHARED, else ignored.
 *   ids      device int32 [M][k]: out (expert ids, descending logit, ties to
 *            the lower id) or, with MOE_FLAG_IDS_GIVEN, in.
 *   topk_w   device FP32 [M][k]: out (softmax of the selected logits) or, with
 *            MOE_FLAG_IDS_GIVEN, in.
 *   plan     device buffer of plan_bytes >= moe_nvfp4_query(...).plan_bytes
 *            for this M; its contents are private to the library.  It must be
 *            zero-filled once before its first use; the library leaves its
 *            internal counters at zero after every call.
 * Logits are FP32 sums of FP16 x FP16 products.  With MOE_FLAG_SHARED the
 * plan also holds gamma = sigmoid(x . w_g) and one extra pair per token for
 * the shared expert.  Given ids outside [0, E) are dropped from the plan and
 * set MOE_ST_INVALID_ID.  Plan calls on one plan buffer must not overlap on
 * the GPU. */
int32_t moe_nvfp4_plan(const moe_nvfp4_config* cfg, int64_t M, const void* x,
                       const void* w_router, const float* bias, const void* w_gate, int32_t* ids,
                       float* topk_w, void* plan, size_t plan_bytes, uint32_t* status,
                       void* stream);

/* The layer forward over a plan made by moe_nvfp4_plan with the same cfg and
 * M (steps "W13/SwiGLU fusion" and "W2/reduction fusion" of the same page):
 *
 *   y[t] = fp16( sum_{j<k} w[t,j] * MLP_{ids[t,j]}(x[t])  +  gamma_t * MLP_shared(x[t]) )
 *   MLP_e(x) = g2_e * W2_e . h,  h = fp16( silu(g13_e * W13_gate_e . x) * (g13_e * W13_up_e . x) )
 *
 * with FP32 accumulation and the slot sum in order j = 0..k-1, then the shared
 * term.  M <= 16 runs the weight-streaming GEMV path, larger M the grouped
 * tcgen05 GEMMs; both give the same results up to FP32 summation order.
 * M == 0 returns MOE_OK at once and ignores every buffer argument.
 *
 *   w13      routed W13, layout MOE_LAYOUT_FRAGMENT_W13, E matrices [2I][H].
 *   w2       routed W2, layout MOE_LAYOUT_FRAGMENT, E matrices [H][I].
 *            Either storage of the scales: raw E4M3, or prepared FP16 with
 *            MOE_SCALES_PREPARED OR-ed into every weight set's layout (all
 *            of them alike, else MOE_ERR_LAYOUT); the output is bitwise the
 *            same ("[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency",
 *            section "Test Result": raw and prepared outputs bitwise equal).
 *   shared13, shared2  shared expert (one matrix each, same layouts); required
 *            with MOE_FLAG_SHARED, else ignored.
 *   y        device FP16 [M][H] out.
 *   ws       device workspace of ws_bytes >= moe_nvfp4_query(...).ws_bytes.
 * Weight pointers need 16-byte alignment; q and s need the sizes above. */
int32_t moe_nvfp4_forward(const moe_nvfp4_config* cfg, int64_t M, const void* x, const void* plan,
                          const moe_nvfp4_weights* w13, const moe_nvfp4_weights* w2,
                          const moe_nvfp4_weights* shared13, const moe_nvfp4_weights* shared2,
                          void* y, void* ws, size_t ws_bytes, uint32_t* status, void* stream);

/* The whole layer in one call: moe_nvfp4_plan followed by moe_nvfp4_forward
 * on the same stream, with the same arguments and results (ids and topk_w
 * written, the plan buffer holding the plan, y the layer output).  The
 * forward's own buffers and weights are checked before the plan is enqueued,
 * so a call that fails launches nothing.  The pages' complete MoE call
 * ("[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Latest
 * grouped-MoE screen": the complete C16 call).  Returns the codes of
 * moe_nvfp4_plan and moe_nvfp4_forward. */
int32_t moe_nvfp4_layer(const moe_nvfp4_config* cfg, int64_t M, const void* x,
                        const void* w_router, const float* bias, const void* w_gate, int32_t* ids,
                        float* topk_w, void* plan, size_t plan_bytes, const moe_nvfp4_weights* w13,
                        const moe_nvfp4_weights* w2, const moe_nvfp4_weights* shared13,
                        const moe_nvfp4_weights* shared2, void* y, void* ws, size_t ws_bytes,
                        uint32_t* status, void* stream);

/* moe_nvfp4_forward without a workspace argument, for callers that cannot
 * allocate device memory (a host runtime that owns every allocation, a phase
 * in which a framework forbids allocation, a fixed C signature with no room
 * for a workspace).  The pages have no counterpart: this is an interface
 * addition of this library, not a step of the method.
 *
 * Same arguments, results and rules as moe_nvfp4_forward, except that the
 * workspace is a 4 MiB array inside the library (allocated when the library
 * is loaded and held by every GPU that loads it until the process exits).
 * Calls whose workspace would exceed it (M * k_eff * (2*I + 2*H) bytes plus
 * alignment) return MOE_ERR_WORKSPACE and launch nothing.  At H 2048, I 512,
 * top-10 that admits M <= 81 (M <= 16 on the decode kernels, above that the
 * grouped kernels); at small layers larger M fits (e.g. H 256, I 128, top-2:
 * M <= 2730).
 * The first call on a device looks the array's device address up
 * (cudaGetSymbolAddress) with that device current and keeps it for the life
 * of the process; make that first call before any stream capture.  A device
 * reset between calls is not supported.  All calls share the array and it
 * keeps the last call's contents (nothing in it needs to start at zero), so
 * calls whose GPU work overlaps race: order them on one stream.  Allocates
 * nothing. */
int32_t moe_nvfp4_forward_noalloc(const moe_nvfp4_config* cfg, int64_t M, const void* x,
                                  const void* plan, const moe_nvfp4_weights* w13,
                                  const moe_nvfp4_weights* w2, const moe_nvfp4_weights* shared13,
                                  const moe_nvfp4_weights* shared2, void* y, uint32_t* status,
                                  void* stream);

/* Dequantises NVFP4 matrices to FP16 (exact: every E2M1 x E4M3 product is an
 * FP16 value), applying no global scale.  q, s in `layout`; out FP16
 * [n_mats][rows][k] in canonical row order.  Same shape rules as
 * moe_nvfp4_quantize.  A diagnostic of the decode that every GEMM kernel
 * applies to its weight operand. */
int32_t moe_nvfp4_dequantize(const uint8_t* q, const uint8_t* s, int64_t n_mats, int64_t rows,
                             int64_t k, int32_t layout, void* out, void* stream);

/* Diagnostic kernel timing (no counterpart in the pages: a measurement aid).
 * With `events` non-NULL, every later plan and
 * forward call records events[2*i] on its stream just before and
 * events[2*i+1] just after step i, for i < n_steps:
 *   i = 0  the whole plan call (router and plan kernels),
 *   i = 1  the W13 kernel (decode GEMV or grouped tcgen05 GEMM),
 *   i = 2  the W2 kernel,
 *   i = 3  the combine kernel.
 * `events` are cudaEvent_t handles created by the caller (with timing
 * enabled).  The records are external event records, so a call captured in
 * a CUDA graph records them at every replay.  The records separate the kernels on the stream, so a traced call
 * does not overlap its kernels through programmatic dependent launch.  NULL
 * turns tracing off.  Process-wide setting; not thread-safe. */
int32_t moe_nvfp4_set_trace_events(void* const* events, int32_t n_steps);

/* ---- dense few-row projections (M <= 32) ------------------------------------
 *
 * The QPN2 / QPN8 projections of "[SM70][Draft] Extend Qwen3.8 DFlash2
 * concurrency paths" (section "Purpose": NVFP4 QPN2 in independent
 * eight-row tiles, admitted through M <= 32; section "TP4-only NVFP4 verifier
 * follow-up": split-K with the FP32 reduction order preserved, M9 / M15 / M16
 * bitwise equal to concatenated M8 calls; section "Follow-up: exact
 * channel-FP8 QPN8 concurrency paths": the same over FP8 weights with one
 * scale per output channel):
 *
 *   y[m][n] = fp16( scale_n * sum_k x[m][k] * w16[n][k] )
 *
 * with FP32 accumulation.  Every output row is computed by the same
 * operations whatever M is, so a call's rows are bitwise equal to the same
 * rows computed in any other batch.  Shapes: 0 <= M <= 32 (M == 0 returns
 * MOE_OK and touches nothing), N % 256 == 0 with 256 <= N <= 65536, K % 64 == 0
 * with 64 <= K <= 65536; anything else MOE_ERR_SHAPE (larger M belongs to a
 * GEMM, not to this weight-streaming path).  x is FP16 [M][K] and y FP16
 * [M][N], row-major, device, 16-byte aligned. */

/* Workspace bytes a dense call of this shape needs: 0 for every shape (each
 * block of the kernel owns whole 16-row output tiles over all of K, so no
 * partial sums are kept between blocks); the query and the ws arguments stay
 * so that callers need not change if a later kernel asks for one.
 * Host-only; MOE_ERR_SHAPE as above, MOE_ERR_INVALID_ARG for a NULL out. */
int32_t moe_nvfp4_dense_query(int64_t M, int64_t N, int64_t K, size_t* ws_bytes);

/* NVFP4 dense projection (QPN2).  w: one N x K matrix in MOE_LAYOUT_FRAGMENT
 * (optionally | MOE_SCALES_PREPARED), w->g one FP32 global scale (scale_n =
 * g for all n).  ws: device workspace of at least moe_nvfp4_dense_query bytes
 * (NULL when that is 0, as it is for every shape), borrowed for the call's
 * stream work.  Returns MOE_ERR_LAYOUT for another layout, MOE_ERR_WORKSPACE
 * for a short ws, MOE_ERR_ALIGNMENT / MOE_ERR_INVALID_ARG as usual.  Bounded
 * device waits set MOE_ST_TIMEOUT in *status if they give up. */
int32_t moe_nvfp4_dense(int64_t M, int64_t N, int64_t K, const void* x,
                        const moe_nvfp4_weights* w, void* y, void* ws, size_t ws_bytes,
                        uint32_t* status, void* stream);

/* Channel-FP8 quantiser (the load-time step of QPN8, same section).  w:
 * device FP32 [rows][k]; q: device out, rows * k E4M3 codes in `layout`
 * (MOE_LAYOUT_CANONICAL: [rows][k]; MOE_LAYOUT_FP8_FRAGMENT: as above);
 * channel_scale: device out FP32 [rows].  Per row, every step one correctly
 * rounded FP32 operation: cs = amax / 448 (1 for an all-zero row),
 * q = E4M3_rne_satfinite(x / cs).  NaN or infinite input is quantised as zero
 * and sets MOE_ST_NONFINITE.  Requires k % 64 == 0 (64 <= k <= 65536),
 * rows % 16 == 0 (rows % 256 == 0 for the fragment layout). */
int32_t moe_fp8_quantize(const float* w, int64_t rows, int64_t k, int32_t layout, uint8_t* q,
                         float* channel_scale, uint32_t* status, void* stream);

/* Channel-FP8 dense projection (QPN8): q is N x K in MOE_LAYOUT_FP8_FRAGMENT,
 * channel_scale FP32 [N] (scale_n), applied to the FP32 sum.  Otherwise as
 * moe_nvfp4_dense. */
int32_t moe_fp8_dense(int64_t M, int64_t N, int64_t K, const void* x, const uint8_t* q,
                      const float* channel_scale, void* y, void* ws, size_t ws_bytes,
                      uint32_t* status, void* stream);

/* Prepared-scale storage ("[Kernel][SM70] Improve Qwen3.8 no-MTP
 * concurrency", sections "Purpose" and "Scope and related PRs": prepared
 * effective decode scales beside raw E4M3 scale residency; section "Test
 * Result": raw and prepared outputs bitwise equal).  s16[i] = the FP16 bit
 * pattern of E4M3 code s[i], for i < n, in the same order (any layout).  The
 * NaN codes 0x7F / 0xFF give 0x7E00 and set MOE_ST_NONFINITE.  s: device n
 * bytes; s16: device out, 2n bytes; both 16-byte aligned.  n == 0 returns
 * MOE_OK. */
int32_t moe_nvfp4_prepare_scales(const uint8_t* s, int64_t n, void* s16, uint32_t* status,
                                 void* stream);

/* Diagnostic router selection for M <= 16 (no counterpart in the pages; a test
 * aid).  mode 0: automatic (one thread-block cluster when the device can
 * co-schedule it, else the 128-block router); mode 1: always the 128-block
 * router with arrival tickets, the fallback of devices where a cluster of 8
 * CTAs cannot be scheduled.  Both give bit-identical ids, weights and plans.
 * Process-wide; takes effect at the next moe_nvfp4_plan call; not
 * thread-safe.  Returns MOE_ERR_INVALID_ARG for another mode. */
int32_t moe_nvfp4_set_small_router(int32_t mode);

/* Failure-path test switch (no counterpart in the pages beyond their safe
 * fallback of an unsafe launch: "[Kernel][SM70] Improve Qwen3.8 no-MTP
 * concurrency", section "Test Result").  With hold_raw_producer = 1 the
 * grouped W13 kernel (the forward at M > 16) issues none of its raw weight
 * copies, so its consumers' bounded waits run out: they set MOE_ST_TIMEOUT in
 * *status, stop, let copies in flight land, free tensor memory and return;
 * the output is then invalid, the context stays usable.  wait_limit_cycles
 * sets the grouped GEMMs' wait limit in SM clock cycles (<= 0: the default,
 * 4e8 ~ 200 ms).  Set on the current device through `stream`, synchronously;
 * process-wide; call with (0, 0) to restore.  MOE_ERR_INVALID_ARG for another
 * hold value. */
int32_t moe_nvfp4_set_wait_test(int32_t hold_raw_producer, int64_t wait_limit_cycles,
                                void* stream);

/* Diagnostic M bucket of moe_nvfp4_forward (no counterpart in the pages' text
 * beyond their M-bucketed dispatch: "[Kernel][SM70] Improve Qwen3.8 no-MTP
 * concurrency", section "Scope and related PRs", dynamic M2-M16 dispatch; a
 * measurement aid).  Calls with M <= m run the weight-streaming decode
 * kernels, larger M the grouped tensor-core GEMMs; 0 <= m <= 16 (default 16,
 * the measured crossover), else MOE_ERR_INVALID_ARG.  Both give results
 * within the acceptance bar of each other.  Process-wide; not thread-safe. */
int32_t moe_nvfp4_set_decode_max_tokens(int32_t m);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
