// Shared device helpers of the NVFP4 MoE library: status bits, the plan
// buffer layout, and thin inline-PTX wrappers for sm_103a (mbarrier, bulk
// and per-thread async copies, tcgen05, programmatic dependent launch).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_nvfp4.h"

namespace moe {

constexpr int kDecodeMaxTokens = 16;     // M <= this runs the streaming GEMV path
constexpr int kTileRows = 192;           // plan tile height (N of the grouped MMAs)
constexpr int kPlanChunk = 2048;         // pairs per histogram block in the plan
constexpr int kRouterChunk = 8192;       // tokens per large-M router logits pass
constexpr uint64_t kWaitTimeoutNs = 200ull * 1000 * 1000;  // bounded spins: 200 ms
// The same bound in SM clock cycles, for spins that time themselves with the
// SM-local cycle counter (cheap to read): 200 ms at 2 GHz, longer if slower.
constexpr long long kWaitTimeoutCycles = 400ll * 1000 * 1000;
// Decode work table entry (one per active expert, M <= 16): expert, first plan
// position, rows, then the pair id of each of the first 16 rows; entries past
// the active experts hold expert -1.
constexpr int kDtabInts = 20;
constexpr int kDtabEntries = kDecodeMaxTokens * 33;

// ---------------------------------------------------------------------------
// Plan buffer: a header followed by int32/float arrays, all carved by
// plan_layout() on the host and re-derived identically on the device.
// ---------------------------------------------------------------------------
struct PlanHeader {
  int32_t M;          // tokens
  int32_t k_eff;      // slots per token (top_k, +1 with a shared expert)
  int32_t e_eff;      // experts in the plan (n_experts, +1 with a shared expert)
  int32_t n_active;   // experts with at least one pair
  int32_t n_tiles;    // tiles of at most kTileRows rows
  int32_t n_valid;    // pairs with a valid expert id
  int32_t pad[10];
};

struct PlanView {
  PlanHeader* hdr;
  int32_t* ids;       // [M][k_eff] expert of each pair (slot k = shared expert)
  float* w;           // [M][k_eff] combine weight of each pair (slot k = gamma)
  int32_t* counts;    // [e_eff]
  int32_t* offsets;   // [e_eff + 1]
  int32_t* active;    // [e_eff] experts with count > 0, ascending
  int32_t* perm;      // [M * k_eff] plan position -> pair id
  int32_t* inv;       // [M * k_eff] pair id -> plan position, -1 if dropped
  int32_t* tiles;     // [max_tiles][4] (expert, first row, rows, first plan position)
  int32_t* chunk_hist;// [n_chunks][e_eff] scratch of the large-M plan
  int32_t* rank;      // [M * k_eff] scratch: rank of a pair inside its chunk
  float* partial;     // [n_hchunks][kDecodeMaxTokens][n_experts] scratch (128-block router)
  float* logits;      // [kDecodeMaxTokens][n_experts] scratch (128-block router)
  uint32_t* tickets;  // [64] self-resetting arrival counters of the 128-block small-M
                      // router: [0, 8) expert slices, 63 finaliser
  int32_t* dtab;      // [kDecodeMaxTokens * 33][kDtabInts] decode work table (M <= 16)
  float* rlogits;     // [min(M, kRouterChunk)][n_experts] router logits (M > 16)
  __half* wrt;        // [n_experts][hidden] transposed router weight (M > 16)
  float* rpart;       // [ksplit][M][n_experts] partial logits of the split mma.sync router
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// K splits of the mma.sync router (M > 16 where the tensor-core router does
// not run: E < 256, E % 16 != 0 or M < 128): enough 32-row K splits that
// token tiles of 64 x splits fill ~128 SMs; 1 = no split (top-k in the
// router's epilogue).  The same for every call with this M, H, E.
constexpr int kRouterSplitRows = 32;
__host__ __device__ inline int router_ksplit(int64_t M, int H, int E) {
  if (M <= kDecodeMaxTokens) return 1;
  if (E >= 256 && E % 16 == 0 && M >= 128) return 1;  // tensor-core router
  const int64_t tiles = (M + 63) / 64;
  int64_t s = (128 + tiles - 1) / tiles;
  const int64_t smax = H / kRouterSplitRows;
  if (s > smax) s = smax;
  return s < 1 ? 1 : (int)s;
}

__host__ __device__ inline int max_tiles_for(int64_t pairs, int e_eff) {
  return (int)(e_eff + (pairs + kTileRows - 1) / kTileRows);
}

// Carves a plan buffer starting at `base` (nullptr => sizes only).  Returns
// the number of bytes used.
__host__ __device__ inline size_t plan_layout(char* base, int64_t M, int k_eff, int e_eff,
                                              int n_experts, int hidden, PlanView* v) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off = align_up(off + bytes, 256);
    return p;
  };
  int64_t P = M * k_eff;
  int64_t Pc = P > 0 ? P : 1;
  int n_chunks = (int)((Pc + kPlanChunk - 1) / kPlanChunk);
  int n_hchunks = (hidden + 127) / 128;
  PlanView t;
  t.hdr = (PlanHeader*)take(sizeof(PlanHeader));
  t.tickets = (uint32_t*)take(64 * sizeof(uint32_t));
  t.ids = (int32_t*)take(sizeof(int32_t) * Pc);
  t.w = (float*)take(sizeof(float) * Pc);
  t.counts = (int32_t*)take(sizeof(int32_t) * e_eff);
  t.offsets = (int32_t*)take(sizeof(int32_t) * (e_eff + 1));
  t.active = (int32_t*)take(sizeof(int32_t) * e_eff);
  t.perm = (int32_t*)take(sizeof(int32_t) * Pc);
  t.inv = (int32_t*)take(sizeof(int32_t) * Pc);
  t.tiles = (int32_t*)take(sizeof(int32_t) * 4 * max_tiles_for(P, e_eff));
  t.chunk_hist = (int32_t*)take(sizeof(int32_t) * (size_t)n_chunks * e_eff);
  t.rank = (int32_t*)take(sizeof(int32_t) * Pc);
  t.partial = (float*)take(sizeof(float) * (size_t)n_hchunks * kDecodeMaxTokens * n_experts);
  t.logits = (float*)take(sizeof(float) * (size_t)kDecodeMaxTokens * n_experts);
  t.dtab = (int32_t*)take(sizeof(int32_t) * kDtabEntries * kDtabInts);
  const int64_t Mr = M > kDecodeMaxTokens ? (M < kRouterChunk ? M : kRouterChunk) : 0;
  t.rlogits = (float*)take(sizeof(float) * (size_t)Mr * n_experts);
  t.wrt = (__half*)take(Mr > 0 ? sizeof(__half) * (size_t)n_experts * hidden : 0);
  const int ks = router_ksplit(M, hidden, n_experts);
  t.rpart = (float*)take(ks > 1 ? sizeof(float) * (size_t)ks * M * n_experts : 0);
  if (v) *v = t;
  return off;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- timeline instrumentation (built only with -DMOE_TIMELINE) -------------
// Per kernel slot: [0] earliest block start, [1] earliest block past its
// programmatic-launch wait, [2] latest block end, [3] blocks that ran.  Read
// with moe_nvfp4_timeline_read() in that build; compiled out otherwise.
enum TimelineSlot { kTlRouter = 0, kTlPlan = 1, kTlW13 = 2, kTlW2 = 3, kTlCombine = 4 };
#ifdef MOE_TIMELINE
extern __device__ unsigned long long g_timeline[64];
struct TlScope {
  int slot;
  __device__ explicit TlScope(int s) : slot(s) {
    if (threadIdx.x == 0) {
      atomicMin(&g_timeline[4 * s], (unsigned long long)globaltimer());
      atomicAdd(&g_timeline[4 * s + 3], 1ull);
    }
  }
  __device__ void waited() const {
    if (threadIdx.x == 0) atomicMin(&g_timeline[4 * slot + 1], (unsigned long long)globaltimer());
  }
  __device__ ~TlScope() {
    if (threadIdx.x == 0) atomicMax(&g_timeline[4 * slot + 2], (unsigned long long)globaltimer());
  }
};
#define MOE_TL(slot) ::moe::TlScope tl_scope_(slot)
#define MOE_TL_WAITED() tl_scope_.waited()
// per-role cycle accounting of the grouped GEMM (summed over blocks)
extern __device__ unsigned long long g_prof[32];
// per-event clock64 stamps of block 0 of the grouped GEMM (timeline build),
// 2048 per kind: [0] MMA K step issued, [1] B stage seen ready by the MMA
// thread, [2] A stage seen ready, [3] / [4] dequantise start / end (K step x 8
// + warp), [5] B stage loads issued, [6] raw stage issued, [7] epilogue
// accumulator seen ready / epilogue done (2 x unit, 2 x unit + 1), [8] raw
// stage landed, [9] B stage landed
extern __device__ unsigned long long g_dbg[20480];
#define MOE_DBG(slot, idx)                                                   \
  do {                                                                        \
    if (blockIdx.x == 0 && (idx) < 2048) g_dbg[(slot) * 2048 + (idx)] = clock64(); \
  } while (0)
#define MOE_PROF(stmt) stmt
// raw stamps on timeline cells 20..63 (earliest / latest over the threads that pass)
#define MOE_TL_MIN(cell) atomicMin(&::moe::g_timeline[cell], (unsigned long long)::moe::globaltimer())
#define MOE_TL_MAX(cell) atomicMax(&::moe::g_timeline[cell], (unsigned long long)::moe::globaltimer())
#else
#define MOE_DBG(slot, idx) \
  do {                     \
  } while (0)
#define MOE_PROF(stmt)
#define MOE_TL_MIN(cell) \
  do {                   \
  } while (0)
#define MOE_TL_MAX(cell) \
  do {                   \
  } while (0)
#define MOE_TL(slot) \
  do {               \
  } while (0)
#define MOE_TL_WAITED() \
  do {                  \
  } while (0)
#endif

// ---- mbarrier ------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete.  Gives up after
// kWaitTimeoutNs, sets MOE_ST_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > kWaitTimeoutCycles) {
      set_status(status, MOE_ST_TIMEOUT);
      return false;
    }
  }
}

// ---- copies ---------------------------------------------------------------
// One bulk (TMA-engine) copy global -> shared, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// One 2-D tiled TMA load of the box at (x, y) (x in elements of the map)
// into shared memory, completing on `bar`.  `map` is a kernel parameter.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// One 3-D tiled TMA load of the box at (x, y, z) into shared memory.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// 16-byte per-thread async copy; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// Arrives on `bar` (without changing its expected count) once every cp.async
// this thread issued before has landed.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---- programmatic dependent launch -----------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Starts an HBM -> L2 transfer of [p, p + bytes) (16-byte aligned, bytes a
// multiple of 16) on the TMA engine; no completion is tracked.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- NVFP4 decode ----------------------------------------------------------
// Byte b (0..3, a compile-time constant at every call) of w, zero-extended,
// with one byte permute.
__device__ __forceinline__ uint32_t byte_of(uint32_t w, int b) {
  return __byte_perm(w, 0u, 0x4440u | (uint32_t)b);
}
// Two E2M1 codes (low nibble -> low half) to an FP16 pair.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n"
      : "=r"(r)
      : "r"(byte));
  return r;
}
// Two E4M3 codes (low byte -> low half) to an FP16 pair.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
      : "=r"(r)
      : "r"(two));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Dequantises 8 E2M1 codes held in `word` (element 0 in the low nibble) with
// the FP16 scale splat in `sc2`; returns 4 FP16 pairs.  Exact: every product
// of an E2M1 value and an E4M3 value is representable in FP16.
__device__ __forceinline__ void dequant8(uint32_t word, uint32_t sc2, uint32_t out[4]) {
#pragma unroll
  for (int b = 0; b < 4; ++b) out[b] = hmul2_u32(e2m1x2_to_f16x2(byte_of(word, b)), sc2);
}

// Dequantised A fragment of k-step `s` (0..3) of a 16x64 fragment-layout block:
// q = {row g codes 0-7, row g codes 8-15, row g+8 codes 0-7, row g+8 codes 8-15}
// of this thread's 16-element run; sg / sg8 the FP16 scale splats.  The
// m16n8k16 K index 2c + {0, 1} (c = lane % 4) holds element 16c + 4s + {0, 1}
// of the run and 2c + 8 + {0, 1} element 16c + 4s + {2, 3}; the B operand
// (token rows) is read in the same K order.
__device__ __forceinline__ void a_frag(const uint4& q, uint32_t sg, uint32_t sg8, int s,
                                       uint32_t a[4]) {
  const uint32_t wg = (s < 2) ? q.x : q.y;
  const uint32_t wg8 = (s < 2) ? q.z : q.w;
  const int sh = 16 * (s & 1);
  const int b0 = sh >> 3;
  a[0] = hmul2_u32(e2m1x2_to_f16x2(byte_of(wg, b0)), sg);
  a[2] = hmul2_u32(e2m1x2_to_f16x2(byte_of(wg, b0 + 1)), sg);
  a[1] = hmul2_u32(e2m1x2_to_f16x2(byte_of(wg8, b0)), sg8);
  a[3] = hmul2_u32(e2m1x2_to_f16x2(byte_of(wg8, b0 + 1)), sg8);
}

// FP16 scale splats of rows g (sg) and g + 8 (sg8) from their two E4M3 codes
// (row g in the low byte).
__device__ __forceinline__ void scale_splats(uint32_t sc16, uint32_t* sg, uint32_t* sg8) {
  const uint32_t f = e4m3x2_to_f16x2(sc16);
  *sg = __byte_perm(f, f, 0x1010);
  *sg8 = __byte_perm(f, f, 0x3232);
}

// The same from two prepared FP16 scales (row g in the low half).
__device__ __forceinline__ void scale_splats_f16(uint32_t f, uint32_t* sg, uint32_t* sg8) {
  *sg = __byte_perm(f, f, 0x1010);
  *sg8 = __byte_perm(f, f, 0x3232);
}

// ---- legacy warp MMA (decode GEMV and small router) --------------------------
__device__ __forceinline__ void mma_16816(float c[4], const uint32_t a[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---- tcgen05 -----------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, issued by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16, issued by one thread: A is
// read from tensor memory (lane m = row m, column j = K elements 2j, 2j+1).
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 32 columns of 32-bit TMEM cells: thread i of the warp receives
// lane (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t v[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 lanes x 32 columns of 32-bit TMEM cells from the warp's registers, in the
// layout of the mma.sync accumulator fragment repeated along the columns:
// thread 4g + c writes, for repetition r (columns [8r, 8r + 8)), lane g columns
// 8r + 2c and 8r + 2c + 1 from r[4r], r[4r + 1] and lane g + 8 the same two
// columns from r[4r + 2], r[4r + 3].  `taddr` carries the first lane (the
// warp's lane quadrant or its upper half) and the first column.
__device__ __forceinline__ void tmem_st16x256_x4(uint32_t taddr, const uint32_t r[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
// Waits until this thread's tensor-memory stores have completed.
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand with the 128-byte swizzle:
// rows of 128 bytes (64 FP16 along K), 8-row groups 1024 bytes apart.  The
// tile must start on a 1024-byte boundary.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                      // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                      // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                      // swizzle mode: 128-byte
  return d;
}
// Instruction descriptor of kind::f16: FP16 A and B (both K-major), FP32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                      // D format F32
         | (0u << 7) | (0u << 10)       // A, B format F16
         | ((uint32_t)(N >> 3) << 17)   // N / 8
         | ((uint32_t)(M >> 4) << 24);  // M / 16
}
// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128B-swizzled,
// K-major tile of 128-byte rows.
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c) {
  return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

}  // namespace moe
