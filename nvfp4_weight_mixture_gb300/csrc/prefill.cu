// Prefill path (M > 16): expert-grouped GEMMs on the 5th-generation tensor
// cores (tcgen05, kind::f16, FP32 accumulators in tensor memory).
//
// "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Scope and
// related PRs": grouped W13 with SwiGLU and grouped W2 with the reduction,
// both driven by the same integer plan.  A work unit is one plan tile (one
// expert, up to 192 of its routed rows) times a block of weight rows:
//
//   D[weight row][token] = sum_k W[weight row][k] * X[token][k]     (swap-AB)
//
// so the weight rows are the MMA's M = 128 and the tokens are N (<= 192).  The
// dequantised weights (A) go to tensor memory (`tcgen05.st`), not shared
// memory, which leaves the shared-memory bandwidth to the token rows (B) and
// the raw weights.  Blocks are persistent (one per SM) and walk the units with
// a static stride; each role runs ahead as far as its ring allows.
//
// grouped_w13_kernel: units of 256 weight rows (two A tiles, gate and up
// interleaved); tensor memory holds the two accumulators (2 x 192 columns)
// and two A stages of one K step (2 x 64 columns).  Warp roles:
//   warp 13    one lane streams the unit's raw NVFP4 blocks (fragment layout:
//              16 blocks of 512 + 64 bytes per K step of 64) into a shared
//              ring with two bulk asynchronous copies per K step;
//   warps 0-7  dequantise each raw stage into tensor memory (two fragment
//              blocks per warp: warp w owns lanes 32 (w % 4) .. +31 of A tile
//              w / 4, the lanes its sub-partition may access), then run the
//              unit's SwiGLU epilogue on the same lanes of accumulator w / 4,
//              staging the unit's h in shared memory and releasing tensor
//              memory right after their last read;
//   warp 8     one lane fills the token-row operand, one ring stage per K step
//              (128-byte swizzled, K-major), with 64-row tensor-map loads of
//              the token rows gathered into plan order beforehand;
//   warps 9-11 write each unit's staged h rows out (whole 256-byte token
//              rows), while the dequantising warps go on with the next unit;
//   warp 12    allocates tensor memory; one lane issues the MMAs: per K step
//              one wait (A and B stages share one barrier), then per A tile and
//              16-element K slice one MMA with N = all of the unit's rows, then
//              one commit that frees both stages.
// grouped_w2_kernel (further below): units of 128 output rows with
// double-buffered accumulators and separate epilogue warps.
//
// K order inside each 64-element K step.  A warp's dequantised values sit in
// the mma.sync fragment order (thread 4g + c: rows g, g + 8, elements
// [16c, 16c + 16)), and the 16x256b tensor-memory store puts that thread's
// 4-element group r at K positions [16r + 4c, 16r + 4c + 4).  So position
// 16r + 4c + e of A holds element 16c + 4r + e; the token-row operands are
// written in the same order (the row gather for W13, the W13 epilogue for
// h), and the products pair up as in the natural order.
//
// W13: the fragment layout interleaves 16-row gate and up tiles, so TMEM lanes
// [32q, 32q+16) hold gate rows and [32q+16, 32q+32) the matching up rows; the
// epilogue pairs them with one shuffle and writes h = fp16(silu(G) * U).
// W2:  the epilogue scales the FP32 sums by g2 and the pair's combine weight
// and writes each pair's partial row, rounded to FP16 (the activations' type),
// at its plan position (rows of a unit are consecutive); a separate pass adds
// each token's slots in order in FP32.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBK = 64;                   // K per step (128 bytes of FP16)
constexpr int kAS = 2;                    // A (dequantised) stages in tensor memory
constexpr int kBChunkRows = 64;           // rows per tensor-map load: 64 token rows x 128 bytes
constexpr int kBChunk = kBChunkRows * 128;
constexpr int kBStage = kTileRows * 128;  // B ring stage: one K step of up to 192 rows
constexpr int kBStages = 4;               // B ring stages (96 KiB)
constexpr int kRS = 8;                    // raw weight stages
constexpr int kRawQ = 16 * 512;           // raw q bytes per K step (16 fragment blocks)
// + their scales: 16 x 64 bytes raw E4M3, 16 x 128 bytes prepared FP16
constexpr int kRawBytes = kRawQ + 16 * 128;
// Warp roles: 0-7 dequantise and run the epilogue, 8 fills the token-row
// operand, 9-11 write the staged h rows out, 12 issues the MMAs (and owns
// tensor memory), 13 streams raw weights.
constexpr int kDqWarps = 8;
constexpr int kBWarp0 = 8;
constexpr int kOutWarp0 = 9;
constexpr int kOutWarps = 3;
constexpr int kMmaWarp = 12;
constexpr int kRawWarp = 13;
constexpr int kGemmThreads = 14 * 32;
// Tensor memory: accumulator t at column t * kTileRows, A stage s, tile t at
// column kAOff + s * 64 + t * 32 (64 FP16 of K per row = 32 columns).
constexpr int kTmemCols = 512;
constexpr int kAOff = 2 * kTileRows;
static_assert(kAOff + kAS * 2 * (kBK / 2) <= kTmemCols, "tensor memory over-committed");
static_assert(kTileRows % kBChunkRows == 0 && kTileRows % 16 == 0 && kTileRows <= 256,
              "plan tile height must be a multiple of 64 and a valid MMA N");
constexpr int kOffB = 0;
constexpr int kOffRaw = kOffB + kBStages * kBStage;
constexpr int kOffMeta = kOffRaw + kRS * kRawBytes;
static_assert(kBStage % 1024 == 0, "B stages must stay 1024-byte aligned for the swizzle");
static_assert(kBStages % kAS == 0 && kBStages >= 2 * kAS,
              "one barrier per K step serves both rings: B ring a multiple of, and at least twice, the A ring");

constexpr int kHStageHalfs = kTileRows * 16 + 16;

struct GemmSmem {
  uint64_t raw_full[kRS], raw_empty[kRS];
  // K step k: full[k % kBStages] completes when A stage k % kAS is in tensor
  // memory (one arrival per dequantising warp) and B stage k % kBStages has
  // landed (the loading thread's arrival plus the transaction bytes); the MMA
  // thread commits K step k to empty[k % kBStages], which frees both.
  uint64_t full[kBStages], empty[kBStages];
  uint64_t accf, tmem_empty, drain;
  // W13 epilogue, once per unit: every dequantising warp has staged its tile
  // of the unit's h (ep_staged) / the output warps have written the unit's
  // token rows out (ep_free)
  uint64_t ep_staged, ep_free;
  uint32_t tmem;
  int abort;
  int n_units;
  // epilogue staging of a whole unit: per dequantising warp h values
  // [kTileRows tokens][16 i] (FP16); the 32-byte pad after each tile makes
  // the output warps' 8-byte reads of one half-warp hit 32 different banks
  __align__(16) __half hstage[kDqWarps][kHStageHalfs];
};

constexpr size_t gemm_smem_bytes() {
  return 1024 /* alignment slack */ + (size_t)kOffMeta + sizeof(GemmSmem);
}
static_assert(gemm_smem_bytes() <= 232448, "grouped GEMM shared memory above the sm_103 limit");

// Wait limit of the grouped GEMMs' bounded waits (SM cycles) and a test switch
// that holds back W13's raw-weight producer (so that its consumers' waits run
// out): both set only by moe_nvfp4_set_wait_test; the defaults are the
// library's 200 ms bound and no hold.
static __device__ long long g_pf_wait_limit = kWaitTimeoutCycles;
static __device__ int g_pf_hold_raw = 0;

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* status,
                                              volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > g_pf_wait_limit) {
      set_status(status, MOE_ST_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// Waits (bounded by the same limit) for a phase whose completion is only
// awaited so that copies in flight land before the block leaves.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < g_pf_wait_limit) {
  }
}

// Every lane of the warp waits; the outcome is made the same for the whole
// warp (the tensor-memory instructions that follow are warp-wide, so the
// warp goes on, or leaves after an abort, together).
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t* bar, uint32_t parity,
                                                   uint32_t* status, volatile int* abort) {
  return __all_sync(0xffffffffu, wait_or_abort(bar, parity, status, abort));
}

// Profiling cells (timeline build): [0..1] raw producer wait/issue, [2..3]
// MMA thread total / unit bookkeeping, [4..7]
// MMA wait-A / wait-B / issue / wait-TMEM, [8..9] B wait/issue, [10..14]
// dequant wait-raw / wait-A / work, epilogue wait / work (W13); W2 at 16 + the
// same offsets.
// Each thread sums its cells in registers and adds them to g_prof once, at
// exit, so that no global atomic sits inside a pipeline loop.
#ifdef MOE_TIMELINE
#define PROF_ADD(cell, t0) (pacc[(cell) - poff] += (unsigned long long)(clock64() - (t0)))
#else
#define PROF_ADD(cell, t0)
#endif

struct Unit {
  int e, rows, npad, sub, pos0;
  const uint8_t* q;  // the expert's q bytes
  const uint8_t* s;  // the expert's s bytes
  float g;
};

// Scale storage: SB = 1 raw E4M3 bytes, SB = 2 prepared FP16 scales (every
// scale offset doubles; the two scales of a fragment lane become one 32-bit word).
template <int SB>
__device__ __forceinline__ uint32_t lane_scale_word(const char* p) {
  if constexpr (SB == 1)
    return *reinterpret_cast<const unsigned short*>(p);
  else
    return *reinterpret_cast<const uint32_t*>(p);
}
template <int SB>
__device__ __forceinline__ uint32_t lane_scale_f16x2(uint32_t v) {
  if constexpr (SB == 1)
    return e4m3x2_to_f16x2(v);
  else
    return v;
}

// The tile entry of unit u (all zero past the last unit).  Every role walks
// the units u = blockIdx.x, + gridDim.x, ... and loads the entry of its next
// unit while it works on the current one, so that the entry's L2 latency
// hides behind the unit instead of stalling the role at each unit boundary.
__device__ __forceinline__ int4 unit_tile(const PlanView& pv, int u, int upt, int n_units) {
  return u < n_units ? __ldcg(reinterpret_cast<const int4*>(pv.tiles) + u / upt)
                     : make_int4(0, 0, 0, 0);
}

// Unit u from its tile entry tl = (expert, first row, rows, first plan
// position); nxt receives the entry of the role's next unit.
template <bool kW13, int SB>
__device__ __forceinline__ Unit load_unit(const LayerDims& d, const PlanView& pv, Weights w,
                                          Weights ws, int u, int upt, int n_units, int4& nxt) {
  Unit un;
  const int4 tl = nxt;
  nxt = unit_tile(pv, u + (int)gridDim.x, upt, n_units);
  un.sub = u - (u / upt) * upt;
  un.e = tl.x;
  un.rows = tl.z;
  un.npad = (tl.z + 15) & ~15;
  un.pos0 = tl.w;
  const bool sh = (un.e == d.E);
  const size_t mat_q = kW13 ? (size_t)d.I * d.H : (size_t)d.H * d.I / 2;
  un.q = sh ? ws.q : w.q + (size_t)un.e * mat_q;
  un.s = sh ? ws.s : w.s + (size_t)un.e * mat_q / 8 * SB;
  un.g = sh ? ws.g[0] : w.g[un.e];
  return un;
}

template <int SB>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_w13_kernel(LayerDims d, PlanView pv, const __grid_constant__ CUtensorMap bmap,
                       Weights w, Weights ws, __half* __restrict__ h_out, uint32_t* status) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  GemmSmem* sm = reinterpret_cast<GemmSmem*>(base + kOffMeta);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  MOE_TL(kTlW13);
  MOE_PROF(constexpr int poff = 0);
  MOE_PROF(unsigned long long pacc[15] = {});

  const int K = d.H;                        // reduction length
  const int S = K / kBK;                     // K steps per unit
  const int upt = (2 * d.I) / 256;          // units per plan tile

  if (tid == 0) {
    for (int i = 0; i < kRS; ++i) {
      mbar_init(&sm->raw_full[i], 1);
      mbar_init(&sm->raw_empty[i], kDqWarps);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&sm->full[i], kDqWarps + 1);
      mbar_init(&sm->empty[i], 1);
    }
    mbar_init(&sm->accf, 1);
    mbar_init(&sm->tmem_empty, kDqWarps);
    mbar_init(&sm->ep_staged, kDqWarps);
    mbar_init(&sm->ep_free, kOutWarps);
    mbar_init(&sm->drain, 1);
    sm->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&sm->tmem, kTmemCols);
  // everything above is independent of the previous grid's results
  pdl_wait();
  MOE_TL_WAITED();
  if (tid == 0) sm->n_units = __ldcg(&pv.hdr->n_tiles) * upt;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem;
  const int n_units = sm->n_units;
  volatile int* abort = &sm->abort;

  if (warp == kRawWarp) {
    // ---- raw weight producer (one lane; held back only by the test switch) ---
    if (lane == 0 && !g_pf_hold_raw) {
      uint32_t kr = 0;
      int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
      for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
        const Unit un = load_unit<true, SB>(d, pv, w, ws, u, upt, n_units, nxt);
        const int grp = un.sub;  // the unit's 256 weight rows are one fragment group
        bool ok = true;
        for (int ks = 0; ks < S; ++ks) {
          const int slot = kr % kRS;
          MOE_PROF(long long t0 = clock64());
          if (!wait_or_abort(&sm->raw_empty[slot], ((kr / kRS) & 1) ^ 1, status, abort)) {
            ok = false;
            break;
          }
          MOE_PROF(PROF_ADD(poff + 0, t0); t0 = clock64());
          char* dst = base + kOffRaw + slot * kRawBytes;
          mbar_expect_tx(&sm->raw_full[slot], kRawQ + 16 * 64 * SB);
          // the group's 16 tiles are contiguous for each segment: two copies
          const size_t blk = ((size_t)grp * S + ks) * 16;
          bulk_g2s(dst, un.q + blk * 512, kRawQ, &sm->raw_full[slot]);
          bulk_g2s(dst + kRawQ, un.s + blk * 64 * SB, 16 * 64 * SB, &sm->raw_full[slot]);
          MOE_DBG(6, kr);
          MOE_PROF(PROF_ADD(poff + 1, t0));
          ++kr;
        }
        if (!ok) break;
      }
      // copies still in flight must land before the block exits: wait for the
      // most recent stages (consumed ones completed long ago)
      for (uint32_t k = (kr > (uint32_t)kRS ? kr - kRS : 0); k < kr; ++k)
        wait_or_abort(&sm->raw_full[k % kRS], (k / kRS) & 1, status, abort);
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer (one lane) --------------------------------------------------
    if (lane == 0) {
      uint32_t ka = 0, it = 0;
      MOE_PROF(const long long t_all = clock64());
      int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
      for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++it) {
        MOE_PROF(long long t0 = clock64());
        const Unit un = load_unit<true, SB>(d, pv, w, ws, u, upt, n_units, nxt);
        const uint32_t idesc = idesc_f16_f32(128, un.npad);
        MOE_PROF(PROF_ADD(poff + 3, t0); t0 = clock64());
        if (it > 0 && !wait_or_abort(&sm->tmem_empty, (it - 1) & 1, status, abort)) break;
        MOE_PROF(PROF_ADD(poff + 7, t0));
        tc_fence_after();
        bool ok = true;
        // per K step: one wait (A stage and B stage of the step), then per A
        // tile and 16-element K slice one MMA with N = all of the unit's rows,
        // then one commit that frees both stages
        for (int ks = 0; ks < S; ++ks, ++ka) {
          const int as = ka % kAS, bs = ka % kBStages;
          MOE_PROF(t0 = clock64());
          if (!wait_or_abort(&sm->full[bs], (ka / kBStages) & 1, status, abort)) {
            ok = false;
            break;
          }
          MOE_DBG(2, ka);
          MOE_PROF(PROF_ADD(poff + 4, t0); t0 = clock64());
          tc_fence_after();
          const uint32_t ta = tmem + kAOff + as * kBK;
          const uint64_t db = sdesc_sw128(smem_u32(base + kOffB + bs * kBStage));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (ks | kk) ? 1u : 0u;
            // B: +32 bytes along K inside the 128-byte swizzle atom (start
            // address + 2); A: +8 tensor-memory columns; tile t in accumulator t
            tc_mma_f16_ts(tmem, ta + 8 * kk, db + 2 * kk, idesc, acc);
            tc_mma_f16_ts(tmem + kTileRows, ta + kBK / 2 + 8 * kk, db + 2 * kk, idesc, acc);
          }
          tc_commit(&sm->empty[bs]);
          MOE_DBG(0, ka);
          MOE_PROF(PROF_ADD(poff + 6, t0));
        }
        if (!ok) break;
        tc_commit(&sm->accf);
      }
      MOE_PROF(PROF_ADD(poff + 2, t_all));
      // every MMA issued has completed before tensor memory is released
      tc_commit(&sm->drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(&sm->drain, 0) && clock64() - t0 < g_pf_wait_limit) {
      }
    }
  } else if (warp == kBWarp0) {
    // ---- B producer (one thread): the unit's token rows, one ring stage per K
    // step (up to 192 rows, 128-byte swizzle), loaded as 64-row tiles of the
    // plan-ordered operand (x rows gathered into plan order for W13, h for W2).
    if (lane == 0) {
      uint32_t kb = 0;
      bool ok = true;
      int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
      for (int u = blockIdx.x; u < n_units && ok && !*abort; u += gridDim.x) {
        const Unit un = load_unit<true, SB>(d, pv, w, ws, u, upt, n_units, nxt);
        const int nch = (un.npad + kBChunkRows - 1) / kBChunkRows;
        for (int ks = 0; ks < S; ++ks, ++kb) {
          const int bs = kb % kBStages;
          MOE_PROF(long long t0 = clock64());
          if (!wait_or_abort(&sm->empty[bs], ((kb / kBStages) & 1) ^ 1, status, abort)) {
            ok = false;
            break;
          }
          MOE_PROF(PROF_ADD(poff + 8, t0); t0 = clock64());
          mbar_expect_tx(&sm->full[bs], (uint32_t)(nch * kBChunk));
          for (int ch = 0; ch < nch; ++ch)
            tma_load_2d(base + kOffB + bs * kBStage + ch * kBChunk, &bmap, ks * kBK,
                        un.pos0 + ch * kBChunkRows, &sm->full[bs]);
          MOE_DBG(5, kb);
          MOE_PROF(PROF_ADD(poff + 9, t0));
        }
      }
      // loads still in flight land before the block exits (bounded waits; each
      // of these phases completes once the dequantisers have arrived too, or
      // the wait gives up after an abort)
      for (uint32_t k = (kb > (uint32_t)kBStages ? kb - kBStages : 0); k < kb; ++k)
        drain_wait(&sm->full[k % kBStages], (k / kBStages) & 1);
    }
  } else if (warp >= kOutWarp0 && warp < kOutWarp0 + kOutWarps) {
    // ---- output warps: write each unit's staged h rows out (whole 256-byte
    // token rows, one 8-byte store per lane); lane l carries positions
    // 4 l .. 4 l + 3 of a row, held by dequantising warp (q = l % 4,
    // t = l / 16) at values 4 ((l % 16) / 4) .. + 3 ----
    const int I = d.I;
    const char* src_tile = reinterpret_cast<const char*>(sm->hstage[(lane & 3) + 4 * (lane >> 4)]) +
                           8 * ((lane & 15) >> 2);
    uint32_t it = 0;
    int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
    for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++it) {
      const Unit un = load_unit<true, SB>(d, pv, w, ws, u, upt, n_units, nxt);
      MOE_PROF(long long t0 = clock64());
      if (!warp_wait_or_abort(&sm->ep_staged, it & 1, status, abort)) break;
      MOE_PROF(if (lane == 0 && warp == kOutWarp0) PROF_ADD(poff + 5, t0));
      __half* hrow = h_out + (int64_t)un.pos0 * I + un.sub * 128 + 4 * lane;
      for (int n = warp - kOutWarp0; n < un.rows; n += kOutWarps)
        *reinterpret_cast<uint2*>(hrow + (int64_t)n * I) =
            *reinterpret_cast<const uint2*>(src_tile + n * 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->ep_free);
    }
  } else {
    // ---- warps 0-7: dequantise, then the unit's epilogue ---------------------------
    uint32_t kd = 0, it = 0;
    int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
    for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++it) {
      const Unit un = load_unit<true, SB>(d, pv, w, ws, u, upt, n_units, nxt);
      bool ok = true;
      // this warp's two fragment blocks j = 2 warp + jj: rows 32 (warp % 4) + 16 jj
      // .. + 15 of A tile warp / 4
      const uint32_t ta_warp = ((uint32_t)(32 * (warp & 3)) << 16) + kAOff + (warp >> 2) * (kBK / 2);
      for (int ks = 0; ks < S; ++ks, ++kd) {
        const int rs = kd % kRS, as = kd % kAS;
        MOE_PROF(long long t0 = clock64());
        if (!warp_wait_or_abort(&sm->raw_full[rs], (kd / kRS) & 1, status, abort)) {
          ok = false;
          break;
        }
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 10, t0); t0 = clock64());
        const char* raw = base + kOffRaw + rs * kRawBytes;
        uint4 q[2];
        uint32_t sc[2];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int j = warp * 2 + jj;
          q[jj] = *reinterpret_cast<const uint4*>(raw + j * 512 + lane * 16);
          sc[jj] = lane_scale_word<SB>(raw + kRawQ + (j * 64 + lane * 2) * SB);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->raw_empty[rs]);  // the stage is in registers
        // A stage kd % kAS was last read by the MMAs of K step kd - kAS
        if (kd >= (uint32_t)kAS) {
          const uint32_t kp = kd - kAS;
          if (!warp_wait_or_abort(&sm->empty[kp % kBStages], (kp / kBStages) & 1, status, abort)) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 11, t0); t0 = clock64());
        if (lane == 0) MOE_DBG(3, kd * kDqWarps + warp);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const uint32_t f = lane_scale_f16x2<SB>(sc[jj]);
          const uint32_t sg = __byte_perm(f, f, 0x1010), sg8 = __byte_perm(f, f, 0x3232);
          uint32_t x[4], y[4], z[4], w4[4];
          dequant8(q[jj].x, sg, x);   // row g,     elements 16c + 0..7
          dequant8(q[jj].y, sg, y);   // row g,     elements 16c + 8..15
          dequant8(q[jj].z, sg8, z);  // row g + 8, elements 16c + 0..7
          dequant8(q[jj].w, sg8, w4); // row g + 8, elements 16c + 8..15
          const uint32_t r[16] = {x[0], x[1], z[0], z[1], x[2], x[3], z[2], z[3],
                                  y[0], y[1], w4[0], w4[1], y[2], y[3], w4[2], w4[3]};
          tmem_st16x256_x4(tmem + ta_warp + ((uint32_t)(16 * jj) << 16) + as * kBK, r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) MOE_DBG(4, kd * kDqWarps + warp);
        if (lane == 0) mbar_arrive(&sm->full[kd % kBStages]);
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 12, t0));
      }
      if (!ok) break;
      // ---- epilogue of this unit: warp w reads TMEM lanes 32 (w % 4) .. +31 of
      // accumulator w / 4 ----
      const int q4 = warp & 3, at = warp >> 2;
      MOE_PROF(long long te = clock64());
      if (!warp_wait_or_abort(&sm->accf, it & 1, status, abort)) break;
      if (tid == 0) MOE_DBG(7, 2 * it);
      // the staging tiles are free once the output warps have written unit
      // it - 1 out (long before, in the steady state: a unit's K loop)
      if (it > 0 && !warp_wait_or_abort(&sm->ep_free, (it - 1) & 1, status, abort)) break;
      MOE_PROF(if (tid == 0) PROF_ADD(poff + 13, te); te = clock64());
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q4 * 32) << 16) + at * kTileRows;
      // Lane r < 16 of warp q holds gate row (16q + r) and lane r + 16 the
      // matching up row, for 32 token columns per load.  One exchange per
      // pair of columns gives each lane 16 (G, U) pairs: gate lanes take
      // columns 0-15, up lanes 16-31.  A token row's 16 values of warp (q, t)
      // belong at positions 64 t + 16 r + 4 q + (0..3), r = 0..3, of the
      // unit's 128 h values (the K order of the W2 operand).  Tensor memory
      // is released right after the last read, so that the next unit's MMAs
      // need not wait for the SwiGLU of the last chunk or the row writes.
      const int r16 = lane & 15;
      const bool is_gate = lane < 16;
      __half(*stg)[16] = reinterpret_cast<__half(*)[16]>(sm->hstage[warp]);
#pragma unroll 1
      for (int c0 = 0; c0 < un.npad; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + c0, v);
        if (c0 + 32 >= un.npad) {  // the unit's accumulators are read
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm->tmem_empty);
        }
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const float lo = __uint_as_float(v[jj]), hi = __uint_as_float(v[jj + 16]);
          const float recv = __shfl_xor_sync(0xffffffffu, is_gate ? hi : lo, 16);
          const float G = (is_gate ? lo : recv) * un.g;
          const float U = (is_gate ? recv : hi) * un.g;
          const float hv = __fdividef(G, 1.f + __expf(-G)) * U;
          stg[c0 + (is_gate ? jj : jj + 16)][r16] = __float2half_rn(hv);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->ep_staged);
      if (tid == 0) MOE_DBG(7, 2 * it + 1);
      MOE_PROF(if (tid == 0) PROF_ADD(poff + 14, te));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
#ifdef MOE_TIMELINE
#pragma unroll
  for (int i = 0; i < 15; ++i)
    if (pacc[i]) atomicAdd(&g_prof[poff + i], pacc[i]);
#endif
}

// ---------------------------------------------------------------------------
// Grouped W2.  A unit is one plan tile times 128 output rows (one A tile), so
// that tensor memory holds two accumulator buffers (2 x 192 columns) beside
// two A stages of a 128-element K step (2 x 64 columns): the epilogue of unit
// u drains one buffer while the MMAs of unit u + 1 fill the other.  A K step
// is two 64-element fragment segments (8 MMAs per wait and commit).  20 warps:
//   warps 0-7    dequantise one fragment block of each segment per K step
//                (warp w owns lanes 16 (2 (w % 4) + w / 4) .. + 15 of the A tile);
//   warps 8-15   epilogue: warp 8 + q + 4 p reads lanes 32 q .. + 31 of the
//                unit's buffer, the 32-column chunks of parity p;
//   warp 16      tensor memory owner, one lane issues the MMAs;
//   warp 17      raw NVFP4 bulk copies (8 fragment blocks per segment);
//   warp 18      token rows (h) by 64-row tensor-map loads, one 24 KiB half
//                stage per segment;
//   warp 19      g2 x combine weight of each row, one unit ahead.
// ---------------------------------------------------------------------------
constexpr int kW2Threads = 20 * 32;
constexpr int kW2Seg = 2;              // 64-element fragment segments per W2 K step
constexpr int kW2KS = kW2Seg * kBK;    // K per W2 step
constexpr int kW2AS = 4 / kW2Seg;      // A stages (128 tensor-memory columns in all)
constexpr int kW2BStages = kW2AS;      // B stages of one step (kW2Seg 24 KiB halves each)
constexpr int kW2EpiWarp0 = 8;
constexpr int kW2MmaWarp = 16;
constexpr int kW2RawWarp = 17;
constexpr int kW2BWarp = 18;
constexpr int kW2ScaleWarp = 19;
constexpr int kW2RawQ = 8 * 512;  // raw q bytes per segment (8 fragment blocks)
constexpr int kW2RawS = 8 * 64;   // their raw scale bytes (x 2 when prepared)
// raw slot of one K step: the segments' q, then their scales (room for FP16)
constexpr int kW2RawSlot = kW2Seg * (kW2RawQ + 2 * kW2RawS);
constexpr int kW2RS = kRS * kRawBytes / kW2RawSlot;  // raw stages in the raw region
static_assert(kW2RawSlot % 16 == 0 && kW2RS * kW2RawSlot <= kRS * kRawBytes, "W2 raw slot");
static_assert(kAOff + kW2AS * (kW2KS / 2) <= kTmemCols, "W2 tensor memory over-committed");
static_assert(kW2BStages == kW2AS, "one barrier per K step serves both rings");
static_assert(kW2BStages * kW2Seg * kBStage <= kBStages * kBStage, "W2 B ring inside the B region");

struct W2Smem {
  uint64_t raw_full[kW2RS], raw_empty[kW2RS];
  uint64_t full[kW2BStages], empty[kW2BStages];
  // per accumulator buffer b: accf[b] completes when a unit's MMAs into b are
  // done, tmem_empty[b] when its epilogue has read b, wsc_full[b] when the
  // unit's scales are in wsc[b]
  uint64_t accf[2], tmem_empty[2], wsc_full[2], drain;
  __align__(16) float wsc[2][kTileRows];
  uint32_t tmem;
  int abort;
  int n_units;
  __align__(16) float stage[8][512];  // epilogue staging, [16 pairs][32 rows] per warp
};

constexpr size_t w2_smem_bytes() { return 1024 + (size_t)kOffMeta + sizeof(W2Smem); }
static_assert(w2_smem_bytes() <= 232448, "grouped W2 shared memory above the sm_103 limit");

template <int SB>
__global__ void __launch_bounds__(kW2Threads, 1)
    grouped_w2_kernel(LayerDims d, PlanView pv, const __grid_constant__ CUtensorMap bmap,
                      Weights w, Weights ws, __half* __restrict__ partial, uint32_t* status) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  W2Smem* sm = reinterpret_cast<W2Smem*>(base + kOffMeta);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  MOE_TL(kTlW2);
  MOE_PROF(constexpr int poff = 16);
  MOE_PROF(unsigned long long pacc[15] = {});
  const int S = d.I / kW2KS;   // K steps per unit (I % 128 == 0)
  static_assert(128 % kW2KS == 0, "W2 K step divides 128");
  const int upt = d.H / 128;   // units per plan tile

  if (tid == 0) {
    for (int i = 0; i < kW2RS; ++i) {
      mbar_init(&sm->raw_full[i], 1);
      mbar_init(&sm->raw_empty[i], kDqWarps);
    }
    for (int i = 0; i < kW2BStages; ++i) {
      mbar_init(&sm->full[i], kDqWarps + 1);
      mbar_init(&sm->empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm->accf[b], 1);
      mbar_init(&sm->tmem_empty[b], 8);
      mbar_init(&sm->wsc_full[b], 1);
    }
    mbar_init(&sm->drain, 1);
    sm->abort = 0;
    fence_mbar_init();
  }
  if (warp == kW2MmaWarp) tmem_alloc(&sm->tmem, kTmemCols);
  pdl_wait();
  MOE_TL_WAITED();
  if (tid == 0) sm->n_units = __ldcg(&pv.hdr->n_tiles) * upt;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem;
  const int n_units = sm->n_units;
  volatile int* abort = &sm->abort;

  if (warp == kW2RawWarp) {
    // ---- raw weights: the unit's 8 fragment blocks of each K step ----
    if (lane == 0) {
      uint32_t kr = 0;
      bool ok = true;
      int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
      for (int u = blockIdx.x; u < n_units && ok && !*abort; u += gridDim.x) {
        const Unit un = load_unit<false, SB>(d, pv, w, ws, u, upt, n_units, nxt);
        const int grp = un.sub >> 1, half = un.sub & 1;
        for (int ks = 0; ks < S; ++ks, ++kr) {
          const int slot = kr % kW2RS;
          if (!wait_or_abort(&sm->raw_empty[slot], ((kr / kW2RS) & 1) ^ 1, status, abort)) {
            ok = false;
            break;
          }
          char* dst = base + kOffRaw + slot * kW2RawSlot;
          mbar_expect_tx(&sm->raw_full[slot], kW2Seg * (kW2RawQ + kW2RawS * SB));
          // segments kW2Seg ks + c: q of segment c at c * kW2RawQ, s at
          // kW2Seg * kW2RawQ + c * kW2RawS
#pragma unroll
          for (int c = 0; c < kW2Seg; ++c) {
            const size_t blk = ((size_t)grp * (kW2Seg * S) + kW2Seg * ks + c) * 16 + 8 * half;
            bulk_g2s(dst + c * kW2RawQ, un.q + blk * 512, kW2RawQ, &sm->raw_full[slot]);
            bulk_g2s(dst + kW2Seg * kW2RawQ + c * kW2RawS * SB, un.s + blk * 64 * SB,
                     kW2RawS * SB, &sm->raw_full[slot]);
          }
        }
      }
      for (uint32_t k = (kr > (uint32_t)kW2RS ? kr - kW2RS : 0); k < kr; ++k)
        wait_or_abort(&sm->raw_full[k % kW2RS], (k / kW2RS) & 1, status, abort);
    }
  } else if (warp == kW2MmaWarp) {
    // ---- MMAs: per K step one wait, 4 MMAs (K 16 each), one commit ----
    if (lane == 0) {
      uint32_t ka = 0, it = 0;
      MOE_PROF(const long long t_all = clock64());
      int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
      for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++it) {
        MOE_PROF(long long t0 = clock64());
        const Unit un = load_unit<false, SB>(d, pv, w, ws, u, upt, n_units, nxt);
        const uint32_t idesc = idesc_f16_f32(128, un.npad);
        const int b = it & 1;
        MOE_PROF(PROF_ADD(poff + 3, t0); t0 = clock64());
        if (it >= 2 && !wait_or_abort(&sm->tmem_empty[b], ((it - 2) >> 1) & 1, status, abort))
          break;
        MOE_PROF(PROF_ADD(poff + 7, t0));
        tc_fence_after();
        bool ok = true;
        for (int ks = 0; ks < S; ++ks, ++ka) {
          const int st = ka % kW2BStages, as = ka % kW2AS;
          MOE_PROF(t0 = clock64());
          if (!wait_or_abort(&sm->full[st], (ka / kW2BStages) & 1, status, abort)) {
            ok = false;
            break;
          }
          MOE_PROF(PROF_ADD(poff + 4, t0); t0 = clock64());
          tc_fence_after();
          const uint32_t ta = tmem + kAOff + as * (kW2KS / 2);
#pragma unroll
          for (int c = 0; c < kW2Seg; ++c) {
            // segment c: A columns [32 c, 32 c + 32) of the stage, B half c
            const uint64_t db =
                sdesc_sw128(smem_u32(base + kOffB + (st * kW2Seg + c) * kBStage));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              tc_mma_f16_ts(tmem + b * kTileRows, ta + 32 * c + 8 * kk, db + 2 * kk, idesc,
                            (ks | c | kk) ? 1u : 0u);
          }
          tc_commit(&sm->empty[st]);
          MOE_PROF(PROF_ADD(poff + 6, t0));
        }
        if (!ok) break;
        tc_commit(&sm->accf[b]);
      }
      MOE_PROF(PROF_ADD(poff + 2, t_all));
      tc_commit(&sm->drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(&sm->drain, 0) && clock64() - t0 < g_pf_wait_limit) {
      }
    }
  } else if (warp == kW2BWarp) {
    // ---- token rows (h in plan order): one ring stage per K step ----
    if (lane == 0) {
      uint32_t kb = 0;
      bool ok = true;
      int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
      for (int u = blockIdx.x; u < n_units && ok && !*abort; u += gridDim.x) {
        const Unit un = load_unit<false, SB>(d, pv, w, ws, u, upt, n_units, nxt);
        const int nch = (un.npad + kBChunkRows - 1) / kBChunkRows;
        for (int ks = 0; ks < S; ++ks, ++kb) {
          const int bs = kb % kW2BStages;
          MOE_PROF(long long t0 = clock64());
          if (!wait_or_abort(&sm->empty[bs], ((kb / kW2BStages) & 1) ^ 1, status, abort)) {
            ok = false;
            break;
          }
          MOE_PROF(PROF_ADD(poff + 8, t0));
          mbar_expect_tx(&sm->full[bs], (uint32_t)(kW2Seg * nch * kBChunk));
          for (int c = 0; c < kW2Seg; ++c)
            for (int ch = 0; ch < nch; ++ch)
              tma_load_2d(base + kOffB + (bs * kW2Seg + c) * kBStage + ch * kBChunk, &bmap,
                          ks * kW2KS + c * kBK, un.pos0 + ch * kBChunkRows, &sm->full[bs]);
        }
      }
      for (uint32_t k = (kb > (uint32_t)kW2BStages ? kb - kW2BStages : 0); k < kb; ++k)
        drain_wait(&sm->full[k % kW2BStages], (k / kW2BStages) & 1);
    }
  } else if (warp == kW2ScaleWarp) {
    // ---- g2 x combine weight of each row, one unit ahead (buffer it & 1 is
    // free once the epilogue of unit it - 2 is done) ----
    uint32_t it = 0;
    int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
    for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++it) {
      const Unit un = load_unit<false, SB>(d, pv, w, ws, u, upt, n_units, nxt);
      if (it >= 2 &&
          !warp_wait_or_abort(&sm->tmem_empty[it & 1], ((it - 2) >> 1) & 1, status, abort))
        break;
      float* wsc = sm->wsc[it & 1];
      int pr[kTileRows / 32];
#pragma unroll
      for (int i = 0; i < kTileRows / 32; ++i) {
        const int n = lane + 32 * i;
        pr[i] = n < un.rows ? __ldcg(pv.perm + un.pos0 + n) : -1;
      }
#pragma unroll
      for (int i = 0; i < kTileRows / 32; ++i)
        if (pr[i] >= 0) wsc[lane + 32 * i] = un.g * __ldcg(pv.w + pr[i]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->wsc_full[it & 1]);
    }
  } else if (warp >= kW2EpiWarp0 && warp < kW2EpiWarp0 + 8) {
    // ---- epilogue: lane r of warp (q, p) holds output row 32 q + r of the
    // unit (H row sub * 128 + 32 q + r) for the chunks c0 = 32 p, 32 p + 64, ...
    // A per-warp staging tile turns 16 columns at a time into rows of 32
    // contiguous FP32 values, scaled and written as FP16 (8-byte stores) into
    // the pairs' partial rows (at the pairs' plan positions) ----
    const int q = warp & 3, pr = (warp - kW2EpiWarp0) >> 2;
    const int H = d.H;
    float(*stg)[32] = reinterpret_cast<float(*)[32]>(sm->stage[warp - kW2EpiWarp0]);
    uint32_t it = 0;
    int4 nxt = unit_tile(pv, blockIdx.x, upt, n_units);
    for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++it) {
      const Unit un = load_unit<false, SB>(d, pv, w, ws, u, upt, n_units, nxt);
      const int b = it & 1;
      MOE_PROF(long long te = clock64());
      if (!warp_wait_or_abort(&sm->accf[b], (it >> 1) & 1, status, abort)) break;
      if (!warp_wait_or_abort(&sm->wsc_full[b], (it >> 1) & 1, status, abort)) break;
      MOE_PROF(if (tid == kW2EpiWarp0 * 32) PROF_ADD(poff + 13, te); te = clock64());
      tc_fence_after();
      const float* wsc = sm->wsc[b];
      __half* pbase = partial + (int64_t)un.pos0 * H + un.sub * 128 + q * 32;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + b * kTileRows;
#pragma unroll 1
      for (int c0 = 32 * pr; c0 < un.npad; c0 += 64) {
        uint32_t v[32];
        tmem_ld32(tbase + c0, v);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int j = 0; j < 16; ++j) stg[j][lane] = __uint_as_float(v[16 * hf + j]);
          __syncwarp();
          // lanes 8p .. 8p+7 write column (pair) p0 + p: 8 x 16 bytes
          const int cl = lane >> 3, part = lane & 7;
#pragma unroll
          for (int p4 = 0; p4 < 4; ++p4) {
            const int j = p4 * 4 + cl;
            const int n = c0 + 16 * hf + j;
            if (n < un.rows) {
              const float4 o = reinterpret_cast<const float4*>(stg[j])[part];
              const float sc = wsc[n];
              const __half2 lo = __floats2half2_rn(o.x * sc, o.y * sc);
              const __half2 hi = __floats2half2_rn(o.z * sc, o.w * sc);
              uint2 hv;
              hv.x = *reinterpret_cast<const uint32_t*>(&lo);
              hv.y = *reinterpret_cast<const uint32_t*>(&hi);
              __stcs(reinterpret_cast<uint2*>(pbase + (int64_t)n * H) + part, hv);
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->tmem_empty[b]);
      MOE_PROF(if (tid == kW2EpiWarp0 * 32) PROF_ADD(poff + 14, te));
    }
  } else if (warp < kDqWarps) {
    // ---- dequantise: one fragment block per warp and K step into the A stage ----
    const int jl = 2 * (warp & 3) + (warp >> 2);  // block of the unit's 8 (rows 16 jl ..)
    const uint32_t ta_warp = ((uint32_t)(16 * jl) << 16) + kAOff;
    uint32_t kd = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok && !*abort; u += gridDim.x) {
      for (int ks = 0; ks < S; ++ks, ++kd) {
        const int rs = kd % kW2RS, as = kd % kW2AS;
        MOE_PROF(long long t0 = clock64());
        if (!warp_wait_or_abort(&sm->raw_full[rs], (kd / kW2RS) & 1, status, abort)) {
          ok = false;
          break;
        }
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 10, t0); t0 = clock64());
        const char* raw = base + kOffRaw + rs * kW2RawSlot;
        uint4 qv[kW2Seg];
        uint32_t sc[kW2Seg];
#pragma unroll
        for (int c = 0; c < kW2Seg; ++c) {
          qv[c] = *reinterpret_cast<const uint4*>(raw + c * kW2RawQ + jl * 512 + lane * 16);
          sc[c] = lane_scale_word<SB>(raw + kW2Seg * kW2RawQ + (c * kW2RawS + jl * 64 + lane * 2) * SB);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->raw_empty[rs]);  // the stage is in registers
        // A stage kd % kW2AS was last read by the MMAs of K step kd - kW2AS
        if (kd >= (uint32_t)kW2AS) {
          const uint32_t kp = kd - kW2AS;
          if (!warp_wait_or_abort(&sm->empty[kp % kW2BStages], (kp / kW2BStages) & 1, status,
                                  abort)) {
            ok = false;
            break;
          }
        }
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 11, t0); t0 = clock64());
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kW2Seg; ++c) {
          const uint32_t f = lane_scale_f16x2<SB>(sc[c]);
          const uint32_t sg = __byte_perm(f, f, 0x1010), sg8 = __byte_perm(f, f, 0x3232);
          uint32_t x[4], y[4], z[4], w4[4];
          dequant8(qv[c].x, sg, x);
          dequant8(qv[c].y, sg, y);
          dequant8(qv[c].z, sg8, z);
          dequant8(qv[c].w, sg8, w4);
          const uint32_t r[16] = {x[0], x[1], z[0], z[1], x[2], x[3], z[2], z[3],
                                  y[0], y[1], w4[0], w4[1], y[2], y[3], w4[2], w4[3]};
          tmem_st16x256_x4(tmem + ta_warp + as * (kW2KS / 2) + 32 * c, r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->full[kd % kW2BStages]);
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 12, t0));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kW2MmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
#ifdef MOE_TIMELINE
#pragma unroll
  for (int i = 0; i < 15; ++i)
    if (pacc[i]) atomicAdd(&g_prof[poff + i], pacc[i]);
#endif
}

// xg[pos] = x[perm[pos] / k_eff]: the token rows in plan order, the operand of
// the grouped W13 GEMM (positions past the valid pairs are left alone), with
// each 64-element K step in the order of the tensor-memory A operand: output
// position 16r + 4c + e takes element 16c + 4r + e.  One warp per row; each
// lane writes 16 bytes (positions [8m, 8m + 8): r = m / 2, c = 2 (m % 2) and
// 2 (m % 2) + 1) from two 8-byte loads.
__global__ void gather_rows_kernel(LayerDims d, PlanView pv, const __half* __restrict__ x,
                                   __half* __restrict__ xg) {
  MOE_TL(kTlPlan);
  pdl_wait();
  pdl_launch_dependents();
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= __ldcg(&pv.hdr->n_valid)) return;
  const int t = __ldcg(pv.perm + row) / d.k_eff;
  const __half* src = x + (int64_t)t * d.H;
  uint4* dst = reinterpret_cast<uint4*>(xg + row * d.H);
  for (int ch = lane; ch < d.H / 8; ch += 32) {
    const int k0 = (ch >> 3) * 64, m = ch & 7;
    const int r = m >> 1, c = 2 * (m & 1);
    const uint2 lo = __ldg(reinterpret_cast<const uint2*>(src + k0 + 16 * c + 4 * r));
    const uint2 hi = __ldg(reinterpret_cast<const uint2*>(src + k0 + 16 * (c + 1) + 4 * r));
    dst[ch] = make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
}

cudaError_t prefill_set_wait_test(int hold_raw, long long limit_cycles, cudaStream_t stream) {
  const long long lim = limit_cycles > 0 ? limit_cycles : kWaitTimeoutCycles;
  cudaError_t e = cudaMemcpyToSymbolAsync(g_pf_hold_raw, &hold_raw, sizeof(int), 0,
                                          cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_pf_wait_limit, &lim, sizeof(long long), 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

cudaError_t prefill_device_init() {
  for (auto f : {(const void*)grouped_w13_kernel<1>, (const void*)grouped_w13_kernel<2>}) {
    cudaError_t e =
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemm_smem_bytes());
    if (e != cudaSuccess) return e;
  }
  for (auto f : {(const void*)grouped_w2_kernel<1>, (const void*)grouped_w2_kernel<2>}) {
    cudaError_t e =
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)w2_smem_bytes());
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_prefill_forward(const LayerDims& d, int64_t M, const __half* x,
                                   const PlanView& pv, Weights w13, Weights w2, Weights s13,
                                   Weights s2, __half* y, __half* h, __half* partial,
                                   uint32_t* status, cudaStream_t stream, int num_sms,
                                   bool prepared) {
  const int64_t P = M * d.k_eff;
  const int max_tiles = max_tiles_for(P, d.e_eff);
  const size_t smem = gemm_smem_bytes();
  const int g13 = (int)std::min<int64_t>((int64_t)max_tiles * ((2 * d.I) / 256), num_sms);  // 256 weight rows per unit
  const int g2 = (int)std::min<int64_t>((int64_t)max_tiles * (d.H / 128), num_sms);
  const bool pdl = !trace_on();
  // Token-row operands in plan order, read as 64-row tensor-map tiles (128-byte
  // swizzled): W13 reads x rows gathered into the partials buffer (unused until
  // the W2 grid, which starts after W13 has finished), W2 reads h.
  __half* xg = partial;
  CUtensorMap xmap, hmap;
  cudaError_t e = make_fp16_map(&xmap, xg, d.H, (uint64_t)P, kBK, kBChunkRows, true);
  if (e != cudaSuccess) return e;
  e = make_fp16_map(&hmap, h, d.I, (uint64_t)P, kBK, kBChunkRows, true);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW13, false);
  e = launch_k(gather_rows_kernel, dim3((unsigned)((P + 7) / 8)), dim3(256), 0, stream, pdl, d, pv,
               x, xg);
  if (e != cudaSuccess) return e;
  e = launch_k(prepared ? grouped_w13_kernel<2> : grouped_w13_kernel<1>, dim3(g13),
               dim3(kGemmThreads), smem, stream, pdl, d, pv, xmap, w13, s13, h, status);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW13, true);
  trace_mark(stream, kTraceW2, false);
  e = launch_k(prepared ? grouped_w2_kernel<2> : grouped_w2_kernel<1>, dim3(g2),
               dim3(kW2Threads), w2_smem_bytes(), stream, pdl, d, pv, hmap, w2, s2, partial, status);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW2, true);
  trace_mark(stream, kTraceCombine, false);
  e = launch_combine(d, M, pv, partial, y, stream, pdl);
  trace_mark(stream, kTraceCombine, true);
  return e;
}

}  // namespace moe
