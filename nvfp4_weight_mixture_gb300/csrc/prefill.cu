// Prefill path (M > 16): expert-grouped GEMMs on the 5th-generation tensor
// cores (tcgen05, kind::f16, FP32 accumulators in tensor memory).
//
// "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Scope and
// related PRs": grouped W13 with SwiGLU and grouped W2 with the reduction,
// both driven by the same integer plan.  A work unit is one plan tile (one
// expert, up to 256 of its routed rows) times 256 weight rows:
//
//   D[weight row][token] = sum_k W[weight row][k] * X[token][k]     (swap-AB)
//
// so the weight rows are the MMA's M = 128 (two accumulators of N <= 256
// columns fill the 512 tensor-memory columns) and the tokens are N.  Blocks
// are persistent (one per SM) and walk the units with a static stride.
// Warp roles, each running ahead as far as its ring allows:
//   warp 13    one lane streams the unit's raw NVFP4 blocks (fragment layout:
//              16 blocks of 512 + 64 bytes per K step of 64) into a 4-deep
//              shared ring with two bulk asynchronous copies per K step;
//   warps 0-7  dequantise each raw stage into 128-byte-swizzled K-major FP16
//              A tiles (2-deep ring; two fragment blocks per warp), then run
//              the unit's epilogue, warp w on TMEM lanes 32 (w % 4) .. +31 of
//              accumulator w / 4;
//   warp 8     one lane fills the token-row operand, one 3-deep ring stage per
//              K step (same swizzled layout), with 64-row tensor-map loads of
//              the plan-ordered rows: x gathered beforehand for W13, h for W2
//              (warps 9-11 are spare);
//   warp 12    allocates tensor memory; one lane issues the MMAs: per K step
//              one wait on each ring, then per A tile and 16-element K slice one
//              MMA with N = all of the unit's rows, then one commit per ring.
//              (The issuing thread shares its SM sub-partition with busy
//              dequantise and gather warps, so its per-step instruction chain
//              is kept short.)
//
// W13: the fragment layout interleaves 16-row gate and up tiles, so TMEM lanes
// [32q, 32q+16) hold gate rows and [32q+16, 32q+32) the matching up rows; the
// epilogue pairs them with one shuffle and writes h = fp16(silu(G) * U).
// W2:  the epilogue scales by g2 and the pair's combine weight and writes the
// FP32 partial row of each pair; a separate pass sums the slots in order.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kBK = 64;                   // K per step (128 bytes of FP16)
constexpr int kATile = 128 * 128;         // one 128-row FP16 A tile, bytes
constexpr int kBTile = kTileRows * 128;   // the B tile, bytes
constexpr int kAS = 2;                    // A (dequantised) stages
constexpr int kBChunkRows = 64;           // one gather warp's share: 64 token rows x 128 bytes
constexpr int kBChunk = kBChunkRows * 128;
constexpr int kBStage = 4 * kBChunk;      // B ring stage: one K step of up to 256 rows
constexpr int kBStages = 3;               // B ring stages (96 KiB)
constexpr int kRS = 4;                    // raw weight stages
constexpr int kRawQ = 16 * 512;           // raw q bytes per K step (16 fragment blocks)
constexpr int kRawBytes = kRawQ + 16 * 64;
// Warp roles: 0-7 dequantise and run the epilogue, 8-11 fill the token-row
// operand, 12 issues the MMAs (and owns tensor memory), 13 streams raw weights.
constexpr int kDqWarps = 8;
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kBWarp0 = 8;
constexpr int kMmaWarp = 12;
constexpr int kRawWarp = 13;
constexpr int kGemmThreads = 14 * 32;
constexpr int kTmemCols = 512;
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kAS * 2 * kATile;
constexpr int kOffRaw = kOffB + kBStages * kBStage;
constexpr int kOffMeta = kOffRaw + kRS * kRawBytes;

struct GemmSmem {
  uint64_t raw_full[kRS], raw_empty[kRS];
  uint64_t a_full[kAS], a_empty[kAS];
  uint64_t b_full[kBStages], b_empty[kBStages];
  uint64_t accf, tmem_empty, drain;
  uint32_t tmem;
  int abort;
  int n_units;
  int epair[2][kTileRows];   // epilogue (W2): pair id of each row
  float ewsc[2][kTileRows];  // epilogue (W2): g2 * combine weight of each row
  // epilogue staging, 2 KiB per warp: W13 h values [32 tokens][16 i] (FP16),
  // W2 partial values [16 pairs][32 rows] (FP32)
  __align__(16) float stage[kDqWarps][512];
};

constexpr size_t gemm_smem_bytes() {
  return 1024 /* alignment slack */ + (size_t)kOffMeta + sizeof(GemmSmem);
}
static_assert(gemm_smem_bytes() <= 232448, "grouped GEMM shared memory above the sm_103 limit");

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* status,
                                              volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitTimeoutCycles) {
      set_status(status, MOE_ST_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Profiling cells (timeline build): [0..1] raw producer wait/issue, [2..3]
// MMA thread total / unit bookkeeping, [4..7]
// MMA wait-A / wait-B / issue / wait-TMEM, [8..9] B wait/issue, [10..14]
// dequant wait-raw / wait-A / work, epilogue wait / work; [16 + 2k] = calls.
#ifdef MOE_TIMELINE
#define PROF_ADD(cell, t0) atomicAdd(&g_prof[cell], (unsigned long long)(clock64() - (t0)))
#else
#define PROF_ADD(cell, t0)
#endif

struct Unit {
  int e, rows, npad, sub, pos0;
  const uint8_t* q;  // the expert's q bytes
  const uint8_t* s;  // the expert's s bytes
  float g;
};

template <bool kW13>
__device__ __forceinline__ Unit load_unit(const LayerDims& d, const PlanView& pv, Weights w,
                                          Weights ws, int u, int upt) {
  Unit un;
  const int tile = u / upt;
  un.sub = u - tile * upt;
  const int4 tl = __ldcg(reinterpret_cast<const int4*>(pv.tiles) + tile);
  un.e = tl.x;
  un.rows = tl.z;
  un.npad = (tl.z + 15) & ~15;
  un.pos0 = __ldcg(pv.offsets + tl.x) + tl.y;
  const bool sh = (un.e == d.E);
  const size_t mat_q = kW13 ? (size_t)d.I * d.H : (size_t)d.H * d.I / 2;
  un.q = sh ? ws.q : w.q + (size_t)un.e * mat_q;
  un.s = sh ? ws.s : w.s + (size_t)un.e * mat_q / 8;
  un.g = sh ? ws.g[0] : w.g[un.e];
  return un;
}

template <bool kW13>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(LayerDims d, PlanView pv, const __grid_constant__ CUtensorMap bmap,
                        Weights w, Weights ws, __half* __restrict__ h_out,
                        float* __restrict__ partial, uint32_t* status) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  GemmSmem* sm = reinterpret_cast<GemmSmem*>(base + kOffMeta);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  MOE_TL(kW13 ? kTlW13 : kTlW2);
  MOE_PROF(constexpr int poff = kW13 ? 0 : 16);

  const int K = kW13 ? d.H : d.I;           // reduction length
  const int S = K / kBK;                     // K steps per unit
  const int upt = kW13 ? (2 * d.I) / 256 : d.H / 256;  // units per plan tile

  if (tid == 0) {
    for (int i = 0; i < kRS; ++i) {
      mbar_init(&sm->raw_full[i], 1);
      mbar_init(&sm->raw_empty[i], kDqThreads);
    }
    for (int i = 0; i < kAS; ++i) {
      mbar_init(&sm->a_full[i], kDqThreads);
      mbar_init(&sm->a_empty[i], 1);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&sm->b_full[i], 1);  // the loading thread, plus the transaction bytes
      mbar_init(&sm->b_empty[i], 1);
    }
    mbar_init(&sm->accf, 1);
    mbar_init(&sm->tmem_empty, kDqThreads);
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
    // ---- raw weight producer (one lane) ---------------------------------------
    if (lane == 0) {
      uint32_t kr = 0;
      for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
        const Unit un = load_unit<kW13>(d, pv, w, ws, u, upt);
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
          mbar_expect_tx(&sm->raw_full[slot], kRawBytes);
          // the group's 16 tiles are contiguous for each segment: two copies
          const size_t blk = ((size_t)grp * S + ks) * 16;
          bulk_g2s(dst, un.q + blk * 512, kRawQ, &sm->raw_full[slot]);
          bulk_g2s(dst + kRawQ, un.s + blk * 64, kRawBytes - kRawQ, &sm->raw_full[slot]);
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
      for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++it) {
        MOE_PROF(long long t0 = clock64());
        const Unit un = load_unit<kW13>(d, pv, w, ws, u, upt);
        const uint32_t idesc = idesc_f16_f32(128, un.npad);
        MOE_PROF(PROF_ADD(poff + 3, t0); t0 = clock64());
        if (it > 0 && !wait_or_abort(&sm->tmem_empty, (it - 1) & 1, status, abort)) break;
        MOE_PROF(PROF_ADD(poff + 7, t0));
        tc_fence_after();
        bool ok = true;
        // per K step: one A stage (two 128-row tiles) and one B stage (all of
        // the unit's token rows); one MMA per tile and 16-element K slice
        for (int ks = 0; ks < S; ++ks, ++ka) {
          const int as = ka % kAS, bs = ka % kBStages;
          MOE_PROF(t0 = clock64());
          if (!wait_or_abort(&sm->a_full[as], (ka / kAS) & 1, status, abort)) {
            ok = false;
            break;
          }
          if (kW13) MOE_DBG(2, ka);
          MOE_PROF(PROF_ADD(poff + 4, t0); t0 = clock64());
          if (!wait_or_abort(&sm->b_full[bs], (ka / kBStages) & 1, status, abort)) {
            ok = false;
            break;
          }
          if (kW13) MOE_DBG(1, ka);
          MOE_PROF(PROF_ADD(poff + 5, t0); t0 = clock64());
          tc_fence_after();
          const uint64_t da0 = sdesc_sw128(smem_u32(base + kOffA + as * 2 * kATile));
          const uint64_t da1 = sdesc_sw128(smem_u32(base + kOffA + as * 2 * kATile + kATile));
          const uint64_t db = sdesc_sw128(smem_u32(base + kOffB + bs * kBStage));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (ks | kk) ? 1u : 0u;
            // +32 bytes along K inside the 128-byte swizzle atom: start address + 2
            tc_mma_f16(tmem, da0 + 2 * kk, db + 2 * kk, idesc, acc);
            tc_mma_f16(tmem + 256, da1 + 2 * kk, db + 2 * kk, idesc, acc);
          }
          tc_commit(&sm->b_empty[bs]);
          tc_commit(&sm->a_empty[as]);
          MOE_PROF(PROF_ADD(poff + 6, t0));
        }
        if (!ok) break;
        tc_commit(&sm->accf);
      }
      MOE_PROF(PROF_ADD(poff + 2, t_all));
      // every MMA issued has completed before tensor memory is released
      tc_commit(&sm->drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(&sm->drain, 0) && clock64() - t0 < kWaitTimeoutCycles) {
      }
    }
  } else if (warp == kBWarp0) {
    // ---- B producer (one thread): the unit's token rows, one ring stage per K
    // step (up to 256 rows, 128-byte swizzle), loaded as 64-row tiles of the
    // plan-ordered operand (x rows gathered into plan order for W13, h for W2).
    if (lane == 0) {
      uint32_t kb = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok && !*abort; u += gridDim.x) {
        const Unit un = load_unit<kW13>(d, pv, w, ws, u, upt);
        const int nch = (un.npad + kBChunkRows - 1) / kBChunkRows;
        for (int ks = 0; ks < S; ++ks, ++kb) {
          const int bs = kb % kBStages;
          MOE_PROF(long long t0 = clock64());
          if (!wait_or_abort(&sm->b_empty[bs], ((kb / kBStages) & 1) ^ 1, status, abort)) {
            ok = false;
            break;
          }
          MOE_PROF(PROF_ADD(poff + 8, t0); t0 = clock64());
          mbar_expect_tx(&sm->b_full[bs], (uint32_t)(nch * kBChunk));
          for (int ch = 0; ch < nch; ++ch)
            tma_load_2d(base + kOffB + bs * kBStage + ch * kBChunk, &bmap, ks * kBK,
                        un.pos0 + ch * kBChunkRows, &sm->b_full[bs]);
          MOE_PROF(PROF_ADD(poff + 9, t0));
        }
      }
      // loads still in flight land before the block exits (bounded waits)
      for (uint32_t k = (kb > (uint32_t)kBStages ? kb - kBStages : 0); k < kb; ++k)
        mbar_wait(&sm->b_full[k % kBStages], (k / kBStages) & 1, status);
    }
  } else if (warp > kBWarp0) {
    // spare warps
  } else {
    // ---- warps 0-7: dequantise, then the unit's epilogue ---------------------------
    const int g = lane >> 2, c = lane & 3;
    uint32_t kd = 0, it = 0;
    for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x, ++it) {
      const Unit un = load_unit<kW13>(d, pv, w, ws, u, upt);
      if (!kW13) {
        for (int n = tid; n < un.rows; n += kDqThreads) {
          const int pair = __ldcg(pv.perm + un.pos0 + n);
          sm->epair[it & 1][n] = pair;
          sm->ewsc[it & 1][n] = un.g * __ldcg(pv.w + pair);
        }
      }
      bool ok = true;
      for (int ks = 0; ks < S; ++ks, ++kd) {
        const int rs = kd % kRS, as = kd % kAS;
        MOE_PROF(long long t0 = clock64());
        if (!wait_or_abort(&sm->raw_full[rs], (kd / kRS) & 1, status, abort)) {
          ok = false;
          break;
        }
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 10, t0); t0 = clock64());
        if (!wait_or_abort(&sm->a_empty[as], ((kd / kAS) & 1) ^ 1, status, abort)) {
          ok = false;
          break;
        }
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 11, t0); t0 = clock64());
        if (kW13 && lane == 0) MOE_DBG(3, kd * kDqWarps + warp);
        const char* raw = base + kOffRaw + rs * kRawBytes;
        char* stage = base + kOffA + as * 2 * kATile;
#pragma unroll
        for (int jj = 0; jj < 16 / kDqWarps; ++jj) {
          // fragment block j: A tile j / 8, local row tile j % 8
          const int j = warp * (16 / kDqWarps) + jj;
          const uint4 q = *reinterpret_cast<const uint4*>(raw + j * 512 + lane * 16);
          const uint32_t sc =
              *reinterpret_cast<const unsigned short*>(raw + kRawQ + j * 64 + lane * 2);
          char* at = stage + (j >> 3) * kATile;
          const int r = (j & 7) * 16 + g;
          const uint32_t f = e4m3x2_to_f16x2(sc);
          const uint32_t sg = __byte_perm(f, f, 0x1010), sg8 = __byte_perm(f, f, 0x3232);
          uint32_t o[4];
          dequant8(q.x, sg, o);
          *reinterpret_cast<uint4*>(at + sw128_off(r, 2 * c)) = make_uint4(o[0], o[1], o[2], o[3]);
          dequant8(q.y, sg, o);
          *reinterpret_cast<uint4*>(at + sw128_off(r, 2 * c + 1)) =
              make_uint4(o[0], o[1], o[2], o[3]);
          dequant8(q.z, sg8, o);
          *reinterpret_cast<uint4*>(at + sw128_off(r + 8, 2 * c)) =
              make_uint4(o[0], o[1], o[2], o[3]);
          dequant8(q.w, sg8, o);
          *reinterpret_cast<uint4*>(at + sw128_off(r + 8, 2 * c + 1)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async();
        if (kW13 && lane == 0) MOE_DBG(4, kd * kDqWarps + warp);
        mbar_arrive(&sm->a_full[as]);
        mbar_arrive(&sm->raw_empty[rs]);
        MOE_PROF(if (tid == 0) PROF_ADD(poff + 12, t0));
      }
      if (!ok) break;
      // ---- epilogue of this unit: warp w reads TMEM lanes 32 (w % 4) .. +31 of
      // accumulator w / 4 ----
      named_bar_sync(1, kDqThreads);  // epair / ewsc of this unit visible to every warp
      const int q4 = warp & 3, at = warp >> 2;
      MOE_PROF(long long te = clock64());
      if (!wait_or_abort(&sm->accf, it & 1, status, abort)) break;
      MOE_PROF(if (tid == 0) PROF_ADD(poff + 13, te); te = clock64());
      tc_fence_after();
      if (kW13) {
        // Lane r < 16 of warp q holds gate row (16q + r) and lane r + 16 the
        // matching up row, for 32 token columns per load.  One exchange per
        // pair of columns gives each lane 16 (G, U) pairs: gate lanes take
        // columns 0-15, up lanes 16-31.  h goes through a per-warp staging
        // tile so that each token row leaves as two 16-byte stores.
        const int I = d.I;
        const int r16 = lane & 15;
        const bool is_gate = lane < 16;
        __half(*stg)[16] = reinterpret_cast<__half(*)[16]>(sm->stage[warp]);
        {
          const int i0 = un.sub * 128 + at * 64 + q4 * 16;
#pragma unroll 1
          for (int c0 = 0; c0 < un.npad; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(q4 * 32) << 16) + at * 256 + c0, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float lo = __uint_as_float(v[jj]), hi = __uint_as_float(v[jj + 16]);
              const float recv = __shfl_xor_sync(0xffffffffu, is_gate ? hi : lo, 16);
              const float G = (is_gate ? lo : recv) * un.g;
              const float U = (is_gate ? recv : hi) * un.g;
              const float hv = __fdividef(G, 1.f + __expf(-G)) * U;
              stg[is_gate ? jj : jj + 16][r16] = __float2half_rn(hv);
            }
            __syncwarp();
            const int n = c0 + lane;
            if (n < un.rows) {
              const uint4* s4 = reinterpret_cast<const uint4*>(stg[lane]);
              uint4* dst = reinterpret_cast<uint4*>(h_out + (int64_t)(un.pos0 + n) * I + i0);
              dst[0] = s4[0];
              dst[1] = s4[1];
            }
            __syncwarp();
          }
        }
      } else {
        // Lane r of warp q holds output row hd = ... + 32q + r for 32 pair
        // columns per load; a per-warp staging tile turns 16 columns at a time
        // into rows of 32 contiguous FP32 values, written as 16-byte stores.
        const int H = d.H;
        const int* pr = sm->epair[it & 1];
        const float* wsc = sm->ewsc[it & 1];
        float(*stg)[32] = reinterpret_cast<float(*)[32]>(sm->stage[warp]);
        {
          const int hd0 = un.sub * 256 + at * 128 + q4 * 32;
#pragma unroll 1
          for (int c0 = 0; c0 < un.npad; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(q4 * 32) << 16) + at * 256 + c0, v);
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
                  float4 o = reinterpret_cast<const float4*>(stg[j])[part];
                  const float sc = wsc[n];
                  o.x *= sc;
                  o.y *= sc;
                  o.z *= sc;
                  o.w *= sc;
                  __stcs(reinterpret_cast<float4*>(partial + (int64_t)pr[n] * H + hd0) + part, o);
                }
              }
              __syncwarp();
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm->tmem_empty);
      MOE_PROF(if (tid == 0) PROF_ADD(poff + 14, te));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// xg[pos] = x[perm[pos] / k_eff]: the token rows in plan order, the operand of
// the grouped W13 GEMM (positions past the valid pairs are left alone).
// One warp per row, 16-byte loads and stores.
__global__ void gather_rows_kernel(LayerDims d, PlanView pv, const __half* __restrict__ x,
                                   __half* __restrict__ xg) {
  MOE_TL(kTlPlan);
  pdl_wait();
  pdl_launch_dependents();
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= __ldcg(&pv.hdr->n_valid)) return;
  const int t = __ldcg(pv.perm + row) / d.k_eff;
  const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)t * d.H);
  uint4* dst = reinterpret_cast<uint4*>(xg + row * d.H);
  for (int c = lane; c < d.H / 8; c += 32) dst[c] = __ldg(src + c);
}

cudaError_t launch_prefill_forward(const LayerDims& d, int64_t M, const __half* x,
                                   const PlanView& pv, Weights w13, Weights w2, Weights s13,
                                   Weights s2, __half* y, __half* h, float* partial,
                                   uint32_t* status, cudaStream_t stream, int num_sms) {
  const int64_t P = M * d.k_eff;
  const int max_tiles = max_tiles_for(P, d.e_eff);
  const size_t smem = gemm_smem_bytes();
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(grouped_gemm_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int g13 = (int)std::min<int64_t>((int64_t)max_tiles * ((2 * d.I) / 256), num_sms);
  const int g2 = (int)std::min<int64_t>((int64_t)max_tiles * (d.H / 256), num_sms);
  const bool pdl = !trace_on();
  // Token-row operands in plan order, read as 64-row tensor-map tiles (128-byte
  // swizzled): W13 reads x rows gathered into the partials buffer (unused until
  // the W2 grid, which starts after W13 has finished), W2 reads h.
  __half* xg = reinterpret_cast<__half*>(partial);
  CUtensorMap xmap, hmap;
  cudaError_t e = make_fp16_map(&xmap, xg, d.H, (uint64_t)P, kBK, kBChunkRows, true);
  if (e != cudaSuccess) return e;
  e = make_fp16_map(&hmap, h, d.I, (uint64_t)P, kBK, kBChunkRows, true);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW13, false);
  e = launch_k(gather_rows_kernel, dim3((unsigned)((P + 7) / 8)), dim3(256), 0, stream, pdl, d, pv,
               x, xg);
  if (e != cudaSuccess) return e;
  e = launch_k(grouped_gemm_kernel<true>, dim3(g13), dim3(kGemmThreads), smem, stream, pdl, d, pv,
               xmap, w13, s13, h, partial, status);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW13, true);
  trace_mark(stream, kTraceW2, false);
  e = launch_k(grouped_gemm_kernel<false>, dim3(g2), dim3(kGemmThreads), smem, stream, pdl, d,
               pv, hmap, w2, s2, h, partial, status);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW2, true);
  trace_mark(stream, kTraceCombine, false);
  e = launch_combine(d, M, pv, partial, y, stream, pdl);
  trace_mark(stream, kTraceCombine, true);
  return e;
}

}  // namespace moe
