// Prefill path (M > 16): expert-grouped GEMMs on the 5th-generation tensor
// cores (tcgen05, kind::f16, FP32 accumulators in tensor memory).
//
// "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Scope and
// related PRs": grouped W13 with SwiGLU and grouped W2 with the reduction,
// both driven by the same integer plan.  Here each block takes one plan tile
// (one expert, up to 256 of its routed rows) and 256 weight rows:
//
//   D[weight row][token] = sum_k W[weight row][k] * X[token][k]     (swap-AB)
//
// so the weight rows are the MMA's M = 128 (two accumulators) and the tokens
// are N <= 256.  Warp roles:
//   warps 0-3  dequantise NVFP4 weight blocks (fragment layout, 16-byte loads)
//              to FP16 in 128-byte-swizzled K-major shared tiles, then run the
//              epilogue (TMEM -> registers);
//   warps 4-7  gather the tile's token rows with 16-byte cp.async into the
//              same swizzled layout;
//   warp 8     allocates tensor memory, and one lane issues the MMAs.
// A 3-stage ring of (A0, A1, B) tiles of K = 64 is synchronised with mbarriers.
//
// W13: the fragment layout interleaves 16-row gate and up tiles, so TMEM lanes
// [32q, 32q+16) hold gate rows and [32q+16, 32q+32) the matching up rows; the
// epilogue pairs them with one shuffle and writes h = fp16(silu(G) * U).
// W2:  the epilogue scales by g2 and the pair's combine weight and writes the
// FP32 partial row of each pair; a separate pass sums the slots in order.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kStages = 3;
constexpr int kBK = 64;                       // K per stage (128 bytes of FP16)
constexpr int kATile = 128 * 128;             // one 128-row A tile, bytes
constexpr int kBTile = kTileRows * 128;       // the B tile, bytes
constexpr int kStageBytes = 2 * kATile + kBTile;
constexpr int kGemmThreads = 288;
constexpr int kTmemCols = 512;

struct GemmSmem {
  uint64_t full_a[kStages];
  uint64_t full_b[kStages];
  uint64_t empty[kStages];
  uint64_t accf;
  uint32_t tmem;
  int abort;
  int ep_ok;    // epilogue go/no-go, sampled once
  int rows;     // rows of this tile
  int pos0;     // plan position of the tile's first row
  int src[kTileRows];   // W13: token of each row; W2: pair id of each row
  float wsc[kTileRows]; // W2: g2 * combine weight of each row
};

constexpr size_t gemm_smem_bytes() {
  return 1024 /* alignment slack */ + (size_t)kStages * kStageBytes + sizeof(GemmSmem);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t* status,
                                              volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitTimeoutNs) {
      set_status(status, MOE_ST_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <bool kW13>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(LayerDims d, PlanView pv, const __half* __restrict__ bsrc, Weights w,
                        Weights ws, __half* __restrict__ h_out, float* __restrict__ partial,
                        uint32_t* status) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  GemmSmem* sm = reinterpret_cast<GemmSmem*>(base + (size_t)kStages * kStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work unit ------------------------------------------------------------
  const int K = kW13 ? d.H : d.I;            // reduction length
  const int S = K / kBK;                      // k-steps
  const int units_per_tile = kW13 ? (2 * d.I) / 256 : d.H / 256;
  MOE_TL(kW13 ? kTlW13 : kTlW2);
  pdl_wait();
  MOE_TL_WAITED();
  const int n_tiles = __ldcg(&pv.hdr->n_tiles);
  const int tile = blockIdx.x / units_per_tile;
  const int u = blockIdx.x - tile * units_per_tile;
  if (tile >= n_tiles) return;
  const int4 tl = __ldcg(reinterpret_cast<const int4*>(pv.tiles) + tile);
  const int e = tl.x, r0 = tl.y, rows = tl.z;
  const int npad = (rows + 15) & ~15;
  const bool sh = (e == d.E);
  const size_t mat_q = kW13 ? (size_t)d.I * d.H : (size_t)d.H * d.I / 2;
  const uint8_t* qe = sh ? ws.q : w.q + (size_t)e * mat_q;
  const uint8_t* se = sh ? ws.s : w.s + (size_t)e * mat_q / 8;
  const float gsc = sh ? ws.g[0] : w.g[e];

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm->full_a[s], 128);
      mbar_init(&sm->full_b[s], 128);
      mbar_init(&sm->empty[s], 1);
    }
    mbar_init(&sm->accf, 1);
    sm->abort = 0;
    sm->rows = rows;
    sm->pos0 = __ldcg(pv.offsets + e) + r0;
    fence_mbar_init();
  }
  if (warp == 8) tmem_alloc(&sm->tmem, kTmemCols);
  __syncthreads();
  if (tid >= 128 && tid < 256) {
    for (int n = tid - 128; n < rows; n += 128) {
      const int pair = __ldcg(pv.perm + sm->pos0 + n);
      sm->src[n] = kW13 ? pair / d.k_eff : pair;
      if (!kW13) sm->wsc[n] = gsc * __ldcg(pv.w + pair);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem;
  volatile int* abort = &sm->abort;

  if (warp < 4) {
    // ---- dequantising producer: 16 fragment blocks (2 A tiles x 8) per stage,
    //      4 per warp; raw bytes of the next stage are loaded ahead.
    const int g = lane >> 2, c = lane & 3;
    // packed row tile of block j of this warp: A tile at = j / 8 (j = 4w + jj)
    auto blk_q = [&](int jj, int ks) -> const uint8_t* {
      const int j = warp * 4 + jj;
      const int rt = u * 16 + j;  // A tile j/8, local tile j%8
      return qe + ((size_t)rt * S + ks) * 512 + lane * 16;
    };
    auto blk_s = [&](int jj, int ks) -> const uint8_t* {
      const int j = warp * 4 + jj;
      const int rt = u * 16 + j;
      return se + ((size_t)rt * S + ks) * 64 + lane * 2;
    };
    uint4 qn[4];
    uint32_t sn[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      qn[jj] = ldg_nc_v4(blk_q(jj, 0));
      sn[jj] = __ldg(reinterpret_cast<const unsigned short*>(blk_s(jj, 0)));
    }
    for (int ks = 0; ks < S; ++ks) {
      const int st = ks % kStages;
      uint4 qc[4];
      uint32_t sc[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        qc[jj] = qn[jj];
        sc[jj] = sn[jj];
      }
      if (ks + 1 < S) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          qn[jj] = ldg_nc_v4(blk_q(jj, ks + 1));
          sn[jj] = __ldg(reinterpret_cast<const unsigned short*>(blk_s(jj, ks + 1)));
        }
      }
      if (!wait_or_abort(&sm->empty[st], ((ks / kStages) & 1) ^ 1, status, abort)) break;
      char* stage = base + (size_t)st * kStageBytes;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = warp * 4 + jj;
        char* at = stage + (j >> 3) * kATile;
        const int r = (j & 7) * 16 + g;
        const uint32_t f = e4m3x2_to_f16x2(sc[jj]);
        const uint32_t sg = __byte_perm(f, f, 0x1010), sg8 = __byte_perm(f, f, 0x3232);
        uint32_t o[4];
        dequant8(qc[jj].x, sg, o);
        *reinterpret_cast<uint4*>(at + sw128_off(r, 2 * c)) = make_uint4(o[0], o[1], o[2], o[3]);
        dequant8(qc[jj].y, sg, o);
        *reinterpret_cast<uint4*>(at + sw128_off(r, 2 * c + 1)) =
            make_uint4(o[0], o[1], o[2], o[3]);
        dequant8(qc[jj].z, sg8, o);
        *reinterpret_cast<uint4*>(at + sw128_off(r + 8, 2 * c)) =
            make_uint4(o[0], o[1], o[2], o[3]);
        dequant8(qc[jj].w, sg8, o);
        *reinterpret_cast<uint4*>(at + sw128_off(r + 8, 2 * c + 1)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
      fence_proxy_async();
      mbar_arrive(&sm->full_a[st]);
    }
  } else if (warp < 8) {
    // ---- B producer: gather rows with cp.async; stage ks is announced once
    //      the copies of ks have landed (two stages kept in flight).
    const int t = tid - 128;
    const int chunks = npad * 8;
    int issued = 0, announced = 0;
    bool ok = true;
    for (int ks = 0; ks < S && ok; ++ks) {
      const int st = ks % kStages;
      if (!wait_or_abort(&sm->empty[st], ((ks / kStages) & 1) ^ 1, status, abort)) {
        ok = false;
        break;
      }
      const uint32_t bt = smem_u32(base + (size_t)st * kStageBytes + 2 * kATile);
      for (int i = t; i < chunks; i += 128) {
        const int n = i >> 3, c = i & 7;
        const bool in = n < rows;
        const __half* src;
        if (kW13)
          src = bsrc + (int64_t)(in ? sm->src[n] : 0) * d.H + ks * kBK + c * 8;
        else
          src = bsrc + (int64_t)(in ? sm->pos0 + n : 0) * d.I + ks * kBK + c * 8;
        cp_async16(bt + sw128_off(n, c), src, in ? 16u : 0u);
      }
      cp_async_commit();
      ++issued;
      if (issued - announced > 2) {
        cp_async_wait<2>();
        fence_proxy_async();
        mbar_arrive(&sm->full_b[announced % kStages]);
        ++announced;
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    for (; announced < issued; ++announced) mbar_arrive(&sm->full_b[announced % kStages]);
  } else if (lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = idesc_f16_f32(128, npad);
    for (int ks = 0; ks < S; ++ks) {
      const int st = ks % kStages;
      const uint32_t par = (ks / kStages) & 1;
      if (!wait_or_abort(&sm->full_a[st], par, status, abort)) break;
      if (!wait_or_abort(&sm->full_b[st], par, status, abort)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(base + (size_t)st * kStageBytes);
      const uint32_t a1 = a0 + kATile;
      const uint32_t b0 = a0 + 2 * kATile;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint32_t acc = (ks | kk) ? 1u : 0u;
        tc_mma_f16(tmem, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc, acc);
        tc_mma_f16(tmem + 256, sdesc_sw128(a1 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc, acc);
      }
      tc_commit(&sm->empty[st]);
    }
    tc_commit(&sm->accf);
  }

  // ---- epilogue (warps 0-3: TMEM lanes 32*warp .. +31) -----------------------
  if (warp < 4) {
    wait_or_abort(&sm->accf, 0, status, abort);
    named_bar_sync(1, 128);
    if (tid == 0) sm->ep_ok = !*abort;
    named_bar_sync(1, 128);
    tc_fence_after();
    if (sm->ep_ok) {
      if (kW13) {
        // h staging: [rows][128 i-values] FP16, 272-byte rows, in the dead ring
        __half* hs = reinterpret_cast<__half*>(base);
        const int hst = 136;
        const int r16 = lane & 15;
        const bool is_gate = lane < 16;
#pragma unroll 1
        for (int at = 0; at < 2; ++at) {
          const int il = at * 64 + warp * 16 + r16;
#pragma unroll 1
          for (int c0 = 0; c0 < npad; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + at * 256 + c0, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float mine = __uint_as_float(v[j]);
              const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
              // gate lanes take columns 0..15, up lanes 16..31
              const bool take = is_gate ? (j < 16) : (j >= 16);
              if (take) {
                const float G = (is_gate ? mine : other) * gsc;
                const float U = (is_gate ? other : mine) * gsc;
                const int n = c0 + j;
                if (n < rows) hs[n * hst + il] = __float2half_rn(G / (1.f + expf(-G)) * U);
              }
            }
          }
        }
        named_bar_sync(1, 128);
        const int I = d.I;
        for (int i = tid; i < rows * 16; i += 128) {
          const int n = i >> 4, c = i & 15;
          const uint4 v = *reinterpret_cast<const uint4*>(hs + n * hst + c * 8);
          *reinterpret_cast<uint4*>(h_out + (int64_t)(sm->pos0 + n) * I + u * 128 + c * 8) = v;
        }
      } else {
        const int H = d.H;
#pragma unroll 1
        for (int at = 0; at < 2; ++at) {
          const int hd = u * 256 + at * 128 + warp * 32 + lane;
#pragma unroll 1
          for (int c0 = 0; c0 < npad; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + at * 256 + c0, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int n = c0 + j;
              if (n < rows)
                __stcs(partial + (int64_t)sm->src[n] * H + hd, __uint_as_float(v[j]) * sm->wsc[n]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t launch_prefill_forward(const LayerDims& d, int64_t M, const __half* x,
                                   const PlanView& pv, Weights w13, Weights w2, Weights s13,
                                   Weights s2, __half* y, __half* h, float* partial,
                                   uint32_t* status, cudaStream_t stream, int num_sms) {
  (void)num_sms;
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
  const bool pdl = !trace_on();
  trace_mark(stream, kTraceW13, false);
  cudaError_t e = launch_k(grouped_gemm_kernel<true>, dim3(max_tiles * ((2 * d.I) / 256)),
                           dim3(kGemmThreads), smem, stream, pdl, d, pv, x, w13, s13, h, partial,
                           status);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW13, true);
  trace_mark(stream, kTraceW2, false);
  e = launch_k(grouped_gemm_kernel<false>, dim3(max_tiles * (d.H / 256)), dim3(kGemmThreads),
               smem, stream, pdl, d, pv, (const __half*)h, w2, s2, h, partial, status);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW2, true);
  trace_mark(stream, kTraceCombine, false);
  e = launch_combine(d, M, pv, partial, y, stream, pdl);
  trace_mark(stream, kTraceCombine, true);
  return e;
}

}  // namespace moe
