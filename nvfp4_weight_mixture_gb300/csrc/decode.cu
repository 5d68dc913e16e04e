// Decode path (M <= 16): the weight-streaming forward (W13 + SwiGLU, then W2
// with the fixed-order combine), and the combine kernel of the prefill path.
//
// The layer is HBM-bound here: every touched expert's NVFP4 bytes are read
// once.  Weights are stored in the fragment layout, so each warp reads one
// 512-byte block per 16-row x 64-element piece with a single 16-byte load per
// thread; the thread dequantises its 32 codes in registers (exact E2M1 x E4M3
// products in FP16) straight into mma.sync m16n8k16 A fragments, and the
// tokens of the expert are the N = 8 / 16 columns.
//
// Pages: "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", sections "Scope
// and related PRs" (expert-grouped multi-row W13/SiLU with intra-CTA split-K;
// grouped W2 reusing the integer plan; M2-M16 dynamic dispatch) and "Latest
// grouped-MoE screen" (the complete C16 decode call).
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ uint16_t ldg_u16(const uint8_t* p) {
  return __ldg(reinterpret_cast<const unsigned short*>(p));
}
__device__ __forceinline__ uint32_t ldg_u32(const uint8_t* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// Scale storage: SB = 1 raw E4M3 bytes, SB = 2 prepared FP16 scales (each raw
// byte widened to two bytes in place, so every scale offset doubles).  The
// two scales of a fragment lane (rows g and g + 8) sit at raw byte offset
// `off`: loaded as they are (no wait on the load here) ...
template <int SB>
__device__ __forceinline__ uint32_t lane_scales_ldg(const uint8_t* base, size_t off) {
  if constexpr (SB == 1)
    return ldg_u16(base + off);
  else
    return ldg_u32(base + 2 * off);
}
template <int SB>
__device__ __forceinline__ uint32_t lane_scales_smem(const char* base, size_t off) {
  if constexpr (SB == 1)
    return *reinterpret_cast<const unsigned short*>(base + off);
  else
    return *reinterpret_cast<const uint32_t*>(base + 2 * off);
}
// ... and turned into the FP16 splats when they are used.
template <int SB>
__device__ __forceinline__ void lane_splats(uint32_t v, uint32_t* sg, uint32_t* sg8) {
  if constexpr (SB == 1)
    scale_splats(v, sg, sg8);
  else
    scale_splats_f16(v, sg, sg8);
}

// ---------------------------------------------------------------------------
// Decode forward = two kernels in programmatic dependent launch:
//   W13 + SwiGLU: persistent blocks walk the items (active expert, pair of
//     gate / up 16-row tiles); the block's 8 warps split K, reduce in shared
//     memory in a fixed order and write h[pos][i] = fp16(silu(g13 G) * (g13 U)).
//   W2 + combine: one block per 16-row tile of H; its warps take the active
//     experts in turn, each computing o = g2 * W2[tile] . h for the expert's
//     pairs into shared memory; the block then sums every token's slots in
//     order, y[t][tile] = fp16(sum_j w_j o_j).  Weights (TMA), pair ids and
//     combine weights of a warp's first experts are fetched before waiting on
//     the W13 grid, so only the h rows are read after it.
// ---------------------------------------------------------------------------
struct DecodeArgs {
  LayerDims d;
  PlanView pv;
  const __half* x;
  Weights w13, s13, w2, s2;
  __half* h;
  __half* y;
  uint32_t* status;
  int M;
  int max_active;  // work-table entries that can be valid (min(M * k_eff, e_eff))
  int sb;          // bytes per stored scale (1 raw, 2 prepared)
};

// A work-table entry names a routed expert (or the shared one) and a run of
// plan positions inside [0, M * k_eff); anything else is skipped.
__device__ __forceinline__ bool entry_ok(const DecodeArgs& p, int e, int base, int count) {
  const int P = p.M * p.d.k_eff;
  return e >= 0 && (e < p.d.E || (e == p.d.E && p.d.shared)) && base >= 0 && count >= 0 &&
         base + count <= P;
}

// W13 item (a, rp) for one block of 256 threads.  xs: staged token rows
// (stride 2H + 16).
template <int NT, int SB>
__device__ __forceinline__ void w13_item(const DecodeArgs& p, const int* en, int rp,
                                         const char* xs, float* red, int* s_tok) {
  const LayerDims& d = p.d;
  const int H = d.H, I = d.I;
  const int e = en[0], base = en[1], count = en[2];
  if (!entry_ok(p, e, base, count)) return;
  const bool sh = (e == d.E);
  const uint8_t* qe = sh ? p.s13.q : p.w13.q + (size_t)e * I * H;
  const uint8_t* se = sh ? p.s13.s : p.w13.s + (size_t)e * I * H / 8 * SB;
  const float gsc = sh ? p.s13.g[0] : p.w13.g[e];
  const int ttid = threadIdx.x, warp = ttid >> 5, lane = ttid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int S = H / 64;
  // gate tile 2*rp and up tile 2*rp+1: tiles j0, j0 + 1 of 256-row group rp / 8;
  // block (tile j, segment ks) of a group is number ks * 16 + j within it
  const int j0 = 2 * (rp & 7);
  const uint8_t* qt = qe + (size_t)(rp >> 3) * S * 16 * 512 + j0 * 512;
  const size_t st = (size_t)(rp >> 3) * S * 16 * 64 + j0 * 64;  // raw scale offset
  const int xstride = H * 2 + 16;

  uint4 qv[4][2];
  uint32_t sv[4][2];
  // this warp's segments: ks = warp + 8 * j, in groups of 4
  auto load_group = [&](int ks0) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ks = ks0 + 8 * j;
      if (ks < S) {
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          qv[j][tt] = ldg_nc_v4(qt + ((size_t)ks * 16 + tt) * 512 + lane * 16);
          sv[j][tt] = lane_scales_ldg<SB>(se, st + ((size_t)ks * 16 + tt) * 64 + lane * 2);
        }
      }
    }
  };

  // the expert's rows in chunks of NT * 8 (one chunk unless given ids repeat
  // an expert within a token)
  for (int n0 = 0; n0 < count; n0 += NT * 8) {
    const int n_e = min(count - n0, NT * 8);
    const int pos0 = base + n0;
    load_group(warp);
    if (ttid < n_e) {
      const int pair = (n0 + ttid < 16) ? en[4 + n0 + ttid] : __ldcg(p.pv.perm + pos0 + ttid);
      s_tok[ttid] = min(max(pair / d.k_eff, 0), p.M - 1);
    }
    __syncthreads();
    float acc[2][NT][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[t][n][c] = 0.f;
    for (int ks0 = warp; ks0 < S; ks0 += 32) {
      if (ks0 != warp) load_group(ks0);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ks = ks0 + 8 * j;
        if (ks >= S) break;
        uint32_t xw[NT][8];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int n = nt * 8 + g;
          if (n < n_e) {
            const char* src = xs + s_tok[n] * xstride + (ks * 64 + 16 * t4) * 2;
            const uint4 v0 = *reinterpret_cast<const uint4*>(src);
            const uint4 v1 = *reinterpret_cast<const uint4*>(src + 16);
            xw[nt][0] = v0.x; xw[nt][1] = v0.y; xw[nt][2] = v0.z; xw[nt][3] = v0.w;
            xw[nt][4] = v1.x; xw[nt][5] = v1.y; xw[nt][6] = v1.z; xw[nt][7] = v1.w;
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) xw[nt][u] = 0u;
          }
        }
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
          uint32_t sg, sg8;
          lane_splats<SB>(sv[j][tt], &sg, &sg8);
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            uint32_t af[4];
            a_frag(qv[j][tt], sg, sg8, s, af);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_16816(acc[tt][nt], af, xw[nt][2 * s], xw[nt][2 * s + 1]);
          }
        }
      }
    }
    if (ttid == 0) {
      MOE_TL_MAX(44);
      MOE_TL_MIN(45);
    }
    // red[warp][tt][nt][lane][c]
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          red[(((warp * 2 + tt) * NT + nt) * 32 + lane) * 4 + c] = acc[tt][nt][c];
    __syncthreads();
    if (ttid < NT * 128) {
      const int nt = ttid >> 7, ln = (ttid >> 2) & 31, c = ttid & 3;
      float G = 0.f, U = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        G += red[(((w * 2 + 0) * NT + nt) * 32 + ln) * 4 + c];
        U += red[(((w * 2 + 1) * NT + nt) * 32 + ln) * 4 + c];
      }
      // c0: (row g, col 2t4), c1: (g, 2t4+1), c2: (g+8, 2t4), c3: (g+8, 2t4+1)
      const int row = (ln >> 2) + ((c & 2) ? 8 : 0);
      const int n = nt * 8 + 2 * (ln & 3) + (c & 1);
      if (n < n_e) {
        G *= gsc;
        U *= gsc;
        const float hv = G / (1.f + expf(-G)) * U;
        p.h[(int64_t)(pos0 + n) * I + 16 * rp + row] = __float2half_rn(hv);
      }
    }
    __syncthreads();  // red / s_tok reused by the next chunk or item
  }
}

template <int NT, int SB>
__global__ void __launch_bounds__(256, NT == 1 ? 3 : 2) decode_w13_kernel(const DecodeArgs p) {
  extern __shared__ __align__(16) char dsm[];  // staged token rows, then the reduction area
  __shared__ int s_tok[16];
  __shared__ int s_ent[kDtabInts];
  __shared__ int s_nact;
  MOE_TL(kTlW13);
  const LayerDims& d = p.d;
  const int H = d.H, I = d.I;
  const int tid = threadIdx.x;
  char* xs = dsm;
  const int xstride = H * 2 + 16, cpr = H / 8;
  float* red = reinterpret_cast<float*>(dsm + align_up((size_t)p.M * xstride, 16));
  // token rows: inputs of the layer, staged before waiting on the plan grid
  for (int i = tid; i < p.M * cpr; i += 256) {
    const int n = i / cpr, c = i - n * cpr;
    cp_async16(smem_u32(xs + n * xstride + c * 16), p.x + (int64_t)n * H + c * 8, 16u);
  }
  cp_async_commit();
  pdl_wait();
  MOE_TL_WAITED();
  pdl_launch_dependents();
  const int n_rtp = I / 16;
  if (tid == 0) s_nact = min(__ldcg(&p.pv.hdr->n_active), p.max_active);
  if (tid < kDtabInts && blockIdx.x < p.max_active * n_rtp)
    s_ent[tid] = __ldcg(p.pv.dtab + (blockIdx.x / n_rtp) * kDtabInts + tid);
  cp_async_wait<0>();
  __syncthreads();
  if (tid == 0) {
    MOE_TL_MAX(34);
    MOE_TL_MIN(35);
  }
  const int n13 = s_nact * n_rtp;
  for (int i = blockIdx.x; i < n13; i += gridDim.x) {
    const int a = i / n_rtp, rp = i - a * n_rtp;
    if (i != (int)blockIdx.x) {
      // w13_item ended with a barrier: s_ent of the previous item is no longer read
      if (tid < kDtabInts) s_ent[tid] = __ldcg(p.pv.dtab + a * kDtabInts + tid);
      __syncthreads();
    }
    w13_item<NT, SB>(p, s_ent, rp, xs, red, s_tok);
  }
}

// W2 + combine: grid = H / 16 (one 16-row tile of H per block), 512 threads.
constexpr int kW2Warps = 16;

// Rows of a fragment-layout tensor map: row (m * rows / 256 + G) * (k / 64) + ks
// holds the 16 tile blocks of segment ks of 256-row group G of matrix m.
__device__ __forceinline__ int frag_map_row(int m, int groups, int G, int S, int ks) {
  return (m * groups + G) * S + ks;
}

// W2 + combine.  Warp w < w2_warps takes experts a = w, w + w2_warps, ...; the
// expert's 16-row tile of W2 (codes and scales over the full K = I) arrives by
// two 2-D tensor-map loads into one of the warp's two shared-memory stages,
// the first two issued before waiting on the W13 grid.  Each expert's pairs
// get o = g2 * w_pair * (W2[tile] . h) in shared memory; the block then sums
// every token's slots in order, y[t][tile] = fp16(sum_j o_j).
template <int NT, int SB>
__global__ void __launch_bounds__(kW2Warps * 32, 1)
    decode_w2_kernel(const DecodeArgs p, int w2_warps, int stage_bytes,
                         const __grid_constant__ CUtensorMap mq,
                         const __grid_constant__ CUtensorMap ms,
                         const __grid_constant__ CUtensorMap mqs,
                         const __grid_constant__ CUtensorMap mss) {
  extern __shared__ __align__(1024) char dsm_raw[];
  char* dsm = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                      ~uintptr_t(1023));
  __shared__ uint64_t full[kW2Warps][2];
  MOE_TL(kTlW2);
  // the next layer call's router may start its weight copies now (it waits
  // for this whole grid before it reads anything this call writes)
  pdl_launch_dependents();
  const LayerDims& d = p.d;
  const int H = d.H, I = d.I, k_eff = d.k_eff;
  const int P = p.M * k_eff;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int rt = blockIdx.x;  // 16-row tile of H: tile rt % 16 of 256-row group rt / 16
  const int S = I / 64, groups = H / 256;
  char* wst = dsm + (size_t)warp * 2 * stage_bytes;  // this warp's two stages
  float* o_s = reinterpret_cast<float*>(dsm + (size_t)w2_warps * 2 * stage_bytes);  // [P][16]
  unsigned char* valid = reinterpret_cast<unsigned char*>(o_s + (size_t)P * 16);    // [P]
  const bool worker = warp < w2_warps;
  if (worker && lane == 0) {
    mbar_init(&full[warp][0], 1);
    mbar_init(&full[warp][1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  // ---- everything that comes from the plan grid (complete before W13 began) ----
  for (int q = tid; q < P; q += kW2Warps * 32) valid[q] = __ldcg(p.pv.inv + q) >= 0;
  const int n_act = min(__ldcg(&p.pv.hdr->n_active), p.max_active);
  const uint32_t tx = (uint32_t)S * (512 + 64 * SB);
  // chunk r of this warp = expert a = warp + r * w2_warps, in stage r % 2
  auto entry = [&](int r) {
    const int a = warp + r * w2_warps;
    return (a < n_act && lane < kDtabInts) ? __ldcg(p.pv.dtab + a * kDtabInts + lane) : -1;
  };
  // issues chunk r (entry values in lanes 0..19 of ev); returns, on every
  // lane, whether a copy was issued
  auto issue = [&](int r, int ev) {
    const int e = __shfl_sync(0xffffffffu, ev, 0);
    const int base = __shfl_sync(0xffffffffu, ev, 1);
    const int count = __shfl_sync(0xffffffffu, ev, 2);
    const bool go = warp + r * w2_warps < n_act && entry_ok(p, e, base, count);
    if (go && lane == 0) {
      const bool sh = (e == d.E);
      const int row0 = frag_map_row(sh ? 0 : e, groups, rt >> 4, S, 0);
      char* st = wst + (r & 1) * stage_bytes;
      uint64_t* bar = &full[warp][r & 1];
      mbar_expect_tx(bar, tx);
      tma_load_2d(st, sh ? &mqs : &mq, (rt & 15) * 64, row0, bar);
      tma_load_2d(st + S * 512, sh ? &mss : &ms, (rt & 15) * 8 * SB, row0, bar);
    }
    return go;
  };
  int ent_cur = -1, ent_next = -1;
  float wsc = 0.f;
  int pair_l = -1;
  bool iss_cur = false, iss_next = false;  // chunk r / r + 1 has a copy in flight
  if (worker) {
    ent_cur = entry(0);
    ent_next = entry(1);
    iss_cur = issue(0, ent_cur);
    iss_next = issue(1, ent_next);
  }
  auto pairs_of = [&](int ev) {
    const int e = __shfl_sync(0xffffffffu, ev, 0);
    const int count = __shfl_sync(0xffffffffu, ev, 2);
    const int pr = __shfl_sync(0xffffffffu, ev, (4 + lane) & 31);
    pair_l = (lane < 16 && lane < count && pr >= 0 && pr < P) ? pr : -1;
    const bool sh = (e == d.E);
    const float gsc = (e >= 0 && (e < d.E || (sh && d.shared))) ? (sh ? p.s2.g[0] : p.w2.g[e]) : 0.f;
    wsc = pair_l >= 0 ? gsc * __ldcg(p.pv.w + pair_l) : 0.f;
  };
  if (worker) pairs_of(ent_cur);
  pdl_wait();
  MOE_TL_WAITED();
  bool ok = true;
  int r = 0;
  if (worker) {
    for (; warp + r * w2_warps < n_act; ++r) {
      if (r > 0) pairs_of(ent_cur);
      const int e = __shfl_sync(0xffffffffu, ent_cur, 0);
      const int base = __shfl_sync(0xffffffffu, ent_cur, 1);
      const int count = __shfl_sync(0xffffffffu, ent_cur, 2);
      if (iss_cur) {
        if (!mbar_wait(&full[warp][r & 1], (r >> 1) & 1, p.status)) {
          ok = false;
          break;
        }
        const bool sh = (e == d.E);
        const float gsc = sh ? p.s2.g[0] : p.w2.g[e];
        const char* sq = wst + (r & 1) * stage_bytes;
        const char* ss = sq + S * 512;
        for (int n0 = 0; n0 < count; n0 += 8) {
          const int n = n0 + g;
          int pair_n = __shfl_sync(0xffffffffu, pair_l, n & 15);
          float wsc_n = __shfl_sync(0xffffffffu, wsc, n & 15);
          if (n >= 16 && n < count) {
            pair_n = __ldcg(p.pv.perm + base + n);
            if (pair_n < 0 || pair_n >= P) pair_n = -1;
            wsc_n = pair_n >= 0 ? gsc * __ldcg(p.pv.w + pair_n) : 0.f;
          }
          if (n >= count) pair_n = -1;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int ks0 = 0; ks0 < S; ks0 += 8) {
            uint4 hv[8][2];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (ks0 + j < S && n < count) {
                const __half* src = p.h + (int64_t)(base + n) * I + (ks0 + j) * 64 + 16 * t4;
                hv[j][0] = __ldcg(reinterpret_cast<const uint4*>(src));
                hv[j][1] = __ldcg(reinterpret_cast<const uint4*>(src) + 1);
              } else {
                hv[j][0] = hv[j][1] = make_uint4(0u, 0u, 0u, 0u);
              }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int ks = ks0 + j;
              if (ks >= S) break;
              const uint4 q = *reinterpret_cast<const uint4*>(sq + ks * 512 + lane * 16);
              uint32_t sg, sg8;
              lane_splats<SB>(lane_scales_smem<SB>(ss, (size_t)ks * 64 + lane * 2), &sg, &sg8);
              const uint32_t xw[8] = {hv[j][0].x, hv[j][0].y, hv[j][0].z, hv[j][0].w,
                                      hv[j][1].x, hv[j][1].y, hv[j][1].z, hv[j][1].w};
#pragma unroll
              for (int s = 0; s < 4; ++s) {
                uint32_t af[4];
                a_frag(q, sg, sg8, s, af);
                mma_16816(acc, af, xw[2 * s], xw[2 * s + 1]);
              }
            }
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int col = 2 * t4 + (c & 1);
            const int pr = __shfl_sync(0xffffffffu, pair_n, col * 4);
            const float ws = __shfl_sync(0xffffffffu, wsc_n, col * 4);
            if (pr >= 0) o_s[pr * 16 + g + ((c & 2) ? 8 : 0)] = acc[c] * ws;
          }
        }
      }
      __syncwarp();  // every lane is done with stage r & 1
      ent_cur = ent_next;
      iss_cur = iss_next;
      ent_next = entry(r + 2);
      iss_next = issue(r + 2, ent_next);
    }
    if (!ok && lane == 0) {
      // timed out: let the copies already issued land before the block exits
      // (each wait bounded by the same limit)
      mbar_wait(&full[warp][r & 1], (r >> 1) & 1, p.status);
      if (iss_next) mbar_wait(&full[warp][(r + 1) & 1], ((r + 1) >> 1) & 1, p.status);
    }
  }
  __syncthreads();
  // ---- combine: y[t][tile] = fp16(sum_j o[t * k_eff + j]), slots in order ----
  for (int i = tid; i < p.M * 16; i += kW2Warps * 32) {
    const int t = i >> 4, r = i & 15;
    float sum = 0.f;
    for (int j = 0; j < k_eff; ++j) {
      const int pr = t * k_eff + j;
      if (valid[pr]) sum += o_s[pr * 16 + r];
    }
    p.y[(int64_t)t * H + rt * 16 + r] = __float2half_rn(sum);
  }
}

// ---------------------------------------------------------------------------
// y[t] = fp16( sum_{j < k_eff} partial[inv[t * k_eff + j]] ), slots in order,
// FP32 sums of the FP16 partial rows (which sit at the pairs' plan
// positions); pairs dropped from the plan (invalid ids) contribute nothing.
// ---------------------------------------------------------------------------
__global__ void combine_kernel(int M, int H, int k_eff, const int32_t* __restrict__ inv,
                               const __half* __restrict__ partial, __half* __restrict__ y) {
  MOE_TL(kTlCombine);
  pdl_wait();
  MOE_TL_WAITED();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // 8 elements of y
  const int64_t n8 = (int64_t)M * H / 8;
  if (i >= n8) return;
  const int64_t t = (i * 8) / H;
  const int c = (int)(i * 8 - t * H);
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < k_eff; ++j) {
    const int64_t pos = __ldcg(inv + t * k_eff + j);  // the pair's plan position
    if (pos < 0) continue;
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(partial + pos * H + c));
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w4[q]));
      s[2 * q] += f.x;
      s[2 * q + 1] += f.y;
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2 hq = __floats2half2_rn(s[2 * q], s[2 * q + 1]);
    o[q] = *reinterpret_cast<const uint32_t*>(&hq);
  }
  *reinterpret_cast<uint4*>(y + t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

cudaError_t launch_combine(const LayerDims& d, int64_t M, const PlanView& pv,
                           const __half* partial, __half* y, cudaStream_t stream, bool pdl) {
  const int64_t n8 = M * d.H / 8;
  const unsigned blocks = (unsigned)((n8 + 255) / 256);
  return launch_k(combine_kernel, dim3(blocks), dim3(256), 0, stream, pdl, (int)M, d.H, d.k_eff,
                  (const int32_t*)pv.inv, partial, y);
}

static constexpr size_t kDecSmemLimit = 225 * 1024;

template <int NT, int SB>
static cudaError_t decode_impl(const LayerDims& d, int64_t M, const __half* x, const PlanView& pv,
                               Weights w13, Weights w2, Weights s13, Weights s2, __half* y,
                               __half* h, uint32_t* status, cudaStream_t stream, int num_sms) {
  DecodeArgs a;
  a.status = status;
  a.d = d;
  a.pv = pv;
  a.x = x;
  a.w13 = w13;
  a.s13 = s13;
  a.w2 = w2;
  a.s2 = s2;
  a.h = h;
  a.y = y;
  a.M = (int)M;
  a.max_active = (int)((M * d.k_eff < d.e_eff) ? M * d.k_eff : d.e_eff);
  a.sb = SB;
  const int P = (int)(M * d.k_eff);
  const int S2 = d.I / 64;
  const size_t smem13 =
      align_up((size_t)M * (d.H * 2 + 16), 16) + (size_t)8 * 2 * NT * 32 * 4 * sizeof(float);
  const int st2 = (int)align_up((size_t)S2 * (512 + 64 * SB), 1024);
  const size_t o_b = (size_t)P * 16 * sizeof(float) + P;
  // W2: as many expert warps as two ring stages each allow (at least one:
  // 2 x 37 KB + 34 KB at the largest I and M)
  const int w2_warps =
      (int)std::min<size_t>(kW2Warps, (kDecSmemLimit - 1024 - o_b) / (2 * (size_t)st2));
  if (w2_warps < 1) return cudaErrorInvalidValue;
  int per_sm = 0;
  cudaError_t e =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_w13_kernel<NT, SB>, 256, smem13);
  if (e != cudaSuccess) return e;
  const int n_items = a.max_active * (d.I / 16);
  const int g13 = std::max(1, std::min(n_items, num_sms * std::max(per_sm, 1)));
  const bool pdl = !trace_on();
  trace_mark(stream, kTraceW13, false);
  e = launch_k(decode_w13_kernel<NT, SB>, dim3(g13), dim3(256), smem13, stream, pdl, a);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW13, true);
  trace_mark(stream, kTraceW2, false);
  CUtensorMap mq, ms, mqs, mss;
  const uint64_t rows = (uint64_t)d.E * (d.H / 256) * S2;
  const uint64_t rows_sh = (uint64_t)(d.H / 256) * S2;
  if ((e = make_rows_map(&mq, w2.q, 16 * 512, rows, 512, S2)) != cudaSuccess) return e;
  if ((e = make_rows_map(&ms, w2.s, 16 * 64 * SB, rows, 64 * SB, S2)) != cudaSuccess) return e;
  mqs = mq;
  mss = ms;
  if (d.shared) {
    if ((e = make_rows_map(&mqs, s2.q, 16 * 512, rows_sh, 512, S2)) != cudaSuccess) return e;
    if ((e = make_rows_map(&mss, s2.s, 16 * 64 * SB, rows_sh, 64 * SB, S2)) != cudaSuccess) return e;
  }
  const size_t smem2 = 1024 + (size_t)w2_warps * 2 * st2 + o_b;
  e = launch_k(decode_w2_kernel<NT, SB>, dim3(d.H / 16), dim3(kW2Warps * 32), smem2, stream, pdl, a,
               w2_warps, st2, mq, ms, mqs, mss);
  if (e != cudaSuccess) return e;
  trace_mark(stream, kTraceW2, true);
  // the combine is part of the W2 kernel on this path
  trace_mark(stream, kTraceCombine, false);
  trace_mark(stream, kTraceCombine, true);
  return cudaSuccess;
}

cudaError_t decode_device_init() {
  for (auto f : {(const void*)decode_w13_kernel<1, 1>, (const void*)decode_w2_kernel<1, 1>,
                 (const void*)decode_w13_kernel<2, 1>, (const void*)decode_w2_kernel<2, 1>,
                 (const void*)decode_w13_kernel<1, 2>, (const void*)decode_w2_kernel<1, 2>,
                 (const void*)decode_w13_kernel<2, 2>, (const void*)decode_w2_kernel<2, 2>}) {
    cudaError_t e =
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmemLimit);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_decode_forward(const LayerDims& d, int64_t M, const __half* x,
                                  const PlanView& pv, Weights w13, Weights w2, Weights s13,
                                  Weights s2, __half* y, __half* h, __half* partial,
                                  uint32_t* status, cudaStream_t stream, int num_sms,
                                  bool prepared) {
  (void)partial;
  if (prepared) {
    if (M <= 8)
      return decode_impl<1, 2>(d, M, x, pv, w13, w2, s13, s2, y, h, status, stream, num_sms);
    return decode_impl<2, 2>(d, M, x, pv, w13, w2, s13, s2, y, h, status, stream, num_sms);
  }
  if (M <= 8) return decode_impl<1, 1>(d, M, x, pv, w13, w2, s13, s2, y, h, status, stream, num_sms);
  return decode_impl<2, 1>(d, M, x, pv, w13, w2, s13, s2, y, h, status, stream, num_sms);
}

}  // namespace moe
