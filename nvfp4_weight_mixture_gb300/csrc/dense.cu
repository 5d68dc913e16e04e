// Dense weight-streaming projection of a few FP16 rows (M <= 32), and the
// load-time helpers of its two other weight formats.
//
// "[SM70][Draft] Extend Qwen3.8 DFlash2 concurrency paths": section "Purpose"
// (NVFP4 QPN2 tiled in independent eight-row CTAs, admitted through M <= 32),
// section "TP4-only NVFP4 verifier follow-up" (packed MLP weights reused with
// split-K and the FP32 reduction order preserved; M9 / M15 / M16 bitwise equal
// to concatenated M8 calls) and section "Follow-up: exact channel-FP8 QPN8
// concurrency paths" (the same few-row path over FP8 weights with one scale
// per output channel).  "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency",
// sections "Purpose" and "Scope and related PRs": prepared effective decode
// scales beside raw E4M3 scale storage.
//
//   y[m][n] = fp16( scale_n * sum_k x[m][k] * w16[n][k] )
//
// with w16 the exact FP16 value of the weight (E2M1 x E4M3 for NVFP4, E4M3 for
// FP8), FP32 accumulation, scale_n the FP32 global scale (NVFP4) or the
// channel scale (FP8).
//
// Design.  The weights are the only large operand (HBM-bound), so the kernel
// streams them once.  The work is the (256-row group, 64-element K segment)
// pairs of the fragment layout, G-major; a fixed grid of kDnBlocks blocks
// takes equal contiguous ranges of it, so every block streams the same number
// of bytes.  A block's range falls into one or two "pieces" (the part inside
// one group).  A producer thread fills a ring of stages, each one K segment
// of a group (the group's 16 fragment tiles, contiguous, by one or two bulk
// copies) plus the same segment of every token row (one 128-byte-swizzled
// tensor-map tile).  Sixteen warps own one 16-row tile each (enough warps per
// SM to overlap the dequantise / MMA dependency chains), dequantise their
// fragments in registers straight into mma.sync A operands and multiply with
// up to four 8-token column tiles.  A piece that is a whole group writes y;
// otherwise it writes FP32 partial sums and takes a ticket of its group, and
// the block that completes the group adds the group's pieces in K order and
// writes y.  The ranges depend on N and K only, and a token's column of the
// MMA does not depend on the other columns, so every output row is computed
// by the same operations whatever M is: results are bitwise independent of
// the batch.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDnWarps = 16;                        // consumer warps
constexpr int kDnTpw = 16 / kDnWarps;               // 16-row tiles of a group per consumer warp
constexpr int kDnThreads = (kDnWarps + 1) * 32;     // + one producer warp
constexpr int kDnBlocks = 152;                      // fixed grid (one block per SM of a GB300)
constexpr int kDnRingBudget = 216 * 1024;

// Per weight format: bytes of one (group, segment) of codes (kQ) and scales
// (kS), and kCH, the most consecutive segments one ring stage carries (one
// bulk copy each for codes and scales, one tensor-map copy for the token rows:
// few large copies keep many bytes in flight per SM).
template <int FMT>
struct DnFmt;
template <>
struct DnFmt<kDenseNvfp4> {  // E2M1 codes + raw E4M3 scales
  static constexpr int kQ = 16 * 512, kS = 16 * 64, kCH = 4;
};
template <>
struct DnFmt<kDenseNvfp4Prepared> {  // E2M1 codes + prepared FP16 scales
  static constexpr int kQ = 16 * 512, kS = 16 * 128, kCH = 4;
};
template <>
struct DnFmt<kDenseFp8> {  // E4M3 codes, channel scales applied to the sum
  static constexpr int kQ = 16 * 1024, kS = 0, kCH = 2;
};
// Ring stage: codes of kCH segments | their scales | token rows (kCH tiles of
// up to 32 rows x 128 bytes, 1024-byte aligned for the swizzle).
template <int FMT>
struct DnRing {
  using F = DnFmt<FMT>;
  static constexpr int kSOff = F::kCH * F::kQ;
  static constexpr int kX = (int)((F::kCH * (F::kQ + F::kS) + 1023) / 1024 * 1024);
  static constexpr int kStage = kX + F::kCH * 32 * 128;
  static constexpr int kStages = std::min(8, kDnRingBudget / kStage);
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStage;
};
static_assert(DnRing<kDenseNvfp4>::kSmem + 256 <= 232448 &&
                  DnRing<kDenseFp8>::kSmem + 256 <= 232448 &&
                  DnRing<kDenseNvfp4Prepared>::kSmem + 256 <= 232448,
              "dense ring above the shared-memory limit");
static_assert(DnRing<kDenseNvfp4>::kStages >= 3 && DnRing<kDenseFp8>::kStages >= 3 &&
                  DnRing<kDenseNvfp4Prepared>::kStages >= 3,
              "dense ring too shallow");

// Block b of the grid covers the flattened (group, segment) range
// [b W / B, (b + 1) W / B), W = groups x segments, B = min(W, kDnBlocks).
DenseSplit dense_split(int N, int K) {
  DenseSplit p;
  const int64_t W = (int64_t)(N / 256) * (K / 64);
  p.blocks = (int)std::min<int64_t>(W, kDnBlocks);
  const int len_max = (int)((W + p.blocks - 1) / p.blocks);
  p.pieces = (len_max + (K / 64) - 1) / (K / 64) + 1;  // groups a range can touch
  return p;
}

// Workspace: one ticket per group (zero between calls), then FP32 [M][256]
// partial sums per (block, piece).
static size_t dense_tickets_bytes(int64_t N) { return align_up((size_t)(N / 256) * 4, 256); }

size_t dense_ws_bytes(int64_t M, int64_t N, int64_t K) {
  if (M == 0) return 0;  // nothing is launched
  const DenseSplit p = dense_split((int)N, (int)K);
  const int64_t segs = K / 64, W = (N / 256) * segs;
  bool whole = true;  // every range boundary on a group boundary: no piece to add up
  for (int b = 0; b <= p.blocks; ++b) whole = whole && ((int64_t)b * W / p.blocks) % segs == 0;
  if (whole) return 0;
  return dense_tickets_bytes(N) + (size_t)p.blocks * p.pieces * M * 256 * sizeof(float);
}

__device__ __forceinline__ int dn_block_of(int64_t i, int64_t W, int B) {
  return (int)(((i + 1) * B + W - 1) / W) - 1;  // the block whose range holds index i
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kDnThreads, 1)
    dense_kernel(int M, int N, int K, int pieces, const __grid_constant__ CUtensorMap xmap,
                 const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                 const float* __restrict__ scale, char* __restrict__ ws, __half* __restrict__ y,
                 uint32_t* status) {
  using F = DnFmt<FMT>;
  using R = DnRing<FMT>;
  extern __shared__ __align__(1024) char dn_raw[];
  char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(dn_raw) + 1023) &
                                       ~uintptr_t(1023));
  __shared__ uint64_t full[R::kStages], empty[R::kStages];
  // per split piece: `written` completes when the 8 consumer warps have stored
  // their partial sums, `decided` when warp 0 has taken the group's ticket
  __shared__ uint64_t written, decided;
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int segs = K >> 6;
  const int B = gridDim.x;
  const int64_t W = (int64_t)(N >> 8) * segs;
  const int64_t r0 = (int64_t)blockIdx.x * W / B, r1 = (int64_t)(blockIdx.x + 1) * W / B;
  uint32_t* tickets = reinterpret_cast<uint32_t*>(ws);
  float* part = reinterpret_cast<float*>(ws + align_up((size_t)(N >> 8) * 4, 256));
  if (tid == 0) {
    for (int i = 0; i < R::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDnWarps);
    }
    mbar_init(&written, kDnWarps);
    mbar_init(&decided, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Programmatic dependent launch: the next grid may start as soon as SMs
  // free up.  The weights are inputs of the call, not results of the previous
  // grid, so the first stages' weight copies go out before waiting for it;
  // the token rows, the workspace and y are touched only after the wait.
  pdl_launch_dependents();

  if (warp == kDnWarps) {
    // ---- producer: one stage per K segment of the block's range ----
    if (lane == 0) {
      uint32_t k = 0;
      int pre_seg[R::kStages];  // first K segment of each stage issued before the wait
      bool waited = false;
      for (int64_t i = r0, n; i < r1; i += n, ++k) {
        // up to kCH consecutive segments of one group: (group i / segs,
        // segments i % segs ..): their tiles are contiguous in the fragment layout
        n = min(min((int64_t)F::kCH, r1 - i), (int64_t)(segs - i % segs));
        const int st = k % R::kStages;
        if (!waited && k == (uint32_t)R::kStages) {
          // the ring is full: wait for the previous grid, then the deferred token rows
          pdl_wait();
          waited = true;
          for (uint32_t j = 0; j < k; ++j)
            tma_load_3d(base + j * R::kStage + R::kX, &xmap, 0, 0, pre_seg[j], &full[j]);
        }
        if (!mbar_wait(&empty[st], ((k / R::kStages) & 1) ^ 1, status)) break;
        char* dst = base + st * R::kStage;
        mbar_expect_tx(&full[st], (uint32_t)(n * (F::kQ + F::kS) + F::kCH * NT * 8 * 128));
        bulk_g2s(dst, q + (size_t)i * F::kQ, (uint32_t)(n * F::kQ), &full[st]);
        if (F::kS)
          bulk_g2s(dst + R::kSOff, s + (size_t)i * F::kS, (uint32_t)(n * F::kS), &full[st]);
        // kCH segments of the token rows (those past K read as zeros, unused)
        if (waited)
          tma_load_3d(dst + R::kX, &xmap, 0, 0, (int)(i % segs), &full[st]);
        else
          pre_seg[k] = (int)(i % segs);
      }
      if (!waited) {
        pdl_wait();
        for (uint32_t j = 0; j < k; ++j)
          tma_load_3d(base + j * R::kStage + R::kX, &xmap, 0, 0, pre_seg[j], &full[j]);
      }
      // copies still in flight land before the block exits (bounded waits)
      for (uint32_t j = (k > (uint32_t)R::kStages ? k - R::kStages : 0); j < k; ++j)
        mbar_wait(&full[j % R::kStages], (j / R::kStages) & 1, status);
    }
    return;
  }

  // ---- consumers: warp w owns tiles kDnTpw w .. kDnTpw w + kDnTpw - 1 of the group ----
  pdl_wait();  // the workspace and y of the previous grid are free
  const int tile0 = kDnTpw * warp;
  uint32_t k = 0, n_split = 0;
  int p = 0;
  for (int64_t i0 = r0; i0 < r1; ++p) {
    const int G = (int)(i0 / segs);
    const int64_t i1 = min(r1, (int64_t)(G + 1) * segs);  // this piece: [i0, i1)
    float acc[kDnTpw][NT][4];
#pragma unroll
    for (int a = 0; a < kDnTpw; ++a)
#pragma unroll
      for (int b = 0; b < NT; ++b)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;
    bool ok = true;
    for (int64_t i = i0, n; i < i1; i += n, ++k) {
      n = min((int64_t)F::kCH, i1 - i);
      const int st = k % R::kStages;
      if (!mbar_wait(&full[st], (k / R::kStages) & 1, status)) {
        ok = false;
        break;
      }
      const char* sb = base + st * R::kStage;
#pragma unroll
      for (int c = 0; c < F::kCH; ++c) {
        if (c >= n) break;
        // token rows of segment c: lane (g, t4) reads elements [16 t4, 16 t4 + 16)
        // of token nt * 8 + g (16-byte chunks 2 t4 and 2 t4 + 1, swizzled by row)
        uint32_t xw[NT][8];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const char* xr = sb + R::kX + (c * NT * 8 + nt * 8 + g) * 128;
          const uint4 v0 = *reinterpret_cast<const uint4*>(xr + (((2 * t4) ^ g) << 4));
          const uint4 v1 = *reinterpret_cast<const uint4*>(xr + (((2 * t4 + 1) ^ g) << 4));
          xw[nt][0] = v0.x; xw[nt][1] = v0.y; xw[nt][2] = v0.z; xw[nt][3] = v0.w;
          xw[nt][4] = v1.x; xw[nt][5] = v1.y; xw[nt][6] = v1.z; xw[nt][7] = v1.w;
        }
        const char* qb = sb + c * F::kQ;
        const char* sc_b = sb + R::kSOff + c * F::kS;
#pragma unroll
        for (int tt = 0; tt < kDnTpw; ++tt) {
          const int j = tile0 + tt;
          if constexpr (FMT == kDenseFp8) {
            // block of 1024 bytes: row g's 16 codes at 16 L, row g + 8's at 512 + 16 L
            const uint4 qa = *reinterpret_cast<const uint4*>(qb + j * 1024 + lane * 16);
            const uint4 qc = *reinterpret_cast<const uint4*>(qb + j * 1024 + 512 + lane * 16);
            const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qc.x, qc.y, qc.z, qc.w};
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              uint32_t af[4];
              af[0] = e4m3x2_to_f16x2(wa[s4] & 0xFFFFu);
              af[2] = e4m3x2_to_f16x2(wa[s4] >> 16);
              af[1] = e4m3x2_to_f16x2(wb[s4] & 0xFFFFu);
              af[3] = e4m3x2_to_f16x2(wb[s4] >> 16);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_16816(acc[tt][nt], af, xw[nt][2 * s4], xw[nt][2 * s4 + 1]);
            }
          } else {
            const uint4 qv = *reinterpret_cast<const uint4*>(qb + j * 512 + lane * 16);
            uint32_t sg, sg8;
            if constexpr (FMT == kDenseNvfp4Prepared)
              scale_splats_f16(*reinterpret_cast<const uint32_t*>(sc_b + j * 128 + lane * 4),
                               &sg, &sg8);
            else
              scale_splats(*reinterpret_cast<const unsigned short*>(sc_b + j * 64 + lane * 2),
                           &sg, &sg8);
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              uint32_t af[4];
              a_frag(qv, sg, sg8, s4, af);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_16816(acc[tt][nt], af, xw[nt][2 * s4], xw[nt][2 * s4 + 1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!__all_sync(0xffffffffu, ok)) break;
    const int64_t gs0 = (int64_t)G * segs, gs1 = gs0 + segs;
    const bool whole = (i0 == gs0 && i1 == gs1);
    // c0 (row g, token 2 t4), c1 (g, 2 t4 + 1), c2 (g + 8, 2 t4), c3 (g + 8, 2 t4 + 1)
    float* slot = part + ((size_t)blockIdx.x * pieces + p) * M * 256;
#pragma unroll
    for (int tt = 0; tt < kDnTpw; ++tt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int m = nt * 8 + 2 * t4 + (c & 1);
          const int r = 16 * (tile0 + tt) + g + ((c & 2) ? 8 : 0);  // row inside the group
          if (m < M) {
            if (whole) {
              const float sc = (FMT == kDenseFp8) ? scale[G * 256 + r] : scale[0];
              y[(size_t)m * N + G * 256 + r] = __float2half_rn(acc[tt][nt][c] * sc);
            } else {
              slot[m * 256 + r] = acc[tt][nt][c];
            }
          }
        }
    if (!whole) {
      // the block that brings the group's last piece adds them up in K order
      const int b_first = dn_block_of(gs0, W, B), b_last = dn_block_of(gs1 - 1, W, B);
      // the warps' partial sums reach warp 0 through the mbarrier (CTA scope);
      // warp 0's device-scope fence then orders all of them before the ticket
      __syncwarp();
      if (lane == 0) mbar_arrive(&written);
      if (warp == 0) {
        const bool all_in = mbar_wait(&written, n_split & 1, status);
        if (lane == 0) {
          s_last = 0;
          if (all_in) {
            __threadfence();
            const uint32_t t = atomicAdd(&tickets[G], 1u);
            s_last = (t == (uint32_t)(b_last - b_first));
            if (s_last) {
              tickets[G] = 0u;  // ready for the next call
              // acquire side: the other blocks' pieces are visible to this
              // block's threads, which are ordered after this fence by `decided`
              __threadfence();
            }
          }
          mbar_arrive(&decided);
        }
      }
      const bool dec = mbar_wait(&decided, n_split & 1, status);
      ++n_split;
      if (!__all_sync(0xffffffffu, dec)) break;
      if (s_last) {
        for (int e = tid; e < M * 64; e += kDnWarps * 32) {  // one float4 of y each
          const int m = e >> 6, r = (e & 63) * 4;
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
          // the pieces in K order, eight loads in flight at a time
          for (int b0 = b_first; b0 <= b_last; b0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int b = b0 + u;
              if (b <= b_last) {
                const int pb = G - (int)(((int64_t)b * W / B) / segs);  // piece of block b in G
                v[u] = __ldcg(reinterpret_cast<const float4*>(
                    part + ((size_t)b * pieces + pb) * M * 256 + m * 256 + r));
              }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int b = b0 + u;
              if (b > b_last) break;
              if (b == b_first) {
                a = v[u];
              } else {
                a.x += v[u].x;
                a.y += v[u].y;
                a.z += v[u].z;
                a.w += v[u].w;
              }
            }
          }
          float4 sc;
          if (FMT == kDenseFp8) {
            sc = *reinterpret_cast<const float4*>(scale + G * 256 + r);
          } else {
            const float s0 = scale[0];
            sc = make_float4(s0, s0, s0, s0);
          }
          const __half2 lo = __floats2half2_rn(a.x * sc.x, a.y * sc.y);
          const __half2 hi = __floats2half2_rn(a.z * sc.z, a.w * sc.w);
          uint2 out;
          out.x = *reinterpret_cast<const uint32_t*>(&lo);
          out.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(y + (size_t)m * N + G * 256 + r) = out;
        }
      }
    }
    i0 = i1;
  }
}

template <int FMT, int NT>
static cudaError_t dense_go(int M, int N, int K, const DenseSplit& sp, const CUtensorMap& xmap,
                            const uint8_t* q, const uint8_t* s, const float* scale, char* ws,
                            __half* y, uint32_t* status, cudaStream_t stream) {
  return launch_k(dense_kernel<FMT, NT>, dim3(sp.blocks), dim3(kDnThreads), DnRing<FMT>::kSmem,
                  stream, !trace_on(), M, N, K, sp.pieces, xmap, q, s, scale, ws, y, status);
}

template <int FMT>
static cudaError_t dense_fmt(int M, int N, int K, const DenseSplit& sp, const CUtensorMap& xmap,
                             const uint8_t* q, const uint8_t* s, const float* scale, char* ws,
                             __half* y, uint32_t* status, cudaStream_t stream) {
  switch ((M + 7) / 8) {
    case 1: return dense_go<FMT, 1>(M, N, K, sp, xmap, q, s, scale, ws, y, status, stream);
    case 2: return dense_go<FMT, 2>(M, N, K, sp, xmap, q, s, scale, ws, y, status, stream);
    case 3: return dense_go<FMT, 3>(M, N, K, sp, xmap, q, s, scale, ws, y, status, stream);
    default: return dense_go<FMT, 4>(M, N, K, sp, xmap, q, s, scale, ws, y, status, stream);
  }
}

cudaError_t launch_dense(int fmt, int64_t M, int64_t N, int64_t K, const __half* x,
                         const uint8_t* q, const uint8_t* s, const float* scale, void* ws,
                         __half* y, uint32_t* status, cudaStream_t stream) {
  const int Mi = (int)M, Ni = (int)N, Ki = (int)K;
  const DenseSplit sp = dense_split(Ni, Ki);
  const int nt = (Mi + 7) / 8;
  CUtensorMap xmap;
  const uint32_t ch = fmt == kDenseFp8 ? DnFmt<kDenseFp8>::kCH : DnFmt<kDenseNvfp4>::kCH;
  cudaError_t e = make_fp16_segments_map(&xmap, x, (uint64_t)K, (uint64_t)M, (uint32_t)(nt * 8), ch);
  if (e != cudaSuccess) return e;
  char* w = static_cast<char*>(ws);
  if (fmt == kDenseFp8)
    return dense_fmt<kDenseFp8>(Mi, Ni, Ki, sp, xmap, q, s, scale, w, y, status, stream);
  if (fmt == kDenseNvfp4Prepared)
    return dense_fmt<kDenseNvfp4Prepared>(Mi, Ni, Ki, sp, xmap, q, s, scale, w, y, status, stream);
  return dense_fmt<kDenseNvfp4>(Mi, Ni, Ki, sp, xmap, q, s, scale, w, y, status, stream);
}

// ---------------------------------------------------------------------------
// Channel-FP8 quantiser: one warp per row.  cs = amax / 448 (1 for an all-zero
// row), q = E4M3_rne_satfinite(x / cs), every step one correctly rounded FP32
// operation; non-finite input is quantised as zero and flagged.  Lane l takes
// the 16-element chunks l, l + 32, ... of the row, so each writes 16 bytes in
// either layout.
// ---------------------------------------------------------------------------
__global__ void fp8_quantize_kernel(const float* __restrict__ w, int64_t rows, int64_t k,
                                    int layout, uint8_t* __restrict__ q, float* __restrict__ cs,
                                    uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const float* wr = w + r * k;
  const int64_t nch = k / 16;
  float amax = 0.f;
  bool bad = false;
  for (int64_t ch = lane; ch < nch; ch += 32) {
    const float4* src = reinterpret_cast<const float4*>(wr + ch * 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 v = src[j];
      const float a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (isfinite(a[u]))
          amax = fmaxf(amax, fabsf(a[u]));
        else
          bad = true;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_ST_NONFINITE);
  const float c = amax == 0.f ? 1.f : __fdiv_rn(amax, 448.f);
  if (lane == 0) cs[r] = c;
  // fragment position of row r: 16-row tile rt, row r16 inside it
  const int64_t rt = r >> 4, r16 = r & 15;
  for (int64_t ch = lane; ch < nch; ch += 32) {
    const float4* src = reinterpret_cast<const float4*>(wr + ch * 16);
    uint32_t words[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 v = src[j];
      float a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = isfinite(a[u]) ? __fdiv_rn(a[u], c) : 0.f;
      uint16_t lo, hi;
      // first source -> high byte, second -> low byte
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a[1]), "f"(a[0]));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a[3]), "f"(a[2]));
      words[j] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    const uint4 v4 = make_uint4(words[0], words[1], words[2], words[3]);
    int64_t off;
    if (layout == MOE_LAYOUT_CANONICAL) {
      off = r * k + ch * 16;
    } else {
      const int64_t ks = ch >> 2, cc = ch & 3;
      const int64_t blk = ((rt >> 4) * (k >> 6) + ks) * 16 + (rt & 15);
      off = blk * 1024 + (r16 >= 8 ? 512 : 0) + 16 * (4 * (r16 & 7) + cc);
    }
    *reinterpret_cast<uint4*>(q + off) = v4;
  }
}

cudaError_t launch_fp8_quantize(const float* w, int64_t rows, int64_t k, int layout, uint8_t* q,
                                float* cs, uint32_t* status, cudaStream_t stream) {
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  fp8_quantize_kernel<<<blocks, 256, 0, stream>>>(w, rows, k, layout, q, cs, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Prepared scales: out[i] = FP16 value of E4M3 code s[i] (exact); the NaN codes
// 0x7F / 0xFF give 0x7E00 and flag MOE_ST_NONFINITE.  Each thread widens 8 codes.
// ---------------------------------------------------------------------------
__global__ void prepare_scales_kernel(const uint8_t* __restrict__ s, int64_t n,
                                      uint16_t* __restrict__ out, uint32_t* status) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i >= n) return;
  bool bad = false;
  if (i + 8 <= n) {
    const uint2 v = *reinterpret_cast<const uint2*>(s + i);
    const uint32_t w2[2] = {v.x, v.y};
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const uint32_t two = (w2[h] >> (16 * p)) & 0xFFFFu;
        uint32_t f = e4m3x2_to_f16x2(two);
        if ((two & 0x7Fu) == 0x7Fu) {
          f = (f & 0xFFFF0000u) | 0x7E00u;
          bad = true;
        }
        if (((two >> 8) & 0x7Fu) == 0x7Fu) {
          f = (f & 0x0000FFFFu) | 0x7E000000u;
          bad = true;
        }
        o[2 * h + p] = f;
      }
    *reinterpret_cast<uint4*>(out + i) = make_uint4(o[0], o[1], o[2], o[3]);
  } else {
    for (int64_t j = i; j < n; ++j) {
      const uint32_t c = s[j];
      uint32_t f = e4m3x2_to_f16x2(c) & 0xFFFFu;
      if ((c & 0x7Fu) == 0x7Fu) {
        f = 0x7E00u;
        bad = true;
      }
      out[j] = (uint16_t)f;
    }
  }
  if (bad) set_status(status, MOE_ST_NONFINITE);
}

cudaError_t launch_prepare_scales(const uint8_t* s, int64_t n, uint16_t* out, uint32_t* status,
                                  cudaStream_t stream) {
  const int64_t threads = (n + 7) / 8;
  prepare_scales_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, stream>>>(s, n, out, status);
  return cudaGetLastError();
}

cudaError_t dense_device_init() {
#define MOE_DN_ATTR(F, T)                                                                   \
  {                                                                                         \
    cudaError_t e = cudaFuncSetAttribute(dense_kernel<F, T>,                                \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                                         (int)DnRing<F>::kSmem);                            \
    if (e != cudaSuccess) return e;                                                         \
  }
  MOE_DN_ATTR(kDenseNvfp4, 1) MOE_DN_ATTR(kDenseNvfp4, 2) MOE_DN_ATTR(kDenseNvfp4, 3)
  MOE_DN_ATTR(kDenseNvfp4, 4) MOE_DN_ATTR(kDenseNvfp4Prepared, 1)
  MOE_DN_ATTR(kDenseNvfp4Prepared, 2) MOE_DN_ATTR(kDenseNvfp4Prepared, 3)
  MOE_DN_ATTR(kDenseNvfp4Prepared, 4) MOE_DN_ATTR(kDenseFp8, 1) MOE_DN_ATTR(kDenseFp8, 2)
  MOE_DN_ATTR(kDenseFp8, 3) MOE_DN_ATTR(kDenseFp8, 4)
#undef MOE_DN_ATTR
  return cudaSuccess;
}

}  // namespace moe
