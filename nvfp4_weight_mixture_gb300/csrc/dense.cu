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
// streams them once.  Each of a fixed grid of up to kDnBlocks blocks owns a
// contiguous range of the N / 16 output tiles (16 rows each) over the whole
// of K, so no output is split between blocks.  It takes its tiles kDnTG at a
// time: a producer thread fills a ring of stages, each up to kCH K segments
// of those tiles (two 2-D tensor-map copies per tile: codes and scales) plus
// the same segments of every token row (one 128-byte-swizzled tensor-map
// copy).  The 16 consumer warps split the tiles evenly (16 / T warps per
// tile, T the tiles in hand); warp r of a tile multiplies the tile's K
// segments s with s % (16 / T) == r, dequantising its fragments in registers
// straight into mma.sync A operands with up to four 8-token column tiles.
// The tile's warps then add their sums in warp order and write y.  The tile
// ranges depend on N only and a token's column of the MMA does not depend on
// the other columns, so every output row is computed by the same operations
// whatever M is: results are bitwise independent of the batch.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDnWarps = 16;                     // consumer warps
constexpr int kDnThreads = (kDnWarps + 1) * 32;  // + one producer warp
constexpr int kDnBlocks = 152;                   // fixed grid (one block per SM of a GB300)
constexpr int kDnTG = 4;                         // tiles in hand at a time
constexpr int kDnSmemBudget = 216 * 1024;

// Per weight format: bytes of one (tile, K segment) of codes (kQ) and scales
// (kS) in the fragment layout, and kCH, the K segments of a stage (more for
// the NVFP4 formats, whose expansion costs more instructions per byte: each
// warp then takes more segments per stage wait).
template <int FMT>
struct DnFmt;
template <>
struct DnFmt<kDenseNvfp4> {  // E2M1 codes + raw E4M3 scales
  static constexpr int kQ = 512, kS = 64, kCH = 8;
};
template <>
struct DnFmt<kDenseNvfp4Prepared> {  // E2M1 codes + prepared FP16 scales
  static constexpr int kQ = 512, kS = 128, kCH = 8;
};
template <>
struct DnFmt<kDenseFp8> {  // E4M3 codes, channel scales applied to the sum
  static constexpr int kQ = 1024, kS = 0, kCH = 8;
};
// Shared memory: the reduction area (the 16 warps' sums, [warp][NT][32][4]
// FP32), then the ring.  A stage: codes [tile][segment][kQ] | scales
// [tile][segment][kS] | token rows (kCH segments of NT x 8 rows x 128 bytes,
// 1024-byte aligned for the swizzle).
template <int FMT, int NT>
struct DnRing {
  using F = DnFmt<FMT>;
  // FP8 with 24 or 32 token rows keeps 4 segments a stage (room for 3 stages)
  static constexpr int kCH = (FMT == kDenseFp8 && NT > 2) ? 4 : F::kCH;
  static constexpr int kSOff = kDnTG * kCH * F::kQ;
  static constexpr int kX = (kSOff + kDnTG * kCH * F::kS + 1023) / 1024 * 1024;
  static constexpr int kStage = kX + kCH * NT * 8 * 128;
  static constexpr int kRed = kDnWarps * NT * 32 * 4 * 4;
  static constexpr int kStages = std::min(8, (kDnSmemBudget - kRed) / kStage);
  static constexpr size_t kSmem = 1024 + kRed + (size_t)kStages * kStage;
  static_assert(kSmem + 512 <= 232448, "dense ring above the shared-memory limit");
  static_assert(kStages >= 3, "dense ring too shallow");
};

int dense_blocks(int N) { return std::min(N / 16, kDnBlocks); }

// No output is split between blocks: no workspace.
size_t dense_ws_bytes(int64_t M, int64_t N, int64_t K) {
  (void)M;
  (void)N;
  (void)K;
  return 0;
}

template <int FMT, int NT>
__global__ void __launch_bounds__(kDnThreads, 1)
    dense_kernel(int M, int N, int K, const __grid_constant__ CUtensorMap xmap,
                 const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap smap,
                 const float* __restrict__ scale, __half* __restrict__ y, uint32_t* status) {
  using F = DnFmt<FMT>;
  using R = DnRing<FMT, NT>;
  extern __shared__ __align__(1024) char dn_raw[];
  char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(dn_raw) + 1023) &
                                       ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(base);
  char* ring = base + R::kRed;
  __shared__ uint64_t full[R::kStages], empty[R::kStages];
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int S = K >> 6;
  const int nt_all = N >> 4, B = gridDim.x;
  const int t_begin = (int)((int64_t)blockIdx.x * nt_all / B);
  const int t_end = (int)((int64_t)(blockIdx.x + 1) * nt_all / B);
  const int n_chunks = (S + R::kCH - 1) / R::kCH;  // stages per group of tiles
  if (tid == 0) {
    for (int i = 0; i < R::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDnWarps);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Programmatic dependent launch: the next grid may start as soon as SMs
  // free up.  The weights are inputs of the call, not results of the previous
  // grid, so the first stages' weight copies go out before waiting for it;
  // the token rows and y are touched only after the wait.
  pdl_launch_dependents();

  if (warp == kDnWarps) {
    // ---- producer: stage k = (group of tiles, K chunk), in order ----
    if (lane == 0) {
      uint32_t k = 0;
      int pre_seg[R::kStages];  // first K segment of each stage issued before the wait
      bool waited = false, ok = true;
      for (int t0 = t_begin; ok && t0 < t_end; t0 += kDnTG) {
        const int T = min(kDnTG, t_end - t0);
        for (int ch = 0; ch < n_chunks; ++ch, ++k) {
          const int s0 = ch * R::kCH;
          const int st = k % R::kStages;
          if (!waited && k == (uint32_t)R::kStages) {
            // the ring is full: wait for the previous grid, then the deferred token rows
            pdl_wait();
            waited = true;
            for (uint32_t j = 0; j < k; ++j)
              tma_load_3d(ring + j * R::kStage + R::kX, &xmap, 0, 0, pre_seg[j], &full[j]);
          }
          if (!mbar_wait(&empty[st], ((k / R::kStages) & 1) ^ 1, status)) {
            ok = false;
            break;
          }
          char* dst = ring + st * R::kStage;
          // every copy moves its whole box (segments past K read as zeros)
          mbar_expect_tx(&full[st],
                         (uint32_t)(T * R::kCH * (F::kQ + F::kS) + R::kCH * NT * 8 * 128));
          for (int t = 0; t < T; ++t) {
            const int tile = t0 + t;
            const int row = (tile >> 4) * S + s0;  // (group, segment) row of the fragment layout
            tma_load_2d(dst + t * R::kCH * F::kQ, &qmap, (tile & 15) * (F::kQ / 8), row,
                        &full[st]);
            if (F::kS)
              tma_load_2d(dst + R::kSOff + t * R::kCH * F::kS, &smap, (tile & 15) * (F::kS / 8),
                          row, &full[st]);
          }
          if (waited)
            tma_load_3d(dst + R::kX, &xmap, 0, 0, s0, &full[st]);
          else
            pre_seg[k] = s0;
        }
      }
      if (!waited) {
        pdl_wait();
        for (uint32_t j = 0; j < k; ++j)
          tma_load_3d(ring + j * R::kStage + R::kX, &xmap, 0, 0, pre_seg[j], &full[j]);
      }
      // copies still in flight land before the block exits (bounded waits)
      for (uint32_t j = (k > (uint32_t)R::kStages ? k - R::kStages : 0); j < k; ++j)
        mbar_wait(&full[j % R::kStages], (j / R::kStages) & 1, status);
    }
    return;
  }

  // ---- consumers ----
  pdl_wait();  // y of the previous grid is free
  uint32_t k = 0;
  for (int t0 = t_begin; t0 < t_end; t0 += kDnTG) {
    const int T = min(kDnTG, t_end - t0);
    const int wpt = kDnWarps / T;  // warps per tile
    const int tl = warp / wpt, r = warp - tl * wpt;
    const bool active = tl < T;
    float acc[NT][4];
#pragma unroll
    for (int b = 0; b < NT; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[b][c] = 0.f;
    for (int ch = 0; ch < n_chunks; ++ch, ++k) {
      const int st = k % R::kStages;
      if (!mbar_wait(&full[st], (k / R::kStages) & 1, status)) {
        if (lane == 0) s_abort = 1;
      } else if (active) {
        const char* sb = ring + st * R::kStage;
        const int s0 = ch * R::kCH;
        // this warp's segments of the stage: s % wpt == r
        for (int c = ((r - s0) % wpt + wpt) % wpt; c < R::kCH && s0 + c < S; c += wpt) {
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
          const char* qb = sb + (tl * R::kCH + c) * F::kQ;
          if constexpr (FMT == kDenseFp8) {
            // block of 1024 bytes: row g's 16 codes at 16 L, row g + 8's at 512 + 16 L
            const uint4 qa = *reinterpret_cast<const uint4*>(qb + lane * 16);
            const uint4 qc = *reinterpret_cast<const uint4*>(qb + 512 + lane * 16);
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
                mma_16816(acc[nt], af, xw[nt][2 * s4], xw[nt][2 * s4 + 1]);
            }
          } else {
            const char* sc_b = sb + R::kSOff + (tl * R::kCH + c) * F::kS;
            const uint4 qv = *reinterpret_cast<const uint4*>(qb + lane * 16);
            uint32_t sg, sg8;
            if constexpr (FMT == kDenseNvfp4Prepared)
              scale_splats_f16(*reinterpret_cast<const uint32_t*>(sc_b + lane * 4), &sg, &sg8);
            else
              scale_splats(*reinterpret_cast<const unsigned short*>(sc_b + lane * 2), &sg, &sg8);
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              uint32_t af[4];
              a_frag(qv, sg, sg8, s4, af);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
                mma_16816(acc[nt], af, xw[nt][2 * s4], xw[nt][2 * s4 + 1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // ---- the tile's warps' sums in warp order: red[warp][nt][lane][c] ----
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[((warp * NT + nt) * 32 + lane) * 4 + c] = acc[nt][c];
    asm volatile("bar.sync 1, %0;" ::"r"(kDnWarps * 32) : "memory");
    if (s_abort) break;
    // thread: tile i < T, output element (nt, lane, c) of it
    for (int e = tid; e < T * NT * 128; e += kDnWarps * 32) {
      const int ti = e / (NT * 128), rem = e - ti * (NT * 128);
      const int nt = rem >> 7, ln = (rem >> 2) & 31, c = rem & 3;
      const int m = nt * 8 + 2 * (ln & 3) + (c & 1);
      if (m >= M) continue;
      float a = 0.f;
      for (int rr = 0; rr < wpt; ++rr) a += red[(((ti * wpt + rr) * NT + nt) * 32 + ln) * 4 + c];
      // c0 (row g, token 2 t4), c1 (g, 2 t4 + 1), c2 (g + 8, 2 t4), c3 (g + 8, 2 t4 + 1)
      const int row = 16 * (t0 + ti) + (ln >> 2) + ((c & 2) ? 8 : 0);
      const float sc = (FMT == kDenseFp8) ? scale[row] : scale[0];
      y[(size_t)m * N + row] = __float2half_rn(a * sc);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kDnWarps * 32) : "memory");  // red is reused
  }
}

template <int FMT, int NT>
static cudaError_t dense_go(int M, int N, int K, const __half* x, const uint8_t* q,
                            const uint8_t* s, const float* scale, __half* y, uint32_t* status,
                            cudaStream_t stream) {
  using F = DnFmt<FMT>;
  constexpr int kCH = DnRing<FMT, NT>::kCH;
  // the fragment layout as rows of (256-row group, K segment): 16 tiles of kQ
  // code bytes (kS scale bytes); a box is one tile over kCH segments
  const uint64_t rows = (uint64_t)(N / 256) * (K / 64);
  CUtensorMap xmap, qmap, smap;
  cudaError_t e = make_fp16_segments_map(&xmap, x, (uint64_t)K, (uint64_t)M, (uint32_t)(NT * 8),
                                         (uint32_t)kCH);
  if (e != cudaSuccess) return e;
  if ((e = make_rows_map(&qmap, q, 16 * F::kQ, rows, F::kQ, kCH)) != cudaSuccess) return e;
  smap = qmap;
  if (F::kS && (e = make_rows_map(&smap, s, 16 * F::kS, rows, F::kS, kCH)) != cudaSuccess)
    return e;
  return launch_k(dense_kernel<FMT, NT>, dim3(dense_blocks(N)), dim3(kDnThreads),
                  DnRing<FMT, NT>::kSmem, stream, !trace_on(), M, N, K, xmap, qmap, smap, scale,
                  y, status);
}

template <int FMT>
static cudaError_t dense_fmt(int M, int N, int K, const __half* x, const uint8_t* q,
                             const uint8_t* s, const float* scale, __half* y, uint32_t* status,
                             cudaStream_t stream) {
  switch ((M + 7) / 8) {
    case 1: return dense_go<FMT, 1>(M, N, K, x, q, s, scale, y, status, stream);
    case 2: return dense_go<FMT, 2>(M, N, K, x, q, s, scale, y, status, stream);
    case 3: return dense_go<FMT, 3>(M, N, K, x, q, s, scale, y, status, stream);
    default: return dense_go<FMT, 4>(M, N, K, x, q, s, scale, y, status, stream);
  }
}

cudaError_t launch_dense(int fmt, int64_t M, int64_t N, int64_t K, const __half* x,
                         const uint8_t* q, const uint8_t* s, const float* scale, void* ws,
                         __half* y, uint32_t* status, cudaStream_t stream) {
  (void)ws;
  const int Mi = (int)M, Ni = (int)N, Ki = (int)K;
  if (fmt == kDenseFp8) return dense_fmt<kDenseFp8>(Mi, Ni, Ki, x, q, s, scale, y, status, stream);
  if (fmt == kDenseNvfp4Prepared)
    return dense_fmt<kDenseNvfp4Prepared>(Mi, Ni, Ki, x, q, s, scale, y, status, stream);
  return dense_fmt<kDenseNvfp4>(Mi, Ni, Ki, x, q, s, scale, y, status, stream);
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
                                         (int)DnRing<F, T>::kSmem);                         \
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
