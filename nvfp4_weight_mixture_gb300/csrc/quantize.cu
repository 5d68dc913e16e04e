// NVFP4 quantiser and dequantiser kernels.
//
// Load-time step of the layer: FP32 weights -> E2M1 codes, one E4M3 scale per
// 16 elements along K, one FP32 scale per matrix ("[Kernel][SM70] Improve
// Qwen3.8 no-MTP concurrency", section "Scope and related PRs": native NVFP4
// weights, raw E4M3 scale storage).  Every arithmetic step is a single
// correctly rounded FP32 operation so that the result is bit-reproducible:
//   g = amax / 2688,  s = E4M3((amax_block / g) / 6),  q = E2M1(x / (s * g)).
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Byte offset of the 8 q bytes and the s byte of (packed row rp, 16-element
// block b) of matrix m in the fragment layout: 256-row groups, then 64-element
// segments, then the group's 16 row tiles (512 q bytes + 64 s bytes each).
struct FragPos {
  int64_t q, s;
};
__device__ __forceinline__ FragPos frag_pos(int64_t m, int64_t rows, int64_t k, int64_t rp,
                                            int64_t b) {
  int64_t rt = rp >> 4, r16 = rp & 15, ks = b >> 2, c = b & 3;
  int64_t blk = ((m * (rows >> 8) + (rt >> 4)) * (k >> 6) + ks) * 16 + (rt & 15);
  int64_t L = 4 * (r16 & 7) + c;
  FragPos p;
  p.q = blk * 512 + 16 * L + ((r16 >= 8) ? 8 : 0);
  p.s = blk * 64 + 2 * L + ((r16 >= 8) ? 1 : 0);
  return p;
}

// Packed row of canonical row r for the layout (identity except for the W13
// gate/up tile interleave).
__device__ __forceinline__ int64_t packed_row(int64_t r, int64_t rows, int layout) {
  if (layout != MOE_LAYOUT_FRAGMENT_W13) return r;
  int64_t half = rows >> 1;
  if (r < half) return 32 * (r >> 4) + (r & 15);
  int64_t u = r - half;
  return 32 * (u >> 4) + 16 + (u & 15);
}
__device__ __forceinline__ int64_t canonical_row(int64_t rp, int64_t rows, int layout) {
  if (layout != MOE_LAYOUT_FRAGMENT_W13) return rp;
  int64_t t = rp >> 4, r16 = rp & 15;
  int64_t base = 16 * (t >> 1) + r16;
  return (t & 1) ? (rows >> 1) + base : base;
}

// ---- pass 1: per-matrix amax, stored as FP32 bits in g (zeroed by the host) --
__global__ void quant_amax_kernel(const float* __restrict__ w, int64_t per_mat, float* g,
                                  uint32_t* status) {
  const int64_t m = blockIdx.y;
  const float4* src = reinterpret_cast<const float4*>(w + m * per_mat);
  const int64_t n4 = per_mat / 4;
  float amax = 0.f;
  bool bad = false;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 v = src[i];
    float a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!isfinite(a[j])) {
        bad = true;
      } else {
        amax = fmaxf(amax, fabsf(a[j]));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (bad) set_status(status, MOE_ST_NONFINITE);
  // non-negative floats order like their bit patterns
  if ((threadIdx.x & 31) == 0)
    atomicMax(reinterpret_cast<unsigned int*>(g + m), __float_as_uint(amax));
}

__device__ __forceinline__ float global_scale_from_amax(float amax) {
  return amax == 0.f ? 1.f : __fdiv_rn(amax, 2688.f);
}

// ---- pass 2: block scales and codes ------------------------------------------
// One thread per (row, 16-element block).
__global__ void quant_pack_kernel(const float* __restrict__ w, int64_t n_mats, int64_t rows,
                                  int64_t k, int layout, uint8_t* __restrict__ q,
                                  uint8_t* __restrict__ s, const float* __restrict__ g_amax) {
  const int64_t nb = k >> 4;
  const int64_t total = n_mats * rows * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i % nb;
    const int64_t r = (i / nb) % rows;
    const int64_t m = i / (nb * rows);
    const float gm = global_scale_from_amax(g_amax[m]);
    const float4* src = reinterpret_cast<const float4*>(w + (m * rows + r) * k + b * 16);
    float x[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float4 v = src[j];
      x[4 * j] = v.x;
      x[4 * j + 1] = v.y;
      x[4 * j + 2] = v.z;
      x[4 * j + 3] = v.w;
    }
    float bmax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (!isfinite(x[j])) x[j] = 0.f;
      bmax = fmaxf(bmax, fabsf(x[j]));
    }
    const float sb = __fdiv_rn(__fdiv_rn(bmax, gm), 6.f);
    uint16_t s2;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(s2) : "f"(0.f), "f"(sb));
    const uint32_t sc = s2 & 0xFF;
    // value of the scale (exact in FP32), then d = value * g rounded once
    const uint32_t sf16 = e4m3x2_to_f16x2(sc);
    const float sval = __half2float(__ushort_as_half((unsigned short)(sf16 & 0xFFFF)));
    const float d = __fmul_rn(sval, gm);
    uint32_t codes[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      uint32_t c2;
      if (d == 0.f) {
        c2 = (signbit(x[j]) ? 0x8u : 0u) | (signbit(x[j + 1]) ? 0x80u : 0u);
      } else {
        const float z0 = __fdiv_rn(x[j], d), z1 = __fdiv_rn(x[j + 1], d);
        uint16_t t;
        // first source -> high nibble, second -> low nibble
        asm("{\n .reg .b8 c;\n cvt.rn.satfinite.e2m1x2.f32 c, %1, %2;\n cvt.u16.u8 %0, c;\n}\n"
            : "=h"(t)
            : "f"(z1), "f"(z0));
        c2 = t & 0xFF;
      }
      codes[j >> 3] |= c2 << (8 * ((j >> 1) & 3));
    }
    if (layout == MOE_LAYOUT_CANONICAL) {
      uint2* qd = reinterpret_cast<uint2*>(q + (m * rows + r) * (k >> 1) + b * 8);
      *qd = make_uint2(codes[0], codes[1]);
      s[(m * rows + r) * nb + b] = (uint8_t)sc;
    } else {
      const FragPos p = frag_pos(m, rows, k, packed_row(r, rows, layout), b);
      *reinterpret_cast<uint2*>(q + p.q) = make_uint2(codes[0], codes[1]);
      s[p.s] = (uint8_t)sc;
    }
  }
}

__global__ void quant_finalize_kernel(float* g, int64_t n_mats) {
  int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (m < n_mats) g[m] = global_scale_from_amax(g[m]);
}

// ---- dequantiser (diagnostic) -----------------------------------------------
__global__ void dequant_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                               int64_t n_mats, int64_t rows, int64_t k, int layout,
                               __half* __restrict__ out) {
  const int64_t nb = k >> 4;
  const int64_t total = n_mats * rows * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i % nb;
    const int64_t r = (i / nb) % rows;
    const int64_t m = i / (nb * rows);
    uint2 codes;
    uint32_t sc;
    if (layout == MOE_LAYOUT_CANONICAL) {
      codes = *reinterpret_cast<const uint2*>(q + (m * rows + r) * (k >> 1) + b * 8);
      sc = s[(m * rows + r) * nb + b];
    } else {
      const FragPos p = frag_pos(m, rows, k, packed_row(r, rows, layout), b);
      codes = *reinterpret_cast<const uint2*>(q + p.q);
      sc = s[p.s];
    }
    const uint32_t sf = e4m3x2_to_f16x2(sc);
    const uint32_t s2 = __byte_perm(sf, sf, 0x1010);
    uint32_t o[8];
    dequant8(codes.x, s2, o);
    dequant8(codes.y, s2, o + 4);
    uint4* dst = reinterpret_cast<uint4*>(out + (m * rows + r) * k + b * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ---- launchers --------------------------------------------------------------
cudaError_t launch_quantize(const float* w, int64_t n_mats, int64_t rows, int64_t k, int layout,
                            uint8_t* q, uint8_t* s, float* g, uint32_t* status,
                            cudaStream_t stream, int num_sms) {
  cudaError_t err = cudaMemsetAsync(g, 0, sizeof(float) * n_mats, stream);
  if (err != cudaSuccess) return err;
  const int64_t per_mat = rows * k;
  int64_t bx = (per_mat / 4 + 255) / 256;
  if (bx > 64) bx = 64;
  if (n_mats > 65535) return cudaErrorInvalidValue;
  quant_amax_kernel<<<dim3((unsigned)bx, (unsigned)n_mats), 256, 0, stream>>>(w, per_mat, g,
                                                                              status);
  const int64_t total = n_mats * rows * (k >> 4);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)num_sms * 32) blocks = (int64_t)num_sms * 32;
  quant_pack_kernel<<<(unsigned)blocks, 256, 0, stream>>>(w, n_mats, rows, k, layout, q, s, g);
  quant_finalize_kernel<<<(unsigned)((n_mats + 255) / 256), 256, 0, stream>>>(g, n_mats);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* q, const uint8_t* s, int64_t n_mats, int64_t rows,
                              int64_t k, int layout, void* out, cudaStream_t stream,
                              int num_sms) {
  const int64_t total = n_mats * rows * (k >> 4);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)num_sms * 32) blocks = (int64_t)num_sms * 32;
  if (blocks < 1) blocks = 1;
  dequant_kernel<<<(unsigned)blocks, 256, 0, stream>>>(q, s, n_mats, rows, k, layout,
                                                       reinterpret_cast<__half*>(out));
  return cudaGetLastError();
}

}  // namespace moe
