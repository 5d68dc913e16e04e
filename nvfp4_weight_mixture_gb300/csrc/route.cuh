// Device helpers of the router (top-k, renormalised weights, shared gate,
// route stores, block scan) of the router kernels (router.cu).
#pragma once

#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kMaxEEff = 520;  // >= 512 routed experts + the shared expert

// A pair's expert id is valid if it names a routed expert in a routed slot,
// or the shared expert in the shared slot.
__device__ __forceinline__ bool pair_valid(int e, int slot, const LayerDims& d) {
  return slot < d.k ? (e >= 0 && e < d.E) : (e == d.E);
}

// ---------------------------------------------------------------------------
// Warp top-k over a row of E logits.  Lane j < k receives slot j: the j-th
// largest logit, ties broken towards the lower expert id.  E <= 512.  Each
// round takes the warp maximum of order-preserving integer keys and then the
// lowest expert id holding it (two single-instruction warp reductions).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f2key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <bool kGlobal>
__device__ __forceinline__ void warp_topk(const float* row, int E, int k, int* out_id,
                                          float* out_l) {
  const int lane = threadIdx.x & 31;
  uint32_t v[16];  // key 0 = absent or taken (below every finite or infinite logit)
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? f2key(kGlobal ? __ldcg(row + e) : row[e]) : 0u;
  }
  int my_id = -1;
  float my_l = -INFINITY;
  for (int j = 0; j < k; ++j) {
    uint32_t m8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = max(v[i], v[i + 8]);
#pragma unroll
    for (int i = 0; i < 4; ++i) m8[i] = max(m8[i], m8[i + 4]);
    const uint32_t lm = max(max(m8[0], m8[2]), max(m8[1], m8[3]));
    const uint32_t gm = __reduce_max_sync(0xffffffffu, lm);
    uint32_t li = 0xffffffffu;
#pragma unroll
    for (int i = 15; i >= 0; --i)
      if (v[i] == gm) li = (uint32_t)(lane + 32 * i);
    const uint32_t gi = __reduce_min_sync(0xffffffffu, li);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((uint32_t)(lane + 32 * i) == gi) v[i] = 0u;
    if (lane == j) {
      my_id = (int)gi;
      my_l = key2f(gm);
    }
  }
  *out_id = my_id;
  *out_l = my_l;
}

// The same selection for throughput (one warp per row, many rows): every
// element of the top k is at least T, the k-th largest of the 32 lane maxima
// counted with multiplicity (those k maxima are k distinct elements).  The
// elements >= T, at least k of them and usually few more, are gathered one
// per lane through `slot` (32 entries of this warp), so that the k rounds
// reduce single values instead of selecting over 16 keys per lane.  More than
// 32 such elements (heavy ties) take the rounds of warp_topk.  Lane j < k
// receives the same slot j as from warp_topk.
__device__ __forceinline__ void warp_topk_gathered(const float* row, int E, int k,
                                                   uint32_t (*slot)[2], int* out_id,
                                                   float* out_l) {
  const int lane = threadIdx.x & 31;
  uint32_t v[16];  // key 0 = absent (below every finite or infinite logit)
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? f2key(__ldcg(row + e)) : 0u;
  }
  uint32_t lm = v[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) lm = max(lm, v[i]);
  // T: the k-th largest lane maximum (lanes holding the round's maximum all
  // leave together; their number counts towards k)
  uint32_t rest = lm, T = 0u;
  for (int seen = 0; seen < k;) {
    const uint32_t gm = __reduce_max_sync(0xffffffffu, rest);
    seen += __popc(__ballot_sync(0xffffffffu, rest == gm));
    T = gm;
    if (rest == gm) rest = 0u;
  }
  const uint32_t Tq = max(T, 1u);
  int c = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) c += (int)(v[i] >= Tq);
  const int C = (int)__reduce_add_sync(0xffffffffu, (uint32_t)c);
  int my_id = -1;
  float my_l = -INFINITY;
  if (C <= 32) {
    int off = c;  // exclusive prefix of the lanes' counts
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, off, o);
      if (lane >= o) off += n;
    }
    off -= c;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (v[i] >= Tq) {
        slot[off][0] = v[i];
        slot[off][1] = (uint32_t)(lane + 32 * i);
        ++off;
      }
    __syncwarp();
    uint32_t key = lane < C ? slot[lane][0] : 0u;
    const uint32_t idx = lane < C ? slot[lane][1] : 0xffffffffu;
    __syncwarp();
    for (int j = 0; j < k; ++j) {
      const uint32_t gm = __reduce_max_sync(0xffffffffu, key);
      const uint32_t gi = __reduce_min_sync(0xffffffffu, key == gm ? idx : 0xffffffffu);
      if (idx == gi) key = 0u;
      if (lane == j) {
        my_id = (int)gi;
        my_l = key2f(gm);
      }
    }
  } else {
    for (int j = 0; j < k; ++j) {
      uint32_t m8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) m8[i] = max(v[i], v[i + 8]);
#pragma unroll
      for (int i = 0; i < 4; ++i) m8[i] = max(m8[i], m8[i + 4]);
      const uint32_t l2 = max(max(m8[0], m8[2]), max(m8[1], m8[3]));
      const uint32_t gm = __reduce_max_sync(0xffffffffu, l2);
      uint32_t li = 0xffffffffu;
#pragma unroll
      for (int i = 15; i >= 0; --i)
        if (v[i] == gm) li = (uint32_t)(lane + 32 * i);
      const uint32_t gi = __reduce_min_sync(0xffffffffu, li);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if ((uint32_t)(lane + 32 * i) == gi) v[i] = 0u;
      if (lane == j) {
        my_id = (int)gi;
        my_l = key2f(gm);
      }
    }
  }
  *out_id = my_id;
  *out_l = my_l;
}

// softmax of the k selected logits held by lanes 0..k-1 (lane 0 holds the max)
__device__ __forceinline__ float warp_topk_weight(float my_l, int k) {
  const int lane = threadIdx.x & 31;
  const float lmax = __shfl_sync(0xffffffffu, my_l, 0);
  const float e = (lane < k) ? __expf(my_l - lmax) : 0.f;
  float s = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return __fdividef(e, s);
}

// gamma = sigmoid(x . w_g), one warp, x and w_g FP16 of length H (H % 64 == 0)
__device__ __forceinline__ float warp_gate(const __half* xr, const __half* wg, int H) {
  const int lane = threadIdx.x & 31;
  float z = 0.f;
  for (int c = 2 * lane; c < H; c += 64) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(xr + c));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(wg + c));
    z = fmaf(a.x, b.x, z);
    z = fmaf(a.y, b.y, z);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  return 1.f / (1.f + expf(-z));
}

// Writes slot values of token t (lanes < k), plus the shared slot.
__device__ __forceinline__ void store_route(const LayerDims& d, int t, int id, float w,
                                            float gamma, int32_t* ids_user, float* w_user,
                                            const PlanView& pv) {
  const int lane = threadIdx.x & 31;
  if (lane < d.k) {
    ids_user[(int64_t)t * d.k + lane] = id;
    w_user[(int64_t)t * d.k + lane] = w;
    pv.ids[(int64_t)t * d.k_eff + lane] = id;
    pv.w[(int64_t)t * d.k_eff + lane] = w;
  }
  if (d.shared && lane == 0) {
    pv.ids[(int64_t)t * d.k_eff + d.k] = d.E;
    pv.w[(int64_t)t * d.k_eff + d.k] = gamma;
  }
}

// Exclusive block scan of three counters (blockDim.x == 256).
__device__ __forceinline__ void block_scan3(int& a, int& b, int& c, int* tot) {
  __shared__ int ws[8][3];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b, ic = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ta = __shfl_up_sync(0xffffffffu, ia, o);
    const int tb = __shfl_up_sync(0xffffffffu, ib, o);
    const int tc = __shfl_up_sync(0xffffffffu, ic, o);
    if (lane >= o) {
      ia += ta;
      ib += tb;
      ic += tc;
    }
  }
  if (lane == 31) {
    ws[warp][0] = ia;
    ws[warp][1] = ib;
    ws[warp][2] = ic;
  }
  __syncthreads();
  int oa = 0, ob = 0, oc = 0, sa = 0, sb = 0, sc = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    if (w < warp) {
      oa += ws[w][0];
      ob += ws[w][1];
      oc += ws[w][2];
    }
    sa += ws[w][0];
    sb += ws[w][1];
    sc += ws[w][2];
  }
  a = oa + ia - a;
  b = ob + ib - b;
  c = oc + ic - c;
  tot[0] = sa;
  tot[1] = sb;
  tot[2] = sc;
  __syncthreads();
}

}  // namespace moe
