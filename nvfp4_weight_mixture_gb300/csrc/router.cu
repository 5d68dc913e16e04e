// Router (FP32 logits, top-k, renormalised softmax weights, shared-expert
// gate) and the integer routing plan (per-expert histogram, prefix scan,
// stable permutation, inverse, tile schedule).
//
// "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency", section "Scope and
// related PRs": the router is batched, and one integer plan is built once and
// reused by grouped W13 and grouped W2 ("avoids repeated planning").
//
// Shapes:
//  * M <= 16 (decode): one thread-block cluster (router_cluster_kernel).  CTA
//    r owns an expert slice and computes its complete logits, which it writes
//    into CTA 0's shared memory; CTA 0 takes each token's top-k over all the
//    experts and computes the weights, the gate and the whole plan, decode
//    work table included.  Where such a cluster cannot be scheduled, a
//    128-block router with arrival tickets (router_small_kernel) does the same.
//  * M > 16 (prefill): the logits as a tcgen05 GEMM (router_logits_kernel, W_r
//    transposed once per call) and one warp per token for top-k, weights and
//    gate (router_topk_kernel); an mma.sync router with the top-k in its
//    epilogue (router_mma_kernel) covers E < 256 and M < 128.  Then a
//    three-kernel stable counting sort builds the plan.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "route.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Plan of at most 32 pairs (M <= 16), with no block barrier.  Warp 0 holds
// pair q in lane q: its validity, its rank among the pairs of its expert (a
// match over the lanes), its plan position (valid pairs of a lower expert, by
// comparison with the other lanes, plus that rank), perm and inv; the first
// pair of each expert writes the expert's active entry, its tile (at most 32
// rows: one), its decode work-table entry, and every pair its own id into
// that entry.  The other warps write counts and offsets of every expert
// straight from the pair list.  Same plan as the general path below.
// ---------------------------------------------------------------------------
__device__ void plan_tiny(const LayerDims& d, int M, const int* src, const PlanView& pv,
                          uint32_t* status) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int P = M * d.k_eff, ne = d.e_eff;
  if (tid < 32) {
    const int e_in = lane < P ? src[lane] : -1;
    const bool ok = lane < P && pair_valid(e_in, lane % d.k_eff, d);
    if (__ballot_sync(0xffffffffu, lane < P && !ok) && lane == 0)
      set_status(status, MOE_ST_INVALID_ID);
    const uint32_t vmask = __ballot_sync(0xffffffffu, ok);
    const int e = ok ? e_in : -1 - lane;  // lanes without a valid pair match only themselves
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int before = __popc(same & ((1u << lane) - 1u)), total = __popc(same);
    const uint32_t fmask = __ballot_sync(0xffffffffu, ok && before == 0);
    int less = 0, a = 0;  // valid pairs / experts' first pairs of a lower expert
    for (int q = 0; q < P; ++q) {
      const int eq = __shfl_sync(0xffffffffu, e, q);
      less += (int)((vmask >> q) & 1u) & (int)(eq < e);
      a += (int)((fmask >> q) & 1u) & (int)(eq < e);
    }
    const int pos = less + before, na = __popc(fmask);
    if (lane < P) pv.inv[lane] = ok ? pos : -1;
    if (ok) {
      pv.perm[pos] = lane;
      int* ent = pv.dtab + (size_t)a * kDtabInts;
      if (before < kDtabInts - 4) ent[4 + before] = lane;
      if (before == 0) {
        pv.active[a] = e;
        reinterpret_cast<int4*>(pv.tiles)[a] = make_int4(e, 0, total, pos);
        reinterpret_cast<int4*>(ent)[0] = make_int4(e, pos, total, -1);
        for (int r = total; r < kDtabInts - 4; ++r) ent[4 + r] = -1;
      }
    }
    // entries na .. min(P, ne) - 1 of the work table: unused, all -1
    const int n_pad = (min(P, ne) - na) * 5;
    for (int i = lane; i < n_pad; i += 32)
      reinterpret_cast<int4*>(pv.dtab)[na * 5 + i] = make_int4(-1, -1, -1, -1);
    if (lane == 0) {
      pv.hdr->M = M;
      pv.hdr->k_eff = d.k_eff;
      pv.hdr->e_eff = ne;
      pv.hdr->n_valid = __popc(vmask);
      pv.hdr->n_active = na;
      pv.hdr->n_tiles = na;
    }
  } else {
    // offsets[e] = valid pairs of an expert below e (offsets[ne] = all valid
    // pairs), counts[e] = valid pairs of expert e
    for (int e = tid - 32; e <= ne; e += (int)blockDim.x - 32) {
      int c = 0, l = 0, slot = 0;
      for (int q = 0; q < P; ++q) {
        const int eq = src[q];
        const bool okq = pair_valid(eq, slot, d);
        c += (int)(okq && eq == e);
        l += (int)(okq && eq < e);
        if (++slot == d.k_eff) slot = 0;
      }
      pv.offsets[e] = l;
      if (e < ne) pv.counts[e] = c;
    }
  }
}

// The plan header and the decode work table from the sorted active list
// (expert, first position, rows) and the pair at each plan position, all in
// shared memory.  Work table: every entry up to the largest active-expert
// count, as five 16-byte groups (expert, first position, rows, -1 | first 16
// pair ids, -1 past the expert's rows); entries past the active experts -1.
__device__ void plan_header_and_table(const LayerDims& d, int M, int nv, int na, int nt,
                                      const int* s_ae, const int* s_aoff, const int* s_acnt,
                                      const int* s_perm, const PlanView& pv) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int P = M * d.k_eff, ne = d.e_eff;
  if (tid == 0) {
    pv.hdr->M = M;
    pv.hdr->k_eff = d.k_eff;
    pv.hdr->e_eff = ne;
    pv.hdr->n_valid = nv;
    pv.hdr->n_active = na;
    pv.hdr->n_tiles = nt;
  }
  static_assert(kDtabInts == 20, "a work-table entry is five 16-byte groups");
  const int max_active = min(P, ne);
  for (int i = tid; i < max_active * 5; i += nthr) {
    const int a = i / 5, f4 = i - a * 5;
    int4 v = make_int4(-1, -1, -1, -1);
    if (a < na) {
      const int off = s_aoff[a], cnt = s_acnt[a];
      if (f4 == 0) {
        v = make_int4(s_ae[a], off, cnt, -1);
      } else {
        const int r = 4 * (f4 - 1);
        v.x = r < cnt ? s_perm[off + r] : -1;
        v.y = r + 1 < cnt ? s_perm[off + r + 1] : -1;
        v.z = r + 2 < cnt ? s_perm[off + r + 2] : -1;
        v.w = r + 3 < cnt ? s_perm[off + r + 3] : -1;
      }
    }
    reinterpret_cast<int4*>(pv.dtab)[i] = v;
  }
}

// ---------------------------------------------------------------------------
// Plan of up to kDecodeMaxTokens * (32 + 1) pairs by one block of 256 threads.
// `src` (shared memory) holds the M * k_eff expert ids of the pairs.  Also
// writes the decode work table.  Up to 32 pairs: plan_tiny.  Otherwise each
// expert's token set is gathered first (one bit per token); where no token
// lists an expert twice, one block scan over the experts gives counts,
// offsets, active ranks and tiles, and a pair's position is its expert's
// offset plus the earlier tokens in the expert's set.  Where a token does
// list an expert twice, three steps separated by barriers:
//   1. each pair's plan position, by direct comparison over the pairs (valid
//      pairs of a lower expert, plus those of the same expert and a lower pair
//      id): perm and inv; the first pair of each expert records the expert's
//      row count;
//   2. each active expert's rank and first tile: at up to 64 pairs by direct
//      comparison over the experts' first pairs, above that by a block scan
//      over the plan positions (an expert starts where the expert changes);
//      active, tiles and the sorted active list in shared memory;
//   3. counts and offsets of every expert (binary search in the active list),
//      the header and the decode work table (16-byte stores).
// ---------------------------------------------------------------------------
// Shared-memory scratch of plan_small_block (its caller places it).
struct PlanScratch {
  int ids[kDtabEntries];   // expert of each pair, -1 if invalid
  int perm[kDtabEntries];  // pair at each plan position
  int cnt1[kDtabEntries];  // rows of the pair's expert if it is the first, else 0
  int pos1[kDtabEntries];  // plan position of an expert's first pair
  int ae[kDtabEntries], aoff[kDtabEntries], acnt[kDtabEntries];  // sorted active list
  int nv, na, nt, dup;
};

__device__ void plan_small_block(const LayerDims& d, int M, const int* src, const PlanView& pv,
                                 uint32_t* status, PlanScratch* ps) {
  int* const s_ids = ps->ids;
  int* const s_perm = ps->perm;
  int* const s_cnt1 = ps->cnt1;
  int* const s_pos1 = ps->pos1;
  int* const s_ae = ps->ae;
  int* const s_aoff = ps->aoff;
  int* const s_acnt = ps->acnt;
  int& s_nv = ps->nv;
  int& s_na = ps->na;
  int& s_nt = ps->nt;
  int& s_dup = ps->dup;
  static_assert(kDtabEntries >= kMaxEEff, "per-expert arrays share the per-pair ones");
  // the token set of each expert (bit m for token m) and each expert's first
  // plan position share s_cnt1 / s_pos1, which only the step-by-step path uses
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_cnt1);
  int* s_off = s_pos1;
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;
  const int P = M * d.k_eff, ne = d.e_eff;
  if (P <= 32) {
    plan_tiny(d, M, src, pv, status);
    return;
  }
  if (tid == 0) {
    s_nv = 0;
    s_na = 0;
    s_nt = 0;
    s_dup = 0;
  }
  for (int e = tid; e < ne; e += nthr) s_mask[e] = 0u;
  __syncthreads();
  bool bad = false, dup = false;
  int nvalid = 0;
  for (int p = tid; p < P; p += nthr) {
    const int e = src[p];
    const bool ok = pair_valid(e, p % d.k_eff, d);
    s_ids[p] = ok ? e : -1;
    bad = bad || !ok;
    nvalid += ok;
    if (ok) {
      const uint32_t bit = 1u << (p / d.k_eff);
      dup = dup || (atomicOr(&s_mask[e], bit) & bit);
    }
  }
  if (bad) set_status(status, MOE_ST_INVALID_ID);
  if (dup) s_dup = 1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) nvalid += __shfl_xor_sync(0xffffffffu, nvalid, o);
  if (lane == 0 && nvalid) atomicAdd(&s_nv, nvalid);
  __syncthreads();
  if (tid == 0) MOE_TL_MAX(36);
  const int nv = s_nv;
  if (!s_dup) {
    // No token lists an expert twice (every routed call: the top-k ids are
    // distinct): an expert's pairs come one per token, in token order, so a
    // pair's rank inside its expert is the number of earlier tokens in the
    // expert's token set.  Experts 3 tid .. 3 tid + 2 take their counts,
    // offsets, active ranks and tiles from one block scan.
    int c[3], sa = 0, st = 0, so = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int e = 3 * tid + i;
      c[i] = e < ne ? __popc(s_mask[e]) : 0;
      sa += c[i] != 0;
      st += (c[i] + kTileRows - 1) / kTileRows;
      so += c[i];
    }
    int tot[3];
    block_scan3(sa, st, so, tot);
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int e = 3 * tid + i;
      if (e >= ne) break;
      pv.counts[e] = c[i];
      pv.offsets[e] = so;
      s_off[e] = so;
      if (c[i] != 0) {
        s_ae[sa] = e;
        s_aoff[sa] = so;
        s_acnt[sa] = c[i];
        pv.active[sa] = e;
        for (int r0 = 0; r0 < c[i]; r0 += kTileRows, ++st)
          reinterpret_cast<int4*>(pv.tiles)[st] =
              make_int4(e, r0, min(kTileRows, c[i] - r0), so + r0);
        ++sa;
      }
      so += c[i];
    }
    if (tid == 0) {
      pv.offsets[ne] = nv;
      s_na = tot[0];
      s_nt = tot[1];
    }
    __syncthreads();
    for (int p = tid; p < P; p += nthr) {
      const int e = s_ids[p];
      if (e < 0) {
        pv.inv[p] = -1;
        continue;
      }
      const int m = p / d.k_eff;
      const int pos = s_off[e] + __popc(s_mask[e] & ((1u << m) - 1u));
      pv.perm[pos] = p;
      pv.inv[p] = pos;
      s_perm[pos] = p;
    }
    __syncthreads();
    plan_header_and_table(d, M, nv, s_na, s_nt, s_ae, s_aoff, s_acnt, s_perm, pv);
    return;
  }
  // 1. positions
  for (int p = tid; p < P; p += nthr) {
    const int e = s_ids[p];
    s_cnt1[p] = 0;
    if (e < 0) {
      pv.inv[p] = -1;
      continue;
    }
    int less = 0, before = 0, total = 0;
    for (int q = 0; q < P; ++q) {
      const int eq = s_ids[q];
      less += (eq >= 0 && eq < e);
      before += (eq == e && q < p);
      total += (eq == e);
    }
    const int pos = less + before;
    pv.perm[pos] = p;
    pv.inv[p] = pos;
    s_perm[pos] = p;
    if (before == 0) {
      s_cnt1[p] = total;
      s_pos1[p] = pos;
    }
  }
  __syncthreads();
  if (tid == 0) MOE_TL_MAX(38);
  // 2. active experts and tiles
  if (P <= 64) {
    // one pair per thread: the first pair of each expert counts the lower
    // experts' first pairs and their tiles
    const int p = tid;
    const int c = p < P ? s_cnt1[p] : 0;
    if (c != 0) {
      const int e = s_ids[p];
      int a = 0, t0 = 0, higher = 0;
      for (int q = 0; q < P; ++q) {
        const int cq = s_cnt1[q];
        if (cq == 0) continue;
        const int eq = s_ids[q];
        if (eq < e) {
          ++a;
          t0 += (cq + kTileRows - 1) / kTileRows;
        }
        higher += eq > e;
      }
      s_ae[a] = e;
      s_aoff[a] = s_pos1[p];
      s_acnt[a] = c;
      pv.active[a] = e;
      const int nt_e = (c + kTileRows - 1) / kTileRows;
      for (int r = 0; r < nt_e; ++r)
        reinterpret_cast<int4*>(pv.tiles)[t0 + r] =
            make_int4(e, r * kTileRows, min(kTileRows, c - r * kTileRows),
                      s_pos1[p] + r * kTileRows);
      if (higher == 0) {  // the highest active expert knows the totals
        s_na = a + 1;
        s_nt = t0 + nt_e;
      }
    }
  } else {
    // positions 3 tid .. 3 tid + 2: an expert starts at each position whose
    // pair is its expert's first (the lowest pair id comes first)
    int fl[3], cn[3], sa = 0, st = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const int j = 3 * tid + i;
      cn[i] = j < nv ? s_cnt1[s_perm[j]] : 0;
      fl[i] = cn[i] != 0;
      sa += fl[i];
      st += fl[i] ? (cn[i] + kTileRows - 1) / kTileRows : 0;
    }
    int zero = 0, tot[3];
    block_scan3(sa, st, zero, tot);
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      if (!fl[i]) continue;
      const int j = 3 * tid + i, e = s_ids[s_perm[j]], c = cn[i];
      s_ae[sa] = e;
      s_aoff[sa] = j;
      s_acnt[sa] = c;
      pv.active[sa] = e;
      for (int r0 = 0; r0 < c; r0 += kTileRows, ++st)
        reinterpret_cast<int4*>(pv.tiles)[st] = make_int4(e, r0, min(kTileRows, c - r0), j + r0);
      ++sa;
    }
    if (tid == 0) {
      s_na = tot[0];
      s_nt = tot[1];
    }
  }
  __syncthreads();
  if (tid == 0) MOE_TL_MAX(40);
  // 3. counts / offsets of every expert, header, work table
  const int na = s_na;
  for (int e = tid; e <= ne; e += nthr) {
    int lo = 0, hi = na;  // first active expert >= e
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_ae[mid] < e)
        lo = mid + 1;
      else
        hi = mid;
    }
    if (e == ne) {
      pv.offsets[ne] = nv;
    } else {
      pv.offsets[e] = lo < na ? s_aoff[lo] : nv;
      pv.counts[e] = (lo < na && s_ae[lo] == e) ? s_acnt[lo] : 0;
    }
  }
  plan_header_and_table(d, M, nv, na, s_nt, s_ae, s_aoff, s_acnt, s_perm, pv);
  if (tid == 0) MOE_TL_MAX(42);
}

// ---------------------------------------------------------------------------
// Small-M router + plan (one launch).
// grid = (ceil(E / 64), H / kRsRows), block = 256: warp w of block (s, c)
// streams rows [c*kRsRows + 16w, +16) of W_r for experts [64s, 64s+64).
// ---------------------------------------------------------------------------
constexpr int kRsRows = 128;

__global__ void __launch_bounds__(256) router_small_kernel(LayerDims d, int M,
                                                           const __half* __restrict__ x,
                                                           const __half* __restrict__ wr,
                                                           const float* __restrict__ bias,
                                                           const __half* __restrict__ wg,
                                                           int32_t* ids_user, float* w_user,
                                                           PlanView pv, uint32_t* status) {
  __shared__ float xs[kDecodeMaxTokens][kRsRows];
  __shared__ float red[4][kDecodeMaxTokens][64];
  __shared__ int s_ids[kDecodeMaxTokens * 33];
  __shared__ int is_last;
  MOE_TL(kTlRouter);
  // the forward kernels may become resident now; they wait for this grid
  pdl_launch_dependents();
  const int s = blockIdx.x, hc = blockIdx.y;
  const int E = d.E, H = d.H;
  const int h0 = hc * kRsRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = s * 64 + 2 * lane;
  const bool ev = e0 < E;
  __half2 wv[16];
#pragma unroll
  for (int r = 0; r < 16; ++r)
    wv[r] = ev ? *reinterpret_cast<const __half2*>(wr + (int64_t)(h0 + warp * 16 + r) * E + e0)
               : __float2half2_rn(0.f);
  for (int i = tid; i < kDecodeMaxTokens * kRsRows; i += 256) {
    const int m = i / kRsRows, c = i % kRsRows;
    xs[m][c] = (m < M) ? __half2float(x[(int64_t)m * H + h0 + c]) : 0.f;
  }
  __syncthreads();
  float acc[kDecodeMaxTokens][2];
#pragma unroll
  for (int m = 0; m < kDecodeMaxTokens; ++m) acc[m][0] = acc[m][1] = 0.f;
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float2 f = __half22float2(wv[r]);
#pragma unroll
    for (int m = 0; m < kDecodeMaxTokens; ++m) {
      if (m < M) {
        const float xv = xs[m][warp * 16 + r];
        acc[m][0] = fmaf(xv, f.x, acc[m][0]);
        acc[m][1] = fmaf(xv, f.y, acc[m][1]);
      }
    }
  }
  // fixed-order reduction over the 8 warps: (w, w + 4) pairs, then w = 0..3
  if (warp >= 4) {
#pragma unroll
    for (int m = 0; m < kDecodeMaxTokens; ++m) {
      if (m < M) {
        red[warp - 4][m][2 * lane] = acc[m][0];
        red[warp - 4][m][2 * lane + 1] = acc[m][1];
      }
    }
  }
  __syncthreads();
  if (warp < 4) {
#pragma unroll
    for (int m = 0; m < kDecodeMaxTokens; ++m) {
      if (m < M) {
        red[warp][m][2 * lane] += acc[m][0];
        red[warp][m][2 * lane + 1] += acc[m][1];
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < M * 64; i += 256) {
    const int m = i >> 6, c = i & 63, e = s * 64 + c;
    const float t = (red[0][m][c] + red[1][m][c]) + (red[2][m][c] + red[3][m][c]);
    if (e < E) pv.partial[((int64_t)hc * kDecodeMaxTokens + m) * E + e] = t;
  }
  if (tid == 0) MOE_TL_MAX(20);
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atomicAdd(&pv.tickets[s], 1u);
    is_last = (t == gridDim.y - 1);
    if (is_last) pv.tickets[s] = 0u;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (tid == 0) MOE_TL_MIN(21);
  // slice finaliser: fixed-order sum over the H chunks, + bias
  const int nh = gridDim.y;
  for (int i = tid; i < M * 64; i += 256) {
    const int m = i >> 6, c = i & 63, e = s * 64 + c;
    if (e >= E) continue;
    const float* src = pv.partial + (int64_t)m * E + e;
    const int64_t stride = (int64_t)kDecodeMaxTokens * E;
    float t = 0.f;
    int q = 0;
    for (; q + 8 <= nh; q += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (q + u) * stride);
#pragma unroll
      for (int u = 0; u < 8; ++u) t += v[u];
    }
    for (; q < nh; ++q) t += __ldcg(src + q * stride);
    if (bias) t += bias[e];
    pv.logits[(int64_t)m * E + e] = t;
  }
  if (tid == 0) MOE_TL_MAX(22);
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atomicAdd(&pv.tickets[63], 1u);
    is_last = (t == gridDim.x - 1);
    if (is_last) pv.tickets[63] = 0u;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (tid == 0) MOE_TL_MIN(23);
  for (int m = warp; m < M; m += 8) {
    int id;
    float l;
    warp_topk<true>(pv.logits + (int64_t)m * E, E, d.k, &id, &l);
    if (m == 0 && lane == 0) MOE_TL_MAX(46);
    const float w = warp_topk_weight(l, d.k);
    const float gamma = d.shared ? warp_gate(x + (int64_t)m * H, wg, H) : 0.f;
    store_route(d, m, id, w, gamma, ids_user, w_user, pv);
    if (lane < d.k) s_ids[m * d.k_eff + lane] = id;
    if (d.shared && lane == 0) s_ids[m * d.k_eff + d.k] = d.E;
  }
  __syncthreads();
  if (tid == 0) MOE_TL_MAX(24);
  __shared__ PlanScratch ps;
  plan_small_block(d, M, s_ids, pv, status, &ps);
  if (tid == 0) MOE_TL_MIN(25);
}

// Caller-given ids and weights: copy into the plan (plus the shared slot).
// grid = ceil(M / 8), block = 256 (one warp per token).
__global__ void route_given_kernel(LayerDims d, int M, const __half* __restrict__ x,
                                   const __half* __restrict__ wg, const int32_t* ids_user,
                                   const float* w_user, PlanView pv) {
  MOE_TL(kTlRouter);
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= M) return;
  if (lane < d.k) {
    pv.ids[(int64_t)t * d.k_eff + lane] = ids_user[(int64_t)t * d.k + lane];
    pv.w[(int64_t)t * d.k_eff + lane] = w_user[(int64_t)t * d.k + lane];
  }
  if (d.shared) {
    const float gamma = warp_gate(x + (int64_t)t * d.H, wg, d.H);
    if (lane == 0) {
      pv.ids[(int64_t)t * d.k_eff + d.k] = d.E;
      pv.w[(int64_t)t * d.k_eff + d.k] = gamma;
    }
  }
}

__global__ void __launch_bounds__(256) plan_small_kernel(LayerDims d, int M, PlanView pv,
                                                         uint32_t* status) {
  __shared__ int s_src[kDecodeMaxTokens * 33];
  MOE_TL(kTlPlan);
  pdl_launch_dependents();
  for (int p = threadIdx.x; p < M * d.k_eff; p += blockDim.x) s_src[p] = pv.ids[p];
  __syncthreads();
  __shared__ PlanScratch ps;
  plan_small_block(d, M, s_src, pv, status, &ps);
}

// ---------------------------------------------------------------------------
// Large-M router: 64 tokens x all experts per block, mma.sync m16n8k16 with
// FP32 accumulation, top-k in the epilogue.  block = 512 (16 warps: 2 token
// halves x 8 groups of 64 experts).
// ---------------------------------------------------------------------------
constexpr int kRtTok = 64;
constexpr int kRtK = 32;
static_assert(kRtK == kRouterSplitRows, "router K split granularity");

__device__ __forceinline__ void ldsm_x4(uint32_t r[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

size_t router_mma_smem(int E) {
  const int Ep = (E + 63) / 64 * 64;
  const size_t pipe = 2 * (size_t)(kRtTok * (kRtK + 8) + kRtK * (Ep + 8)) * sizeof(__half);
  const size_t logits = (size_t)kRtTok * (Ep + 1) * sizeof(float);
  return pipe > logits ? pipe : logits;
}

// blockIdx.y = K split: 32-row K steps [y * steps_per_split, ...).  With
// `partial` the block writes its split's FP32 partial logits [split][M][E]
// (no bias; router_split_topk_kernel adds the splits up); without it (one
// split) the top-k runs in the epilogue.
__global__ void __launch_bounds__(512) router_mma_kernel(LayerDims d, int M,
                                                         const __half* __restrict__ x,
                                                         const __half* __restrict__ wr,
                                                         const float* __restrict__ bias,
                                                         const __half* __restrict__ wg,
                                                         int32_t* ids_user, float* w_user,
                                                         PlanView pv, int steps_per_split,
                                                         float* __restrict__ partial) {
  extern __shared__ __align__(16) char smem[];
  MOE_TL(kTlRouter);
  const int E = d.E, H = d.H;
  const int Ep = (E + 63) / 64 * 64;
  const int xst = kRtK + 8, wst = Ep + 8, lst = Ep + 1;
  __half* xs = reinterpret_cast<__half*>(smem);
  __half* ws = xs + 2 * kRtTok * xst;
  float* ls = reinterpret_cast<float*>(smem);
  const int t0 = blockIdx.x * kRtTok;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tg = warp >> 3, eg = warp & 7;
  const int cpr = Ep / 8;

  auto load_stage = [&](int st, int kk) {
    for (int i = tid; i < kRtTok * 4; i += 512) {
      const int r = i >> 2, c = i & 3, t = t0 + r;
      const __half* src = x + (int64_t)(t < M ? t : 0) * H + kk + c * 8;
      cp_async16(smem_u32(xs + (st * kRtTok + r) * xst + c * 8), src, t < M ? 16u : 0u);
    }
    for (int i = tid; i < kRtK * cpr; i += 512) {
      const int r = i / cpr, c = i - r * cpr;
      const bool in = c * 8 < E;
      const __half* src = wr + (int64_t)(kk + r) * E + (in ? c * 8 : 0);
      cp_async16(smem_u32(ws + (st * kRtK + r) * wst + c * 8), src, in ? 16u : 0u);
    }
  };

  float acc[2][8][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;

  const int k_first = blockIdx.y * steps_per_split;
  const int nk = min(H / kRtK - k_first, steps_per_split);
  load_stage(0, k_first * kRtK);
  cp_async_commit();
  for (int it = 0; it < nk; ++it) {
    if (it + 1 < nk) load_stage((it + 1) & 1, (k_first + it + 1) * kRtK);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int st = it & 1;
    if (eg * 64 < E) {
#pragma unroll
      for (int k16 = 0; k16 < 2; ++k16) {
        uint32_t a[2][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
          ldsm_x4(a[mi], xs + (st * kRtTok + tg * 32 + mi * 16 + (lane & 15)) * xst + k16 * 16 +
                             (lane >> 4) * 8);
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) {
          const int n0 = eg * 64 + nj * 16;
          uint32_t b[4];
          ldsm_x4_t(b, ws + (st * kRtK + k16 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * wst +
                           n0 + (lane >> 4) * 8);
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            mma_16816(acc[mi][2 * nj], a[mi], b[0], b[1]);
            mma_16816(acc[mi][2 * nj + 1], a[mi], b[2], b[3]);
          }
        }
      }
    }
    __syncthreads();
  }
  const int g = lane >> 2, t4 = lane & 3;
  if (partial) {
    // this split's partial logits, in the accumulator layout
    if (eg * 64 < E) {
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int e = eg * 64 + nt * 8 + 2 * t4;
          const int r = tg * 32 + mi * 16 + g;
          if (e < E) {
            float* p0 = partial + ((size_t)blockIdx.y * M + t0 + r) * E + e;
            if (t0 + r < M) {
              p0[0] = acc[mi][nt][0];
              p0[1] = acc[mi][nt][1];
            }
            if (t0 + r + 8 < M) {
              p0[8 * (size_t)E] = acc[mi][nt][2];
              p0[8 * (size_t)E + 1] = acc[mi][nt][3];
            }
          }
        }
    }
    return;
  }
  // logits -> shared memory (the pipeline buffers are dead now)
  if (eg * 64 < E) {
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int e = eg * 64 + nt * 8 + 2 * t4;
        const int r = tg * 32 + mi * 16 + g;
        if (e < E) {
          const float b0 = bias ? bias[e] : 0.f, b1 = bias ? bias[e + 1] : 0.f;
          ls[r * lst + e] = acc[mi][nt][0] + b0;
          ls[r * lst + e + 1] = acc[mi][nt][1] + b1;
          ls[(r + 8) * lst + e] = acc[mi][nt][2] + b0;
          ls[(r + 8) * lst + e + 1] = acc[mi][nt][3] + b1;
        }
      }
  }
  __syncthreads();
  for (int r = warp; r < kRtTok; r += 16) {
    const int t = t0 + r;
    if (t >= M) break;
    int id;
    float l;
    warp_topk<false>(ls + r * lst, E, d.k, &id, &l);
    const float w = warp_topk_weight(l, d.k);
    const float gamma = d.shared ? warp_gate(x + (int64_t)t * H, wg, H) : 0.f;
    store_route(d, t, id, w, gamma, ids_user, w_user, pv);
  }
}

// One warp per token: its logits as the K splits' partial sums added in split
// order (+ bias), then top-k, renormalised weights, gate and the route.
// block = 256 (8 tokens), dynamic shared memory 8 x E floats.
__global__ void __launch_bounds__(256) router_split_topk_kernel(
    LayerDims d, int M, int n_split, const float* __restrict__ partial,
    const float* __restrict__ bias, const __half* __restrict__ x, const __half* __restrict__ wg,
    int32_t* ids_user, float* w_user, PlanView pv) {
  extern __shared__ float rs_rows[];
  MOE_TL(kTlPlan);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= M) return;
  const int E = d.E;
  float* row = rs_rows + (size_t)warp * E;
  for (int e = lane; e < E; e += 32) {
    const float* src = partial + (size_t)t * E + e;
    const size_t stride = (size_t)M * E;
    float sum = 0.f;
    int s0 = 0;
    for (; s0 + 8 <= n_split; s0 += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (s0 + u) * stride);
#pragma unroll
      for (int u = 0; u < 8; ++u) sum += v[u];
    }
    for (; s0 < n_split; ++s0) sum += __ldcg(src + s0 * stride);
    row[e] = bias ? sum + bias[e] : sum;
  }
  __syncwarp();
  int id;
  float l;
  warp_topk<false>(row, E, d.k, &id, &l);
  const float w = warp_topk_weight(l, d.k);
  const float gamma = d.shared ? warp_gate(x + (int64_t)t * d.H, wg, d.H) : 0.f;
  store_route(d, t, id, w, gamma, ids_user, w_user, pv);
}

// ---------------------------------------------------------------------------
// Large-M plan: stable counting sort in three kernels.
// ---------------------------------------------------------------------------
// 1. Per chunk of kPlanChunk pairs: per-expert counts and each pair's rank
//    among the earlier pairs of its expert inside the chunk.  block = 1024.
__global__ void __launch_bounds__(1024) plan_hist_kernel(LayerDims d, int64_t P, PlanView pv,
                                                         uint32_t* status) {
  extern __shared__ uint16_t wcnt[];  // [32 warps][e_eff]: counts, then exclusive prefixes
  __shared__ int run[kMaxEEff];       // count of each expert in earlier sub-chunks
  __shared__ int subtot[kMaxEEff];
  MOE_TL(kTlPlan);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ne = d.e_eff;
  for (int i = tid; i < ne; i += 1024) run[i] = 0;
  bool bad = false;
  const int64_t base = (int64_t)blockIdx.x * kPlanChunk;
  for (int sub = 0; sub < kPlanChunk / 1024; ++sub) {
    for (int i = tid; i < 32 * ne; i += 1024) wcnt[i] = 0;
    __syncthreads();
    const int64_t p = base + sub * 1024 + tid;
    int e = -1;
    if (p < P) {
      e = pv.ids[p];
      if (!pair_valid(e, (int)(p % d.k_eff), d)) {
        e = -1;
        bad = true;
      }
    }
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const unsigned lt = mask & ((1u << lane) - 1u);
    if (e >= 0 && lt == 0) wcnt[warp * ne + e] = (uint16_t)__popc(mask);
    __syncthreads();
    for (int ee = tid; ee < ne; ee += 1024) {
      int r = 0;
      for (int w = 0; w < 32; ++w) {
        const int c = wcnt[w * ne + ee];
        wcnt[w * ne + ee] = (uint16_t)r;
        r += c;
      }
      subtot[ee] = r;
    }
    __syncthreads();
    if (p < P) pv.rank[p] = (e >= 0) ? run[e] + (int)wcnt[warp * ne + e] + __popc(lt) : -1;
    __syncthreads();
    for (int ee = tid; ee < ne; ee += 1024) run[ee] += subtot[ee];
    __syncthreads();
  }
  if (bad) set_status(status, MOE_ST_INVALID_ID);
  for (int ee = tid; ee < ne; ee += 1024) pv.chunk_hist[(int64_t)blockIdx.x * ne + ee] = run[ee];
}

// 2. One block: per-expert prefix over chunks, expert offsets, active list,
//    tile schedule and header.  block = 1024.
__global__ void __launch_bounds__(1024) plan_scan_kernel(LayerDims d, int M, int n_chunks,
                                                         PlanView pv) {
  __shared__ int s_cnt[kMaxEEff];
  __shared__ int s_tb[kMaxEEff];
  __shared__ int s_ob[kMaxEEff];
  __shared__ int s_tot[3];
  MOE_TL(kTlPlan);
  const int tid = threadIdx.x, ne = d.e_eff;
  for (int e = tid; e < ne; e += 1024) {
    int r = 0;
    int c = 0;
    // loads in groups of 16, then 8: one dependent round trip per group
    for (; c + 16 <= n_chunks; c += 16) {
      int h[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) h[u] = pv.chunk_hist[(int64_t)(c + u) * ne + e];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        pv.chunk_hist[(int64_t)(c + u) * ne + e] = r;
        r += h[u];
      }
    }
    for (; c + 8 <= n_chunks; c += 8) {
      int h[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) h[u] = pv.chunk_hist[(int64_t)(c + u) * ne + e];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        pv.chunk_hist[(int64_t)(c + u) * ne + e] = r;
        r += h[u];
      }
    }
    for (; c < n_chunks; ++c) {
      const int h = pv.chunk_hist[(int64_t)c * ne + e];
      pv.chunk_hist[(int64_t)c * ne + e] = r;
      r += h;
    }
    s_cnt[e] = r;
  }
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    const int per = (ne + 31) / 32, b = lane * per, end = min(b + per, ne);
    int cs = 0, as = 0, ts = 0;
    for (int i = b; i < end; ++i) {
      const int c = s_cnt[i];
      cs += c;
      as += c > 0;
      ts += (c + kTileRows - 1) / kTileRows;
    }
    int ci = cs, ai = as, ti = ts;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, ci, o);
      const int a2 = __shfl_up_sync(0xffffffffu, ai, o);
      const int a3 = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) {
        ci += a1;
        ai += a2;
        ti += a3;
      }
    }
    if (lane == 31) {
      s_tot[0] = ci;
      s_tot[1] = ai;
      s_tot[2] = ti;
    }
    ci -= cs;
    ai -= as;
    ti -= ts;
    for (int i = b; i < end; ++i) {
      const int c = s_cnt[i];
      s_tb[i] = ti;
      s_ob[i] = ci;
      pv.counts[i] = c;
      pv.offsets[i] = ci;
      if (c > 0) pv.active[ai] = i;
      ci += c;
      ai += c > 0;
      ti += (c + kTileRows - 1) / kTileRows;
    }
  }
  __syncthreads();
  if (tid == 0) {
    pv.offsets[ne] = s_tot[0];
    pv.hdr->M = M;
    pv.hdr->k_eff = d.k_eff;
    pv.hdr->e_eff = ne;
    pv.hdr->n_valid = s_tot[0];
    pv.hdr->n_active = s_tot[1];
    pv.hdr->n_tiles = s_tot[2];
  }
  for (int e = tid; e < ne; e += 1024) {
    const int c = s_cnt[e], o = s_ob[e];
    int t = s_tb[e];
    for (int r0 = 0; r0 < c; r0 += kTileRows, ++t)
      reinterpret_cast<int4*>(pv.tiles)[t] = make_int4(e, r0, min(kTileRows, c - r0), o + r0);
  }
}

// 3. Positions: offset of the expert + rank over earlier chunks + rank in chunk.
__global__ void plan_scatter_kernel(LayerDims d, int64_t P, PlanView pv) {
  MOE_TL(kTlPlan);
  const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= P) return;
  const int r = pv.rank[p];
  if (r < 0) {
    pv.inv[p] = -1;
    return;
  }
  const int e = pv.ids[p];
  const int64_t c = p / kPlanChunk;
  const int pos = pv.offsets[e] + pv.chunk_hist[c * d.e_eff + e] + r;
  pv.perm[pos] = (int)p;
  pv.inv[p] = pos;
}

// ---------------------------------------------------------------------------
// Large-M router on the 5th-generation tensor cores.  The logits are a plain
// FP16 GEMM, D[token][expert] = sum_h x[token][h] W_r[h][expert], with both
// operands K-major: W_r is transposed once per call into the plan buffer.
// One CTA computes 128 tokens x 256 experts: a producer thread loads the
// K steps (64 along H) of both operands by 128-byte-swizzled tensor maps into
// a 4-stage ring, one thread issues tcgen05.mma (M 128, N <= 256, FP32
// accumulator in tensor memory), and four warps move the accumulator (+ bias)
// to the logits rows.  A second kernel, one warp per token over all SMs,
// takes the top-k, the weights and the gate from the logits (resident in L2).
// ---------------------------------------------------------------------------
constexpr int kRlTokens = 128;      // tokens (MMA M) per CTA
constexpr int kRlExperts = 256;     // experts (MMA N) per CTA
constexpr int kRlStages = 4;
constexpr int kRlXBytes = kRlTokens * 128;   // one K step of the token rows
constexpr int kRlWBytes = kRlExperts * 128;  // one K step of the expert rows
constexpr size_t kRlSmem = 1024 + (size_t)kRlStages * (kRlXBytes + kRlWBytes);

// W_r [H][E] -> W_r^T [E][H] through 32 x 32 shared-memory tiles.
__global__ void __launch_bounds__(256) transpose_wr_kernel(const __half* __restrict__ wr, int H,
                                                           int E, __half* __restrict__ wrt) {
  __shared__ __half tile[32][34];
  const int e0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + tx;
    tile[i][tx] = e < E ? wr[(size_t)(h0 + i) * E + e] : __float2half(0.f);
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int e = e0 + i;
    if (e < E) wrt[(size_t)e * H + h0 + tx] = tile[tx][i];
  }
}

__global__ void __launch_bounds__(256, 1)
    router_logits_kernel(LayerDims d, int M0, int Mc, const __grid_constant__ CUtensorMap xmap,
                         const __grid_constant__ CUtensorMap wmap, const float* __restrict__ bias,
                         float* __restrict__ logits, uint32_t* status) {
  extern __shared__ __align__(1024) char rl_raw[];
  char* base = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(rl_raw) + 1023) &
                                       ~uintptr_t(1023));
  __shared__ uint64_t full[kRlStages], empty[kRlStages], accf;
  __shared__ uint32_t tmem_slot;
  MOE_TL(kTlRouter);
  const int E = d.E, H = d.H, S = H / 64;
  const int m0 = blockIdx.x * kRlTokens, e0 = blockIdx.y * kRlExperts;
  const int ne = min(kRlExperts, E - e0);           // experts of this CTA (a multiple of 16)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  char* xs = base;
  char* ws = base + kRlStages * kRlXBytes;
  if (tid == 0) {
    for (int i = 0; i < kRlStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&accf, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, kRlExperts);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (warp == 0) {
    // ---- producer: both operands of each K step into the ring ----
    if (lane == 0) {
      int ks = 0;
      for (; ks < S; ++ks) {
        const int st = ks % kRlStages;
        if (!mbar_wait(&empty[st], ((ks / kRlStages) & 1) ^ 1, status)) break;
        mbar_expect_tx(&full[st], kRlXBytes + kRlWBytes);
        tma_load_2d(xs + st * kRlXBytes, &xmap, ks * 64, M0 + m0, &full[st]);
        tma_load_2d(ws + st * kRlWBytes, &wmap, ks * 64, e0, &full[st]);
      }
      // the copies of the last stages land before the CTA may leave
      for (int k = ks > kRlStages ? ks - kRlStages : 0; k < ks; ++k)
        mbar_wait(&full[k % kRlStages], (k / kRlStages) & 1, status);
    }
  } else if (warp == 1) {
    // ---- MMA issuer: per K step one wait, 4 MMAs of K 16, one commit ----
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(kRlTokens, ne);
      for (int ks = 0; ks < S; ++ks) {
        const int st = ks % kRlStages;
        if (!mbar_wait(&full[st], (ks / kRlStages) & 1, status)) break;
        tc_fence_after();
        const uint64_t dx = sdesc_sw128(smem_u32(xs + st * kRlXBytes));
        const uint64_t dw = sdesc_sw128(smem_u32(ws + st * kRlWBytes));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_f16(tmem, dx + 2 * kk, dw + 2 * kk, idesc, (ks | kk) ? 1u : 0u);
        tc_commit(&empty[st]);
      }
      tc_commit(&accf);  // also after an abort: every MMA issued completes first
    }
  } else if (warp >= 4) {
    // ---- epilogue: lane r of warp q holds token 32 q + r of the tile ----
    const int q = warp & 3;
    if (mbar_wait(&accf, 0, status)) {
      tc_fence_after();
      const int t = m0 + q * 32 + lane;  // token within the chunk
      float* row = logits + (size_t)t * E + e0;
      for (int c0 = 0; c0 < ne; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
        if (t < Mc) {
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const int e = c0 + 4 * j4;
            if (e < ne) {
              float4 o;
              o.x = __uint_as_float(v[4 * j4 + 0]) + (bias ? bias[e0 + e + 0] : 0.f);
              o.y = __uint_as_float(v[4 * j4 + 1]) + (bias ? bias[e0 + e + 1] : 0.f);
              o.z = __uint_as_float(v[4 * j4 + 2]) + (bias ? bias[e0 + e + 2] : 0.f);
              o.w = __uint_as_float(v[4 * j4 + 3]) + (bias ? bias[e0 + e + 3] : 0.f);
              *reinterpret_cast<float4*>(row + e) = o;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kRlExperts);
  }
}

// One warp per token of the chunk: top-k of the logits row, renormalised
// weights, the shared expert's gate, the route.
__global__ void __launch_bounds__(256) router_topk_kernel(LayerDims d, int M0, int Mc,
                                                          const float* __restrict__ logits,
                                                          const __half* __restrict__ x,
                                                          const __half* __restrict__ wg,
                                                          int32_t* ids_user, float* w_user,
                                                          PlanView pv) {
  __shared__ uint32_t s_slot[8][32][2];  // each warp's gathered candidates
  MOE_TL(kTlPlan);
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= Mc) return;
  const int t = M0 + r;
  int id;
  float l;
  warp_topk_gathered(logits + (size_t)r * d.E, d.E, d.k, s_slot[threadIdx.x >> 5], &id, &l);
  const float w = warp_topk_weight(l, d.k);
  const float gamma = d.shared ? warp_gate(x + (int64_t)t * d.H, wg, d.H) : 0.f;
  store_route(d, t, id, w, gamma, ids_user, w_user, pv);
}

// The tensor-core router covers E >= 256 (a multiple of 16) and M >= 128.
static bool router_tc_ok(const LayerDims& d, int64_t M) {
  return d.E >= kRlExperts && d.E % 16 == 0 && M >= kRlTokens;
}

static cudaError_t launch_router_tc(const LayerDims& d, int64_t M, const __half* x,
                                    const __half* w_router, const float* bias,
                                    const __half* w_gate, int32_t* ids_user, float* w_user,
                                    const PlanView& pv, uint32_t* status, cudaStream_t stream) {
  transpose_wr_kernel<<<dim3((d.E + 31) / 32, d.H / 32), 256, 0, stream>>>(w_router, d.H, d.E,
                                                                             pv.wrt);
  CUtensorMap xmap, wmap;
  cudaError_t e = make_fp16_map(&xmap, x, (uint64_t)d.H, (uint64_t)M, 64, kRlTokens, true);
  if (e != cudaSuccess) return e;
  e = make_fp16_map(&wmap, pv.wrt, (uint64_t)d.H, (uint64_t)d.E, 64, kRlExperts, true);
  if (e != cudaSuccess) return e;
  for (int64_t M0 = 0; M0 < M; M0 += kRouterChunk) {
    const int Mc = (int)std::min<int64_t>(kRouterChunk, M - M0);
    const dim3 grid((unsigned)((Mc + kRlTokens - 1) / kRlTokens),
                    (unsigned)((d.E + kRlExperts - 1) / kRlExperts));
    router_logits_kernel<<<grid, 256, kRlSmem, stream>>>(d, (int)M0, Mc, xmap, wmap, bias,
                                                        pv.rlogits, status);
    router_topk_kernel<<<(Mc + 7) / 8, 256, 0, stream>>>(d, (int)M0, Mc, pv.rlogits, x, w_gate,
                                                         ids_user, w_user, pv);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Small-M router + plan as one thread-block cluster of C CTAs (C <= 16).  CTA
// r owns the expert slice [r Es, (r + 1) Es) (Es a multiple of 16) and
// computes those experts' complete logits: each of its 8 warps takes one
// eighth of K, loads its W_r tiles ([K rows][Es experts], swizzled) with 2-D
// tensor-map copies and multiplies them with the staged token rows on
// mma.sync (FP32 accumulate); the 8 partial sums are added in warp order.
// The slice's logits then go straight into CTA 0's shared memory as
// asynchronous remote stores that complete on one of its mbarriers (the
// other CTAs exit after issuing them), and CTA 0 takes every token's top-k
// over all experts (one warp per token), computes the weights and the gate
// and builds the whole plan.
// ---------------------------------------------------------------------------
constexpr int kRcThreads = 256;
constexpr int kRcWarps = kRcThreads / 32;
constexpr int kRcTileBytes = 8192;  // W_r bytes per tensor-map load (at most)
constexpr size_t kRcSmemBudget = 200 * 1024;  // dynamic; the plan builder adds ~15 KB static

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Four FP32 values into the shared memory of another CTA of the cluster (16
// bytes at cluster address `a`), completing as 16 transaction bytes on the
// mbarrier at cluster address `bar` in that CTA.
__device__ __forceinline__ void st_async_f32x4(uint32_t a, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(a),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void st_async_s32(uint32_t a, int v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.s32 [%0], %1, [%2];" ::"r"(a),
               "r"(v), "r"(bar)
               : "memory");
}
// mbarrier wait with acquire at cluster scope (the data came from other CTAs
// of the cluster); bounded like mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  uint32_t* status) {
  const long long t0 = clock64();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], "
        "%2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (clock64() - t0 > kWaitTimeoutCycles) {
      set_status(status, MOE_ST_TIMEOUT);
      return false;
    }
  }
}

// Shape of one cluster launch: experts per CTA, W_r tile rows, ring depth and
// the shared-memory carve (all offsets 1024-byte aligned).
struct RouterClusterPlan {
  int C, Es, tr, ntw, stages;
  size_t xs, cand, ring, stage, total;
};

__host__ __device__ inline RouterClusterPlan router_cluster_plan(int H, int E, int k, int M,
                                                                 int cmax) {
  RouterClusterPlan p;
  p.Es = 16 * ((E + 16 * cmax - 1) / (16 * cmax));
  p.C = (E + p.Es - 1) / p.Es;
  // K rows per warp (a multiple of 32) in ntw tiles of tr rows (tr a multiple
  // of 16 dividing per_warp, at most one tensor-map load of kRcTileBytes)
  const int per_warp = H / kRcWarps;
  const int tr_max = kRcTileBytes / (2 * p.Es);
  int n = (per_warp + tr_max - 1) / tr_max;
  while (per_warp % n != 0 || (per_warp / n) % 16 != 0) ++n;
  p.tr = per_warp / n;
  p.ntw = n;
  // token rows (M x (H + 8) halves) and a 16-byte zero row, then every
  // expert's logit of every token (M x E), which the CTAs write into CTA 0
  // while it may still read its token rows
  (void)k;
  p.xs = align_up((size_t)M * (H + 8) * 2 + 16, 1024);
  p.cand = align_up((size_t)M * E * 4, 1024);
  // a stage also holds the warp's partial sums ([16][Es] FP32) at the end
  const size_t tile = (size_t)p.tr * p.Es * 2, red = (size_t)kDecodeMaxTokens * p.Es * 4;
  p.stage = align_up(tile > red ? tile : red, 1024);
  const size_t fixed = 1024 + p.xs + p.cand;
  int st = (int)((kRcSmemBudget > fixed ? kRcSmemBudget - fixed : 0) / (kRcWarps * p.stage));
  if (st > 2) st = 2;
  if (st > p.ntw) st = p.ntw;
  p.stages = st;
  // the ring also holds CTA 0's plan scratch once the partial sums are read
  const size_t ring = (size_t)kRcWarps * st * p.stage, scratch = align_up(sizeof(PlanScratch), 1024);
  p.ring = ring > scratch ? ring : scratch;
  p.total = fixed + p.ring;
  return p;
}

__global__ void __launch_bounds__(kRcThreads, 1)
    router_cluster_kernel(LayerDims d, int M, const __half* __restrict__ x,
                          const __grid_constant__ CUtensorMap wrmap, const float* __restrict__ bias,
                          const __half* __restrict__ wg, int32_t* ids_user, float* w_user,
                          PlanView pv, uint32_t* status, int cmax) {
  extern __shared__ __align__(1024) char rsm_raw[];
  char* rsm = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(rsm_raw) + 1023) &
                                      ~uintptr_t(1023));
  __shared__ uint64_t full[kRcWarps][2];
  __shared__ uint64_t xch;  // the logits of this CTA's tokens have landed
  __shared__ uint64_t idb;  // CTA 0: the other CTAs' tokens' expert ids have landed
  __shared__ __align__(16) float s_bias[64];
  __shared__ int s_ids[kDecodeMaxTokens * 33];
  MOE_TL(kTlRouter);
  const int E = d.E, H = d.H, k = d.k;
  const uint32_t rank = cluster_ctarank();
  const RouterClusterPlan L = router_cluster_plan(H, E, k, M, cmax);
  const int Es = L.Es, tr = L.tr, ntw = L.ntw, stages = L.stages;
  const int rb = Es * 2;  // bytes of one W_r tile row
  __half* xs = reinterpret_cast<__half*>(rsm);
  const char* zero_row = rsm + (size_t)M * (H + 8) * 2;
  float* all_lg = reinterpret_cast<float*>(rsm + L.xs);      // [M][E] logits, CTA 0
  char* ring = rsm + L.xs + L.cand;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  char* my_ring = ring + (size_t)warp * stages * L.stage;
  const int kw0 = warp * (H / kRcWarps);  // this warp's first K row

  if (tid == 0) {
    for (int w = 0; w < kRcWarps; ++w) {
      mbar_init(&full[w][0], 1);
      mbar_init(&full[w][1], 1);
    }
    // token m belongs to CTA m % C: every expert's logit of its tokens, and
    // to CTA 0 the other CTAs' tokens' expert ids, arrive as transaction bytes
    const int own = (M > (int)rank) ? (M - 1 - (int)rank) / (int)gridDim.x + 1 : 0;
    mbar_init(&xch, 1);
    mbar_expect_tx(&xch, (uint32_t)(own * E * 4));
    if (rank == 0) {
      mbar_init(&idb, 1);
      mbar_expect_tx(&idb, (uint32_t)((M - own) * k * 4));
    }
    fence_mbar_init();
  }
  __syncthreads();
  // every CTA's barriers are initialised before any CTA writes to them: the
  // cluster barrier is arrived at here and waited on just before the first
  // write
  cluster_arrive();
  if (lane == 0)
    for (int i = 0; i < stages; ++i) {
      mbar_expect_tx(&full[warp][i], (uint32_t)(tr * rb));
      tma_load_2d(my_ring + i * L.stage, &wrmap, (int)rank * Es, kw0 + i * tr, &full[warp][i]);
    }
  // The router weight and bias are inputs of the layer, not of the previous
  // kernel: the first weight copies and the bias slice are in flight before
  // waiting for the preceding grid (programmatic dependent launch), whose
  // outputs (the token rows) and buffers (the plan) are only touched after
  // the wait.
  if (tid < Es) {
    const int ge = (int)rank * Es + tid;
    s_bias[tid] = (bias && ge < E) ? bias[ge] : 0.f;
  }
  pdl_wait();
  // token rows (asynchronous copies, all in flight at once) and the zero row
  // (rows >= M of the MMA read it)
  {
    const int rv = H / 8;  // 16-byte vectors per row
    for (int i = tid; i < M * rv; i += kRcThreads) {
      const int m = i / rv, c = i - m * rv;
      cp_async16(smem_u32(xs + (size_t)m * (H + 8) + 8 * c), x + (size_t)m * H + 8 * c, 16u);
    }
    cp_async_commit();
    if (tid == 0) *reinterpret_cast<uint4*>(const_cast<char*>(zero_row)) = make_uint4(0, 0, 0, 0);
    cp_async_wait<0>();
  }
  __syncthreads();

  // ---- this warp's K rows: [16 tokens] x [Es experts] ----
  constexpr int kMaxPairs = 4;  // Es <= 64
  const int npairs = Es / 16;
  float acc[kMaxPairs][2][4];
#pragma unroll
  for (int j = 0; j < kMaxPairs; ++j)
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[j][t][c] = 0.f;
  const int arow = (lane & 7) + 8 * ((lane >> 3) & 1);
  const char* arow_p =
      arow < M ? reinterpret_cast<const char*>(xs + (size_t)arow * (H + 8)) : nullptr;
  int it = 0;
  bool ok = true;
  for (; it < ntw && ok; ++it) {
    const int st = it % stages;
    ok = mbar_wait(&full[warp][st], (it / stages) & 1, status);
    if (!ok) break;
    const char* tb = my_ring + st * L.stage;
    for (int k0 = 0; k0 < tr; k0 += 16) {
      uint32_t a[4];
      {
        const int col = kw0 + it * tr + k0 + 8 * (lane >> 4);
        ldsm_x4(a, arow_p ? arow_p + (size_t)col * 2 : zero_row);
      }
      const int krow = k0 + arow;
      const int swz = ((krow * rb) >> 7) & (rb / 16 - 1);
#pragma unroll
      for (int j = 0; j < kMaxPairs; ++j) {
        if (j < npairs) {
          uint32_t b[4];
          const int cn = 2 * j + (lane >> 4);
          ldsm_x4_t(b, tb + (size_t)krow * rb + ((cn ^ swz) << 4));
          mma_16816(acc[j][0], a, b[0], b[1]);
          mma_16816(acc[j][1], a, b[2], b[3]);
        }
      }
    }
    __syncwarp();  // every lane is done with the stage
    if (lane == 0 && it + stages < ntw) {
      mbar_expect_tx(&full[warp][st], (uint32_t)(tr * rb));
      tma_load_2d(my_ring + st * L.stage, &wrmap, (int)rank * Es, kw0 + (it + stages) * tr,
                  &full[warp][st]);
    }
  }
  if (!ok && lane == 0) {
    // a copy timed out: let the copies already issued land before the ring is
    // reused (each wait bounded by the same limit)
    for (int jt = it; jt < ntw && jt < it + stages; ++jt)
      mbar_wait(&full[warp][jt % stages], (jt / stages) & 1, status);
  }
  __syncwarp();
  // this warp's partial sums into its own (now idle) first ring stage:
  // c0 (token g, expert 2 t4), c1 (g, 2 t4 + 1), c2 (g + 8, 2 t4), c3 (g + 8, 2 t4 + 1)
  float* red = reinterpret_cast<float*>(my_ring);
#pragma unroll
  for (int j = 0; j < kMaxPairs; ++j)
    if (j < npairs)
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int e = j * 16 + t * 8 + 2 * t4 + (c & 1);
          const int m = g + ((c & 2) ? 8 : 0);
          red[m * Es + e] = acc[j][t][c];
        }
  if (tid == 0) MOE_TL_MAX(20);
  __syncthreads();
  cluster_wait();  // every CTA's barriers are initialised
  // ---- logits of the slice, four experts per thread: the 8 warps' partials
  // in warp order (+ bias), stored straight into the CTA that owns the token
  // (all_lg[m / C][rank Es + e] of CTA m % C); E % 8 == 0 and Es % 16 == 0,
  // so four experts are all valid or all past E ----
  const int C = (int)gridDim.x;
  {
    const int q4 = Es / 4;
    for (int i = tid; i < M * q4; i += kRcThreads) {
      const int m = i / q4, e = 4 * (i - m * q4), ge = (int)rank * Es + e;
      if (ge >= E) continue;
      float4 sum = *reinterpret_cast<const float4*>(s_bias + e);
      float4 p[kRcWarps];
#pragma unroll
      for (int w = 0; w < kRcWarps; ++w)
        p[w] = *reinterpret_cast<const float4*>(
            reinterpret_cast<const float*>(ring + (size_t)w * stages * L.stage) + m * Es + e);
      float4 a = p[0];
#pragma unroll
      for (int w = 1; w < kRcWarps; ++w) {
        a.x += p[w].x;
        a.y += p[w].y;
        a.z += p[w].z;
        a.w += p[w].w;
      }
      sum.x += a.x;
      sum.y += a.y;
      sum.z += a.z;
      sum.w += a.w;
      const uint32_t owner = (uint32_t)(m % C);
      st_async_f32x4(dsmem_addr(all_lg + (size_t)(m / C) * E + ge, owner), sum,
                     dsmem_addr(&xch, owner));
    }
  }
  if (tid == 0) MOE_TL_MIN(21);
  const int own = (M > (int)rank) ? (M - 1 - (int)rank) / C + 1 : 0;
  if (own == 0) return;  // nothing writes to this CTA's shared memory
  // every expert's logit of this CTA's tokens is here
  if (!mbar_wait_cluster(&xch, 0, status)) return;
  if (tid == 0) MOE_TL_MAX(24);

  // ---- top-k, weights, gate and route stores of this CTA's tokens: one warp
  // per token over all E logits (largest first; ties: the lower expert id);
  // the expert ids go to CTA 0, which builds the plan ----
  const uint32_t ids0 = dsmem_addr(s_ids, 0), idbar = dsmem_addr(&idb, 0);
  for (int lm = warp; lm < own; lm += kRcWarps) {
    const int m = (int)rank + lm * C;
    int my_id = -1;
    float my_l = -INFINITY;
    warp_topk<false>(all_lg + (size_t)lm * E, E, k, &my_id, &my_l);
    if (tid == 0) MOE_TL_MAX(26);
    const float w = warp_topk_weight(my_l, k);
    const float gamma = d.shared ? warp_gate(x + (size_t)m * H, wg, H) : 0.f;
    store_route(d, m, my_id, w, gamma, ids_user, w_user, pv);
    if (tid == 0) MOE_TL_MAX(28);
    if (lane < k) {
      if (rank == 0)
        s_ids[m * d.k_eff + lane] = my_id;
      else
        st_async_s32(ids0 + 4u * (uint32_t)(m * d.k_eff + lane), my_id, idbar);
    }
  }
  if (rank != 0) return;
  // the other CTAs' tokens' ids; the shared expert's slot of every token
  if (M > own && !mbar_wait_cluster(&idb, 0, status)) return;
  if (d.shared)
    for (int m = tid; m < M; m += kRcThreads) s_ids[m * d.k_eff + k] = d.E;
  __syncthreads();
  if (tid == 0) MOE_TL_MAX(30);
  // the plan's scratch takes the W_r ring, whose partial sums are all read
  plan_small_block(d, M, s_ids, pv, status, reinterpret_cast<PlanScratch*>(ring));
  if (tid == 0) MOE_TL_MIN(25);
}

// Largest cluster (16, else 8, else 0: the 128-block router is used) that each
// device can co-schedule with router_cluster_kernel at its largest
// shared-memory use; written by router_device_init before the device's first
// launch.
static int g_cluster_max[64];
// Diagnostic override (moe_nvfp4_set_small_router): route M <= 16 through the
// 128-block router even where a cluster could be scheduled.
static bool g_force_small_router = false;
void set_force_small_router(bool on) { g_force_small_router = on; }

static int router_cluster_probe() {
  if (cudaFuncSetAttribute(router_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           1) != cudaSuccess ||
      cudaFuncSetAttribute(router_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kRcSmemBudget) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  for (int cand : {16, 8}) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cand);
    cfg.blockDim = dim3(kRcThreads);
    cfg.dynamicSmemBytes = kRcSmemBudget;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cand;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, router_cluster_kernel, &cfg) == cudaSuccess && n >= 1)
      return cand;
    cudaGetLastError();
  }
  return 0;
}

cudaError_t router_device_init(int dev) {
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t e = cudaFuncSetAttribute(router_logits_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRlSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(router_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)router_mma_smem(512));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(plan_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)(sizeof(uint16_t) * 32 * kMaxEEff));
  if (e != cudaSuccess) return e;
  g_cluster_max[dev] = router_cluster_probe();
  return cudaSuccess;
}

// ---------------------------------------------------------------------------
cudaError_t launch_plan(const LayerDims& d, int64_t M, const __half* x, const __half* w_router,
                        const float* bias, const __half* w_gate, int32_t* ids_user,
                        float* w_user, bool ids_given, const PlanView& pv, uint32_t* status,
                        cudaStream_t stream, int num_sms) {
  (void)num_sms;
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  const int Mi = (int)M;
  if (M <= kDecodeMaxTokens) {
    if (ids_given) {
      route_given_kernel<<<(Mi + 7) / 8, 256, 0, stream>>>(d, Mi, x, w_gate, ids_user, w_user, pv);
      plan_small_kernel<<<1, 256, 0, stream>>>(d, Mi, pv, status);
    } else {
      const int cmax =
          (dev >= 0 && dev < 64 && !g_force_small_router) ? g_cluster_max[dev] : 0;
      const RouterClusterPlan L = router_cluster_plan(d.H, d.E, d.k, Mi, cmax > 0 ? cmax : 1);
      if (cmax > 0 && L.stages >= 1 && L.total <= kRcSmemBudget) {
        CUtensorMap wrmap;
        cudaError_t e = make_fp16_map_swz(&wrmap, w_router, (uint64_t)d.E, (uint64_t)d.H,
                                          (uint32_t)L.Es, (uint32_t)L.tr, L.Es * 2);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(L.C);
        cfg.blockDim = dim3(kRcThreads);
        cfg.dynamicSmemBytes = L.total;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = L.C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = trace_on() ? 1 : 2;
        return cudaLaunchKernelEx(&cfg, router_cluster_kernel, d, Mi, x, wrmap, bias, w_gate,
                                  ids_user, w_user, pv, status, cmax);
      }
      dim3 grid((d.E + 63) / 64, d.H / kRsRows);
      router_small_kernel<<<grid, 256, 0, stream>>>(d, Mi, x, w_router, bias, w_gate, ids_user,
                                                     w_user, pv, status);
    }
    return cudaGetLastError();
  }
  if (ids_given) {
    route_given_kernel<<<(Mi + 7) / 8, 256, 0, stream>>>(d, Mi, x, w_gate, ids_user, w_user, pv);
  } else if (router_tc_ok(d, M)) {
    cudaError_t e = launch_router_tc(d, M, x, w_router, bias, w_gate, ids_user, w_user, pv, status,
                                     stream);
    if (e != cudaSuccess) return e;
  } else {
    const size_t smem = router_mma_smem(d.E);
    const int ks = router_ksplit(M, d.H, d.E);
    const int nk = d.H / kRtK, spl = (nk + ks - 1) / ks;
    const int n_split = (nk + spl - 1) / spl;
    const dim3 grid((Mi + kRtTok - 1) / kRtTok, n_split);
    router_mma_kernel<<<grid, 512, smem, stream>>>(d, Mi, x, w_router, bias, w_gate, ids_user,
                                                   w_user, pv, spl,
                                                   n_split > 1 ? pv.rpart : nullptr);
    if (n_split > 1)
      router_split_topk_kernel<<<(Mi + 7) / 8, 256, sizeof(float) * 8 * d.E, stream>>>(
          d, Mi, n_split, pv.rpart, bias, x, w_gate, ids_user, w_user, pv);
  }
  const int64_t P = M * d.k_eff;
  const int n_chunks = (int)((P + kPlanChunk - 1) / kPlanChunk);
  const size_t hsmem = sizeof(uint16_t) * 32 * d.e_eff;
  plan_hist_kernel<<<n_chunks, 1024, hsmem, stream>>>(d, P, pv, status);
  plan_scan_kernel<<<1, 1024, 0, stream>>>(d, Mi, n_chunks, pv);
  plan_scatter_kernel<<<(unsigned)((P + 255) / 256), 256, 0, stream>>>(d, P, pv);
  return cudaGetLastError();
}

}  // namespace moe
