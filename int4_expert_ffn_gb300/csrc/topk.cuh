// Top-k with renormalised softmax gates and the batch-union lists.
//
// Pages: "colibrì 路由遥测全解析" §追踪流 (gates are the normalised values the layer
// applies), §从新引擎接入 (one count per routing decision), §测试与 CI
// (rt_router_pick: an all-NaN score row falls back to the slot index);
// "Colibrì 深度解析" §四 / §十一 (batch union: each used expert read once).
#pragma once

#include "coli_internal.cuh"

namespace coli {

// a ranks before b?  Numbers before NaN, larger first, equal -> lower id.
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib) {
  const bool na = a != a, nb = b != b;
  if (na != nb) return nb;
  if (!na && a != b) return a > b;
  return ia < ib;
}

// Top-k of one token's E logits (any memory space) by one warp.
// Writes idx[0..k) (descending) and gates[0..k); returns true if a logit is NaN.
// `park` is k floats of scratch used when k > 32.
__device__ __noinline__ bool warp_topk(const float *lg, int E, int k, int *idx, float *gates,
                                       float *park) {
  const int lane = threadIdx.x & 31;
  bool any_nan = false;
  float sel_v = 0.0f;
  int sel_i = 0;
  // taken flags: bit i of the lane's mask is its entry e = lane + 32 i (E <= 1024)
  uint32_t taken = 0;
  for (int e = lane; e < E; e += 32)
    if (lg[e] != lg[e]) any_nan = true;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = 0x7FFFFFFF;
    for (int e = lane, i = 0; e < E; e += 32, ++i) {
      if (taken & (1u << i)) continue;
      const float v = lg[e];
      if (bi == 0x7FFFFFFF || ranks_before(v, e, bv, bi)) { bv = v; bi = e; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (oi != 0x7FFFFFFF && (bi == 0x7FFFFFFF || ranks_before(ov, oi, bv, bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j < 32 && lane == j) { sel_v = bv; sel_i = bi; }
    if (j >= 32 && lane == 0) { idx[j] = bi; park[j] = bv; }
  }
  any_nan = __any_sync(0xFFFFFFFFu, any_nan);
  const float l0 = __shfl_sync(0xFFFFFFFFu, sel_v, 0);
  const bool all_nan = (l0 != l0);
  float num = 0.0f;
  if (lane < k) num = (sel_v != sel_v) ? 0.0f : expf(sel_v - l0);
  float extra = 0.0f;
  if (lane == 0)
    for (int j = 32; j < k; ++j) {
      const float lj = park[j];
      extra += (lj != lj) ? 0.0f : expf(lj - l0);
    }
  float den = num;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, off);
  den += __shfl_sync(0xFFFFFFFFu, extra, 0);
  if (lane < k) {
    idx[lane] = sel_i;
    gates[lane] = all_nan ? 1.0f / (float)k : num / den;
  }
  if (lane == 0)
    for (int j = 32; j < k; ++j) {
      const float lj = park[j];
      gates[j] = all_nan ? 1.0f / (float)k : ((lj != lj) ? 0.0f : expf(lj - l0) / den);
    }
  __syncwarp();
  return any_nan;
}

// Union lists (one warp): routed experts in ascending id, each with its slots
// in token order, then the S shared experts with every token.  Slot of (t, j)
// is t*(k+S) + j; shared expert s of token t is slot t*(k+S) + k + s.
//   act_expert[na], act_off[na+1], routes[T*(k+S)], slot_gate[T*(k+S)]; returns na.
__device__ __noinline__ int warp_union(const int *idx, const float *gates, int T, int k, int S,
                                       int E, int *act_expert, int *act_off, int *routes,
                                       float *slot_gate) {
  const int lane = threadIdx.x & 31;
  const int KS = k + S;
  const int n = T * k;
  // rank of each route by (expert, route id): routes[rank] = slot
  for (int r = lane; r < n; r += 32) {
    const int er = idx[r];
    int rank = 0;
    for (int q = 0; q < n; ++q) {
      const int eq = idx[q];
      rank += (eq < er) || (eq == er && q < r);
    }
    const int t = r / k, j = r - t * k;
    routes[rank] = t * KS + j;
    slot_gate[t * KS + j] = gates[r];
  }
  for (int t = lane; t < T; t += 32)
    for (int s = 0; s < S; ++s) {
      slot_gate[t * KS + k + s] = 1.0f;
      routes[n + s * T + t] = t * KS + k + s;
    }
  __syncwarp();
  // expert boundaries in the sorted order
  int na = 0;
  for (int p0 = 0; p0 < n; p0 += 32) {
    const int p = p0 + lane;
    bool start = false;
    int e = -1;
    if (p < n) {
      const int slot = routes[p];
      e = idx[(slot / KS) * k + slot % KS];
      if (p == 0) start = true;
      else {
        const int ps = routes[p - 1];
        start = idx[(ps / KS) * k + ps % KS] != e;
      }
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, start);
    if (start) {
      const int pos = na + __popc(m & ((1u << lane) - 1));
      act_expert[pos] = e;
      act_off[pos] = p;
    }
    na += __popc(m);
  }
  if (lane == 0) {
    for (int s = 0; s < S; ++s) {
      act_expert[na + s] = E + s;
      act_off[na + s] = n + s * T;
    }
    act_off[na + S] = n + S * T;
  }
  __syncwarp();
  return na + S;
}

}  // namespace coli
