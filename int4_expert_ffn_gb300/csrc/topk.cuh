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

// Block-parallel top-k of T tokens x E logits (shared memory), every thread of
// the block taking part.  The rank of logit (t, e) is the number of logits of
// token t that rank before it; the work is split into chunks whose counts are
// added with shared-memory integer atomics, so the result does not depend on
// scheduling.  s_rank: T*E ints of scratch.  Writes idx/gates [T][k]; returns
// true (on every thread) if any logit is NaN.
__device__ __forceinline__ bool block_topk(const float *lg, int T, int E, int k, int *idx,
                                           float *gates, float *vals, int *s_rank, int *s_flag) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int TE = T * E;
  int P = (nthr * 8) / TE;
  if (P < 1) P = 1;
  if (P > E / 8) P = E / 8 > 0 ? E / 8 : 1;
  for (int i = tid; i < TE; i += nthr) s_rank[i] = 0;
  if (tid == 0) *s_flag = 0;
  __syncthreads();
  const int chunk = (E + P - 1) / P;
  for (int i = tid; i < TE * P; i += nthr) {
    const int item = i / P, part = i - item * P;
    const int t = item / E, e = item - t * E;
    const float *lt = lg + t * E;
    const float v = lt[e];
    const int e0 = part * chunk, e1 = e0 + chunk < E ? e0 + chunk : E;
    int r = 0;
    for (int e2 = e0; e2 < e1; ++e2) r += ranks_before(lt[e2], e2, v, e);
    if (r) atomicAdd(s_rank + item, r);
    if (part == 0 && v != v) *s_flag = 1;
  }
  __syncthreads();
  for (int i = tid; i < TE; i += nthr) {
    const int r = s_rank[i];
    if (r < k) {
      const int t = i / E;
      idx[t * k + r] = i - t * E;
      vals[t * k + r] = lg[i];
    }
  }
  __syncthreads();
  // gates = exp(l_j - l_0) / sum_j' exp(l_j' - l_0); NaN picks 0; all NaN -> 1/k
  for (int i = tid; i < T * k; i += nthr) {
    const int t = i / k;
    const float *vt = vals + t * k;
    const float l0 = vt[0];
    float g;
    if (l0 != l0) {
      g = 1.0f / (float)k;
    } else {
      float den = 0.0f;
      for (int j = 0; j < k; ++j) den += (vt[j] != vt[j]) ? 0.0f : expf(vt[j] - l0);
      const float lj = vt[i - t * k];
      g = (lj != lj) ? 0.0f : expf(lj - l0) / den;
    }
    gates[i] = g;
  }
  const bool nan = *(volatile int *)s_flag != 0;
  __syncthreads();
  return nan;
}

// Block-parallel union lists (see warp_union for the layout).  s_sorted: T*k
// ints of scratch.  Returns the number of used experts (routed + shared).
__device__ __forceinline__ int block_union(const int *idx, const float *gates, int T, int k, int S,
                                           int E, int *act, int *act_expert, int *act_off,
                                           int *routes, float *slot_gate, int *s_sorted_e) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int KS = k + S;
  const int n = T * k;
  for (int r = tid; r < n; r += nthr) {
    const int er = idx[r];
    int rank = 0;
    for (int q = 0; q < n; ++q) {
      const int eq = idx[q];
      rank += (eq < er) || (eq == er && q < r);
    }
    const int t = r / k, j = r - t * k;
    routes[rank] = t * KS + j;
    s_sorted_e[rank] = er;
    slot_gate[t * KS + j] = gates[r];
  }
  for (int i = tid; i < T * S; i += nthr) {
    const int s = i / T, t = i - s * T;
    slot_gate[t * KS + k + s] = 1.0f;
    routes[n + s * T + t] = t * KS + k + s;
  }
  __syncthreads();
  if (tid == 0) {
    int na = 0;
    for (int p = 0; p < n; ++p)
      if (p == 0 || s_sorted_e[p] != s_sorted_e[p - 1]) {
        act_expert[na] = s_sorted_e[p];
        act_off[na] = p;
        ++na;
      }
    for (int s = 0; s < S; ++s) {
      act_expert[na + s] = E + s;
      act_off[na + s] = n + s * T;
    }
    act_off[na + S] = n + S * T;
    act[0] = na + S;
  }
  __syncthreads();
  return act[0];
}

}  // namespace coli
