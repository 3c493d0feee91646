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

// Renormalised gates of T tokens from their picked logits (rank order):
// exp(l_j - l_0) / sum_j' exp(l_j' - l_0); a NaN pick gets 0; all NaN -> 1/k.
__device__ __forceinline__ void block_gates(const float *vals, int T, int k, float *gates) {
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
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
}

// The same gates for k <= 32: a warp per token, lane j holds pick j, one
// exponential per lane; the denominator is a butterfly sum, which leaves the
// identical value in every lane (a + b == b + a at every level).
__device__ __forceinline__ void warp_gates(const float *vals, int T, int k, float *gates) {
  const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int t = threadIdx.x >> 5; t < T; t += nw) {
    const float *vt = vals + t * k;
    const float l0 = vt[0];
    const float v = lane < k ? vt[lane] : __int_as_float(0x7FC00000);   // no term
    const float e = (v != v) ? 0.0f : expf(v - l0);
    float den = e;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, off);
    if (lane < k)
      gates[t * k + lane] = (l0 != l0) ? 1.0f / (float)k : ((v != v) ? 0.0f : e / den);
  }
}

// Order key of a logit: the float order mapped onto unsigned integers, NaN
// lowest and -0 folded into +0.  ranks_before(a, ia, b, ib) is exactly
// key(a) > key(b) || (key(a) == key(b) && ia < ib).
__device__ __forceinline__ uint32_t topk_key(float v) {
  v = v + 0.0f;
  const uint32_t b = __float_as_uint(v);
  return (v != v) ? 0u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
}

__device__ __forceinline__ int rank_step(uint32_t o, int j, uint32_t key, int e) {
  return (o > key) | ((o == key) & (j < e));
}

// Top-k of T tokens x E logits (shared memory): one thread per logit counts
// the logits of its token that rank before it (its rank) and, if the rank is
// below k, writes itself to that slot; no atomics, results independent of
// scheduling.  s_key: T*E 32-bit words of scratch (16-byte aligned).  Returns
// true (on every thread) if any logit is NaN.
__device__ __forceinline__ bool rank_topk(const float *lg, int T, int E, int k, int *idx,
                                          float *gates, float *vals, uint32_t *s_key,
                                          int *s_flag) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int TE = T * E;
  if (tid == 0) *s_flag = 0;
  __syncthreads();
  for (int i = tid; i < TE; i += nthr) {
    const float v = lg[i];
    s_key[i] = topk_key(v);
    if (v != v) *s_flag = 1;
  }
  __syncthreads();
  const bool vec = (E & 3) == 0 && ((uintptr_t)s_key & 15) == 0;
  for (int i = tid; i < TE; i += nthr) {
    const int t = i / E, e = i - t * E;
    const uint32_t key = s_key[i];
    const uint32_t *row = s_key + (size_t)t * E;
    int r = 0, j = 0;
    if (vec) {
      const uint4 *row4 = (const uint4 *)row;
      for (; j + 16 <= E; j += 16) {
        uint4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) q[u] = row4[j / 4 + u];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jj = j + 4 * u;
          r += rank_step(q[u].x, jj, key, e) + rank_step(q[u].y, jj + 1, key, e) +
               rank_step(q[u].z, jj + 2, key, e) + rank_step(q[u].w, jj + 3, key, e);
        }
      }
    }
    for (; j < E; ++j) r += rank_step(row[j], j, key, e);
    if (r < k) {
      idx[t * k + r] = e;
      vals[t * k + r] = lg[i];
    }
  }
  __syncthreads();
  block_gates(vals, T, k, gates);
  const bool nan = *(volatile int *)s_flag != 0;
  __syncthreads();
  return nan;
}

// Top-k of one token's E logits by one warp: k rounds of a warp arg-max under
// ranks_before (a total order), each lane scanning its elements e = lane + 32 i
// (E <= 1024) and skipping the ones already taken.  Lane 0 writes idx / vals in
// rank order.  Returns true on every lane if any logit is NaN.
__device__ __forceinline__ bool warp_topk_row(const float *lg, int E, int k, int *idx,
                                              float *vals) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;
  bool nan = false;
  for (int e = lane; e < E; e += 32) nan |= lg[e] != lg[e];
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = -1;
    for (int i = 0, e = lane; e < E; ++i, e += 32) {
      if ((taken >> i) & 1u) continue;
      const float v = lg[e];
      if (bi < 0 || ranks_before(v, e, bv, bi)) {
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (oi >= 0 && (bi < 0 || ranks_before(ov, oi, bv, bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      idx[j] = bi;
      vals[j] = bv;
    }
  }
  return __any_sync(0xFFFFFFFFu, nan) != 0;
}

// Top-k of T tokens by the block's warps (one token per warp at a time), then
// the gates.  Same results as block_topk.  s_flag: one int of scratch.
__device__ __forceinline__ bool warp_topk(const float *lg, int T, int E, int k, int *idx,
                                          float *gates, float *vals, int *s_flag) {
  const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) *s_flag = 0;
  __syncthreads();
  for (int t = warp; t < T; t += nw)
    if (warp_topk_row(lg + (size_t)t * E, E, k, idx + t * k, vals + t * k) &&
        (threadIdx.x & 31) == 0)
      *s_flag = 1;
  __syncthreads();
  block_gates(vals, T, k, gates);
  const bool nan = *(volatile int *)s_flag != 0;
  __syncthreads();
  return nan;
}

// Top-k by a tournament (k <= 32): each warp sorts a 32-logit chunk of one
// token with a shuffle bitonic network on 64-bit keys (order key, then the
// complement of the expert id, so keys are distinct and larger ranks first;
// padding is 0, below every logit) and keeps its k best; one thread per
// candidate then counts the token's larger candidates (a quad of lanes per
// candidate, each over every fourth entry).  s_cand: T * ceil(E/32) * k 64-bit
// words.  Returns true (on every thread) if any logit is NaN.
__device__ __forceinline__ bool tournament_topk(const float *lg, int T, int E, int k, int *idx,
                                                float *gates, float *vals,
                                                unsigned long long *s_cand, int *s_flag) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int nch = (E + 31) >> 5, C = nch * k;
  if (tid == 0) *s_flag = 0;
  __syncthreads();
  for (int task = warp; task < T * nch; task += nw) {
    const int t = task / nch, ch = task - t * nch, e = 32 * ch + lane;
    unsigned long long key = 0ull;
    if (e < E) {
      const float v = lg[(size_t)t * E + e];
      if (v != v) *s_flag = 1;
      key = ((unsigned long long)topk_key(v) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
    }
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, key, stride);
        const bool desc = (lane & size) == 0, first = (lane & stride) == 0;
        const unsigned long long mx = key > o ? key : o, mn = key > o ? o : key;
        key = (first == desc) ? mx : mn;
      }
    if (lane < k) s_cand[(size_t)t * C + ch * k + lane] = key;
  }
  __syncthreads();
  // blockDim is a multiple of 32, so a quad's four lanes share i in every
  // iteration and leave the loop together
  const unsigned qmask = 0xFu << (lane & 28);
  for (int i4 = tid; i4 < 4 * T * C; i4 += blockDim.x) {
    const int i = i4 >> 2, q = i4 & 3;
    const int t = i / C;
    const unsigned long long c = s_cand[i];
    const unsigned long long *row = s_cand + (size_t)t * C;
    int r = 0;
    for (int j = q; j < C; j += 4) r += row[j] > c;
    r += __shfl_xor_sync(qmask, r, 1);
    r += __shfl_xor_sync(qmask, r, 2);
    if (q == 0 && c != 0ull && r < k) {    // c == 0: padding of a short chunk
      const int e = (int)(0xFFFFFFFFu - (uint32_t)c);
      idx[t * k + r] = e;
      vals[t * k + r] = lg[(size_t)t * E + e];
    }
  }
  __syncthreads();
  warp_gates(vals, T, k, gates);
  const bool nan = *(volatile int *)s_flag != 0;
  __syncthreads();
  return nan;
}

// Scratch bytes select_topk needs (16-byte aligned start).
__host__ __device__ constexpr size_t topk_scratch_bytes(int T, int E, int k) {
  return ((size_t)T * E * 4 > (size_t)T * ((E + 31) / 32) * k * 8 ? (size_t)T * E * 4
                                                                   : (size_t)T * ((E + 31) / 32) * k * 8);
}

// The block's top-k by the faster method for the size: the tournament for
// k <= 32, else rank counting for up to 1024 logits, else a warp per token.
__device__ __forceinline__ bool select_topk(const float *lg, int T, int E, int k, int *idx,
                                            float *gates, float *vals, void *scratch,
                                            int *s_flag) {
  if (k <= 32)
    return tournament_topk(lg, T, E, k, idx, gates, vals, (unsigned long long *)scratch, s_flag);
  if (T * E <= 1024) return rank_topk(lg, T, E, k, idx, gates, vals, (uint32_t *)scratch, s_flag);
  return warp_topk(lg, T, E, k, idx, gates, vals, s_flag);
}

// Routing by sigmoid scores with a selection-only bias (the GLM layers'
// n_group = 1 sigmoid + noaux_tc router; with one group the group-limited
// step keeps every expert): s = 1 / (1 + e^-l); experts are ranked by
// s + bias[e] under the select_topk rules; gates = the picked s over their
// sum (a picked NaN gets 0; an all-NaN token gets 1/k).  Used around one
// select_topk call, so the top-k code is not duplicated:
//   sigmoid_keys   lg [T][E] logits -> s (in place), sel [T][E] = s + bias
//   select_topk    on sel
//   sigmoid_gates  gates of the picked experts from s
// bias: E floats (global or shared memory), or null (zero).
__device__ __forceinline__ void sigmoid_keys(float *lg, float *sel, const float *bias, int T,
                                             int E) {
  for (int i = threadIdx.x; i < T * E; i += blockDim.x) {
    const float sc = 1.0f / (1.0f + expf(-lg[i]));
    lg[i] = sc;
    sel[i] = sc + (bias ? bias[i % E] : 0.0f);
  }
  __syncthreads();
}

static __device__ __noinline__ void sigmoid_gates(const float *s, const int *idx, int T, int E, int k,
                                           float *gates) {
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int t = i / k;
    const int *it = idx + t * k;
    const float s0 = s[(size_t)t * E + it[0]];
    float g;
    if (s0 != s0) {
      g = 1.0f / (float)k;
    } else {
      float den = 0.0f;
      for (int j = 0; j < k; ++j) {
        const float sj = s[(size_t)t * E + it[j]];
        den += (sj != sj) ? 0.0f : sj;
      }
      const float si = s[(size_t)t * E + idx[i]];
      g = (si != si) ? 0.0f : si / den;
    }
    gates[i] = g;
  }
  __syncthreads();
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
  if (tid < 32) {
    // group starts in sorted order, 32 positions per step (warp ballot)
    int na = 0;
    for (int p0 = 0; p0 < n; p0 += 32) {
      const int p = p0 + tid;
      const bool first = p < n && (p == 0 || s_sorted_e[p] != s_sorted_e[p - 1]);
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, first);
      if (first) {
        const int gi = na + __popc(m & ((1u << tid) - 1u));
        act_expert[gi] = s_sorted_e[p];
        act_off[gi] = p;
      }
      na += __popc(m);
    }
    for (int s = tid; s < S; s += 32) {
      act_expert[na + s] = E + s;
      act_off[na + s] = n + s * T;
    }
    if (tid == 0) {
      act_off[na + S] = n + S * T;
      act[0] = na + S;
    }
  }
  __syncthreads();
  return act[0];
}

}  // namespace coli
