// Router GEMV, top-k selection with renormalised softmax gates, route counts
// and the batch union of the selected experts.
//
// Pages: "Colibrì 深度解析" §十一 (route -> union: each expert the batch uses is
// read once); "colibrì 路由遥测全解析" §追踪流 (gates are the normalised values the
// layer applies), §从新引擎接入 (one count per routing decision), §测试与 CI
// (rt_router_pick: an all-NaN score row falls back to slot index).
//
// One launch: warps compute logits[t][e] (one warp per expert row and token
// tile, f32 accumulation); the last block to finish (atomic ticket) runs the
// warp-shuffle top-k of every token, the counts, and builds the union lists the
// expert kernels consume.
#include <float.h>

#include "coli_internal.cuh"

namespace coli {
namespace {

constexpr int kRouterThreads = 256;
constexpr int kTokTile = 8;

template <typename T>
__device__ __forceinline__ void load8(const T *p, float v[8]);

template <>
__device__ __forceinline__ void load8<float>(const float *p, float v[8]) {
  const float4 a = __ldg((const float4 *)p);
  const float4 b = __ldg((const float4 *)p + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float v[8]) {
  const uint4 q = __ldg((const uint4 *)p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Ranking: a before b?  Numbers before NaN, larger first, equal -> lower id.
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib) {
  const bool na = a != a, nb = b != b;
  if (na != nb) return nb;
  if (!na && a != b) return a > b;
  return ia < ib;
}

struct RouterArgs {
  const void *x;
  const void *wr;
  int T, H, E, S, k;
  uint8_t *ws;
  WsLayout L;
  int32_t *idx_out;
  float *gates_out;
  uint32_t *counts;
  int build_union;
};

// Top-k of one token by one warp.  EPL = logits held per lane (E <= 32*EPL).
template <int EPL>
__device__ void warp_topk(const float *lg, int E, int k, int32_t *idx, float *gates,
                          uint32_t *counts, uint32_t *flags) {
  const int lane = threadIdx.x & 31;
  float v[EPL];
  bool any_nan = false;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldcg(lg + e) : 0.0f;
    if (e < E && v[i] != v[i]) any_nan = true;
  }
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i >= E) taken |= 1u << i;
  float sel_v = 0.0f;   // lane j keeps the j-th pick
  int sel_i = 0;
  for (int j = 0; j < k; ++j) {
    float bv = 0.0f;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (taken & (1u << i)) continue;
      const int e = lane + 32 * i;
      if (bi == 0x7FFFFFFF || ranks_before(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (oi != 0x7FFFFFFF && (bi == 0x7FFFFFFF || ranks_before(ov, oi, bv, bi))) {
        bv = ov; bi = oi;
      }
    }
    // winner (same on every lane): mark taken by its owner lane
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j < 32 && lane == j) { sel_v = bv; sel_i = bi; }
    if (j >= 32) {  // more than 32 picks: park them in the output directly
      if (lane == 0) { idx[j] = bi; gates[j] = bv; }
    }
  }
  any_nan = __any_sync(0xFFFFFFFFu, any_nan);
  // gates: exp(l_j - l_0) / sum; NaN picks -> 0; all NaN -> 1/k, slot j -> expert j
  const float l0 = __shfl_sync(0xFFFFFFFFu, sel_v, 0);
  const bool all_nan = (l0 != l0);
  float num = 0.0f;
  if (lane < k && lane < 32) num = (sel_v != sel_v) ? 0.0f : expf(sel_v - l0);
  float extra = 0.0f;  // picks beyond 32 (k > 32), parked in gates[32..]
  if (lane == 0)
    for (int j = 32; j < k; ++j) {
      const float lj = gates[j];
      extra += (lj != lj) ? 0.0f : expf(lj - l0);
    }
  float den = num;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, off);
  den += __shfl_sync(0xFFFFFFFFu, extra, 0);
  if (lane < k) {
    idx[lane] = sel_i;
    gates[lane] = all_nan ? 1.0f / (float)k : num / den;
    if (counts) atomicAdd(counts + sel_i, 1u);
  }
  if (lane == 0) {
    for (int j = 32; j < k; ++j) {
      const float lj = gates[j];
      gates[j] = all_nan ? 1.0f / (float)k : ((lj != lj) ? 0.0f : expf(lj - l0) / den);
      if (counts) atomicAdd(counts + idx[j], 1u);
    }
    if (any_nan) atomicOr(flags, COLI_FLAG_NAN_LOGITS);
  }
}

// Union lists: routed experts in ascending id, each with its slots in token
// order; then the shared experts with every token.  Slot of (t, j) is
// t*(k+S) + j; shared expert s of token t is slot t*(k+S) + k + s.
__device__ void build_union(const RouterArgs &a, const int32_t *idx, const float *gates) {
  const int T = a.T, k = a.k, S = a.S, KS = a.k + a.S;
  const int n = T * k;
  int32_t *act = (int32_t *)(a.ws + a.L.act);
  int32_t *act_expert = act + 1;
  int32_t *act_off = act + 1 + (a.E + S);
  int32_t *routes = (int32_t *)(a.ws + a.L.routes);
  float *slot_gate = (float *)(a.ws + a.L.slot_gate);
  __shared__ int s_sorted[kDecodeMaxT * kMaxTopK];
  // rank sort of routes by (expert, route id); keys are distinct
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    const int er = idx[r];
    int rank = 0;
    for (int q = 0; q < n; ++q) {
      const int eq = idx[q];
      rank += (eq < er) || (eq == er && q < r);
    }
    s_sorted[rank] = r;
    const int t = r / k, j = r % k;
    slot_gate[t * KS + j] = gates[r];
  }
  for (int t = threadIdx.x; t < T; t += blockDim.x)
    for (int s = 0; s < S; ++s) slot_gate[t * KS + k + s] = 1.0f;
  __syncthreads();
  if (threadIdx.x == 0) {
    int na = 0, prev = -1;
    for (int p = 0; p < n; ++p) {
      const int r = s_sorted[p];
      const int e = idx[r];
      if (e != prev) { act_expert[na] = e; act_off[na] = p; ++na; prev = e; }
      routes[p] = (r / k) * KS + (r % k);
    }
    int pos = n;
    for (int s = 0; s < S; ++s) {
      act_expert[na] = a.E + s;
      act_off[na] = pos;
      ++na;
      for (int t = 0; t < T; ++t) routes[pos++] = t * KS + k + s;
    }
    act_off[na] = pos;
    act[0] = na;
  }
}

template <typename XT, typename WT, int EPL>
__global__ void __launch_bounds__(kRouterThreads) k_router(RouterArgs a) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nw = kRouterThreads / 32;
  const int T = a.T, H = a.H, E = a.E;
  const XT *x = (const XT *)a.x;
  const WT *wr = (const WT *)a.wr;
  float *logits = (float *)(a.ws + a.L.logits);
  uint32_t *ctrl = (uint32_t *)(a.ws + a.L.ctrl);
  const int n_tt = (T + kTokTile - 1) / kTokTile;
  const int n_items = E * n_tt;
  for (int item = blockIdx.x * nw + warp; item < n_items; item += gridDim.x * nw) {
    const int e = item % E, t0 = (item / E) * kTokTile;
    float acc[kTokTile];
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) acc[t] = 0.0f;
    for (int h = lane * 8; h < H; h += 256) {
      float w8[8];
      load8<WT>(wr + (size_t)e * H + h, w8);
#pragma unroll
      for (int t = 0; t < kTokTile; ++t) {
        if (t0 + t < T) {
          float x8[8];
          load8<XT>(x + (size_t)(t0 + t) * H + h, x8);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[t] = fmaf(w8[i], x8[i], acc[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) {
      float v = acc[t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (lane == 0 && t0 + t < T) logits[(size_t)(t0 + t) * E + e] = v;
    }
  }
  // last block: top-k + union
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned ticket = atomicAdd(ctrl + kCtrlRouterTicket, 1u);
    s_last = (ticket == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  int32_t *idx = (int32_t *)(a.ws + a.L.idx);
  float *gates = (float *)(a.ws + a.L.gates);
  for (int t = warp; t < T; t += nw)
    warp_topk<EPL>(logits + (size_t)t * E, E, a.k, idx + (size_t)t * a.k,
                   gates + (size_t)t * a.k, a.counts, ctrl + kCtrlFlags);
  __syncthreads();
  if (a.idx_out || a.gates_out)
    for (int i = threadIdx.x; i < T * a.k; i += blockDim.x) {
      if (a.idx_out) a.idx_out[i] = idx[i];
      if (a.gates_out) a.gates_out[i] = gates[i];
    }
  if (a.build_union) build_union(a, idx, gates);
  if (threadIdx.x == 0) ctrl[kCtrlRouterTicket] = 0;
}

template <typename XT, typename WT>
cudaError_t launch_epl(const RouterArgs &a, int blocks, cudaStream_t s) {
  const int epl = (a.E + 31) / 32;
  if (epl <= 1) k_router<XT, WT, 1><<<blocks, kRouterThreads, 0, s>>>(a);
  else if (epl <= 2) k_router<XT, WT, 2><<<blocks, kRouterThreads, 0, s>>>(a);
  else if (epl <= 4) k_router<XT, WT, 4><<<blocks, kRouterThreads, 0, s>>>(a);
  else if (epl <= 8) k_router<XT, WT, 8><<<blocks, kRouterThreads, 0, s>>>(a);
  else if (epl <= 16) k_router<XT, WT, 16><<<blocks, kRouterThreads, 0, s>>>(a);
  else k_router<XT, WT, 32><<<blocks, kRouterThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_topk(const void *x, int x_dtype, const void *wr, int w_dtype,
                               int T, int H, int E, int S, int k, uint8_t *ws,
                               const WsLayout &L, int32_t *idx_out, float *gates_out,
                               uint32_t *counts, bool build_union_lists, cudaStream_t s) {
  RouterArgs a{x, wr, T, H, E, S, k, ws, L, idx_out, gates_out, counts,
               build_union_lists ? 1 : 0};
  const int nw = kRouterThreads / 32;
  const int n_items = E * ((T + kTokTile - 1) / kTokTile);
  int blocks = (n_items + nw - 1) / nw;
  const int cap = num_sms() * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (x_dtype == COLI_F32 && w_dtype == COLI_F32) return launch_epl<float, float>(a, blocks, s);
  if (x_dtype == COLI_F32 && w_dtype == COLI_BF16)
    return launch_epl<float, __nv_bfloat16>(a, blocks, s);
  if (x_dtype == COLI_BF16 && w_dtype == COLI_F32)
    return launch_epl<__nv_bfloat16, float>(a, blocks, s);
  return launch_epl<__nv_bfloat16, __nv_bfloat16>(a, blocks, s);
}

}  // namespace coli
