// Decode path of the routed-MoE layer over int4-grouped experts (T <= 16 tokens).
//
// Pages: "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战" (matmul_i4_grouped
// consumes packed rows: W = s (u - 8); expert_ffn.h's dot(u,x) - 8 sum(x) with
// unsigned nibbles against signed 8-bit activations), "Colibrì 深度解析" §四 (an
// expert's three matrices adjacent; batch union reads each used expert once),
// §十一 (route -> union -> compute), "colibrì 路由遥测全解析" (route counts, gates).
//
// Per layer two kernels, chained with programmatic dependent launch:
//   k_gateup: every CTA reduces the router partial logits (fixed order), runs
//     the top-k and builds the union lists itself; CTA 0 publishes them and
//     the route counts.  The CTA then streams its share of the used experts'
//     gate/up rows through a bulk-copy (TMA) ring in shared memory, forms
//     h = silu(g) * u * gate, and prefetches into L2 the down rows that the
//     same-index CTA of k_down will read.
//   k_down: each CTA owns a block of output rows; it streams those rows of
//     every used expert's down matrix, sums the experts in ascending id order,
//     adds the residual, and forms the next layer's router partial logits
//     from its rows (the router GEMV split by rows).
// k_route forms the partial logits of the first layer.
//
// Arithmetic: each lane owns 32 consecutive columns.  Its 32 activations are
// quantised to 15-bit fixed point (scale = max|x| / 16319), split into signed
// 8-bit high and low planes (xq = 128 xh + xl), and dotted with the unsigned
// nibbles by dp4a; the exact integer sum sum_i (u_i - 8) xq_i is scaled by the
// group scale and the activation scale.  Activation rounding is at most
// max|x| / 32638 per element; all accumulation is exact or f32.
#include <mutex>
#include <unordered_map>

#include "coli_internal.cuh"
#include "ptx.cuh"
#include "topk.cuh"
#include "trace.cuh"

namespace coli {

namespace {

constexpr int kQ = 16319;
constexpr int kChunkCols = 1024;  // columns per warp pass (32 lanes x 32)

struct Planes {
  uint32_t eh[4], el[4], oh[4], ol[4];
  int sq;
  float sx;
};

__device__ __forceinline__ void quantize32(const float (&v)[32], Planes &p) {
  float m = 0.0f;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    m = fmaxf(m, fabsf(v[i]));
    bad |= (v[i] != v[i]);
  }
  const float inv = m > 0.0f ? (float)kQ / m : 0.0f;
  p.sx = bad ? __int_as_float(0x7FC00000) : m / (float)kQ;
  int sq = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t eh = 0, el = 0, oh = 0, ol = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int qe = (int)fminf(fmaxf(rintf(v[8 * i + 2 * b] * inv), -(float)kQ), (float)kQ);
      const int qo = (int)fminf(fmaxf(rintf(v[8 * i + 2 * b + 1] * inv), -(float)kQ), (float)kQ);
      const int he = (qe + 64) >> 7, ho = (qo + 64) >> 7;
      const int le = qe - (he << 7), lo = qo - (ho << 7);
      eh |= (uint32_t)(he & 0xFF) << (8 * b);
      el |= (uint32_t)(le & 0xFF) << (8 * b);
      oh |= (uint32_t)(ho & 0xFF) << (8 * b);
      ol |= (uint32_t)(lo & 0xFF) << (8 * b);
      sq += qe + qo;
    }
    p.eh[i] = eh; p.el[i] = el; p.oh[i] = oh; p.ol[i] = ol;
  }
  p.sq = sq;
}

// sum over the 32 columns of (u - 8) * x, for 16 packed bytes w.
__device__ __forceinline__ float dot32(const uint4 w, const Planes &p) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  int aeh = 0, ael = 0, aoh = 0, aol = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = ws[i] & 0x0F0F0F0Fu;   // even columns: u
    const uint32_t hi = ws[i] & 0xF0F0F0F0u;   // odd columns: 16 u
    aeh = dp4a_us(lo, p.eh[i], aeh);
    ael = dp4a_us(lo, p.el[i], ael);
    aoh = dp4a_us(hi, p.oh[i], aoh);
    aol = dp4a_us(hi, p.ol[i], aol);
  }
  const int q = ((aeh + (aoh >> 4)) << 7) + ael + (aol >> 4) - 8 * p.sq;
  return (float)q * p.sx;
}

template <typename XT>
__device__ __forceinline__ void load32(const XT *p, float (&v)[32]);

template <>
__device__ __forceinline__ void load32<float>(const float *p, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 q = __ldcg((const float4 *)p + i);
    v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
  }
}

template <>
__device__ __forceinline__ void load32<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 q = __ldcg((const uint4 *)p + i);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ void load32_smem(const float *p, float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 q = ((const float4 *)p)[i];
    v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
  }
}

// Reduce 8 values across the warp in 9 shuffles; lane l ends with the total of
// value (l >> 2).
__device__ __forceinline__ float reduce8(float (&v)[8]) {
  const int lane = threadIdx.x & 31;
  float a[4];
  const bool b4 = lane & 16;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b4 ? v[i + 4] : v[i];
    const float give = b4 ? v[i] : v[i + 4];
    a[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 16);
  }
  float c[2];
  const bool b3 = lane & 8;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b3 ? a[i + 2] : a[i];
    const float give = b3 ? a[i] : a[i + 2];
    c[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 8);
  }
  const bool b2 = lane & 4;
  const float keep = b2 ? c[1] : c[0];
  const float give = b2 ? c[0] : c[1];
  float d = keep + __shfl_xor_sync(0xFFFFFFFFu, give, 4);
  d += __shfl_xor_sync(0xFFFFFFFFu, d, 2);
  d += __shfl_xor_sync(0xFFFFFFFFu, d, 1);
  return d;
}

// Quantise n_vec f32 vectors of length F (global, row-major [n_vec][F]) into
// activation planes in shared memory, transposed for conflict-free reads:
// word w (0..15 planes, 16 = sq, 17 = sx bits) of 32-column block b of vector v
// is at planes[(v * 18 + w) * nbp + b].  One warp handles 4 blocks at a time;
// lane q of a block's 8 lanes holds its columns 4q..4q+3.
__device__ void build_planes_impl(const float *src, int n_vec, int F, const int *list,
                                  uint32_t *planes, int nbp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int groups_per_vec = (F + 127) / 128;
  const int n_groups = n_vec * groups_per_vec;
  const int q = lane & 7;
  for (int g0 = warp; g0 < n_groups; g0 += 8 * nw) {
    // issue up to eight independent loads before using any of them
    float4 xs[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int g = g0 + u * nw;
      xs[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g < n_groups) {
        const int v = g / groups_per_vec, gc = g - v * groups_per_vec;
        const int col = gc * 128 + 4 * lane;
        const int64_t row = list ? list[v] : v;
        if (col < F) xs[u] = __ldcg((const float4 *)(src + row * F + col));
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
    const int g = g0 + u * nw;
    if (g >= n_groups) break;
    const int v = g / groups_per_vec, gc = g - v * groups_per_vec;
    const int col = gc * 128 + 4 * lane;
    const bool act = col < F;
    const float4 x = xs[u];
    float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
    bool bad = (x.x != x.x) | (x.y != x.y) | (x.z != x.z) | (x.w != x.w);
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
      bad |= __shfl_xor_sync(0xFFFFFFFFu, (int)bad, off) != 0;
    }
    const float inv = m > 0.0f ? (float)kQ / m : 0.0f;
    const float sx = bad ? __int_as_float(0x7FC00000) : m / (float)kQ;
    int qv[4];
    const float xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      qv[i] = (int)fminf(fmaxf(rintf(xv[i] * inv), -(float)kQ), (float)kQ);
    int hv[4], lv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      hv[i] = (qv[i] + 64) >> 7;
      lv[i] = qv[i] - (hv[i] << 7);
    }
    // 16-bit halves of the plane words: even columns are elements 0, 2; odd 1, 3
    const uint32_t eh = (uint32_t)(hv[0] & 0xFF) | ((uint32_t)(hv[2] & 0xFF) << 8);
    const uint32_t el = (uint32_t)(lv[0] & 0xFF) | ((uint32_t)(lv[2] & 0xFF) << 8);
    const uint32_t oh = (uint32_t)(hv[1] & 0xFF) | ((uint32_t)(hv[3] & 0xFF) << 8);
    const uint32_t ol = (uint32_t)(lv[1] & 0xFF) | ((uint32_t)(lv[3] & 0xFF) << 8);
    const uint32_t eh2 = __shfl_down_sync(0xFFFFFFFFu, eh, 1);
    const uint32_t el2 = __shfl_down_sync(0xFFFFFFFFu, el, 1);
    const uint32_t oh2 = __shfl_down_sync(0xFFFFFFFFu, oh, 1);
    const uint32_t ol2 = __shfl_down_sync(0xFFFFFFFFu, ol, 1);
    int sq = qv[0] + qv[1] + qv[2] + qv[3];
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) sq += __shfl_xor_sync(0xFFFFFFFFu, sq, off);
    const int b = (gc * 128 + 32 * (lane >> 3)) / 32;   // block index within the vector
    if (act && (q & 1) == 0) {
      const int i = q >> 1;
      uint32_t *pv = planes + (size_t)v * 18 * nbp + b;
      pv[(size_t)i * nbp] = eh | (eh2 << 16);
      pv[(size_t)(4 + i) * nbp] = el | (el2 << 16);
      pv[(size_t)(8 + i) * nbp] = oh | (oh2 << 16);
      pv[(size_t)(12 + i) * nbp] = ol | (ol2 << 16);
      if (q == 0) {
        pv[(size_t)16 * nbp] = (uint32_t)sq;
        pv[(size_t)17 * nbp] = __float_as_uint(sx);
      }
    }
    }
  }
}

// build_planes over a list of source rows: vector p is row list[p] of src.
__device__ void build_planes_list(const float *src, int F, const int *list, int n, uint32_t *planes,
                                  int nbp);

__device__ void build_planes(const float *src, int n_vec, int F, uint32_t *planes, int nbp) {
  build_planes_impl(src, n_vec, F, nullptr, planes, nbp);
}

__device__ void build_planes_list(const float *src, int F, const int *list, int n, uint32_t *planes,
                                  int nbp) {
  build_planes_impl(src, n, F, list, planes, nbp);
}

__device__ __forceinline__ void load_planes(const uint32_t *planes, int v, int b, int nbp,
                                            Planes &p) {
  const uint32_t *pv = planes + (size_t)v * 18 * nbp + b;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    p.eh[i] = pv[(size_t)i * nbp];
    p.el[i] = pv[(size_t)(4 + i) * nbp];
    p.oh[i] = pv[(size_t)(8 + i) * nbp];
    p.ol[i] = pv[(size_t)(12 + i) * nbp];
  }
  p.sq = (int)pv[(size_t)16 * nbp];
  p.sx = __uint_as_float(pv[(size_t)17 * nbp]);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ int part_lo(int c, int n, int parts) {
  return (int)(((long long)c * n) / parts);
}

__device__ __forceinline__ void set_flag(uint32_t *ctrl, uint32_t f) {
  atomicOr(ctrl + kCtrlFlags, f);
}

// The pointers that change from layer to layer (the rest of Dec2Args stays in
// kernel-parameter space).
struct LayerPtrs {
  const uint8_t *packed;
  const float *scales;
  uint32_t *route_counts;
  float *layer_out;
  const float *partials;
  float *out;
  float *xrep;
};

__device__ __forceinline__ LayerPtrs layer_ptrs(const Dec2Args &a) {
  LayerPtrs p;
  p.packed = a.packed;
  p.scales = a.scales;
  p.route_counts = a.route_counts;
  p.layer_out = a.layer_out;
  p.partials = a.partials;
  p.out = a.out;
  p.xrep = a.xrep;
  return p;
}


}  // namespace

// ---------------------------------------------------------------------------
// Router partial logits: CTA c of G sums its rows [h0, h1) of every expert's
// router row against x:  partials[c][t][e] = sum_{h in [h0,h1)} Wr[e][h] x[t][h].

template <typename XT, typename WT>
__global__ void __launch_bounds__(kDec2MaxThreads) k_route(Dec2Args a) {
  grid_dependents_launch();
  grid_dependency_wait();
  const int c = blockIdx.x, G = gridDim.x;
  const int U = a.H / 4;
  const int h0 = 4 * part_lo(c, U, G), h1 = 4 * part_lo(c + 1, U, G);
  const XT *x = (const XT *)a.x;
  const WT *wr = (const WT *)a.wr;
  for (int o = threadIdx.x; o < a.T * a.E; o += blockDim.x) {
    const int t = o / a.E, e = o - t * a.E;
    float s = 0.0f;
    for (int h = h0; h < h1; ++h)
      s = fmaf(to_f32(wr[(size_t)e * a.H + h]), to_f32(x[(size_t)t * a.H + h]), s);
    a.partials[(size_t)c * a.T * a.E + o] = s;
  }
  // the layer input, widened to f32, in every replica (read by all gate/up CTAs)
  if (a.xrep) {
    const int nr = h1 - h0;
    for (int i = threadIdx.x; i < a.T * nr; i += blockDim.x) {
      const int t = i / nr, h = h0 + (i - t * nr);
      const float v = to_f32(x[(size_t)t * a.H + h]);
      for (int r = 0; r < a.n_rep; ++r) a.xrep[r * a.x_stride + (size_t)t * a.H + h] = v;
    }
  }
  extern __shared__ __align__(128) uint8_t smem_route[];
  route_if_last(a, layer_ptrs(a), smem_route);
}

// ---------------------------------------------------------------------------
// Routing shared by k_gateup and k_topk: logits from the partials (fixed
// order), top-k per token by warps, NaN flag.

// Routing shared by k_gateup and k_topk: logits from this CTA's replica of the
// router partials (fixed summation order), block-parallel top-k, NaN flag and,
// if `publish`, the user-visible idx/gates and route counts.
__device__ void route_block(const Dec2Args &a, const LayerPtrs &lp, float *s_logits, int *s_idx,
                            float *s_gates, float *s_vals, int *s_rank, float *s_scratch,
                            float *s_stage, bool publish) {
  const int T = a.T, E = a.E, k = a.k;
  const int TE = T * E;
  const int nthr = blockDim.x;
  const float *src = lp.partials;
  if (s_stage) {
    // all threads copy the partials into shared memory, every load in flight at once
    const int n4 = (a.n_part * TE) / 4, tail = (a.n_part * TE) & 3;
    const float4 *s4 = (const float4 *)src;
    float4 *d4 = (float4 *)s_stage;
    for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * nthr) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * nthr < n4) v[u] = __ldcg(s4 + i0 + u * nthr);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u * nthr < n4) d4[i0 + u * nthr] = v[u];
    }
    if (threadIdx.x < tail) s_stage[4 * n4 + threadIdx.x] = __ldcg(src + 4 * n4 + threadIdx.x);
    __syncthreads();
    src = s_stage;
  }
  int nsplit = nthr / TE;
  if (nsplit > 8) nsplit = 8;
  if (nsplit <= 1) {
    for (int o = threadIdx.x; o < TE; o += nthr) {
      float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
      int p = 0;
      for (; p + 4 <= a.n_part; p += 4) {
        s0 += src[(size_t)p * TE + o];
        s1 += src[(size_t)(p + 1) * TE + o];
        s2 += src[(size_t)(p + 2) * TE + o];
        s3 += src[(size_t)(p + 3) * TE + o];
      }
      for (; p < a.n_part; ++p) s0 += src[(size_t)p * TE + o];
      s_logits[o] = (s0 + s1) + (s2 + s3);
    }
  } else {
    // nsplit * TE <= nthr: one partial sum per thread, combined in fixed order
    for (int i = threadIdx.x; i < TE * nsplit; i += nthr) {
      const int o = i % TE, part = i / TE;
      const int p0 = part_lo(part, a.n_part, nsplit), p1 = part_lo(part + 1, a.n_part, nsplit);
      float s0 = 0.0f, s1 = 0.0f;
      int p = p0;
      for (; p + 2 <= p1; p += 2) {
        s0 += src[(size_t)p * TE + o];
        s1 += src[(size_t)(p + 1) * TE + o];
      }
      if (p < p1) s0 += src[(size_t)p * TE + o];
      s_scratch[part * TE + o] = s0 + s1;
    }
    __syncthreads();
    for (int o = threadIdx.x; o < TE; o += nthr) {
      float s = 0.0f;
      for (int part = 0; part < nsplit; ++part) s += s_scratch[part * TE + o];
      s_logits[o] = s;
    }
  }
  __syncthreads();
  const bool nan = block_topk(s_logits, T, E, k, s_idx, s_gates, s_vals, s_rank,
                              (int *)s_scratch);
  if (publish) {
    if (threadIdx.x == 0 && nan) set_flag(a.ctrl, COLI_FLAG_NAN_LOGITS);
    for (int i = threadIdx.x; i < T * k; i += nthr) {
      a.g_idx[i] = s_idx[i];
      a.g_gates[i] = s_gates[i];
      if (lp.route_counts) atomicAdd(lp.route_counts + s_idx[i], 1u);
    }
  }
}

// Routing of one layer from its router partials, run by the last CTA of the
// kernel that produced them: logits (fixed summation order), top-k, gates,
// route counts, and the union lists the expert kernels read.  `smem` holds
// at least route_smem_bytes(a) bytes.
__device__ void route_finish(const Dec2Args &a, const LayerPtrs &lp, uint8_t *smem) {
  const int T = a.T, E = a.E, k = a.k, S = a.S, KS = k + S;
  float *s_stage = (float *)smem;
  float *s_logits = s_stage + (a.stage_partials ? (size_t)a.n_part * T * E : 0);
  int *s_rank = (int *)(s_logits + T * E);
  int *s_idx = s_rank + T * E;
  float *s_gates = (float *)(s_idx + T * k);
  float *s_vals = s_gates + T * k;
  float *s_scratch = s_vals + T * k;
  route_block(a, lp, s_logits, s_idx, s_gates, s_vals, s_rank, s_scratch,
              a.stage_partials ? s_stage : nullptr, true);
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    if (a.idx_out) a.idx_out[i] = s_idx[i];
    if (a.gates_out) a.gates_out[i] = s_gates[i];
  }
  if (a.build_union) {
    int *s_act = (int *)(s_scratch + kDec2MaxThreads);
    int *s_routes = s_act + 2 + 2 * (E + S);
    float *s_slot_gate = (float *)(s_routes + T * KS);
    block_union(s_idx, s_gates, T, k, S, E, s_act, s_act + 1, s_act + 1 + (E + S), s_routes,
                s_slot_gate, s_rank);
    for (int i = threadIdx.x; i < 2 + 2 * (E + S); i += blockDim.x) a.g_act[i] = s_act[i];
    for (int i = threadIdx.x; i < T * KS; i += blockDim.x) {
      a.g_routes[i] = s_routes[i];
      a.g_slot_gate[i] = s_slot_gate[i];
    }
  }
}

// Every CTA has written its partials: the last one to arrive (atomic ticket)
// routes the layer and resets the ticket for the next use.
__device__ void route_if_last(const Dec2Args &a, const LayerPtrs &lp, uint8_t *smem) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned t = atomicAdd(a.ctrl + kCtrlRouterTicket, 1u);
    s_last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  route_finish(a, lp, smem);
  if (threadIdx.x == 0) a.ctrl[kCtrlRouterTicket] = 0;
}

// ---------------------------------------------------------------------------
// gate/up phase: each compute warp owns one 1024-column chunk (cg) of every
// row congruent to rg modulo nrg within the CTA's row range, issues the loads
// of kGuBatch rows before computing any of them, and leaves per-row partial
// sums in shared memory; after one barrier the block finalises
// h = silu(g) * u * gate and writes it to every replica.  The union lists are
// already in shared memory.

constexpr int kGuBatch = 4;

__device__ void gu_phase(const Dec2Args &a, const LayerPtrs &lp, const int *s_act,
                         const int *s_routes, const float *s_slot_gate, float *red,
                         uint32_t *s_xpl) {
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int *s_act_expert = s_act + 1;
  const int *s_act_off = s_act + 1 + (E + S);
  const int n_active = s_act[0];
  const int G = gridDim.x, c = blockIdx.x;
  const int64_t rb = H / 2, ngr = H / kGroup;
  // L2 prefetch of the down rows that this CTA index will need in the down phase
  if (warp == 0 && c < a.n_part) {
    const int UH = H / 4;
    const int dh0 = 4 * part_lo(c, UH, a.n_part), dh1 = 4 * part_lo(c + 1, UH, a.n_part);
    for (int q = lane; q < n_active && dh1 > dh0; q += 32) {
      const int e = s_act_expert[q];
      prefetch_l2(lp.packed + (int64_t)e * a.eb + (int64_t)F * H + (int64_t)dh0 * (F / 2),
                  (uint32_t)((dh1 - dh0) * (F / 2)));
      prefetch_l2(lp.scales + (int64_t)e * a.es + (int64_t)2 * F * ngr + (int64_t)dh0 * (F / kGroup),
                  (uint32_t)((dh1 - dh0) * (F / 16)));
    }
  }
  // this CTA's rows in the flattened (used expert, row) space, units of 4 rows
  const int U = n_active * (F / 4);
  const int row0 = 4 * part_lo(c, U, G), nrows = 4 * part_lo(c + 1, U, G) - row0;
  const float *xr = lp.xrep + (size_t)(c % a.n_rep) * a.x_stride;
  const int nbx = H / 32;
  if (a.gu_xpl) {
    build_planes(xr, T, H, s_xpl, nbx);
    __syncthreads();
  }
  if (tid == 0) COLI_TRACE_POINT(0, 4);

  const int ncg = a.gu_ncg, nrg = a.gu_nrg;
  if (warp < ncg * nrg) {
    const int cg = warp % ncg, rg = warp / ncg;
    const int col = cg * kChunkCols + 32 * lane;
    const bool act = col < H;
    const int nq = nrows > rg ? (nrows - rg + nrg - 1) / nrg : 0;
    Planes pl;
    int pl_tok = -1;
    for (int q0 = 0; q0 < nq; q0 += kGuBatch) {
      uint4 wg[kGuBatch], wu[kGuBatch];
      float sg[kGuBatch], su[kGuBatch];
      int ra[kGuBatch];   // used-expert index of each row (-1: none)
#pragma unroll
      for (int b = 0; b < kGuBatch; ++b) {
        ra[b] = -1;
        const int q = q0 + b;
        if (q < nq) {
          const int gr = row0 + rg + q * nrg;
          const int ai = gr / F, f = gr - ai * F;
          ra[b] = ai;
          if (act) {
            const int e = s_act_expert[ai];
            const uint8_t *pg = lp.packed + (int64_t)e * a.eb + (int64_t)f * rb + col / 2;
            const float *pgs = lp.scales + (int64_t)e * a.es + (int64_t)f * ngr + col / kGroup;
            wg[b] = ldg_stream(pg);
            wu[b] = ldg_stream(pg + (int64_t)F * rb);
            sg[b] = __ldg(pgs);
            su[b] = __ldg(pgs + (int64_t)F * ngr);
          }
        }
      }
      if (q0 == 0 && tid == 0) COLI_TRACE_POINT(0, 5);
      int maxtok = 0;
#pragma unroll
      for (int b = 0; b < kGuBatch; ++b)
        if (ra[b] >= 0) {
          const int nt = s_act_off[ra[b] + 1] - s_act_off[ra[b]];
          maxtok = nt > maxtok ? nt : maxtok;
        }
      for (int j = 0; j < maxtok; ++j) {
        float v[8];
#pragma unroll
        for (int b = 0; b < kGuBatch; ++b) {
          v[2 * b] = 0.0f;
          v[2 * b + 1] = 0.0f;
          if (ra[b] >= 0) {
            const int j0 = s_act_off[ra[b]], nt = s_act_off[ra[b] + 1] - j0;
            if (j < nt && act) {
              const int t = s_routes[j0 + j] / KS;
              if (t != pl_tok) {
                if (a.gu_xpl) {
                  load_planes(s_xpl, t, col / 32, nbx, pl);
                } else {
                  float xv[32];
                  load32<float>(xr + (int64_t)t * H + col, xv);
                  quantize32(xv, pl);
                }
                pl_tok = t;
              }
              v[2 * b] = sg[b] * dot32(wg[b], pl);
              v[2 * b + 1] = su[b] * dot32(wu[b], pl);
            }
          }
        }
        const float tot = reduce8(v);
        if ((lane & 3) == 0) {
          const int vi = lane >> 2, b = vi >> 1;
          if (ra[b] >= 0) {
            const int nt = s_act_off[ra[b] + 1] - s_act_off[ra[b]];
            if (j < nt) {
              const int i = rg + (q0 + b) * nrg;
              red[((i * T + j) * ncg + cg) * 2 + (vi & 1)] = tot;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) COLI_TRACE_POINT(0, 6);
  // finalise h for every (row, token) of this CTA
  for (int it = tid; it < nrows * T; it += blockDim.x) {
    const int i = it / T, j = it - i * T;
    const int gr = row0 + i;
    const int ai = gr / F, f = gr - ai * F;
    const int j0 = s_act_off[ai], nt = s_act_off[ai + 1] - j0;
    if (j >= nt) continue;
    float g = 0.0f, u = 0.0f;
    for (int q = 0; q < ncg; ++q) {
      g += red[((i * T + j) * ncg + q) * 2];
      u += red[((i * T + j) * ncg + q) * 2 + 1];
    }
    const int slot_id = s_routes[j0 + j];
    const float hv = silu(g) * u * s_slot_gate[slot_id];
    for (int rr = 0; rr < a.n_rep; ++rr) a.h[rr * a.h_stride + (int64_t)slot_id * F + f] = hv;
  }
  if (tid == 0) COLI_TRACE_POINT(0, 7);
}

// Union lists published by the routing CTA, into shared memory.
__device__ void load_lists(const Dec2Args &a, int *s_act, int *s_routes, float *s_slot_gate) {
  const int KS = a.k + a.S;
  for (int i = threadIdx.x; i < 2 + 2 * (a.E + a.S); i += blockDim.x) s_act[i] = __ldcg(a.g_act + i);
  for (int i = threadIdx.x; i < a.T * KS; i += blockDim.x) {
    s_routes[i] = __ldcg(a.g_routes + i);
    if (s_slot_gate) s_slot_gate[i] = __ldcg(a.g_slot_gate + i);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDec2MaxThreads) k_gateup(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GuSmem &L = a.gu;
  grid_dependents_launch();
  grid_dependency_wait();
  COLI_TRACE_POINT(0, 1);
  int *s_act = (int *)(smem + L.act);
  int *s_routes = (int *)(smem + L.routes);
  float *s_slot_gate = (float *)(smem + L.slot_gate);
  load_lists(a, s_act, s_routes, s_slot_gate);
  if (threadIdx.x == 0) COLI_TRACE_POINT(0, 3);
  gu_phase(a, layer_ptrs(a), s_act, s_routes, s_slot_gate, (float *)(smem + L.red),
           (uint32_t *)(smem + L.xpl));
}

// ---------------------------------------------------------------------------
// down phase: each CTA owns a block of output rows; a warp owns one
// 1024-column chunk (cg) of its rows and walks the used experts in ascending
// order (8 experts' loads in flight), adding each slot's contribution into
// per-token registers.  Writes out (with the residual), layer_out, the x
// replicas, and leaves the new residual-stream rows in s_xn [T][nr].

constexpr int kDnBatch = 8;

template <int TM>   // TM >= a.T: per-token accumulators held in registers
__device__ void dn_phase(const Dec2Args &a, const LayerPtrs &lp, const int *s_act,
                         const int *s_routes, float *red, uint32_t *s_planes, float *s_xn,
                         const float *residual) {
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int UH = H / 4;
  const int dh0 = 4 * part_lo(c, UH, G), dh1 = 4 * part_lo(c + 1, UH, G);
  const int nr = dh1 - dh0;
  const int *s_act_expert = s_act + 1;
  const int *s_act_off = s_act + 1 + (E + S);
  const int ncg = a.dn_ncg, nrg = a.dn_nrg;
  for (int i = tid; i < nr * T * ncg; i += blockDim.x) red[i] = 0.0f;
  const int n_active = s_act[0];
  const float *h_rep = a.h + (size_t)(c % a.n_rep) * a.h_stride;
  const int64_t rb = F / 2, ngr = F / kGroup;
  const int64_t down_b = (int64_t)F * H, down_s = (int64_t)2 * F * (H / kGroup);
  const int nbp = F / 32;
  const int cap = a.dn_slots;     // slots whose planes fit in shared memory at once
  const int cg = warp % ncg, rg = warp / ncg;
  const int col = cg * kChunkCols + 32 * lane;
  const bool act = col < F;
  const bool worker = warp < ncg * nrg;
  // experts in groups whose slots' planes fit; groups run in ascending order
  for (int ga = 0; ga < n_active;) {
    int gb = ga;
    while (gb < n_active && s_act_off[gb + 1] - s_act_off[ga] <= cap) ++gb;
    if (gb == ga) gb = ga + 1;   // cap >= T, so a single expert always fits
    const int p0 = s_act_off[ga], np = s_act_off[gb] - p0;
    build_planes_list(h_rep, F, s_routes + p0, np, s_planes, nbp);
    __syncthreads();
    if (ga == 0 && tid == 0) COLI_TRACE_POINT(1, 2);
    if (worker) {
      for (int r = rg; r < nr; r += nrg) {
        float acc[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) acc[t] = 0.0f;
        for (int a0 = ga; a0 < gb; a0 += kDnBatch) {
          uint4 w[kDnBatch];
          float sc[kDnBatch];
#pragma unroll
          for (int b = 0; b < kDnBatch; ++b)
            if (a0 + b < gb && act) {
              const int e = s_act_expert[a0 + b];
              w[b] = ldg_stream(lp.packed + (int64_t)e * a.eb + down_b + (int64_t)(dh0 + r) * rb +
                                col / 2);
              sc[b] = __ldg(lp.scales + (int64_t)e * a.es + down_s + (int64_t)(dh0 + r) * ngr +
                            col / kGroup);
            }
#pragma unroll
          for (int b = 0; b < kDnBatch; ++b) {
            if (a0 + b >= gb) break;
            if (!act) continue;
            const int j0 = s_act_off[a0 + b], nt = s_act_off[a0 + b + 1] - j0;
            for (int j = 0; j < nt; ++j) {
              Planes pl;
              load_planes(s_planes, j0 + j - p0, col / 32, nbp, pl);
              const float v = sc[b] * dot32(w[b], pl);
              const int t = s_routes[j0 + j] / KS;
#pragma unroll
              for (int tt = 0; tt < TM; ++tt)
                if (tt == t) acc[tt] += v;
            }
          }
        }
        // reduce over lanes, 8 tokens at a time; the owning lane accumulates
        for (int t0 = 0; t0 < T; t0 += 8) {
          float v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[q] = 0.0f;
#pragma unroll
            for (int tt = 0; tt < TM; ++tt)
              if (tt == t0 + q) v[q] = acc[tt];
          }
          const float tot = reduce8(v);
          const int t = t0 + (lane >> 2);
          if ((lane & 3) == 0 && t < T) red[(r * T + t) * ncg + cg] += tot;
        }
      }
    }
    __syncthreads();
    ga = gb;
  }
  if (tid == 0) COLI_TRACE_POINT(1, 4);
  // combine is complete: residual, outputs, replicas of the new layer input
  for (int i = tid; i < T * nr; i += blockDim.x) {
    const int t = i / nr, r = i - t * nr;
    const int64_t o = (int64_t)t * H + dh0 + r;
    float v = 0.0f;
    for (int q = 0; q < ncg; ++q) v += red[(r * T + t) * ncg + q];
    if (lp.layer_out) lp.layer_out[o] = v;
    const float xn = residual ? residual[o] + v : v;
    lp.out[o] = xn;
    s_xn[i] = xn;
    if (lp.xrep)
      for (int rr = 0; rr < a.n_rep; ++rr) lp.xrep[rr * a.x_stride + o] = xn;
  }
  __syncthreads();
}

// Partial logits of the next layer from this CTA's rows of its input:
// partials[c][t][e] = sum_r wr[e][dh0 + r] xn[t][r], written to n_copies copies.
template <typename WT>
__device__ void dn_partials(const Dec2Args &a, float *partials, const WT *s_wr, const float *s_xn,
                            int n_copies, size_t copy_stride) {
  const int T = a.T, H = a.H, E = a.E;
  const int G = gridDim.x, c = blockIdx.x;
  const int UH = H / 4;
  const int nr = 4 * part_lo(c + 1, UH, G) - 4 * part_lo(c, UH, G);
  for (int o = threadIdx.x; o < T * E; o += blockDim.x) {
    const int t = o / E, e = o - t * E;
    float sum = 0.0f;
    for (int r = 0; r < nr; ++r) sum = fmaf(to_f32(s_wr[e * nr + r]), s_xn[t * nr + r], sum);
    for (int rr = 0; rr < n_copies; ++rr)
      partials[rr * copy_stride + (size_t)c * T * E + o] = sum;
  }
}

// This CTA's rows [dh0, dh1) of a router matrix, into shared memory.
template <typename WT>
__device__ void load_router_rows(const Dec2Args &a, const WT *wr, WT *s_wr) {
  const int H = a.H, E = a.E;
  const int G = gridDim.x, c = blockIdx.x;
  const int UH = H / 4;
  const int dh0 = 4 * part_lo(c, UH, G), nr = 4 * part_lo(c + 1, UH, G) - dh0;
  for (int i = threadIdx.x; i < E * nr; i += blockDim.x) {
    const int e = i / nr, r = i - e * nr;
    s_wr[i] = wr[(size_t)e * H + dh0 + r];
  }
}

template <typename WT>
__global__ void __launch_bounds__(kDec2MaxThreads) k_down(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DnSmem &L = a.dn;
  WT *s_wr = (WT *)(smem + L.wr);
  // the next layer's router rows do not depend on the previous kernel
  if (a.wr) load_router_rows<WT>(a, (const WT *)a.wr, s_wr);
  grid_dependents_launch();
  grid_dependency_wait();
  if (threadIdx.x == 0) COLI_TRACE_POINT(1, 1);
  int *s_act = (int *)(smem + L.act);
  int *s_routes = (int *)(smem + L.routes);
  load_lists(a, s_act, s_routes, nullptr);
  float *s_xn = (float *)(smem + L.xn);
  const LayerPtrs lp = layer_ptrs(a);
  if (a.T == 1)
    dn_phase<1>(a, lp, s_act, s_routes, (float *)(smem + L.acc), (uint32_t *)(smem + L.planes),
                s_xn, a.residual);
  else
    dn_phase<kDecodeMaxT>(a, lp, s_act, s_routes, (float *)(smem + L.acc),
                          (uint32_t *)(smem + L.planes), s_xn, a.residual);
  if (a.wr) {
    dn_partials<WT>(a, a.partials, s_wr, s_xn, 1, 0);
    // the last CTA routes the next layer (its shared memory is free again)
    LayerPtrs rp = lp;
    rp.route_counts = a.next_counts;
    route_if_last(a, rp, smem);
  }
  if (threadIdx.x == 0) COLI_TRACE_POINT(1, 6);
}

// ---------------------------------------------------------------------------
// The decode stack in one persistent cooperative kernel: layer after layer,
// every CTA routes the layer itself from its copy of the router partials,
// runs its gate/up share, meets the grid at a barrier (h complete), runs its
// down rows and the next layer's partials, and meets the grid again.  Code and
// launch state stay resident across layers.  Every barrier wait is bounded.

__device__ bool grid_barrier(uint32_t *ctr, uint32_t target, uint32_t *ctrl) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(ctr), "r"(1u) : "memory");
    int ok = 1;
    uint32_t v;
    const long long t0 = clock64();
    for (;;) {
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if (clock64() - t0 > kWaitCycles) {
        ok = 0;
        atomicOr(ctrl + kCtrlFlags, COLI_FLAG_TIMEOUT);
        break;
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

constexpr int kStackThreads = 384;

template <typename XT, typename WT, int TM>
__global__ void __launch_bounds__(kStackThreads) k_stack(Dec2Args a, StackArgs st) {
  extern __shared__ __align__(128) uint8_t smem[];
  const StkSmem &L = st.sm;
  const int T = a.T, H = a.H, E = a.E, S = a.S, k = a.k;
  const int tid = threadIdx.x;
  const int G = gridDim.x, c = blockIdx.x;
  int *s_act = (int *)(smem + L.act);
  int *s_routes = (int *)(smem + L.routes);
  float *s_slot_gate = (float *)(smem + L.slot_gate);
  WT *s_wr = (WT *)(smem + L.wr);
  uint8_t *area = smem + L.area;
  uint32_t *bar = a.ctrl + kCtrlBarrier;
  uint32_t nbar = 0;
  bool ok = true;
  // ---- layer 0: x in every replica (f32) and its router partials
  {
    const int UH = H / 4;
    const int h0 = 4 * part_lo(c, UH, G), nr = 4 * part_lo(c + 1, UH, G) - h0;
    const XT *x = (const XT *)a.x;
    float *s_xn = (float *)area;
    for (int i = tid; i < T * nr; i += blockDim.x) {
      const int t = i / nr, r = i - t * nr;
      const float v = to_f32(x[(size_t)t * H + h0 + r]);
      s_xn[i] = v;
      for (int rr = 0; rr < a.n_rep; ++rr) a.xrep[rr * a.x_stride + (size_t)t * H + h0 + r] = v;
    }
    load_router_rows<WT>(a, (const WT *)st.router, s_wr);
    __syncthreads();
    dn_partials<WT>(a, a.partials, s_wr, s_xn, a.n_rep, st.part_stride);
  }
  ok = grid_barrier(bar, ++nbar * G, a.ctrl);
  for (int l = 0; l < st.n_layers && ok; ++l) {
    LayerPtrs la;
    la.packed = a.packed + (size_t)l * st.pk_stride;
    la.scales = a.scales + (size_t)l * st.sc_stride;
    la.route_counts = st.counts ? st.counts + (size_t)l * E : nullptr;
    la.layer_out = st.layer_out ? st.layer_out + (size_t)l * T * H : nullptr;
    la.partials = a.partials + (size_t)(c % a.n_rep) * st.part_stride;
    la.out = st.x_out;
    la.xrep = a.xrep;
    const bool next = l + 1 < st.n_layers;
    // the next layer's router rows: needed only in the down phase
    if (next)
      load_router_rows<WT>(a, (const WT *)((const uint8_t *)st.router + (size_t)(l + 1) * st.wr_stride),
                           s_wr);
    if (l == 3 && tid == 0) COLI_TRACE_POINT(1, 8);
    // ---- route (every CTA from its own copy of the partials)
    {
      float *s_logits = (float *)area;
      int *s_rank = (int *)(s_logits + T * E);
      int *s_idx = s_rank + T * E;
      float *s_gates = (float *)(s_idx + T * k);
      float *s_vals = s_gates + T * k;
      float *s_scratch = s_vals + T * k;
      float *s_stage = s_scratch + kDec2MaxThreads;
      route_block(a, la, s_logits, s_idx, s_gates, s_vals, s_rank, s_scratch, s_stage, c == 0);
      block_union(s_idx, s_gates, T, k, S, E, s_act, s_act + 1, s_act + 1 + (E + S), s_routes,
                  s_slot_gate, s_rank);
    }
    if (l == 3 && tid == 0) COLI_TRACE_POINT(1, 9);
    // ---- gate/up
    gu_phase(a, la, s_act, s_routes, s_slot_gate, (float *)(area + L.gu_red),
             (uint32_t *)(area + L.gu_xpl));
    if (l == 3 && tid == 0) COLI_TRACE_POINT(1, 10);
    ok = grid_barrier(bar, ++nbar * G, a.ctrl);
    if (!ok) break;
    if (l == 3 && tid == 0) COLI_TRACE_POINT(1, 11);
    // ---- down, residual, next layer's partials
    float *s_xn = (float *)(area + L.dn_xn);
    la.xrep = next ? a.xrep : nullptr;
    dn_phase<TM>(a, la, s_act, s_routes, (float *)(area + L.dn_acc),
                 (uint32_t *)(area + L.dn_planes), s_xn, a.xrep);   // replica 0: this layer's input
    if (l == 3 && tid == 0) COLI_TRACE_POINT(1, 12);
    if (next) {
      dn_partials<WT>(a, a.partials, s_wr, s_xn, a.n_rep, st.part_stride);
      if (l == 3 && tid == 0) COLI_TRACE_POINT(1, 13);
      ok = grid_barrier(bar, ++nbar * G, a.ctrl);
      if (l == 3 && tid == 0) COLI_TRACE_POINT(1, 14);
    }
  }
  // the last CTA out resets the barrier counters for the next launch
  __syncthreads();
  if (tid == 0) {
    const unsigned t = atomicAdd(a.ctrl + kCtrlExit, 1u);
    if (t == (unsigned)G - 1) {
      a.ctrl[kCtrlBarrier] = 0;
      a.ctrl[kCtrlExit] = 0;
    }
  }
}

// ---------------------------------------------------------------------------
// host side

#ifdef COLI_TRACE
extern "C" int coli_trace_read(void *points, void *stages, void *issues) {
  if (cudaMemcpyFromSymbol(points, g_trace, sizeof(g_trace)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(stages, g_trace_stage, sizeof(g_trace_stage)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(issues, g_trace_issue, sizeof(g_trace_issue)) != cudaSuccess) return -1;
  return 0;
}
#endif

namespace {

template <typename K>
cudaError_t launch(K kernel, int grid, int block, size_t smem, cudaStream_t s, bool pdl,
                   const Dec2Args &args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

size_t al16(size_t v) { return (v + 15) & ~(size_t)15; }
size_t al128(size_t v) { return (v + 127) & ~(size_t)127; }

int max_smem() {
  static int v = 0;
  if (!v) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      v = 227 * 1024;
  }
  return v;
}

// Raise a kernel's dynamic shared-memory limit once per device (the limit is
// only ever raised, so later smaller launches need no call).
template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
  static std::mutex mu;
  static std::unordered_map<const void *, size_t> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  size_t &cur = done[dev][(const void *)kernel];
  if (bytes <= cur) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cur = bytes;
  return e;
}

}  // namespace

// Geometry and shared-memory plans of both kernels for one layer shape.
cudaError_t plan_decode(Dec2Args &a, int n_part) {
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const size_t budget = (size_t)max_smem() - 4096;
  const int G = num_sms();
  a.n_part = n_part;
  // ---- gate/up
  a.gu_ncg = (H + kChunkCols - 1) / kChunkCols;
  a.gu_nrg = 16 / a.gu_ncg;
  if (a.gu_nrg < 1) a.gu_nrg = 1;
  if (a.gu_ncg * a.gu_nrg > kDec2MaxThreads / 32) return cudaErrorInvalidValue;
  const int n_used = ((E < T * k) ? E : T * k) + S;
  const int max_rows = 4 * ((n_used * (F / 4) + G - 1) / G);
  GuSmem g{};
  size_t o = 0;
  g.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  g.routes = o; o = al16(o + (size_t)T * KS * 4);
  g.slot_gate = o; o = al16(o + (size_t)T * KS * 4);
  g.red = o; o = al16(o + (size_t)max_rows * T * a.gu_ncg * 2 * 4);
  if (o > budget) return cudaErrorInvalidValue;
  const size_t xpl_bytes = (size_t)T * 18 * (H / 32) * 4;
  a.gu_xpl = o + al16(xpl_bytes) <= budget;
  g.xpl = o; o = al16(o + (a.gu_xpl ? xpl_bytes : 0));
  g.total = o;
  a.gu = g;
  // ---- down
  a.dn_ncg = (F + kChunkCols - 1) / kChunkCols;
  a.dn_nrg = 16 / a.dn_ncg;
  if (a.dn_nrg < 1) a.dn_nrg = 1;
  if (a.dn_ncg * a.dn_nrg > kDec2MaxThreads / 32) return cudaErrorInvalidValue;
  const int UH = H / 4;
  const int max_nr = 4 * ((UH + n_part - 1) / n_part);
  DnSmem d{};
  o = 0;
  d.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  d.routes = o; o = al16(o + (size_t)T * KS * 4);
  d.acc = o; o = al16(o + (size_t)max_nr * T * a.dn_ncg * 4);
  d.xn = o; o = al16(o + (size_t)T * max_nr * 4);
  d.wr = o; o = al16(o + (size_t)E * max_nr * 4);
  const size_t per_slot = (size_t)18 * (F / 32) * 4;
  size_t room = budget > o ? budget - o : 0;
  int slots = (int)(room / per_slot);
  if (slots > T * KS) slots = T * KS;
  if (slots < T) return cudaErrorInvalidValue;   // one expert's tokens must fit
  a.dn_slots = slots;
  d.planes = o; o = al16(o + (size_t)slots * per_slot);
  d.total = o;
  a.dn = d;
  return cudaSuccess;
}

// Shared memory the last CTA needs to route a layer (see route_finish).
size_t route_smem_bytes(const Dec2Args &a, bool *stage) {
  const size_t rest = (size_t)(2 * a.T * a.E + 3 * a.T * a.k + kDec2MaxThreads + 2 +
                               2 * (a.E + a.S) + 2 * a.T * (a.k + a.S)) * 4;
  const size_t st = (size_t)a.n_part * a.T * a.E * 4;
  *stage = st + rest <= (size_t)max_smem() - 4096;
  return (*stage ? st : 0) + rest;
}

cudaError_t launch_route_partials(const Dec2Args &a_in, int x_bf16, int w_bf16, cudaStream_t s,
                                  bool pdl) {
  Dec2Args a = a_in;
  bool stage = false;
  const size_t smem = route_smem_bytes(a, &stage);
  a.stage_partials = stage;
  const int threads = kDec2MaxThreads;
  cudaError_t e;
#define COLI_LAUNCH_ROUTE(XT, WT)                                             \
  if ((e = allow_smem(k_route<XT, WT>, smem)) != cudaSuccess) return e;      \
  return launch(k_route<XT, WT>, a.n_part, threads, smem, s, pdl, a);
  if (!x_bf16 && !w_bf16) { COLI_LAUNCH_ROUTE(float, float) }
  if (!x_bf16 && w_bf16) { COLI_LAUNCH_ROUTE(float, __nv_bfloat16) }
  if (x_bf16 && !w_bf16) { COLI_LAUNCH_ROUTE(__nv_bfloat16, float) }
  COLI_LAUNCH_ROUTE(__nv_bfloat16, __nv_bfloat16)
#undef COLI_LAUNCH_ROUTE
}

cudaError_t plan_stack(Dec2Args &a, StackArgs &st) {
  cudaError_t e = plan_decode(a, a.n_part);
  if (e != cudaSuccess) return e;
  // the persistent kernel runs kStackThreads threads: fewer warps per phase
  const int nw = kStackThreads / 32;
  a.gu_nrg = nw / a.gu_ncg;
  a.dn_nrg = nw / a.dn_ncg;
  if (a.gu_nrg < 1 || a.dn_nrg < 1) return cudaErrorInvalidValue;
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const size_t budget = (size_t)max_smem() - 4096;
  const int G = a.n_part;
  StkSmem m{};
  size_t o = 0;
  m.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  m.routes = o; o = al16(o + (size_t)T * KS * 4);
  m.slot_gate = o; o = al16(o + (size_t)T * KS * 4);
  const int UH = H / 4;
  const int max_nr = 4 * ((UH + G - 1) / G);
  m.wr = o; o = al16(o + (size_t)E * max_nr * 4);
  m.area = al128(o);
  const size_t route_b = (size_t)(2 * T * E + 3 * T * k + kDec2MaxThreads + (size_t)G * T * E) * 4;
  const int n_used = ((E < T * k) ? E : T * k) + S;
  const int max_rows = 4 * ((n_used * (F / 4) + G - 1) / G);
  size_t go = 0;
  m.gu_red = go; go = al16(go + (size_t)max_rows * T * a.gu_ncg * 2 * 4);
  m.gu_xpl = go; go = al16(go + (a.gu_xpl ? (size_t)T * 18 * (H / 32) * 4 : 0));
  size_t dof = 0;
  m.dn_acc = dof; dof = al16(dof + (size_t)max_nr * T * a.dn_ncg * 4);
  m.dn_xn = dof; dof = al16(dof + (size_t)T * max_nr * 4);
  m.dn_planes = dof;
  size_t area = route_b > go ? route_b : go;
  if (dof > area) area = dof;
  if (m.area + area > budget) return cudaErrorInvalidValue;
  const size_t per_slot = (size_t)18 * (F / 32) * 4;
  int slots = (int)((budget - m.area - dof) / per_slot);
  if (slots > T * KS) slots = T * KS;
  if (slots < T) return cudaErrorInvalidValue;
  a.dn_slots = slots;
  const size_t dn_b = dof + (size_t)slots * per_slot;
  if (dn_b > area) area = dn_b;
  m.total = al16(m.area + area);
  st.sm = m;
  return cudaSuccess;
}

cudaError_t launch_stack(const Dec2Args &a, const StackArgs &st, int x_bf16, int wr_bf16,
                         cudaStream_t s) {
  const int threads = kStackThreads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_part);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = st.sm.total;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e;
#define COLI_LAUNCH_STACK(XT, WT)                                                        \
  if (a.T == 1) {                                                                         \
    if ((e = allow_smem(k_stack<XT, WT, 1>, st.sm.total)) != cudaSuccess) return e;       \
    return cudaLaunchKernelEx(&cfg, k_stack<XT, WT, 1>, a, st);                            \
  }                                                                                       \
  if ((e = allow_smem(k_stack<XT, WT, kDecodeMaxT>, st.sm.total)) != cudaSuccess) return e; \
  return cudaLaunchKernelEx(&cfg, k_stack<XT, WT, kDecodeMaxT>, a, st);
  if (!x_bf16 && !wr_bf16) { COLI_LAUNCH_STACK(float, float) }
  if (!x_bf16 && wr_bf16) { COLI_LAUNCH_STACK(float, __nv_bfloat16) }
  if (x_bf16 && !wr_bf16) { COLI_LAUNCH_STACK(__nv_bfloat16, float) }
  COLI_LAUNCH_STACK(__nv_bfloat16, __nv_bfloat16)
#undef COLI_LAUNCH_STACK
}

cudaError_t launch_gateup(const Dec2Args &a, int grid, cudaStream_t s, bool pdl) {
  const int threads = a.gu_ncg * a.gu_nrg * 32;
  cudaError_t e = allow_smem(k_gateup, a.gu.total);
  if (e != cudaSuccess) return e;
  return launch(k_gateup, grid, threads, a.gu.total, s, pdl, a);
}

cudaError_t launch_down(const Dec2Args &a_in, int wr_bf16, cudaStream_t s, bool pdl) {
  Dec2Args a = a_in;
  const int threads = a.dn_ncg * a.dn_nrg * 32;
  size_t smem = a.dn.total;
  if (a.wr) {
    bool stage = false;
    const size_t rs = route_smem_bytes(a, &stage);
    a.stage_partials = stage;
    if (rs > smem) smem = rs;
  }
  cudaError_t e;
  if (wr_bf16) {
    if ((e = allow_smem(k_down<__nv_bfloat16>, smem)) != cudaSuccess) return e;
    return launch(k_down<__nv_bfloat16>, a.n_part, threads, smem, s, pdl, a);
  }
  if ((e = allow_smem(k_down<float>, smem)) != cudaSuccess) return e;
  return launch(k_down<float>, a.n_part, threads, smem, s, pdl, a);
}

}  // namespace coli
