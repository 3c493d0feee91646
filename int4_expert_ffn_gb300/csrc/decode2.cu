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
__device__ void build_planes(const float *src, int n_vec, int F, uint32_t *planes, int nbp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int groups_per_vec = (F + 127) / 128;
  const int n_groups = n_vec * groups_per_vec;
  const int q = lane & 7;
  for (int g = warp; g < n_groups; g += nw) {
    const int v = g / groups_per_vec, gc = g - v * groups_per_vec;
    const int col = gc * 128 + 4 * lane;
    const bool act = col < F;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (act) x = __ldcg((const float4 *)(src + (int64_t)v * F + col));
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

struct StageIter {
  int u, u1, seg4, rs4;
  __device__ StageIter(int u0_, int u1_, int seg4_, int rs4_)
      : u(u0_), u1(u1_), seg4(seg4_), rs4(rs4_) {}
  // next (segment index, first row in segment, rows) in units of 4 rows
  __device__ bool next(int &a, int &r0, int &n) {
    if (u >= u1) return false;
    a = u / seg4;
    const int ru = u - a * seg4;
    int nu = rs4;
    if (nu > u1 - u) nu = u1 - u;
    if (nu > seg4 - ru) nu = seg4 - ru;
    r0 = ru * 4;
    n = nu * 4;
    u += nu;
    return true;
  }
};

}  // namespace

// ---------------------------------------------------------------------------
// Router partial logits: CTA c of G sums its rows [h0, h1) of every expert's
// router row against x:  partials[c][t][e] = sum_{h in [h0,h1)} Wr[e][h] x[t][h].

template <typename XT, typename WT>
__global__ void __launch_bounds__(256) k_route(Dec2Args a) {
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
    for (int r = 0; r < a.n_rep; ++r)
      a.partials[r * a.part_stride + (size_t)c * a.T * a.E + o] = s;
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
}

// ---------------------------------------------------------------------------
// Routing shared by k_gateup and k_topk: logits from the partials (fixed
// order), top-k per token by warps, NaN flag.

__device__ void route_block(const Dec2Args &a, float *s_logits, int *s_idx, float *s_gates,
                            float *s_vals, int *s_rank, float *s_scratch, float *s_stage,
                            uint64_t *pbar, bool publish) {
  const int T = a.T, E = a.E, k = a.k;
  const int TE = T * E;
  const int nthr = blockDim.x;
  const float *src = a.partials + (size_t)(blockIdx.x % a.n_rep) * a.part_stride;
  if (s_stage) {
    // one bulk copy of all partials into shared memory, then reduce there
    if (threadIdx.x == 0) {
      const uint32_t bytes = (uint32_t)((size_t)a.n_part * TE * 4);
      mbar_arrive_expect_tx(pbar, bytes);
      bulk_g2s(s_stage, src, bytes, pbar);
    }
    if (!mbar_wait(pbar, 0)) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
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
      if (a.counts) atomicAdd(a.counts + s_idx[i], 1u);
    }
  }
}

__global__ void __launch_bounds__(256) k_topk(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  grid_dependents_launch();
  uint64_t *pbar = (uint64_t *)smem;
  if (threadIdx.x == 0) {
    mbar_init(pbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();
  const int T = a.T, E = a.E, k = a.k;
  float *s_stage = (float *)(smem + 128);
  float *s_logits = s_stage + (a.gu_stage_partials ? (size_t)a.n_part * T * E : 0);
  int *s_rank = (int *)(s_logits + T * E);
  int *s_idx = s_rank + T * E;
  float *s_gates = (float *)(s_idx + T * k);
  float *s_vals = s_gates + T * k;
  float *s_scratch = s_vals + T * k;
  route_block(a, s_logits, s_idx, s_gates, s_vals, s_rank, s_scratch,
              a.gu_stage_partials ? s_stage : nullptr, pbar, true);
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    if (a.idx_out) a.idx_out[i] = s_idx[i];
    if (a.gates_out) a.gates_out[i] = s_gates[i];
  }
}

// ---------------------------------------------------------------------------
// gate/up

__global__ void __launch_bounds__(kDec2MaxThreads) k_gateup(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GuSmem &L = a.gu;
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwc = a.gu_ncg * a.gu_nrg;   // compute warps; warp nwc is the producer
  const int ns = a.gu_ns;
  uint64_t *full = (uint64_t *)(smem + L.bar);
  uint64_t *done = full + ns;
  uint64_t *pbar = done + ns;
  int *s_abort = (int *)(pbar + 1);
  int *s_desc = (int *)(smem + L.desc);   // [3][16]: segment, first row, rows per slot
  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(full + i, 1);
      mbar_init(done + i, nwc);
    }
    mbar_init(pbar, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependents_launch();
  if (tid == 0) COLI_TRACE_POINT(0, 0);
  grid_dependency_wait();
  if (tid == 0) COLI_TRACE_POINT(0, 1);

  float *s_logits = (float *)(smem + L.logits);
  int *s_idx = (int *)(smem + L.idx);
  float *s_gates = (float *)(smem + L.gates);
  float *s_vals = (float *)(smem + L.vals);
  int *s_rank = (int *)(smem + L.rank);
  float *s_scratch = (float *)(smem + L.scratch);
  int *s_act = (int *)(smem + L.act);          // [0] n_active, act_expert, act_off
  int *s_act_expert = s_act + 1;
  int *s_act_off = s_act + 1 + (E + S);
  int *s_routes = (int *)(smem + L.routes);
  float *s_slot_gate = (float *)(smem + L.slot_gate);
  const bool cta0 = blockIdx.x == 0;

  // partials are staged in the (not yet used) weight ring
  route_block(a, s_logits, s_idx, s_gates, s_vals, s_rank, s_scratch,
              a.gu_stage_partials ? (float *)(smem + L.ring) : nullptr, pbar, cta0);
  if (tid == 0) COLI_TRACE_POINT(0, 2);
  const int n_active = block_union(s_idx, s_gates, T, k, S, E, s_act, s_act_expert, s_act_off,
                                   s_routes, s_slot_gate, s_rank);
  if (tid == 0) COLI_TRACE_POINT(0, 3);
  if (cta0) {
    for (int i = tid; i < 1 + 2 * (E + S) + 1; i += blockDim.x) a.g_act[i] = s_act[i];
    for (int i = tid; i < T * KS; i += blockDim.x) {
      a.g_routes[i] = s_routes[i];
      a.g_slot_gate[i] = s_slot_gate[i];
    }
  }

  // this CTA's rows in the flattened (used expert, row) space, units of 4 rows
  const int G = gridDim.x, c = blockIdx.x;
  const int F4 = F / 4;
  const int U = n_active * F4;
  const int u0 = part_lo(c, U, G), u1 = part_lo(c + 1, U, G);
  const int rs4 = a.gu_rs / 4;
  const int64_t rb = H / 2, ngr = H / kGroup;
  const int stage_bytes = a.gu_rs * (H + H / 8);
  float *red = (float *)(smem + L.red);
  const int red_stride = a.gu_rs * T * a.gu_ncg * 2;

  if (warp == nwc) {
    // ---------------- producer warp: issue copies, finalise h ----------------
    fence_proxy_async();   // the ring held the staged partials
    StageIter it(u0, u1, F4, rs4);
    int s = 0, fin = 0, ai, r0, n;
    bool ok = true, prefetched = false;
    for (;;) {
      const bool more = ok && it.next(ai, r0, n);
      // finalise the oldest stage when its slot is needed again, or at the end
      while (ok && fin < s && (!more || s - fin >= ns)) {
        const int slot = fin % ns;
        if (!mbar_wait(done + slot, (fin / ns) & 1)) { ok = false; break; }
        const int fa = s_desc[slot], f0 = s_desc[16 + slot], fn = s_desc[32 + slot];
        const int j0 = s_act_off[fa], ntok = s_act_off[fa + 1] - j0;
        const float *rd = red + slot * red_stride;
        for (int i = lane; i < fn * ntok; i += 32) {
          const int r = i / ntok, j = i - r * ntok;
          float g = 0.0f, u = 0.0f;
          for (int cg = 0; cg < a.gu_ncg; ++cg) {
            g += rd[((r * T + j) * a.gu_ncg + cg) * 2];
            u += rd[((r * T + j) * a.gu_ncg + cg) * 2 + 1];
          }
          const int slot_id = s_routes[j0 + j];
          const float hv = silu(g) * u * s_slot_gate[slot_id];
          for (int rr = 0; rr < a.n_rep; ++rr)
            a.h[rr * a.h_stride + (int64_t)slot_id * F + f0 + r] = hv;
        }
        __syncwarp();
        ++fin;
      }
      if (!more) {
        if (lane == 0) COLI_TRACE_POINT(0, 6);
        break;
      }
      const int slot = s % ns;
      if (lane == 0) {
        s_desc[slot] = ai;
        s_desc[16 + slot] = r0;
        s_desc[32 + slot] = n;
        const int e = s_act_expert[ai];
        const uint8_t *pg = a.packed + (int64_t)e * a.eb + (int64_t)r0 * rb;
        const uint8_t *pu = pg + (int64_t)F * rb;
        const float *sg = a.scales + (int64_t)e * a.es + (int64_t)r0 * ngr;
        const float *su = sg + (int64_t)F * ngr;
        uint8_t *dst = smem + L.ring + (size_t)slot * stage_bytes;
        const uint32_t nb = (uint32_t)(n * rb), sb = (uint32_t)(n * ngr * 4);
        mbar_arrive_expect_tx(full + slot, 2 * nb + 2 * sb);
        bulk_g2s(dst, pg, nb, full + slot);
        bulk_g2s(dst + a.gu_rs * rb, pu, nb, full + slot);
        bulk_g2s(dst + 2 * a.gu_rs * rb, sg, sb, full + slot);
        bulk_g2s(dst + 2 * a.gu_rs * rb + a.gu_rs * ngr * 4, su, sb, full + slot);
      }
      __syncwarp();
      ++s;
      if (!prefetched && (s == ns || it.u >= it.u1)) {
        prefetched = true;
        if (lane == 0) COLI_TRACE_POINT(0, 4);
        // L2 prefetch of the down rows the same-index k_down CTA will read
        if (lane == 0 && c < a.n_part) {
          const int UH = H / 4;
          const int dh0 = 4 * part_lo(c, UH, a.n_part), dh1 = 4 * part_lo(c + 1, UH, a.n_part);
          for (int q = 0; q < n_active && dh1 > dh0; ++q) {
            const int e = s_act_expert[q];
            prefetch_l2(a.packed + (int64_t)e * a.eb + (int64_t)F * H + (int64_t)dh0 * (F / 2),
                        (uint32_t)((dh1 - dh0) * (F / 2)));
            prefetch_l2(a.scales + (int64_t)e * a.es + (int64_t)2 * F * ngr +
                            (int64_t)dh0 * (F / kGroup),
                        (uint32_t)((dh1 - dh0) * (F / 16)));
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
      *(volatile int *)s_abort = 1;
      // drain copies still in flight before the CTA may exit
      for (int st = fin; st < s; ++st) (void)mbar_wait(full + (st % ns), (st / ns) & 1);
    }
  } else if (warp < nwc) {
    // ---------------- compute warps ----------------
    const int cg = warp % a.gu_ncg, rg = warp / a.gu_ncg, nrg = a.gu_nrg;
    const int col = cg * kChunkCols + 32 * lane;
    const bool act = col < H;
    const float *x = a.xrep + (size_t)(c % a.n_rep) * a.x_stride;
    Planes pl;
    int cached = -1;
    if (u1 > u0) {
      // quantise the first stage's token now, while the first weights are in flight
      const int t = s_routes[s_act_off[u0 / F4]] / KS;
      float v[32];
      if (act) load32<float>(x + (int64_t)t * H + col, v);
      else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      }
      quantize32(v, pl);
      cached = t;
    }
    StageIter it(u0, u1, F4, rs4);
    int s = 0, ai, r0, n;
    while (it.next(ai, r0, n)) {
      const int slot = s % ns;
      if (!mbar_wait(full + slot, (s / ns) & 1)) {
        if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
        break;
      }
      if (*(volatile int *)s_abort) break;
      if (warp == 0 && lane == 0) {
        if (s == 0) COLI_TRACE_POINT(0, 5);
        COLI_TRACE_STAGE(0, s);
      }
      const uint8_t *stg = smem + L.ring + (size_t)slot * stage_bytes;
      const uint8_t *wg = stg, *wu = stg + a.gu_rs * rb;
      const float *sgp = (const float *)(stg + 2 * a.gu_rs * rb);
      const float *sup = sgp + a.gu_rs * ngr;
      float *rd = red + slot * red_stride;
      const int j0 = s_act_off[ai], ntok = s_act_off[ai + 1] - j0;
      const int nrows = n > rg ? (n - rg + nrg - 1) / nrg : 0;
      for (int j = 0; j < ntok; ++j) {
        const int t = s_routes[j0 + j] / KS;
        if (t != cached) {
          float v[32];
          if (act) load32<float>(x + (int64_t)t * H + col, v);
          else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
          }
          quantize32(v, pl);
          cached = t;
        }
        for (int q0 = 0; q0 < nrows; q0 += 4) {
          float v[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            v[2 * q] = 0.0f;
            v[2 * q + 1] = 0.0f;
            const int r = rg + (q0 + q) * nrg;
            if (q0 + q < nrows && act) {
              const uint4 g4 = *(const uint4 *)(wg + r * rb + col / 2);
              const uint4 u4 = *(const uint4 *)(wu + r * rb + col / 2);
              v[2 * q] = sgp[r * ngr + col / kGroup] * dot32(g4, pl);
              v[2 * q + 1] = sup[r * ngr + col / kGroup] * dot32(u4, pl);
            }
          }
          const float tot = reduce8(v);
          if ((lane & 3) == 0) {
            const int vi = lane >> 2, q = vi >> 1;
            if (q0 + q < nrows) {
              const int r = rg + (q0 + q) * nrg;
              rd[((r * T + j) * a.gu_ncg + cg) * 2 + (vi & 1)] = tot;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(done + slot);
      ++s;
    }
  }
}

// ---------------------------------------------------------------------------
// down + combine + residual + next layer's router partials

template <typename WT>
__global__ void __launch_bounds__(kDec2MaxThreads) k_down(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DnSmem &L = a.dn;
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwc = a.dn_ncg * a.dn_nrg;
  const int G = gridDim.x, c = blockIdx.x;
  const int UH = H / 4;
  const int dh0 = 4 * part_lo(c, UH, G), dh1 = 4 * part_lo(c + 1, UH, G);
  const int nr = dh1 - dh0;
  const int ns = a.dn_ns;
  uint64_t *full = (uint64_t *)(smem + L.bar);
  uint64_t *done = full + ns;
  int *s_abort = (int *)(done + ns);
  int *s_desc = (int *)(smem + L.desc);
  WT *s_wr = (WT *)(smem + L.wr);
  if (tid == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(full + i, 1);
      mbar_init(done + i, nwc);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  // the next layer's router rows [dh0, dh1) do not depend on the previous kernel
  if (a.wr) {
    const WT *wr = (const WT *)a.wr;
    for (int i = tid; i < E * nr; i += blockDim.x) {
      const int e = i / nr, r = i - e * nr;
      s_wr[i] = wr[(size_t)e * H + dh0 + r];
    }
  }
  __syncthreads();
  grid_dependents_launch();
  if (tid == 0) COLI_TRACE_POINT(1, 0);
  grid_dependency_wait();
  if (tid == 0) COLI_TRACE_POINT(1, 1);
  int *s_act = (int *)(smem + L.act);
  int *s_act_expert = s_act + 1;
  int *s_act_off = s_act + 1 + (E + S);
  int *s_routes = (int *)(smem + L.routes);
  float *s_acc = (float *)(smem + L.acc);   // [T][nr]
  uint32_t *s_planes = (uint32_t *)(smem + L.planes);
  const int nbp = a.dn_nbp;
  for (int i = tid; i < 1 + 2 * (E + S) + 1; i += blockDim.x) s_act[i] = __ldcg(a.g_act + i);
  for (int i = tid; i < T * KS; i += blockDim.x) s_routes[i] = __ldcg(a.g_routes + i);
  for (int i = tid; i < T * nr; i += blockDim.x) s_acc[i] = 0.0f;
  // the slots' h vectors, quantised once for the whole CTA
  const float *h_rep = a.h + (size_t)(c % a.n_rep) * a.h_stride;
  if (a.dn_planes) build_planes(h_rep, T * KS, F, s_planes, nbp);
  __syncthreads();
  if (tid == 0) COLI_TRACE_POINT(1, 2);
  const int n_active = s_act[0];
  const int rs4 = a.dn_rs / 4;
  const int64_t rb = F / 2, ngr = F / kGroup;
  const int stage_bytes = a.dn_rs * (F / 2 + F / 16);
  float *red = (float *)(smem + L.red);
  const int red_stride = a.dn_rs * T * a.dn_ncg;
  const int64_t down_b = (int64_t)F * H, down_s = (int64_t)2 * F * (H / kGroup);
  const int seg4 = nr / 4;
  const int n_units = seg4 > 0 ? n_active * seg4 : 0;

  if (warp == nwc) {
    StageIter it(0, n_units, seg4 > 0 ? seg4 : 1, rs4);
    int s = 0, fin = 0, ai, r0, n;
    bool ok = true;
    for (;;) {
      const bool more = ok && it.next(ai, r0, n);
      while (ok && fin < s && (!more || s - fin >= ns)) {
        const int slot = fin % ns;
        if (!mbar_wait(done + slot, (fin / ns) & 1)) { ok = false; break; }
        const int fa = s_desc[slot], f0 = s_desc[16 + slot], fn = s_desc[32 + slot];
        const int j0 = s_act_off[fa], ntok = s_act_off[fa + 1] - j0;
        const float *rd = red + slot * red_stride;
        for (int i = lane; i < fn * ntok; i += 32) {
          const int r = i / ntok, j = i - r * ntok;
          float v = 0.0f;
          for (int cg = 0; cg < a.dn_ncg; ++cg) v += rd[(r * T + j) * a.dn_ncg + cg];
          const int t = s_routes[j0 + j] / KS;
          s_acc[t * nr + f0 + r] += v;   // experts finalised in ascending order
        }
        __syncwarp();
        ++fin;
      }
      if (!more) break;
      const int slot = s % ns;
      if (lane == 0) {
        s_desc[slot] = ai;
        s_desc[16 + slot] = r0;
        s_desc[32 + slot] = n;
        const int e = s_act_expert[ai];
        const uint8_t *pd = a.packed + (int64_t)e * a.eb + down_b + (int64_t)(dh0 + r0) * rb;
        const float *sd = a.scales + (int64_t)e * a.es + down_s + (int64_t)(dh0 + r0) * ngr;
        uint8_t *dst = smem + L.ring + (size_t)slot * stage_bytes;
        const uint32_t nb = (uint32_t)(n * rb), sb = (uint32_t)(n * ngr * 4);
        mbar_arrive_expect_tx(full + slot, nb + sb);
        bulk_g2s(dst, pd, nb, full + slot);
        bulk_g2s(dst + a.dn_rs * rb, sd, sb, full + slot);
      }
      __syncwarp();
      ++s;
    }
    if (!ok) {
      if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
      *(volatile int *)s_abort = 1;
      for (int st = fin; st < s; ++st) (void)mbar_wait(full + (st % ns), (st / ns) & 1);
    }
  } else if (warp < nwc) {
    const int cg = warp % a.dn_ncg, rg = warp / a.dn_ncg, nrg = a.dn_nrg;
    const int col = cg * kChunkCols + 32 * lane;
    const bool act = col < F;
    StageIter it(0, n_units, seg4 > 0 ? seg4 : 1, rs4);
    int s = 0, ai, r0, n;
    while (it.next(ai, r0, n)) {
      const int slot = s % ns;
      if (!mbar_wait(full + slot, (s / ns) & 1)) {
        if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
        break;
      }
      if (*(volatile int *)s_abort) break;
      if (warp == 0 && lane == 0) {
        if (s == 0) COLI_TRACE_POINT(1, 3);
        COLI_TRACE_STAGE(1, s);
      }
      const uint8_t *stg = smem + L.ring + (size_t)slot * stage_bytes;
      const float *sdp = (const float *)(stg + a.dn_rs * rb);
      float *rd = red + slot * red_stride;
      const int j0 = s_act_off[ai], ntok = s_act_off[ai + 1] - j0;
      const int nrows = n > rg ? (n - rg + nrg - 1) / nrg : 0;
      for (int j = 0; j < ntok; ++j) {
        const int slot_id = s_routes[j0 + j];
        Planes pl;
        if (a.dn_planes) {
          if (act) load_planes(s_planes, slot_id, col / 32, nbp, pl);
          else { pl = Planes{}; }
        } else {
          float v[32];
          if (act) load32<float>(h_rep + (int64_t)slot_id * F + col, v);
          else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
          }
          quantize32(v, pl);
        }
        for (int q0 = 0; q0 < nrows; q0 += 8) {
          float v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[q] = 0.0f;
            const int r = rg + (q0 + q) * nrg;
            if (q0 + q < nrows && act) {
              const uint4 w4 = *(const uint4 *)(stg + r * rb + col / 2);
              v[q] = sdp[r * ngr + col / kGroup] * dot32(w4, pl);
            }
          }
          const float tot = reduce8(v);
          if ((lane & 3) == 0) {
            const int q = lane >> 2;
            if (q0 + q < nrows) {
              const int r = rg + (q0 + q) * nrg;
              rd[(r * T + j) * a.dn_ncg + cg] = tot;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(done + slot);
      ++s;
    }
  }
  if (tid == 0) COLI_TRACE_POINT(1, 4);
  __syncthreads();
  if (tid == 0) COLI_TRACE_POINT(1, 5);
  // combine is complete: residual, outputs, next layer's partial logits
  float *s_xn = (float *)(smem + L.xn);   // [T][nr]
  for (int i = tid; i < T * nr; i += blockDim.x) {
    const int t = i / nr, r = i - t * nr;
    const int64_t o = (int64_t)t * H + dh0 + r;
    const float v = s_acc[i];
    if (a.layer_out) a.layer_out[o] = v;
    const float xn = a.residual ? a.residual[o] + v : v;
    a.out[o] = xn;
    s_xn[i] = xn;
    if (a.xrep)
      for (int rr = 0; rr < a.n_rep; ++rr) a.xrep[rr * a.x_stride + o] = xn;
  }
  if (a.wr) {
    __syncthreads();
    for (int o = tid; o < T * E; o += blockDim.x) {
      const int t = o / E, e = o - t * E;
      float sum = 0.0f;
      for (int r = 0; r < nr; ++r) sum = fmaf(to_f32(s_wr[e * nr + r]), s_xn[t * nr + r], sum);
      for (int rr = 0; rr < a.n_rep; ++rr)
        a.partials[rr * a.part_stride + (size_t)c * T * E + o] = sum;
    }
  }
#ifdef COLI_TRACE
  __syncthreads();
  if (tid == 0) COLI_TRACE_POINT(1, 6);
#endif
}

// ---------------------------------------------------------------------------
// host side

#ifdef COLI_TRACE
extern "C" int coli_trace_read(void *points, void *stages) {
  if (cudaMemcpyFromSymbol(points, g_trace, sizeof(g_trace)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(stages, g_trace_stage, sizeof(g_trace_stage)) != cudaSuccess) return -1;
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

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

// Geometry and shared-memory plans of both kernels for one layer shape.
cudaError_t plan_decode(Dec2Args &a, int n_part) {
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const size_t budget = (size_t)max_smem() - 2048;
  a.n_part = n_part;
  // ---- gate/up
  a.gu_ncg = (H + kChunkCols - 1) / kChunkCols;
  a.gu_nrg = 12 / a.gu_ncg;
  if (a.gu_nrg < 1) a.gu_nrg = 1;
  if (a.gu_ncg * a.gu_nrg > kDec2MaxThreads / 32 - 1) a.gu_nrg = (kDec2MaxThreads / 32 - 1) / a.gu_ncg;
  if (a.gu_nrg < 1) return cudaErrorInvalidValue;
  GuSmem g{};
  size_t o = 0;
  g.logits = o; o = al16(o + (size_t)T * E * 4);
  g.idx = o; o = al16(o + (size_t)T * k * 4);
  g.gates = o; o = al16(o + (size_t)T * k * 4);
  g.vals = o; o = al16(o + (size_t)T * k * 4);
  g.rank = o; o = al16(o + (size_t)(T * E > T * k ? T * E : T * k) * 4);
  g.scratch = o; o = al16(o + (size_t)kDec2MaxThreads * 4);
  g.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  g.routes = o; o = al16(o + (size_t)T * KS * 4);
  g.slot_gate = o; o = al16(o + (size_t)T * KS * 4);
  g.desc = o; o = al16(o + 48 * 4);
  const size_t fixed = o;
  const size_t row_bytes = (size_t)H + H / 8;   // gate + up nibbles and scales per row pair
  int rs = (int)(40960 / row_bytes) / 4 * 4;
  if (rs < 4) rs = 4;
  if (rs > 32) rs = 32;
  const size_t red_row = (size_t)T * a.gu_ncg * 2 * 4;
  int ns = 0;
  for (ns = 16; ns >= 2; --ns) {
    const size_t need = al128(fixed) + ns * rs * row_bytes + ns * rs * red_row + ns * 16 + 64;
    if (need <= budget) break;
  }
  if (ns < 2) return cudaErrorInvalidValue;
  a.gu_rs = rs;
  a.gu_ns = ns;
  o = al128(fixed);
  g.ring = o; o += (size_t)ns * rs * row_bytes;
  g.red = o; o = al16(o + (size_t)ns * rs * red_row);
  g.bar = o; o += (size_t)(2 * ns + 1) * 8 + 16;
  g.total = al16(o);
  a.gu = g;
  a.gu_stage_partials = (size_t)n_part * T * E * 4 <= (size_t)ns * rs * row_bytes;
  // ---- down
  a.dn_ncg = (F + kChunkCols - 1) / kChunkCols;
  a.dn_nrg = 12 / a.dn_ncg;
  if (a.dn_nrg < 1) a.dn_nrg = 1;
  if (a.dn_ncg * a.dn_nrg > kDec2MaxThreads / 32 - 1) a.dn_nrg = (kDec2MaxThreads / 32 - 1) / a.dn_ncg;
  if (a.dn_nrg < 1) return cudaErrorInvalidValue;
  const int UH = H / 4;
  const int max_nr = 4 * ((UH + n_part - 1) / n_part);
  a.dn_nbp = F / 32;
  const size_t planes_bytes = (size_t)T * KS * 18 * a.dn_nbp * 4;
  a.dn_planes = planes_bytes <= 98304;
  DnSmem d{};
  o = 0;
  d.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  d.routes = o; o = al16(o + (size_t)T * KS * 4);
  d.acc = o; o = al16(o + (size_t)T * max_nr * 4);
  d.xn = o; o = al16(o + (size_t)T * max_nr * 4);
  d.wr = o; o = al16(o + (size_t)E * max_nr * 4);
  d.desc = o; o = al16(o + 48 * 4);
  d.planes = o; o = al16(o + (a.dn_planes ? planes_bytes : 0));
  const size_t fixed_d = o;
  const size_t drow = (size_t)F / 2 + F / 16;
  int rsd = max_nr;
  while ((size_t)rsd * drow > 65536 && rsd > 4) rsd -= 4;
  const size_t red_drow = (size_t)T * a.dn_ncg * 4;
  int nsd = 0;
  for (nsd = 16; nsd >= 2; --nsd) {
    const size_t need = al128(fixed_d) + nsd * rsd * drow + nsd * rsd * red_drow + nsd * 16 + 96;
    if (need <= budget) break;
  }
  if (nsd < 2) return cudaErrorInvalidValue;
  // no more stages than the CTA can use
  const int n_used = ((E < T * k) ? E : T * k) + S;
  const int stages_needed = n_used * ((max_nr / 4 + rsd / 4 - 1) / (rsd / 4));
  if (nsd > stages_needed && stages_needed >= 2) nsd = stages_needed;
  a.dn_rs = rsd;
  a.dn_ns = nsd;
  o = al128(fixed_d);
  d.ring = o; o += (size_t)nsd * rsd * drow;
  d.red = o; o = al16(o + (size_t)nsd * rsd * red_drow);
  d.bar = o; o += (size_t)nsd * 16 + 32;
  d.total = al16(o);
  a.dn = d;
  return cudaSuccess;
}

cudaError_t launch_route_partials(const Dec2Args &a, int x_bf16, int w_bf16, cudaStream_t s,
                                  bool pdl) {
  if (!x_bf16 && !w_bf16) return launch(k_route<float, float>, a.n_part, 256, 0, s, pdl, a);
  if (!x_bf16 && w_bf16) return launch(k_route<float, __nv_bfloat16>, a.n_part, 256, 0, s, pdl, a);
  if (x_bf16 && !w_bf16) return launch(k_route<__nv_bfloat16, float>, a.n_part, 256, 0, s, pdl, a);
  return launch(k_route<__nv_bfloat16, __nv_bfloat16>, a.n_part, 256, 0, s, pdl, a);
}

cudaError_t launch_topk(const Dec2Args &a_in, cudaStream_t s, bool pdl) {
  Dec2Args a = a_in;
  const size_t rest = (size_t)(2 * a.T * a.E + 3 * a.T * a.k + 256) * 4;
  const size_t stage = (size_t)a.n_part * a.T * a.E * 4;
  a.gu_stage_partials = 128 + stage + rest <= (size_t)max_smem() - 2048;
  const size_t smem = 128 + (a.gu_stage_partials ? stage : 0) + rest;
  cudaError_t e = allow_smem(k_topk, smem);
  if (e != cudaSuccess) return e;
  return launch(k_topk, 1, 256, smem, s, pdl, a);
}

cudaError_t launch_gateup(const Dec2Args &a, int grid, cudaStream_t s, bool pdl) {
  const int threads = (a.gu_ncg * a.gu_nrg + 1) * 32;
  cudaError_t e = allow_smem(k_gateup, a.gu.total);
  if (e != cudaSuccess) return e;
  return launch(k_gateup, grid, threads, a.gu.total, s, pdl, a);
}

cudaError_t launch_down(const Dec2Args &a, int wr_bf16, cudaStream_t s, bool pdl) {
  const int threads = (a.dn_ncg * a.dn_nrg + 1) * 32;
  cudaError_t e;
  if (wr_bf16) {
    if ((e = allow_smem(k_down<__nv_bfloat16>, a.dn.total)) != cudaSuccess) return e;
    return launch(k_down<__nv_bfloat16>, a.n_part, threads, a.dn.total, s, pdl, a);
  }
  if ((e = allow_smem(k_down<float>, a.dn.total)) != cudaSuccess) return e;
  return launch(k_down<float>, a.n_part, threads, a.dn.total, s, pdl, a);
}

}  // namespace coli
