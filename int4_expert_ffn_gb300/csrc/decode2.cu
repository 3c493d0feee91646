// Decode path of the routed-MoE layer over int4-grouped experts (T <= 16 tokens).
//
// Pages: "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战" (matmul_i4_grouped
// consumes packed rows: W = s (u - 8); expert_ffn.h's dot(u,x) - 8 sum(x) with
// unsigned nibbles against signed 8-bit activations), "Colibrì 深度解析" §四 (an
// expert's three matrices adjacent; batch union reads each used expert once),
// §十一 (route -> union -> compute), "colibrì 路由遥测全解析" (route counts, gates).
//
// Per layer, kernels chained with programmatic dependent launch inside one
// CUDA graph per step:
//   k_route (first layer of a several-token pass): the router partial logits
//     of each CTA's slice of the hidden dimension, added as fixed-point
//     integers.  With one token the first layer's gate/up CTAs form the
//     logits themselves instead (gu_router_logits: each CTA the whole logits
//     of its own experts, published as never-zero words every CTA waits for).
//   k_gateup (one token) / k_gateup_multi (several): every CTA routes the
//     layer itself from the logits (top-k, union lists; CTA 0 publishes them
//     and the route counts), then streams its share of the used experts'
//     gate/up rows through per-warp cp.async rings in shared memory and
//     writes h = silu(g) * u * gate.
//   k_down (one token): each CTA owns a block of output rows of every used
//     expert's down matrix, sums the experts in a fixed order, adds the
//     residual, and adds its rows' share of the next layer's router logits;
//     its warp count makes the largest number of tasks per warp smallest.
//   k_down_multi + k_down (several tokens): the down GEMVs split by expert
//     and cost into per-slot outputs, then k_down adds each token's slots.
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
#include "decode_common.cuh"
#include "ptx.cuh"
#include "topk.cuh"
#include "trace.cuh"

namespace coli {


// ---------------------------------------------------------------------------
// Router partial logits: CTA c of G sums its rows [h0, h1) of every expert's
// router row against x:  partials[c][t][e] = sum_{h in [h0,h1)} Wr[e][h] x[t][h].

// Four consecutive router weights as floats (the row slice start and every
// offset used here are multiples of four elements).
__device__ __forceinline__ void load4w(const float *p, float (&v)[4]) {
  const float4 q = __ldg((const float4 *)p);
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
__device__ __forceinline__ void load4w(const __nv_bfloat16 *p, float (&v)[4]) {
  const uint2 q = __ldg((const uint2 *)p);
  v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xFFFF0000u);
  v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xFFFF0000u);
}

template <typename XT, typename WT>
__global__ void __launch_bounds__(kDec2MaxThreads) k_route(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem_route[];
  grid_dependents_launch();
  grid_dependency_wait();
  const int c = blockIdx.x, G = gridDim.x, T = a.T, E = a.E, H = a.H;
  const int U = H / 4;
  const int h0 = 4 * part_lo(c, U, G), h1 = 4 * part_lo(c + 1, U, G), nr = h1 - h0;
  const XT *x = (const XT *)a.x;
  const WT *wr = (const WT *)a.wr;
  // this CTA's columns of the layer input, widened to f32: into shared memory
  // and into every replica (read by all gate/up CTAs)
  float *s_x = (float *)smem_route;   // [T][nr]
  for (int i = threadIdx.x; i < T * nr; i += blockDim.x) {
    const int t = i / nr, h = h0 + (i - t * nr);
    const float v = to_f32(x[(size_t)t * H + h]);
    s_x[i] = v;
    if (a.xrep)
      for (int r = 0; r < a.n_rep; ++r) a.xrep[r * a.x_stride + (size_t)t * H + h] = v;
  }
  __syncthreads();
  // one thread per expert: its row slice in 16-element pieces (four vector
  // loads in flight), against up to four tokens at a time
  constexpr int kTok = 4;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const WT *w = wr + (size_t)e * H + h0;
    for (int t0 = 0; t0 < T; t0 += kTok) {
      float acc[kTok] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int r0 = 0; r0 < nr; r0 += 16) {
        float wv[4][4];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          if (r0 + 4 * v < nr) {
            load4w(w + r0 + 4 * v, wv[v]);
          } else {
            wv[v][0] = wv[v][1] = wv[v][2] = wv[v][3] = 0.0f;
          }
        }
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt) {
          if (t0 + tt < T) {
            const float *xs = s_x + (t0 + tt) * nr + r0;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              if (r0 + 4 * v < nr)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[tt] = fmaf(wv[v][j], xs[4 * v + j], acc[tt]);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kTok; ++tt) {
        if (t0 + tt >= T) break;
        const int o = (t0 + tt) * E + e;
        if (a.fx) fx_add(a, o, acc[tt]);
        else a.partials[(size_t)c * T * E + o] = acc[tt];
      }
    }
  }
  __syncthreads();   // s_x is dead; the routing below may reuse the memory
  if (!a.route_gu) route_if_last(a, layer_ptrs(a), smem_route);
}

// ---------------------------------------------------------------------------
// Routing shared by k_gateup and k_topk: logits from the partials (fixed
// order), top-k per token by warps, NaN flag.

// Partial logits were written by other CTAs of this kernel: global reads go
// through L2 (never a stale L1 line).
__device__ __forceinline__ float ld_part(const float *src, size_t i, bool staged) {
  return staged ? src[i] : __ldcg(src + i);
}

// Routing shared by k_gateup and k_topk: logits from this CTA's replica of the
// router partials (fixed summation order), block-parallel top-k, NaN flag and,
// if `publish`, the user-visible idx/gates and route counts.
__device__ void route_block(const Dec2Args &a, const LayerPtrs &lp, float *s_logits, float *s_sel,
                            int *s_idx, float *s_gates, float *s_vals, int *s_rank,
                            float *s_scratch, float *s_stage, bool publish) {
  const int T = a.T, E = a.E, k = a.k;
  const int TE = T * E;
  const int nthr = blockDim.x;
  const float *src = lp.partials;
  if (a.fx) {
    // fixed-point sums: read once and cleared for the next use
    for (int i = threadIdx.x; i < TE; i += nthr) {
      const long long v = __ldcg(a.fx_acc + i);
      const uint32_t f = __ldcg(a.fx_flag + i);
      s_logits[i] = f ? __int_as_float(0x7FC00000) : fx_to_float(v);
      a.fx_acc[i] = 0;
      a.fx_flag[i] = 0u;
    }
    __syncthreads();
    COLI_TRACE_POINT(a.layer, kTpRtLogits);
  } else if (s_stage) {
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
  const bool staged = s_stage != nullptr;
  int nsplit = a.fx ? 0 : nthr / TE;
  if (nsplit > 8) nsplit = 8;
  if (a.fx) {
    // logits already in shared memory
  } else if (nsplit <= 1) {
    for (int o = threadIdx.x; o < TE; o += nthr) {
      float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
      int p = 0;
      for (; p + 4 <= a.n_part; p += 4) {
        s0 += ld_part(src, (size_t)p * TE + o, staged);
        s1 += ld_part(src, (size_t)(p + 1) * TE + o, staged);
        s2 += ld_part(src, (size_t)(p + 2) * TE + o, staged);
        s3 += ld_part(src, (size_t)(p + 3) * TE + o, staged);
      }
      for (; p < a.n_part; ++p) s0 += ld_part(src, (size_t)p * TE + o, staged);
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
        s0 += ld_part(src, (size_t)p * TE + o, staged);
        s1 += ld_part(src, (size_t)(p + 1) * TE + o, staged);
      }
      if (p < p1) s0 += ld_part(src, (size_t)p * TE + o, staged);
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
  const bool sig = a.router_fn == COLI_ROUTER_SIGMOID_BIAS;
  if (sig) sigmoid_keys(s_logits, s_sel, a.router_bias, T, E);
  const bool nan = select_topk(sig ? s_sel : s_logits, T, E, k, s_idx, s_gates, s_vals, s_rank,
                               (int *)s_scratch);
  if (sig) sigmoid_gates(s_logits, s_idx, T, E, k, s_gates);
  COLI_TRACE_POINT(a.layer, kTpRtTopk);
  if (publish) {
    if (threadIdx.x == 0 && nan) set_flag(a.ctrl, COLI_FLAG_NAN_LOGITS);
    for (int i = threadIdx.x; i < T * k; i += nthr) {
      a.g_idx[i] = s_idx[i];
      a.g_gates[i] = s_gates[i];
      if (lp.route_counts) atomicAdd(lp.route_counts + COLI_CHK(s_idx[i], a.E, a.ctrl), 1u);
    }
  }
}

// Shared-memory layout of the routing CTA (byte offsets).
struct RouteSmem {
  size_t logits, sel, topk, idx, gates, vals, scratch, act, routes, slot_gate, total;
};
__host__ __device__ inline RouteSmem route_smem(int T, int E, int k, int S, int n_part, bool stage) {
  auto a16 = [](size_t v) { return (v + 15) & ~(size_t)15; };
  RouteSmem R{};
  size_t o = stage ? (size_t)n_part * T * E * 4 : 0;
  R.logits = a16(o); o = R.logits + (size_t)T * E * 4;
  R.sel = a16(o); o = R.sel + (size_t)T * E * 4;
  R.topk = a16(o);
  size_t tk = topk_scratch_bytes(T, E, k);
  if (tk < (size_t)T * k * 4) tk = (size_t)T * k * 4;       // the union's sort scratch
  o = R.topk + tk;
  R.idx = a16(o); o = R.idx + (size_t)T * k * 4;
  R.gates = o; o += (size_t)T * k * 4;
  R.vals = o; o += (size_t)T * k * 4;
  R.scratch = a16(o); o = R.scratch + (size_t)kDnMaxThreads * 4;   // one float per thread, any kernel
  R.act = o; o += (size_t)(2 + 2 * (E + S)) * 4;
  R.routes = o; o += (size_t)T * (k + S) * 4;
  R.slot_gate = o; o += (size_t)T * (k + S) * 4;
  R.total = a16(o);
  return R;
}

// Routing of one layer from its router partials, run by the last CTA of the
// kernel that produced them: logits (fixed summation order), top-k, gates,
// route counts, and the union lists the expert kernels read.  `smem` holds
// at least route_smem_bytes(a) bytes.
__device__ void route_finish(const Dec2Args &a, const LayerPtrs &lp, uint8_t *smem) {
  const int T = a.T, E = a.E, k = a.k, S = a.S, KS = k + S;
  const RouteSmem R = route_smem(T, E, k, S, a.n_part, a.stage_partials);
  float *s_stage = (float *)smem;
  float *s_logits = (float *)(smem + R.logits);
  int *s_rank = (int *)(smem + R.topk);
  int *s_idx = (int *)(smem + R.idx);
  float *s_gates = (float *)(smem + R.gates);
  float *s_vals = (float *)(smem + R.vals);
  float *s_scratch = (float *)(smem + R.scratch);
  route_block(a, lp, s_logits, (float *)(smem + R.sel), s_idx, s_gates, s_vals, s_rank, s_scratch,
              a.stage_partials ? s_stage : nullptr, true);
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    if (a.idx_out) a.idx_out[i] = s_idx[i];
    if (a.gates_out) a.gates_out[i] = s_gates[i];
  }
  COLI_TRACE_POINT(a.layer, kTpRtPublish);
  if (a.build_union) {
    int *s_act = (int *)(smem + R.act);
    int *s_routes = (int *)(smem + R.routes);
    float *s_slot_gate = (float *)(smem + R.slot_gate);
    block_union(s_idx, s_gates, T, k, S, E, s_act, s_act + 1, s_act + 1 + (E + S), s_routes,
                s_slot_gate, s_rank);
    for (int i = threadIdx.x; i < 2 + 2 * (E + S); i += blockDim.x) a.g_act[i] = s_act[i];
    for (int i = threadIdx.x; i < T * KS; i += blockDim.x) {
      a.g_routes[i] = s_routes[i];
      a.g_slot_gate[i] = s_slot_gate[i];
    }
    COLI_TRACE_POINT(a.layer, kTpRtUnion);
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
  COLI_TRACE_POINT(a.layer, kTpRouteStart);
  route_finish(a, lp, smem);
  if (threadIdx.x == 0) a.ctrl[kCtrlRouterTicket] = 0;
}

// ---------------------------------------------------------------------------
// gate/up (one token; several tokens: k_gateup_multi below): the CTA owns a
// contiguous range of rows in the flattened (used expert, f) space, after
// routing the layer itself (gu_lists); a row is gate row f and up row f of
// that expert.  Work is
// cut into tasks of (4-row group, 1024-column chunk).  Each warp runs its
// tasks (a round robin over the warps) through a private multi-stage
// cp.async pipeline, gu_slots - 1 tasks ahead: lane l copies the 16-byte
// slice of each of the 8 rows that it consumes, and the warp copies the 8
// rows' scales of the chunk, so tens of KB per SM stay in flight without
// holding registers.  Partial sums per (row, chunk) go to shared memory;
// rows are finalised in batches of gu_rows into h = silu(g) * u * gate,
// written to every replica.

// slot: weights [8 rows][32 lanes][16 B] | scales: [8 rows][16 groups] f32 when
// the row's scales are 16-byte aligned (K % 256 == 0), else [8 rows][32 lanes]
constexpr int kGuSlotWeights = 8 * 32 * 16;
__host__ __device__ constexpr int slot_bytes(int K) {
  return kGuSlotWeights + (K % 256 == 0 ? 8 * 16 * 4 : 8 * 32 * 4);
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    default: cp_async_wait<5>(); break;
  }
}

// Position of a warp's task in its row batch, stepped without divisions:
// task l = warp + i * NW is (4-row group g = l / ncg, chunk cg = l % ncg);
// the group's first row is expert ai, row f (f a multiple of 4).
struct GuTask {
  int g, cg, ai, f;
  __device__ __forceinline__ void init(int l, int ncg, int gr_base, int F) {
    g = l / ncg;
    cg = l - g * ncg;
    const int gr = gr_base + 4 * g;
    ai = gr / F;
    f = gr - ai * F;
  }
  __device__ __forceinline__ void next(int dg, int dcg, int ncg, int F) {
    int d = dg;
    cg += dcg;
    if (cg >= ncg) { cg -= ncg; ++d; }
    g += d;
    f += 4 * d;
    while (f >= F) { f -= F; ++ai; }
  }
};

// Issue the copies of one task into `slot`.
__device__ __forceinline__ void gu_copy(const Dec2Args &a, const LayerPtrs &lp,
                                        const int *s_act_expert, uint8_t *slot, const GuTask &k,
                                        bool vec_scales) {
  const int H = a.H, F = a.F, lane = threadIdx.x & 31;
  const int64_t rb = H / 2, ngr = H / kGroup;
  const int e = COLI_CHK(s_act_expert[k.ai], a.E + a.S, a.ctrl);
  const int col = k.cg * kChunkCols + 32 * lane;
  const uint8_t *pe;
  const float *se;
  expert_record(a.tier, lp.packed, lp.scales, a.eb, a.es, e, &pe, &se);
  const uint8_t *pg = pe + (int64_t)k.f * rb;
  const float *ps = se + (int64_t)k.f * ngr + k.cg * 16;
  float *ss = (float *)(slot + kGuSlotWeights);
  if (col < H) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      cp_async16(slot + ((2 * b) * 32 + lane) * 16, pg + b * rb + col / 2);
      cp_async16(slot + ((2 * b + 1) * 32 + lane) * 16, pg + (int64_t)F * rb + b * rb + col / 2);
    }
  }
  if (vec_scales) {
    // 16 groups of the chunk for 8 rows: lane l copies row l / 4, groups 4 (l % 4) .. + 3
    const int q = lane >> 2, b = q >> 1, m = q & 1, gq = 4 * (lane & 3);
    if (k.cg * 16 + gq < ngr)
      cp_async16(ss + q * 16 + gq, ps + (m ? (int64_t)F * ngr : 0) + b * ngr + gq);
  } else if (col < H) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      cp_async4(ss + (2 * b) * 32 + lane, ps + b * ngr + lane / 2);
      cp_async4(ss + (2 * b + 1) * 32 + lane, ps + (int64_t)F * ngr + b * ngr + lane / 2);
    }
  }
}

__device__ __forceinline__ void gu_slot_values(const uint8_t *slot, bool act, bool vec_scales,
                                               uint4 (&w)[8], float (&sc)[8]) {
  const int lane = threadIdx.x & 31;
  const float *ss = (const float *)(slot + kGuSlotWeights);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    w[q] = act ? *(const uint4 *)(slot + (q * 32 + lane) * 16) : make_uint4(0, 0, 0, 0);
    sc[q] = act ? (vec_scales ? ss[q * 16 + (lane >> 1)] : ss[q * 32 + lane]) : 0.0f;
  }
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


// The union lists of this layer in the gate/up CTA's shared memory: routed
// here from the fixed-point logits (every CTA alike, same integers, same
// result; CTA 0 also publishes the lists for the down kernel, the counts and
// the NaN flag), else loaded from the routing CTA's.  `scratch` is free
// shared memory (the pipeline ring, not yet in use).  Ends with __syncthreads.
__device__ void gu_lists(const Dec2Args &a, const LayerPtrs &lp, uint8_t *scratch, int *s_act,
                         int *s_routes, float *s_slot_gate) {
  if (!a.route_gu) {
    load_lists(a, s_act, s_routes, s_slot_gate);
    return;
  }
  const int T = a.T, E = a.E, k = a.k, S = a.S, KS = k + S, TE = T * E;
  const GuRouteSmem R = gu_route_smem(T, E, k);
  float *s_logits = (float *)(scratch + R.logits);
  int *s_idx = (int *)(scratch + R.idx);
  float *s_gates = (float *)(scratch + R.gates);
  bool late = false;
  for (int i = threadIdx.x; i < TE; i += blockDim.x) {
    if (a.gu_router) {
      // published whole by the owning CTAs (gu_router_logits): wait for the
      // word to become nonzero (bounded), then undo the sign flip
      const uint32_t *wp = (const uint32_t *)a.fx_rd_acc + i;
      uint32_t w = ld_acquire(wp);
      if (w == 0u) {
        const uint32_t lw = ld_acquire(a.ctrl + kCtrlWaitLimit);
        const long long limit = lw ? (long long)lw : kWaitCycles;
        const long long t0 = clock64();
        while ((w = ld_acquire(wp)) == 0u) {
          if (clock64() - t0 > limit) { late = true; break; }
          __nanosleep(32);
        }
      }
      s_logits[i] = __uint_as_float(w ^ 0x80000000u);
    } else {
      const long long v = __ldcg(a.fx_rd_acc + i);
      const uint32_t f = __ldcg(a.fx_rd_flag + i);
      s_logits[i] = f ? __int_as_float(0x7FC00000) : fx_to_float(v);
    }
  }
  if (late) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
  __syncthreads();
  COLI_TRACE_POINT(a.layer, kTpRtLogits);
  const bool sig = a.router_fn == COLI_ROUTER_SIGMOID_BIAS;
  float *s_keys = s_logits;
  if (sig) {
    s_keys = (float *)(scratch + R.sel);
    sigmoid_keys(s_logits, s_keys, a.router_bias ? (const float *)(scratch + R.bias) : nullptr,
                 T, E);
  }
  const bool nan = select_topk(s_keys, T, E, k, s_idx, s_gates, (float *)(scratch + R.vals),
                               scratch + R.topk, (int *)(scratch + R.flag));
  if (sig) sigmoid_gates(s_logits, s_idx, T, E, k, s_gates);
  COLI_TRACE_POINT(a.layer, kTpRtTopk);
  block_union(s_idx, s_gates, T, k, S, E, s_act, s_act + 1, s_act + 1 + (E + S), s_routes,
              s_slot_gate, (int *)(scratch + R.topk));
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0 && nan) set_flag(a.ctrl, COLI_FLAG_NAN_LOGITS);
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
      a.g_idx[i] = s_idx[i];
      a.g_gates[i] = s_gates[i];
      if (lp.route_counts) atomicAdd(lp.route_counts + COLI_CHK(s_idx[i], a.E, a.ctrl), 1u);
    }
    for (int i = threadIdx.x; i < 2 + 2 * (E + S); i += blockDim.x) a.g_act[i] = s_act[i];
    for (int i = threadIdx.x; i < T * KS; i += blockDim.x) {
      a.g_routes[i] = s_routes[i];
      a.g_slot_gate[i] = s_slot_gate[i];
    }
  }
  __syncthreads();
}

// The sigmoid router's bias does not depend on the previous kernel: the
// gate/up CTAs copy it into gu_lists' scratch before their dependency wait.
__device__ __forceinline__ void gu_bias_prefetch(const Dec2Args &a, uint8_t *scratch) {
  if (!a.route_gu || a.router_fn != COLI_ROUTER_SIGMOID_BIAS || !a.router_bias) return;
  float *s_bias = (float *)(scratch + gu_route_smem(a.T, a.E, a.k).bias);
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) s_bias[i] = __ldg(a.router_bias + i);
}

// First layer of a one-token call without a k_route launch.  CTA c of G owns
// the experts e = c, c + G, ... and forms their logits whole,
// l_e = sum_h Wr[e][h] x[h] in f32 (each thread its columns h = tid + i *
// blockDim in order, four experts' sums side by side, then a fixed reduction
// tree).  It publishes each as one 32-bit word over the layer's fixed-point
// buffer, which holds zeros at the start of the call (its down kernel clears
// it): the bits of l + 0 (so -0 becomes +0; a NaN becomes the quiet NaN) with
// the sign bit flipped, a word that is never zero.  Every CTA then waits for
// all E words to be nonzero (gu_lists), so no grid barrier is needed; the
// gate/up warps of this layer read x directly (no replicas).
// The owned router rows go to shared memory before the dependency wait (the
// weights do not depend on the previous kernel); x is read after it.
// Shared memory at `buf`: owned rows [ceil(E/G)][H] (router dtype), x f32
// [H], 32 x 4 floats of reduction scratch.
__device__ __forceinline__ uint32_t logit_word(float v) {
  v = v + 0.0f;
  return (v != v ? 0x7FC00000u : __float_as_uint(v)) ^ 0x80000000u;
}

__device__ __forceinline__ void gu_router_prefetch(const Dec2Args &a, uint8_t *buf) {
  const int E = a.E, G = gridDim.x, c = blockIdx.x;
  const int row16 = a.H * (a.wr_bf16 ? 2 : 4) / 16;       // H is a multiple of 64
  const uint8_t *wr = (const uint8_t *)a.wr;
  int n = 0;
  for (int e = c; e < E; e += G, ++n)
    for (int i = threadIdx.x; i < row16; i += blockDim.x)
      cp_async16(buf + ((size_t)n * row16 + i) * 16, wr + ((size_t)e * row16 + i) * 16);
  cp_async_commit();
}

template <typename WT>
__device__ __forceinline__ void router_dots4(const WT *w, int H, const float *s_x, int n,
                                             float (&sum)[4]) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int i = tid; i < H; i += nthr) {
    const float xv = s_x[i];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < n) sum[q] = fmaf(to_f32(w[(size_t)q * H + i]), xv, sum[q]);
  }
}

__device__ void gu_router_logits(const Dec2Args &a, uint8_t *buf) {
  const int E = a.E, H = a.H, G = gridDim.x, c = blockIdx.x;
  const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int nw = nthr >> 5;
  const int wsz = a.wr_bf16 ? 2 : 4;
  const int n_max = (E + G - 1) / G;
  const int n_own = c < E ? (E - c + G - 1) / G : 0;
  float *s_x = (float *)(buf + al16c((size_t)n_max * H * wsz));
  float *s_red = s_x + H;                        // [32][4]
  // x in groups of four elements, up to four 8- or 16-byte loads per thread in
  // flight before any is used (one memory round trip for H <= 16 blockDim)
  const int n4 = H / 4;
  for (int i0 = tid; i0 < n4; i0 += 4 * nthr) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * nthr;
      if (i >= n4) break;
      if (a.x_bf16) {
        const uint2 q = __ldcg((const uint2 *)a.x + i);
        v[u] = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                           __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u));
      } else {
        v[u] = __ldcg((const float4 *)a.x + i);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * nthr;
      if (i >= n4) break;
      ((float4 *)s_x)[i] = v[u];
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  COLI_TRACE_POINT(a.layer, kTpGuSplit);
  uint32_t *words = (uint32_t *)const_cast<long long *>(a.fx_rd_acc);
  for (int n0 = 0; n0 < n_own; n0 += 4) {
    const int n = n_own - n0 < 4 ? n_own - n0 : 4;
    float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (wsz == 2) router_dots4((const __nv_bfloat16 *)buf + (size_t)n0 * H, H, s_x, n, sum);
    else router_dots4((const float *)buf + (size_t)n0 * H, H, s_x, n, sum);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum[q] += __shfl_xor_sync(0xFFFFFFFFu, sum[q], off);
    }
    if (lane == 0)
#pragma unroll
      for (int q = 0; q < 4; ++q) s_red[warp * 4 + q] = sum[q];
    __syncthreads();
    if (tid < n) {
      float t = 0.0f;
      for (int w = 0; w < nw; ++w) t += s_red[w * 4 + tid];
      words[c + (n0 + tid) * G] = logit_word(t);
    }
    __syncthreads();
  }
  COLI_TRACE_POINT(a.layer, kTpGuNeed);
}

// The down kernel of a layer clears the fixed-point buffer that the layer's
// gate/up CTAs routed from (they have all finished): CTA c its share.
__device__ __forceinline__ void clear_fx(const Dec2Args &a) {
  if (!a.route_gu) return;
  const int TE = a.T * a.E, G = gridDim.x, c = blockIdx.x;
  const int i0 = part_lo(c, TE, G), i1 = part_lo(c + 1, TE, G);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    a.fx_clr_acc[i] = 0;
    a.fx_clr_flag[i] = 0u;
  }
}


// One token per call: every used expert serves token 0, each warp quantises
// the 1024-column slice of x that its chunk needs once (kept in registers),
// and there is no token loop.
// kFast: H a multiple of 1024 (every lane of every chunk active, 16-byte
// aligned scale rows), checks folded away.
// At most 12 warps (the plan's choices), so the compiler may use up to 168 registers.
constexpr int kGuOneMaxThreads = 384;

template <bool kFast>
__global__ void __launch_bounds__(kGuOneMaxThreads) k_gateup(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GuSmem &L = a.gu;
  COLI_TRACE_POINT(a.layer, kTpGuEntry);
  int *s_act = (int *)(smem + L.act);
  int *s_routes = (int *)(smem + L.routes);
  float *s_slot_gate = (float *)(smem + L.slot_gate);
  float *red = (float *)(smem + L.red);
  gu_bias_prefetch(a, smem + L.ring);
  if (a.gu_router) gu_router_prefetch(a, smem + L.ring + a.gu_rt_off);
  grid_dependents_launch();
  grid_dependency_wait();
  COLI_TRACE_POINT(a.layer, kTpGuDepWait);
  const LayerPtrs lp = layer_ptrs(a);
  if (a.gu_router) gu_router_logits(a, smem + L.ring + a.gu_rt_off);
  gu_lists(a, lp, smem + L.ring, s_act, s_routes, s_slot_gate);   // ends with __syncthreads
  COLI_TRACE_POINT(a.layer, kTpGuLists);
  const int H = a.H, F = a.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, NW = blockDim.x >> 5;
  const int n_active = s_act[0];
  const int *s_act_expert = s_act + 1;
  const int *s_act_off = s_act + 1 + (a.E + a.S);
  const int G = gridDim.x, c = blockIdx.x;
  const int U = n_active * (F / 4);
  const int row0 = 4 * part_lo(c, U, G), nrows = 4 * part_lo(c + 1, U, G) - row0;
  const float *xr = lp.xrep + (size_t)(c % a.n_rep) * a.x_stride;
  // with the router formed here (first layer), x comes from the caller's input
  const bool x_direct = a.gu_router != 0;
  const int ncg = a.gu_ncg, S = a.gu_slots;
  const int dg = NW / ncg, dcg = NW - dg * ncg;
  const bool vec_scales = kFast || (H % 256) == 0;
  const int SB = a.gu_slot_bytes;
  uint8_t *ring = smem + L.ring + (size_t)warp * S * SB;

  for (int rb0 = 0; rb0 < nrows; rb0 += a.gu_rows) {
    const int nrb = nrows - rb0 < a.gu_rows ? nrows - rb0 : a.gu_rows;
    const int n_tasks = (nrb / 4) * ncg;
    const int my_tasks = n_tasks > warp ? (n_tasks - warp + NW - 1) / NW : 0;
    GuTask ci, cc;      // the next task to copy, the next task to compute
    ci.init(warp, ncg, row0 + rb0, F);
    cc = ci;
    if (rb0 == 0) COLI_TRACE_POINT(a.layer, kTpGuPlanes);
    // prologue: the first S - 1 tasks of this warp in flight
    for (int p = 0; p < S - 1; ++p) {
      if (p < my_tasks) {
        gu_copy(a, lp, s_act_expert, ring + (size_t)p * SB, ci, vec_scales);
        ci.next(dg, dcg, ncg, F);
      }
      cp_async_commit();
    }
    if (rb0 == 0) COLI_TRACE_POINT(a.layer, kTpGuFirstLoads);
    Planes pl;
    int pl_cg = -1;             // chunk whose planes are in `pl`
    int ld = S - 1, cs = 0;     // ring slots of the next copy / the next compute
    for (int i = 0; i < my_tasks; ++i) {
      if (i + S - 1 < my_tasks) {
        gu_copy(a, lp, s_act_expert, ring + (size_t)ld * SB, ci, vec_scales);
        ci.next(dg, dcg, ncg, F);
      }
      if (++ld == S) ld = 0;
      cp_async_commit();
      cp_async_wait_dyn(S - 1);      // this lane's copies of task i have landed
      if (vec_scales) __syncwarp();  // scales were copied by other lanes
      const uint8_t *slot = ring + (size_t)cs * SB;
      if (++cs == S) cs = 0;
      const int col = cc.cg * kChunkCols + 32 * lane;
      const bool act = kFast || col < H;
      uint4 w[8];
      float sc[8];
      gu_slot_values(slot, act, vec_scales, w, sc);
      float v[8];
      if (act) {
        if (cc.cg != pl_cg) {
          float xv[32];
          if (!x_direct) load32<float>(xr + col, xv);
          else if (a.x_bf16) load32<__nv_bfloat16>((const __nv_bfloat16 *)a.x + col, xv);
          else load32<float>((const float *)a.x + col, xv);
          quantize32(xv, pl);
          pl_cg = cc.cg;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = sc[q] * dot32(w[q], pl);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.0f;
      }
      const float tot = reduce8(v);    // lane 4 vi: value vi = 2 * row + (0 gate | 1 up)
      if ((lane & 3) == 0) {
        const int vi = lane >> 2;
        red[((4 * cc.g + (vi >> 1)) * ncg + cc.cg) * 2 + (vi & 1)] = tot;
      }
      __syncwarp();                  // the slot is refilled by the next iteration's copy
      cc.next(dg, dcg, ncg, F);
    }
    cp_async_wait<0>();
    __syncthreads();
    if (rb0 == 0) COLI_TRACE_POINT(a.layer, kTpGuCompute);
    // finalise h for every row of this batch
    for (int i = tid; i < nrb; i += blockDim.x) {
      const int gr = row0 + rb0 + i;
      const int ai = gr / F, f = gr - ai * F;
      float gs = 0.0f, us = 0.0f;
      for (int q = 0; q < ncg; ++q) {
        gs += red[(i * ncg + q) * 2];
        us += red[(i * ncg + q) * 2 + 1];
      }
      const int slot_id = COLI_CHK(s_routes[s_act_off[ai]], a.T * (a.k + a.S), a.ctrl);
      const float hv = silu(gs) * us * s_slot_gate[slot_id];
      for (int rr = 0; rr < a.n_rep; ++rr) a.h[rr * a.h_stride + (int64_t)slot_id * F + f] = hv;
    }
    __syncthreads();
  }
  COLI_TRACE_POINT(a.layer, kTpGuEnd);
}

// Several tokens per call.  A used expert serving nt tokens costs more per
// row than one serving a single token (the shared expert serves all of them),
// so the (used expert, 4-row group) space is split over the CTAs by cost,
// 1 + 2 nt units per group, not by rows.  A warp owns whole groups: it runs
// their chunks in order through its pipeline, adds each chunk's partial sums
// per (token, row) in its own shared-memory accumulator, and after the last
// chunk writes h = silu(g) * u * gate for the group's rows.  The CTA quantises
// only the tokens its experts serve (into shared memory when they fit, else
// per task in registers).
// The (used expert, group) space split by cost: a group of an expert that
// serves nt tokens costs 1 + 2 nt units; CTA c of G gets the groups [u0, u1)
// whose cost prefix starts in [c C / G, (c + 1) C / G), C the total.  Warp 0
// scans the experts 32 at a time and leaves the bounds in s_u (2 ints); all
// threads read them after the barrier.
__device__ void cost_split(const int *s_act_off, int n_active, int gpe, int c, int G, int *s_u,
                           int *u0, int *u1) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    long long total = 0;
    for (int a0 = 0; a0 < n_active; a0 += 32) {
      const int ai = a0 + lane;
      const long long span =
          ai < n_active ? (1 + 2LL * (s_act_off[ai + 1] - s_act_off[ai])) * gpe : 0;
      total += span;   // per-lane partial, reduced below
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xFFFFFFFFu, total, off);
    // first group whose cost prefix reaches b, for the two bounds
    for (int k = 0; k < 2; ++k) {
      const long long b = total * (c + k) / G;
      long long before = 0;
      int u = n_active * gpe;
      for (int a0 = 0; a0 < n_active; a0 += 32) {
        const int ai = a0 + lane;
        const long long w = ai < n_active ? 1 + 2LL * (s_act_off[ai + 1] - s_act_off[ai]) : 0;
        long long incl = w * gpe;   // inclusive scan of the spans over the lanes
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const long long o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
          if (lane >= off) incl += o;
        }
        const long long excl = before + incl - w * gpe;
        const bool hit = ai < n_active && b < before + incl;
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, hit);
        if (m) {
          const int src = __ffs(m) - 1;
          const long long e_b = __shfl_sync(0xFFFFFFFFu, excl, src);
          const long long w_b = __shfl_sync(0xFFFFFFFFu, w, src);
          u = (a0 + src) * gpe + (int)((b - e_b + w_b - 1) / w_b);
          break;
        }
        before += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      if (lane == 0) s_u[k] = u;
    }
  }
  __syncthreads();
  *u0 = s_u[0];
  *u1 = s_u[1];
}

struct MTask {
  int u, cg, ai, f;   // 4-row group (flattened), chunk, used expert, first row
  __device__ __forceinline__ void set(int u_, int gpe) {
    u = u_;
    cg = 0;
    ai = u / gpe;
    f = 4 * (u - ai * gpe);
  }
  __device__ __forceinline__ void next(int NW, int ncg, int gpe) {
    if (++cg == ncg) set(u + NW, gpe);
  }
  __device__ __forceinline__ GuTask gu() const { return GuTask{0, cg, ai, f}; }
};

// At most 8 warps: the task loop then keeps its state in registers (no spills).
constexpr int kGuMultiMaxThreads = 256;

template <bool kFast, bool kXpl>
__global__ void __launch_bounds__(kGuMultiMaxThreads) k_gateup_multi(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GuSmem &L = a.gu;
  COLI_TRACE_POINT(a.layer, kTpGuEntry);
  int *s_act = (int *)(smem + L.act);
  int *s_routes = (int *)(smem + L.routes);
  float *s_slot_gate = (float *)(smem + L.slot_gate);
  int *s_tok = (int *)(smem + L.tok);            // [T] needed tokens, then [T] token -> plane
  uint32_t *s_xpl = (uint32_t *)(smem + L.xpl);  // the needed tokens' planes, then the ring
  gu_bias_prefetch(a, smem + L.xpl);
  grid_dependents_launch();
  grid_dependency_wait();
  COLI_TRACE_POINT(a.layer, kTpGuDepWait);
  const LayerPtrs lp = layer_ptrs(a);
  gu_lists(a, lp, smem + L.xpl, s_act, s_routes, s_slot_gate);   // ends with __syncthreads
  COLI_TRACE_POINT(a.layer, kTpGuLists);
  const int T = a.T, H = a.H, F = a.F, KS = a.k + a.S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, NW = blockDim.x >> 5;
  const int n_active = s_act[0];
  const int *s_act_expert = s_act + 1;
  const int *s_act_off = s_act + 1 + (a.E + a.S);
  const int G = gridDim.x, c = blockIdx.x;
  const int gpe = F / 4;
  int u0, u1;
  cost_split(s_act_off, n_active, gpe, c, G, (int *)(smem + L.tok) + 2 * T + 1, &u0, &u1);
  COLI_TRACE_POINT(a.layer, kTpGuSplit);
  const float *xr = lp.xrep + (size_t)(c % a.n_rep) * a.x_stride;
  // with the router formed here (first layer), x comes from the caller's input
  const bool x_direct = a.gu_router != 0;
  const int ncg = a.gu_ncg, nbx = H / 32;
  const bool vec_scales = kFast || (H % 256) == 0;
  const bool xpl = kXpl;   // a.gu_xpl
  const int SB = a.gu_slot_bytes;
  float *acc = (float *)(smem + L.red) + (size_t)warp * T * 8;   // [T][8] of this warp
  int n_need = 0;

  // the tokens that the experts of groups [u0, u1) serve, in token order
  if (u1 > u0 && xpl) {
    if (warp == 0) {
      const int r0 = s_act_off[u0 / gpe], r1 = s_act_off[(u1 - 1) / gpe + 1];
      uint32_t need = 0;
      for (int r = r0 + lane; r < r1; r += 32) need |= 1u << (COLI_CHK(s_routes[r], T * KS, a.ctrl) / KS);
      need = __reduce_or_sync(0xFFFFFFFFu, need);
      if (lane < T) {
        const bool mine = (need >> lane) & 1u;
        const int pos = __popc(need & ((1u << lane) - 1u));
        if (mine) s_tok[pos] = lane;
        s_tok[T + lane] = mine ? pos : -1;
      }
      if (lane == 0) s_tok[2 * T] = __popc(need);
    }
    __syncthreads();
    COLI_TRACE_POINT(a.layer, kTpGuNeed);
    n_need = s_tok[2 * T];
    build_planes_impl(xr, n_need, H, s_tok, s_xpl, nbx, warp, NW);
    __syncthreads();
  }
  COLI_TRACE_POINT(a.layer, kTpGuPlanes);
  // the ring after this CTA's planes, as deep as the rest of shared memory allows
  const size_t ring_off = (L.xpl + (size_t)n_need * 18 * nbx * 4 + 127) & ~(size_t)127;
  int S = (int)((L.total - ring_off) / ((size_t)NW * SB));
  S = S < a.gu_slots ? S : a.gu_slots;
  uint8_t *ring = smem + ring_off + (size_t)warp * S * SB;

  const int n_groups = u1 - u0;
  const int my_groups = n_groups > warp ? (n_groups - warp + NW - 1) / NW : 0;
  const int my_tasks = my_groups * ncg;
  MTask ci, cc;
  ci.set(u0 + warp, gpe);
  cc = ci;
  for (int p = 0; p < S - 1; ++p) {
    if (p < my_tasks) {
      gu_copy(a, lp, s_act_expert, ring + (size_t)p * SB, ci.gu(), vec_scales);
      ci.next(NW, ncg, gpe);
    }
    cp_async_commit();
  }
  COLI_TRACE_POINT(a.layer, kTpGuFirstLoads);
  Planes pl;
  int pl_key = -1;            // (token, chunk) whose planes are in `pl`
  int ld = S - 1, cs = 0;     // ring slots of the next copy / the next compute
  for (int i = 0; i < my_tasks; ++i) {
    if (i + S - 1 < my_tasks) {
      gu_copy(a, lp, s_act_expert, ring + (size_t)ld * SB, ci.gu(), vec_scales);
      ci.next(NW, ncg, gpe);
    }
    if (++ld == S) ld = 0;
    cp_async_commit();
    cp_async_wait_dyn(S - 1);
    if (vec_scales) __syncwarp();
    const uint8_t *slot = ring + (size_t)cs * SB;
    if (++cs == S) cs = 0;
    const int col = cc.cg * kChunkCols + 32 * lane;
    const bool act = kFast || col < H;
    uint4 w[8];
    float sc[8];
    gu_slot_values(slot, act, vec_scales, w, sc);
    const int j0 = s_act_off[cc.ai], nt = s_act_off[cc.ai + 1] - j0;
    for (int j = 0; j < nt; ++j) {
      const int t = COLI_CHK(s_routes[j0 + j], T * KS, a.ctrl) / KS;
      float v[8];
      if (act) {
        const int key = t * ncg + cc.cg;
        if (key != pl_key) {
          if (xpl) {
            load_planes(s_xpl, s_tok[T + t], col / 32, nbx, pl);
          } else {
            float xv[32];
            load32<float>(xr + (int64_t)t * H + col, xv);
            quantize32(xv, pl);
          }
          pl_key = key;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = sc[q] * dot32(w[q], pl);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.0f;
      }
      const float tot = reduce8(v);    // lane 4 vi: value vi = 2 * row + (0 gate | 1 up)
      if ((lane & 3) == 0) {
        float *p = acc + j * 8 + (lane >> 2);
        *p = (cc.cg == 0 ? 0.0f : *p) + tot;   // chunks added in order
      }
    }
    if (cc.cg == ncg - 1) {
      __syncwarp();
      for (int it = lane; it < 4 * nt; it += 32) {
        const int j = it >> 2, r = it & 3;
        const float gs = acc[j * 8 + 2 * r], us = acc[j * 8 + 2 * r + 1];
        const int slot_id = COLI_CHK(s_routes[j0 + j], T * KS, a.ctrl);
        const float hv = silu(gs) * us * s_slot_gate[slot_id];
        for (int rr = 0; rr < a.n_rep; ++rr)
          a.h[rr * a.h_stride + (int64_t)slot_id * F + cc.f + r] = hv;
      }
    }
    __syncwarp();                  // the slot (and the accumulator) are reused next
    cc.next(NW, ncg, gpe);
  }
  cp_async_wait<0>();
  COLI_TRACE_POINT(a.layer, kTpGuEnd);
}

// ---------------------------------------------------------------------------
// down: each CTA owns output rows [dh0, dh1) (one token: of every used
// expert's down matrix).  Work is cut into tasks of (expert, 8-row group,
// 1024-column chunk) that run, like the gate/up tasks, through each warp's
// cp.async pipeline (the same slot layout: 8 rows x 16 bytes per lane, plus
// scales); each warp takes a contiguous run of tasks and quantises the h slice
// of its task's expert in registers.  A task leaves the partial sum of each
// (row, chunk) in shared memory, and every row then adds its experts' and
// chunks' partial sums in a fixed order.  With several tokens k_down_multi
// has already produced the per-slot outputs y and this kernel only adds each
// token's slots.  The combine then writes out (with the residual), layer_out,
// the x replicas, and leaves the new residual-stream rows in s_xn [T][nr].

struct DnTask {
  int a, gi, cg;     // expert (index into the used list), 8-row group, chunk
};

__device__ __forceinline__ void dn_copy(const Dec2Args &a, const LayerPtrs &lp,
                                        const int *s_act_expert, uint8_t *slot, const DnTask &k,
                                        int dh0, int nr, bool vec_scales) {
  const int H = a.H, F = a.F, lane = threadIdx.x & 31;
  const int64_t rb = F / 2, ngr = F / kGroup;
  const int e = COLI_CHK(s_act_expert[k.a], a.E + a.S, a.ctrl);
  const int col = k.cg * kChunkCols + 32 * lane;
  const int r0 = 8 * k.gi, nq = nr - r0 < 8 ? nr - r0 : 8;
  const uint8_t *pe;
  const float *se;
  expert_record(a.tier, lp.packed, lp.scales, a.eb, a.es, e, &pe, &se);
  const uint8_t *pw = pe + (int64_t)F * H + (int64_t)(dh0 + r0) * rb;
  const float *ps = se + (int64_t)2 * F * (H / kGroup) + (int64_t)(dh0 + r0) * ngr + k.cg * 16;
  float *ss = (float *)(slot + kGuSlotWeights);
  if (col < F) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < nq) cp_async16(slot + (q * 32 + lane) * 16, pw + q * rb + col / 2);
  }
  if (vec_scales) {
    const int q = lane >> 2, gq = 4 * (lane & 3);
    if (q < nq && k.cg * 16 + gq < ngr) cp_async16(ss + q * 16 + gq, ps + q * ngr + gq);
  } else if (col < F) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < nq) cp_async4(ss + q * 32 + lane, ps + q * ngr + lane / 2);
  }
}

// A warp's run of one-token down tasks in (expert, chunk, 8-row group) order.
struct DnSeq {
  int a, cg, gi;
  __device__ __forceinline__ void init(int l, int ncg, int gpe) {
    gi = l % gpe;
    const int u = l / gpe;
    cg = u % ncg;
    a = u / ncg;
  }
  __device__ __forceinline__ void next(int ncg, int gpe) {
    if (++gi == gpe) {
      gi = 0;
      if (++cg == ncg) { cg = 0; ++a; }
    }
  }
  __device__ __forceinline__ DnTask task() const { return DnTask{a, gi, cg}; }
};

template <bool kOne, bool kFast>
__device__ void dn_phase(const Dec2Args &a, const LayerPtrs &lp, const int *s_act,
                         const int *s_routes, uint8_t *smem, float *s_xn, const float *residual) {
  const DnSmem &L = a.dn;
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, KS = a.k + S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, NW = blockDim.x >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int UH = H / 4;
  const int dh0 = 4 * part_lo(c, UH, G), dh1 = 4 * part_lo(c + 1, UH, G);
  const int nr = dh1 - dh0;
  float *acc = (float *)(smem + L.acc);          // [nr][T]
  if (!kOne) {
    // several tokens: k_down_multi left each slot's down output in y; a
    // token's rows add its slots in slot order (routed by rank, then shared)
    for (int i = tid; i < nr * T; i += blockDim.x) {
      const int t = i / nr, r = i - t * nr;
      float sum = 0.0f;
      for (int p = 0; p < KS; ++p) sum += __ldcg(a.y + (size_t)(t * KS + p) * H + dh0 + r);
      acc[r * T + t] = sum;
    }
    __syncthreads();
  } else {
    // one token: every used expert's (8-row group, chunk) tasks at once; a
    // warp quantises the h slice of a task's expert in registers when the
    // (expert, chunk) changes, so no block-wide plane build precedes the work
    const int *s_act_expert = s_act + 1;
    const int *s_act_off = s_act + 1 + (E + S);
    const int n_active = s_act[0];
    const float *h_rep = a.h + (size_t)(c % a.n_rep) * a.h_stride;
    const int ncg = a.dn_ncg, Sl = a.dn_slots_pipe;
    const int gpe = (nr + 7) / 8;                  // 8-row groups per expert
    const bool vec_scales = kFast || (F % 256) == 0;
    float *red = (float *)(smem + L.red);          // [expert][nr][ncg]
    const int SB = a.dn_slot_bytes;
    uint8_t *ring = smem + L.ring + (size_t)warp * Sl * SB;
    // warp w takes tasks [l0, l1) in (expert, chunk, group) order, so its
    // consecutive tasks share the expert's h slice
    const int n_tasks = n_active * gpe * ncg;
    const int l0 = part_lo(warp, n_tasks, NW);
    const int my_tasks = part_lo(warp + 1, n_tasks, NW) - l0;
    DnSeq ci, cc;
    ci.init(l0, ncg, gpe);
    cc = ci;
    COLI_TRACE_POINT(a.layer, kTpDnPlanes);
    for (int p = 0; p < Sl - 1; ++p) {
      if (p < my_tasks) {
        dn_copy(a, lp, s_act_expert, ring + (size_t)p * SB, ci.task(), dh0, nr, vec_scales);
        ci.next(ncg, gpe);
      }
      cp_async_commit();
    }
    Planes pl;
    int pl_key = -1;
    int ld = Sl - 1, cs = 0;    // ring slots of the next copy / the next compute
    for (int i = 0; i < my_tasks; ++i) {
      if (i + Sl - 1 < my_tasks) {
        dn_copy(a, lp, s_act_expert, ring + (size_t)ld * SB, ci.task(), dh0, nr, vec_scales);
        ci.next(ncg, gpe);
      }
      if (++ld == Sl) ld = 0;
      cp_async_commit();
      const int col = cc.cg * kChunkCols + 32 * lane;
      const bool act = kFast || col < F;
      const int key = cc.a * 64 + cc.cg;
      if (act && key != pl_key) {
        // the h loads go out before this task's weights are waited for
        float xv[32];
        load32<float>(h_rep + (int64_t)COLI_CHK(s_routes[s_act_off[cc.a]], T * KS, a.ctrl) * F + col,
                      xv);
        quantize32(xv, pl);
        pl_key = key;
      }
      cp_async_wait_dyn(Sl - 1);
      if (vec_scales) __syncwarp();
      const uint8_t *slot = ring + (size_t)cs * SB;
      if (++cs == Sl) cs = 0;
      const int r0 = 8 * cc.gi, nq = nr - r0 < 8 ? nr - r0 : 8;
      uint4 w[8];
      float sc[8];
      gu_slot_values(slot, act, vec_scales, w, sc);
      float v[8];
      if (act) {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = q < nq ? sc[q] * dot32(w[q], pl) : 0.0f;
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.0f;
      }
      const float tot = reduce8(v);   // lane 4 q ends with row q
      if ((lane & 3) == 0) {
        const int q = lane >> 2;
        if (q < nq) red[(cc.a * nr + r0 + q) * ncg + cc.cg] = tot;
      }
      __syncwarp();
      cc.next(ncg, gpe);
    }
    cp_async_wait<0>();
    __syncthreads();
    // every row adds its experts' and chunks' partial sums in a fixed order
    for (int r = tid; r < nr; r += blockDim.x) {
      float sum = 0.0f;
      for (int x = 0; x < n_active; ++x)
        for (int q = 0; q < ncg; ++q) sum += red[(x * nr + r) * ncg + q];
      acc[r] = sum;
    }
    __syncthreads();
  }
  COLI_TRACE_POINT(a.layer, kTpDnCompute);
  // combine is complete: residual, outputs, replicas of the new layer input
  for (int i = tid; i < T * nr; i += blockDim.x) {
    const int t = i / nr, r = i - t * nr;
    const int64_t o = (int64_t)t * H + dh0 + r;
    const float v = acc[r * T + t];
    if (lp.layer_out) lp.layer_out[o] = v;
    const float xn = residual ? residual[o] + v : v;
    lp.out[o] = xn;
    s_xn[i] = xn;
    if (lp.xrep)
      for (int rr = 0; rr < a.n_rep; ++rr) lp.xrep[rr * a.x_stride + o] = xn;
  }
  __syncthreads();
}


template <typename WT, bool kOne, bool kFast>
__global__ void __launch_bounds__(kOne ? kDnMaxThreads : kDec2MaxThreads) k_down(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DnSmem &L = a.dn;
  WT *s_wr = (WT *)(smem + L.wr);
  COLI_TRACE_POINT(a.layer, kTpDnEntry);
  // the next layer's router rows do not depend on the previous kernel
  if (a.wr) load_router_rows<WT>(a, (const WT *)a.wr, s_wr);
  grid_dependents_launch();
  grid_dependency_wait();
  COLI_TRACE_POINT(a.layer, kTpDnDepWait);
  clear_fx(a);
  int *s_act = (int *)(smem + L.act);
  int *s_routes = (int *)(smem + L.routes);
  load_lists(a, s_act, s_routes, nullptr);
  COLI_TRACE_POINT(a.layer, kTpDnLists);
  float *s_xn = (float *)(smem + L.xn);
  const LayerPtrs lp = layer_ptrs(a);
  dn_phase<kOne, kFast>(a, lp, s_act, s_routes, smem, s_xn, a.residual);
  COLI_TRACE_POINT(a.layer, kTpDnCombine);
  if (a.wr) {
    if (a.fx) dn_partials_fx<WT>(a, s_wr, s_xn);
    else dn_partials<WT>(a, a.partials, s_wr, s_xn, 1, 0);
    COLI_TRACE_POINT(a.layer, kTpDnPartials);
    // without fixed-point logits the last CTA routes the next layer (its
    // shared memory is free again); with them the next gate/up does
    if (!a.route_gu) {
      LayerPtrs rp = lp;
      rp.route_counts = a.next_counts;
      route_if_last(a, rp, smem);
    }
  }
  COLI_TRACE_POINT(a.layer, kTpEnd);
}

// The task loop of k_down_multi, compiled apart for planes in shared memory
// (kXpl) and for planes quantised per task, so that the common case does not
// carry the fallback's registers.
template <bool kFast, bool kXpl>
__device__ __forceinline__ void dm_loop(const Dec2Args &a, const LayerPtrs &lp,
                                        const int *s_act_expert, const int *s_act_off,
                                        const int *s_routes, const uint32_t *s_planes,
                                        const float *h_rep, int u0, int u1, int r0,
                                        uint8_t *ring, float *acc) {
  const int H = a.H, F = a.F;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, NW = blockDim.x >> 5;
  const int gpe = H / 8;
  const int ncg = a.dn_ncg, Sl = a.dm_slots_pipe, nbp = F / 32;
  const bool vec_scales = kFast || (F % 256) == 0;
  const int SB = a.dn_slot_bytes;
  const int n_groups = u1 - u0;
  const int my_groups = n_groups > warp ? (n_groups - warp + NW - 1) / NW : 0;
  const int my_tasks = my_groups * ncg;
  // task: group u (expert u / gpe, rows 8 (u % gpe) ..), chunk cg
  int ci_u = u0 + warp, ci_cg = 0, cc_u = ci_u, cc_cg = 0;
  auto task = [&](int u, int cg) { return DnTask{u / gpe, u - (u / gpe) * gpe, cg}; };
  for (int p = 0; p < Sl - 1; ++p) {
    if (p < my_tasks) {
      dn_copy(a, lp, s_act_expert, ring + (size_t)p * SB, task(ci_u, ci_cg), 0, H, vec_scales);
      if (++ci_cg == ncg) { ci_cg = 0; ci_u += NW; }
    }
    cp_async_commit();
  }
  Planes pl;
  int pl_key = -1;
  int ld = Sl - 1, cs = 0;    // ring slots of the next copy / the next compute
  for (int i = 0; i < my_tasks; ++i) {
    if (i + Sl - 1 < my_tasks) {
      dn_copy(a, lp, s_act_expert, ring + (size_t)ld * SB, task(ci_u, ci_cg), 0, H, vec_scales);
      if (++ci_cg == ncg) { ci_cg = 0; ci_u += NW; }
    }
    if (++ld == Sl) ld = 0;
    cp_async_commit();
    cp_async_wait_dyn(Sl - 1);
    if (vec_scales) __syncwarp();
    const uint8_t *slot = ring + (size_t)cs * SB;
    if (++cs == Sl) cs = 0;
    const int col = cc_cg * kChunkCols + 32 * lane;
    const bool act = kFast || col < F;
    uint4 w[8];
    float sc[8];
    gu_slot_values(slot, act, vec_scales, w, sc);
    const int ai = cc_u / gpe, row0 = 8 * (cc_u - ai * gpe);
    const int j0 = s_act_off[ai], nt = s_act_off[ai + 1] - j0;
    for (int j = 0; j < nt; ++j) {
      float v[8];
      if (act) {
        const int key = (j0 + j) * 64 + cc_cg;
        if (key != pl_key) {
          if (kXpl) {
            load_planes(s_planes, j0 + j - r0, col / 32, nbp, pl);
          } else {
            float xv[32];
            load32<float>(h_rep + (int64_t)COLI_CHK(s_routes[j0 + j], a.T * (a.k + a.S), a.ctrl) * F + col, xv);
            quantize32(xv, pl);
          }
          pl_key = key;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = sc[q] * dot32(w[q], pl);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.0f;
      }
      const float tot = reduce8(v);   // lane 4 q ends with row q
      if ((lane & 3) == 0) {
        float *p = acc + j * 8 + (lane >> 2);
        *p = (cc_cg == 0 ? 0.0f : *p) + tot;   // chunks added in order
      }
    }
    if (cc_cg == ncg - 1) {
      __syncwarp();
      for (int it = lane; it < 8 * nt; it += 32) {
        const int j = it >> 3, q = it & 7;
        a.y[(size_t)COLI_CHK(s_routes[j0 + j], a.T * (a.k + a.S), a.ctrl) * H + row0 + q] = acc[j * 8 + q];
      }
    }
    __syncwarp();
    if (++cc_cg == ncg) { cc_cg = 0; cc_u += NW; }
  }
  cp_async_wait<0>();
}

// Down GEMVs of a several-token call, split like k_gateup_multi: the (used
// expert, 8-row group) space goes to the CTAs by cost (1 + 2 nt units per
// group); a warp owns whole groups, runs their chunks in order, and after the
// last one writes y[slot][row] = sum_f down[row][f] h[slot][f] for each token
// slot of the expert.  The CTA's slots' h rows are quantised once into shared
// memory when they fit (else per task in registers).  k_down then adds each
// token's slots.
template <bool kFast>
__global__ void __launch_bounds__(kDec2MaxThreads) k_down_multi(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const DmSmem &L = a.dm;
  int *s_act = (int *)(smem + L.act);
  int *s_routes = (int *)(smem + L.routes);
  uint32_t *s_planes = (uint32_t *)(smem + L.planes);
  grid_dependents_launch();
  grid_dependency_wait();
  load_lists(a, s_act, s_routes, nullptr);   // ends with __syncthreads
  const LayerPtrs lp = layer_ptrs(a);
  const int H = a.H, F = a.F, T = a.T;
  const int warp = threadIdx.x >> 5;
  const int n_active = s_act[0];
  const int *s_act_expert = s_act + 1;
  const int *s_act_off = s_act + 1 + (a.E + a.S);
  const int G = gridDim.x, c = blockIdx.x;
  const int gpe = H / 8;
  int u0, u1;
  cost_split(s_act_off, n_active, gpe, c, G, (int *)(smem + L.u), &u0, &u1);
  const float *h_rep = a.h + (size_t)(c % a.n_rep) * a.h_stride;
  const int Sl = a.dm_slots_pipe, nbp = F / 32;
  const int SB = a.dn_slot_bytes;
  uint8_t *ring = smem + L.ring + (size_t)warp * Sl * SB;
  float *acc = (float *)(smem + L.acc) + (size_t)warp * T * 8;   // [T][8] of this warp
  // h rows (slots) of the experts of groups [u0, u1): routes [r0, r1)
  const int r0 = u1 > u0 ? s_act_off[u0 / gpe] : 0;
  const int r1 = u1 > u0 ? s_act_off[(u1 - 1) / gpe + 1] : 0;
  const bool xpl = r1 - r0 <= a.dm_cap;
  if (u1 > u0 && xpl) {
    build_planes_list(h_rep, F, s_routes + r0, r1 - r0, s_planes, nbp);
    __syncthreads();
  }
  if (xpl) {
    dm_loop<kFast, true>(a, lp, s_act_expert, s_act_off, s_routes, s_planes, h_rep, u0, u1, r0,
                         ring, acc);
  } else {
    dm_loop<kFast, false>(a, lp, s_act_expert, s_act_off, s_routes, s_planes, h_rep, u0, u1, r0,
                          ring, acc);
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// host side

#ifdef COLI_TRACE
extern "C" int coli_trace_reset() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_trace) != cudaSuccess) return -1;
  return cudaMemset(p, 0, sizeof(g_trace)) == cudaSuccess ? 0 : -1;
}
// [layer][point][cta] timestamps (0: not reached).
extern "C" int coli_trace_read_raw(void *buf) {
  return cudaMemcpyFromSymbol(buf, g_trace, sizeof(g_trace)) == cudaSuccess ? 0 : -1;
}
// Earliest / latest timestamp per [layer][point] over the CTAs that reached it.
extern "C" int coli_trace_read(void *lo, void *hi) {
  static unsigned long long raw[kTraceLayers][kTracePoints][kTraceCtas];
  if (coli_trace_read_raw(raw) != 0) return -1;
  auto *L = (unsigned long long *)lo, *Hh = (unsigned long long *)hi;
  for (int l = 0; l < kTraceLayers; ++l)
    for (int p = 0; p < kTracePoints; ++p) {
      unsigned long long mn = ~0ull, mx = 0;
      for (int c = 0; c < kTraceCtas; ++c) {
        const unsigned long long t = raw[l][p][c];
        if (!t) continue;
        mn = t < mn ? t : mn;
        mx = t > mx ? t : mx;
      }
      L[l * kTracePoints + p] = mn;
      Hh[l * kTracePoints + p] = mx;
    }
  return 0;
}
#endif


static cudaError_t plan_down_multi(Dec2Args &a);

// Geometry and shared-memory plans of both kernels for one layer shape.
cudaError_t plan_decode(Dec2Args &a, int n_part) {
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const size_t budget = (size_t)max_smem() - 4096;
  const int G = n_part;
  a.n_part = n_part;
  // ---- gate/up: gu_nw warps, each with a gu_slots-deep cp.async pipeline
  a.gu_ncg = (H + kChunkCols - 1) / kChunkCols;
  a.gu_slot_bytes = slot_bytes(H);
  GuSmem g{};
  size_t o = 0;
  g.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  g.routes = o; o = al16(o + (size_t)T * KS * 4);
  g.slot_gate = o; o = al16(o + (size_t)T * KS * 4);
  // warps x slots (measured: 12 x 2 and 12 x 3 within 1-2 %; the smaller
  // ring leaves more of the SM's unified memory to L1), then 16 x 2, ...
  static const int kNw[] = {12, 12, 8, 8, 4, 4};
  static const int kSl[] = {2, 3, 3, 2, 3, 2};
  bool ok = false;
  if (T == 1) {
    // one token: partial sums per (row, chunk) in shared memory, rows in
    // batches of gu_rows.  x is quantised per warp for the chunk it works on,
    // so warp counts that keep every warp on one chunk (NW % gu_ncg == 0) come first.
    const int n_used = (E < k ? E : k) + S;
    const int max_rows = 4 * ((n_used * (F / 4) + G - 1) / G);
    const size_t row_bytes = (size_t)a.gu_ncg * 2 * 4;
    const int min_batch = max_rows < 64 ? max_rows : 64;
    for (int pass = 0; pass < 2 && !ok; ++pass)
      for (int c = 0; c < 6 && !ok; ++c) {
        if (pass == 0 && kNw[c] % a.gu_ncg != 0) continue;
        const size_t ring = (size_t)kNw[c] * kSl[c] * a.gu_slot_bytes;
        if (al128(o) + ring + 128 + (size_t)min_batch * row_bytes <= budget) {
          a.gu_nw = kNw[c];
          a.gu_slots = kSl[c];
          ok = true;
        }
      }
    if (!ok) return cudaErrorInvalidValue;
    a.gu_xpl = 0;
    g.xpl = g.tok = o;
    g.ring = al128(o); o = g.ring + (size_t)a.gu_nw * a.gu_slots * a.gu_slot_bytes;
    g.red = al16(o);
    const size_t fit = (budget - g.red) / row_bytes;
    int rows = fit < (size_t)max_rows ? (int)fit : max_rows;
    rows &= ~3;
    if (rows < 4) return cudaErrorInvalidValue;
    a.gu_rows = rows;
    g.total = al16(g.red + (size_t)rows * row_bytes);
  } else {
    // several tokens: one [T][8] accumulator per warp, then the planes of the
    // tokens the CTA serves and the ring.  Each CTA sizes its ring from what
    // its planes leave (up to gu_slots deep); the plan makes sure a CTA that
    // serves all T tokens still gets two slots.  Without room for that, no
    // planes (x quantised per task).
    g.tok = o; o = al16(o + (size_t)(2 * T + 3) * 4);
    const size_t xpl_bytes = (size_t)T * 18 * (H / 32) * 4;
    static const int kNwM[] = {kGuMultiMaxThreads / 32, 4};
    for (int xpl = 1; xpl >= 0 && !ok; --xpl)
      for (int c = 0; c < 2 && !ok; ++c) {
        const size_t acc = (size_t)kNwM[c] * T * 8 * 4;
        const size_t ring2 = (size_t)kNwM[c] * 2 * a.gu_slot_bytes;
        if (al128(al16(o + acc) + (xpl ? xpl_bytes : 0)) + ring2 <= budget) {
          a.gu_xpl = xpl;
          a.gu_nw = kNwM[c];
          a.gu_slots = 4;
          ok = true;
        }
      }
    if (!ok) return cudaErrorInvalidValue;
    a.gu_rows = 0;
    g.red = o; o = al16(g.red + (size_t)a.gu_nw * T * 8 * 4);
    g.xpl = g.ring = o;
    g.total = budget;
  }
  a.gu = g;
  // routing scratch: the T = 1 kernel's ring, the several-token kernel's plane area
  a.gu_route_fits = gu_route_smem(T, E, k).total <=
                    (T == 1 ? (size_t)a.gu_nw * a.gu_slots * a.gu_slot_bytes : g.total - g.xpl);
  // one token: room in the ring, after the routing scratch, for a CTA's owned
  // router rows, x and the reduction scratch (the first layer's logits formed
  // in k_gateup, gu_router_logits); -1: none
  a.gu_rt_off = -1;
  if (T == 1) {
    const int n_max = (E + G - 1) / G;
    const size_t off = al16(gu_route_smem(T, E, k).total);
    const size_t need = off + al16((size_t)n_max * H * (a.wr_bf16 ? 2 : 4)) + (size_t)H * 4 + 512;
    if (need <= (size_t)a.gu_nw * a.gu_slots * a.gu_slot_bytes) a.gu_rt_off = (int)off;
  }
  // ---- down: dn_nw warps with dn_slots_pipe-deep cp.async pipelines
  a.dn_ncg = (F + kChunkCols - 1) / kChunkCols;
  a.dn_slot_bytes = slot_bytes(F);
  if (T > 1) return plan_down_multi(a);
  const int UH = H / 4;
  const int max_nr = 4 * ((UH + n_part - 1) / n_part);
  DnSmem d{};
  o = 0;
  d.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  d.routes = o; o = al16(o + (size_t)T * KS * 4);
  d.acc = o; o = al16(o + (size_t)max_nr * T * 4);
  d.xn = o; o = al16(o + (size_t)T * max_nr * 4);
  d.wr = o; o = al16(o + (a.chain ? (size_t)E * max_nr * (a.wr_bf16 ? 2 : 4) : 0));
  // one token: every used expert's partial sums [expert][row][chunk] at once
  const int n_exp = (E < k ? E : k) + S;
  const size_t red_bytes = (size_t)n_exp * max_nr * a.dn_ncg * 4;
  // Each warp works its tasks (an expert's 8-row group x 1024-column chunk) in
  // order, one in flight while it computes another, so the down phase lasts
  // about as long as the largest number of tasks any warp has: the warp count
  // that fits makes that number smallest, and the fewest warps among equals
  // (measured on the GLM-like layer: 18 warps, 6 tasks each, 4 % faster than
  // 16 warps with up to 7, and faster than 20 with up to 6).
  static const int kDnNw[] = {4, 8, 8, 8, 12, 12, 16, 18, 20};
  static const int kDnSl[] = {2, 2, 3, 4, 2, 3, 2, 2, 2};
  const int n_dn_tasks = n_exp * ((max_nr + 7) / 8) * a.dn_ncg;
  int dn_pick = -1, dn_best = 0;
  for (int c = 0; c < 9; ++c) {
    const size_t ring = (size_t)kDnNw[c] * kDnSl[c] * a.dn_slot_bytes;
    if (al128(o) + ring + 16 + red_bytes > budget) continue;
    const int per_warp = (n_dn_tasks + kDnNw[c] - 1) / kDnNw[c];
    if (dn_pick < 0 || per_warp < dn_best) {
      dn_pick = c;
      dn_best = per_warp;
    }
  }
  if (dn_pick < 0) return cudaErrorInvalidValue;
  a.dn_nw = kDnNw[dn_pick];
  a.dn_slots_pipe = kDnSl[dn_pick];
  d.ring = al128(o); o = d.ring + (size_t)a.dn_nw * a.dn_slots_pipe * a.dn_slot_bytes;
  d.red = al16(o); o = d.red + red_bytes;
  d.total = al16(o);
  a.dn = d;
  return cudaSuccess;
}

// Several tokens: k_down_multi runs the expert GEMVs and k_down only adds the
// slots (no ring, planes or partial sums of its own).
static cudaError_t plan_down_multi(Dec2Args &a) {
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, KS = a.k + S;
  const size_t budget = (size_t)max_smem() - 4096;
  const int G = a.n_part;
  const int max_nr = 4 * ((H / 4 + G - 1) / G);
  DnSmem d{};
  size_t o = 0;
  d.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  d.routes = o; o = al16(o + (size_t)T * KS * 4);
  d.acc = o; o = al16(o + (size_t)max_nr * T * 4);
  d.xn = o; o = al16(o + (size_t)T * max_nr * 4);
  d.wr = o; o = al16(o + (a.chain ? (size_t)E * max_nr * (a.wr_bf16 ? 2 : 4) : 0));
  d.ring = d.red = o;
  d.total = o;
  a.dn = d;
  a.dn_nw = 16;
  a.dn_slots_pipe = 2;
  // k_down_multi: warps x slots, then as many h rows' planes as fit (at least
  // one expert's tokens plus one more, else planes per task)
  DmSmem m{};
  o = 0;
  m.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  m.routes = o; o = al16(o + (size_t)T * KS * 4);
  m.u = o; o += 16;
  const size_t per_slot = (size_t)18 * (F / 32) * 4;
  static const int kNw[] = {16, 12, 8, 12, 8, 8, 4};
  static const int kSl[] = {2, 3, 4, 2, 3, 2, 2};
  int pick = -1, cap = 0;
  for (int pass = 0; pass < 2 && pick < 0; ++pass)
    for (int c = 0; c < 7 && pick < 0; ++c) {
      const size_t fixed = al128(o + (size_t)kNw[c] * T * 8 * 4) +
                           (size_t)kNw[c] * kSl[c] * a.dn_slot_bytes;
      if (fixed + 128 > budget) continue;
      const size_t n = (budget - fixed - 128) / per_slot;   // 128: alignment slack
      if (pass == 0 && n < (size_t)(T + 1)) continue;
      pick = c;
      cap = n > (size_t)(T * KS) ? T * KS : (int)n;
    }
  if (pick < 0) return cudaErrorInvalidValue;
  a.dm_nw = kNw[pick];
  a.dm_slots_pipe = kSl[pick];
  a.dm_cap = cap;
  m.planes = o; o = al16(o + (size_t)cap * per_slot);
  m.acc = o; o = o + (size_t)a.dm_nw * T * 8 * 4;
  m.ring = al128(o); o = m.ring + (size_t)a.dm_nw * a.dm_slots_pipe * a.dn_slot_bytes;
  m.total = al16(o);
  a.dm = m;
  return cudaSuccess;
}

// Shared memory the last CTA needs to route a layer (see route_finish).
size_t route_smem_bytes(const Dec2Args &a, bool *stage) {
  const RouteSmem plain = route_smem(a.T, a.E, a.k, a.S, a.n_part, false);
  const RouteSmem staged = route_smem(a.T, a.E, a.k, a.S, a.n_part, true);
  *stage = !a.fx && staged.total <= (size_t)max_smem() - 4096;
  return *stage ? staged.total : plain.total;
}

cudaError_t launch_route_partials(const Dec2Args &a_in, int x_bf16, int w_bf16, cudaStream_t s,
                                  bool pdl) {
  Dec2Args a = a_in;
  bool stage = false;
  size_t smem = route_smem_bytes(a, &stage);
  a.stage_partials = stage;
  const size_t x_bytes = (size_t)a.T * 4 * ((a.H / 4 + a.n_part - 1) / a.n_part) * 4;
  if (smem < x_bytes) smem = x_bytes;
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

cudaError_t launch_gateup(const Dec2Args &a, int grid, cudaStream_t s, bool pdl) {
  const int threads = 32 * a.gu_nw;
  cudaError_t e;
  const bool fast = a.H % kChunkCols == 0;
#define COLI_LAUNCH_GU(K)                                                                \
  if ((e = allow_smem(K, a.gu.total)) != cudaSuccess) return e;                         \
  return launch(K, grid, threads, a.gu.total, s, pdl, a);
  if (a.T == 1 && fast) { COLI_LAUNCH_GU(k_gateup<true>) }
  if (a.T == 1) { COLI_LAUNCH_GU(k_gateup<false>) }
  if (fast && a.gu_xpl) { COLI_LAUNCH_GU((k_gateup_multi<true, true>)) }
  if (fast) { COLI_LAUNCH_GU((k_gateup_multi<true, false>)) }
  if (a.gu_xpl) { COLI_LAUNCH_GU((k_gateup_multi<false, true>)) }
  COLI_LAUNCH_GU((k_gateup_multi<false, false>))
#undef COLI_LAUNCH_GU
}

cudaError_t launch_down_multi(const Dec2Args &a, cudaStream_t s, bool pdl) {
  cudaError_t e;
  if (a.F % kChunkCols == 0) {
    if ((e = allow_smem(k_down_multi<true>, a.dm.total)) != cudaSuccess) return e;
    return launch(k_down_multi<true>, a.n_part, 32 * a.dm_nw, a.dm.total, s, pdl, a);
  }
  if ((e = allow_smem(k_down_multi<false>, a.dm.total)) != cudaSuccess) return e;
  return launch(k_down_multi<false>, a.n_part, 32 * a.dm_nw, a.dm.total, s, pdl, a);
}

cudaError_t launch_down(const Dec2Args &a_in, int wr_bf16, cudaStream_t s, bool pdl) {
  Dec2Args a = a_in;
  const int threads = a.dn_nw * 32;
  size_t smem = a.dn.total;
  if (a.wr) {
    bool stage = false;
    const size_t rs = route_smem_bytes(a, &stage);
    a.stage_partials = stage;
    if (rs > smem) smem = rs;
  }
  cudaError_t e;
#define COLI_LAUNCH_DOWN(WT, ONE, FAST)                                                  \
  if ((e = allow_smem(k_down<WT, ONE, FAST>, smem)) != cudaSuccess) return e;            \
  return launch(k_down<WT, ONE, FAST>, a.n_part, threads, smem, s, pdl, a);
  // the several-token k_down only adds slots: no chunked loop to specialise
  const bool fast = a.F % kChunkCols == 0;
  if (wr_bf16 && a.T == 1 && fast) { COLI_LAUNCH_DOWN(__nv_bfloat16, true, true) }
  if (wr_bf16 && a.T == 1) { COLI_LAUNCH_DOWN(__nv_bfloat16, true, false) }
  if (wr_bf16) { COLI_LAUNCH_DOWN(__nv_bfloat16, false, false) }
  if (a.T == 1 && fast) { COLI_LAUNCH_DOWN(float, true, true) }
  if (a.T == 1) { COLI_LAUNCH_DOWN(float, true, false) }
  COLI_LAUNCH_DOWN(float, false, false)
#undef COLI_LAUNCH_DOWN
}

}  // namespace coli
