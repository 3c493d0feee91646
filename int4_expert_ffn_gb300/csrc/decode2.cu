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
    for (int h = h0; h < h1; ++h) s = fmaf(to_f32(wr[(size_t)e * a.H + h]), to_f32(x[(size_t)t * a.H + h]), s);
    a.partials[(size_t)c * a.T * a.E + o] = s;
  }
}

// ---------------------------------------------------------------------------
// Routing shared by k_gateup and k_topk: logits from the partials (fixed
// order), top-k per token by warps, NaN flag.

__device__ void route_block(const Dec2Args &a, float *s_logits, int *s_idx, float *s_gates,
                            float *s_park, float *s_scratch, bool publish) {
  const int T = a.T, E = a.E, k = a.k;
  const int TE = T * E;
  const int nthr = blockDim.x;
  int nsplit = nthr / TE;
  if (nsplit > 8) nsplit = 8;
  if (nsplit <= 1) {
    for (int o = threadIdx.x; o < TE; o += nthr) {
      float s = 0.0f;
#pragma unroll 4
      for (int p = 0; p < a.n_part; ++p) s += __ldcg(a.partials + (size_t)p * TE + o);
      s_logits[o] = s;
    }
  } else {
    // nsplit * TE <= nthr: one partial sum per thread, combined in fixed order
    for (int i = threadIdx.x; i < TE * nsplit; i += nthr) {
      const int o = i % TE, part = i / TE;
      const int p0 = part_lo(part, a.n_part, nsplit), p1 = part_lo(part + 1, a.n_part, nsplit);
      float s = 0.0f;
#pragma unroll 4
      for (int p = p0; p < p1; ++p) s += __ldcg(a.partials + (size_t)p * TE + o);
      s_scratch[part * TE + o] = s;
    }
    __syncthreads();
    for (int o = threadIdx.x; o < TE; o += nthr) {
      float s = 0.0f;
      for (int part = 0; part < nsplit; ++part) s += s_scratch[part * TE + o];
      s_logits[o] = s;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, nw = nthr >> 5, lane = threadIdx.x & 31;
  bool nan = false;
  for (int t = warp; t < T; t += nw)
    nan |= warp_topk(s_logits + t * E, E, k, s_idx + t * k, s_gates + t * k, s_park + warp * k);
  if (publish && lane == 0 && nan) set_flag(a.ctrl, COLI_FLAG_NAN_LOGITS);
  __syncthreads();
  if (publish) {
    for (int i = threadIdx.x; i < T * k; i += nthr) {
      a.g_idx[i] = s_idx[i];
      a.g_gates[i] = s_gates[i];
      if (a.counts) atomicAdd(a.counts + s_idx[i], 1u);
    }
  }
}

__global__ void __launch_bounds__(256) k_topk(Dec2Args a) {
  extern __shared__ __align__(16) uint8_t smem[];
  grid_dependents_launch();
  grid_dependency_wait();
  float *s_logits = (float *)smem;
  int *s_idx = (int *)(s_logits + a.T * a.E);
  float *s_gates = (float *)(s_idx + a.T * a.k);
  float *s_park = s_gates + a.T * a.k;
  float *s_scratch = s_park + 8 * a.k;
  route_block(a, s_logits, s_idx, s_gates, s_park, s_scratch, true);
  __syncthreads();
  for (int i = threadIdx.x; i < a.T * a.k; i += blockDim.x) {
    if (a.idx_out) a.idx_out[i] = s_idx[i];
    if (a.gates_out) a.gates_out[i] = s_gates[i];
  }
}

// ---------------------------------------------------------------------------
// gate/up

template <typename XT>
__global__ void __launch_bounds__(kDec2MaxThreads) k_gateup(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GuSmem &L = a.gu;
  const int T = a.T, H = a.H, F = a.F, E = a.E, S = a.S, k = a.k, KS = k + S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwc = a.gu_ncg * a.gu_nrg;   // compute warps; warp nwc is the producer
  uint64_t *full = (uint64_t *)(smem + L.bar);
  uint64_t *done = full + a.gu_ns;
  int *s_abort = (int *)(done + a.gu_ns);
  if (tid == 0) {
    for (int i = 0; i < a.gu_ns; ++i) {
      mbar_init(full + i, 1);
      mbar_init(done + i, nwc);
    }
    *s_abort = 0;
    fence_mbar_init();
  }
  grid_dependents_launch();
  grid_dependency_wait();

  float *s_logits = (float *)(smem + L.logits);
  int *s_idx = (int *)(smem + L.idx);
  float *s_gates = (float *)(smem + L.gates);
  float *s_park = (float *)(smem + L.park);
  float *s_scratch = (float *)(smem + L.scratch);
  int *s_act = (int *)(smem + L.act);          // [0] n_active, act_expert, act_off
  int *s_act_expert = s_act + 1;
  int *s_act_off = s_act + 1 + (E + S);
  int *s_routes = (int *)(smem + L.routes);
  float *s_slot_gate = (float *)(smem + L.slot_gate);
  const bool cta0 = blockIdx.x == 0;

  route_block(a, s_logits, s_idx, s_gates, s_park, s_scratch, cta0);
  if (warp == 0) {
    const int na = warp_union(s_idx, s_gates, T, k, S, E, s_act_expert, s_act_off, s_routes,
                              s_slot_gate);
    if (lane == 0) s_act[0] = na;
  }
  __syncthreads();
  const int n_active = s_act[0];
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
  const int rs4 = a.gu_rs / 4, ns = a.gu_ns;
  const int64_t rb = H / 2, ngr = H / kGroup;
  const int stage_bytes = a.gu_rs * (H + H / 8);
  float *red = (float *)(smem + L.red);
  const int red_stride = a.gu_rs * T * a.gu_ncg * 2;

  if (warp == nwc) {
    // ---------------- producer warp ----------------
    StageIter it(u0, u1, F4, rs4);
    int sa[16], sr[16], sn[16];   // descriptors of stages in flight (ns <= 16)
    int s = 0, fin = 0;
    int ai, r0, n;
    bool ok = true;
    // L2 prefetch of the down rows that the same-index k_down CTA will read
    auto prefetch_down = [&]() {
      if (lane != 0 || c >= a.n_part) return;
      const int UH = H / 4;
      const int dh0 = 4 * part_lo(c, UH, a.n_part), dh1 = 4 * part_lo(c + 1, UH, a.n_part);
      for (int q = 0; q < n_active && dh1 > dh0; ++q) {
        const int e = s_act_expert[q];
        prefetch_l2(a.packed + (int64_t)e * a.eb + (int64_t)F * H + (int64_t)dh0 * (F / 2),
                    (uint32_t)((dh1 - dh0) * (F / 2)));
        prefetch_l2(a.scales + (int64_t)e * a.es + (int64_t)2 * F * ngr + (int64_t)dh0 * (F / kGroup),
                    (uint32_t)((dh1 - dh0) * (F / 16)));
      }
    };
    auto finalize = [&](int st) {
      const int slot = st % ns;
      const int fa = sa[slot], f0 = sr[slot], fn = sn[slot];
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
        a.h[(int64_t)slot_id * F + f0 + r] = silu(g) * u * s_slot_gate[slot_id];
      }
    };
    while (ok && it.next(ai, r0, n)) {
      const int slot = s % ns;
      if (s >= ns) {
        if (!mbar_wait(done + slot, ((s / ns) - 1) & 1)) { ok = false; break; }
        finalize(fin++);
      }
      sa[slot] = ai; sr[slot] = r0; sn[slot] = n;
      if (lane == 0) {
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
      ++s;
      if (s == ns) prefetch_down();
      __syncwarp();
    }
    if (s < ns) prefetch_down();
    if (ok) {
      for (; fin < s; ++fin) {
        const int slot = fin % ns;
        if (!mbar_wait(done + slot, (fin / ns) & 1)) { ok = false; break; }
        finalize(fin);
      }
    }
    if (!ok) {
      if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
      *s_abort = 1;
      // drain copies still in flight before the CTA may exit
      for (int st = (s > ns ? s - ns : 0); st < s; ++st)
        (void)mbar_wait(full + (st % ns), (st / ns) & 1);
    }
  } else if (warp < nwc) {
    // ---------------- compute warps ----------------
    const int cg = warp % a.gu_ncg, rg = warp / a.gu_ncg, nrg = a.gu_nrg;
    const int col = cg * kChunkCols + 32 * lane;
    const bool act = col < H;
    const XT *x = (const XT *)a.x;
    Planes pl;
    int cached = -1;
    StageIter it(u0, u1, F4, rs4);
    int s = 0, ai, r0, n;
    while (it.next(ai, r0, n)) {
      const int slot = s % ns;
      if (!mbar_wait(full + slot, (s / ns) & 1)) {
        if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
        break;
      }
      if (*(volatile int *)s_abort) break;
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
          if (act) load32<XT>(x + (int64_t)t * H + col, v);
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
  uint64_t *full = (uint64_t *)(smem + L.bar);
  uint64_t *done = full + a.dn_ns;
  uint64_t *hbar = done + a.dn_ns;
  int *s_abort = (int *)(hbar + 1);
  WT *s_wr = (WT *)(smem + L.wr);
  if (tid == 0) {
    for (int i = 0; i < a.dn_ns; ++i) {
      mbar_init(full + i, 1);
      mbar_init(done + i, nwc);
    }
    mbar_init(hbar, 1);
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
  grid_dependents_launch();
  grid_dependency_wait();
  int *s_act = (int *)(smem + L.act);
  int *s_act_expert = s_act + 1;
  int *s_act_off = s_act + 1 + (E + S);
  int *s_routes = (int *)(smem + L.routes);
  float *s_acc = (float *)(smem + L.acc);   // [T][nr]
  for (int i = tid; i < 1 + 2 * (E + S) + 1; i += blockDim.x) s_act[i] = __ldcg(a.g_act + i);
  for (int i = tid; i < T * KS; i += blockDim.x) s_routes[i] = __ldcg(a.g_routes + i);
  for (int i = tid; i < T * nr; i += blockDim.x) s_acc[i] = 0.0f;
  __syncthreads();
  const int n_active = s_act[0];
  const int ns = a.dn_ns, rs4 = a.dn_rs / 4;
  const int64_t rb = F / 2, ngr = F / kGroup;
  const int stage_bytes = a.dn_rs * (F / 2 + F / 16);
  float *red = (float *)(smem + L.red);
  const int red_stride = a.dn_rs * T * a.dn_ncg;
  const float *s_h = (const float *)(smem + L.h);
  const int64_t down_b = (int64_t)F * H, down_s = (int64_t)2 * F * (H / kGroup);
  const int seg4 = nr / 4;

  if (warp == nwc) {
    StageIter it(0, n_active * seg4, seg4 > 0 ? seg4 : 1, rs4);
    if (seg4 == 0) it.u1 = 0;
    int sa[16], sr[16], sn[16];
    int s = 0, fin = 0, ai, r0, n;
    bool ok = true;
    if (a.dn_h_smem && lane == 0) {
      const uint32_t hb = (uint32_t)(T * KS * F * 4);
      mbar_arrive_expect_tx(hbar, hb);
      bulk_g2s((void *)s_h, a.h, hb, hbar);
    }
    auto finalize = [&](int st) {
      const int slot = st % ns;
      const int fa = sa[slot], f0 = sr[slot], fn = sn[slot];
      const int j0 = s_act_off[fa], ntok = s_act_off[fa + 1] - j0;
      const float *rd = red + slot * red_stride;
      for (int i = lane; i < fn * ntok; i += 32) {
        const int r = i / ntok, j = i - r * ntok;
        float v = 0.0f;
        for (int cg = 0; cg < a.dn_ncg; ++cg) v += rd[(r * T + j) * a.dn_ncg + cg];
        const int t = s_routes[j0 + j] / KS;
        s_acc[t * nr + f0 + r] += v;   // experts finalised in ascending order
      }
    };
    while (ok && it.next(ai, r0, n)) {
      const int slot = s % ns;
      if (s >= ns) {
        if (!mbar_wait(done + slot, ((s / ns) - 1) & 1)) { ok = false; break; }
        finalize(fin++);
      }
      sa[slot] = ai; sr[slot] = r0; sn[slot] = n;
      if (lane == 0) {
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
    if (ok)
      for (; fin < s; ++fin) {
        const int slot = fin % ns;
        if (!mbar_wait(done + slot, (fin / ns) & 1)) { ok = false; break; }
        finalize(fin);
      }
    if (!ok) {
      if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
      *s_abort = 1;
      for (int st = (s > ns ? s - ns : 0); st < s; ++st)
        (void)mbar_wait(full + (st % ns), (st / ns) & 1);
    }
    if (a.dn_h_smem) (void)mbar_wait(hbar, 0);
  } else if (warp < nwc) {
    const int cg = warp % a.dn_ncg, rg = warp / a.dn_ncg, nrg = a.dn_nrg;
    const int col = cg * kChunkCols + 32 * lane;
    const bool act = col < F;
    bool h_ready = !a.dn_h_smem;
    StageIter it(0, n_active * seg4, seg4 > 0 ? seg4 : 1, rs4);
    if (seg4 == 0) it.u1 = 0;
    int s = 0, ai, r0, n;
    while (it.next(ai, r0, n)) {
      const int slot = s % ns;
      if (!h_ready) {
        if (!mbar_wait(hbar, 0)) { if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT); break; }
        h_ready = true;
      }
      if (!mbar_wait(full + slot, (s / ns) & 1)) {
        if (lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
        break;
      }
      if (*(volatile int *)s_abort) break;
      const uint8_t *stg = smem + L.ring + (size_t)slot * stage_bytes;
      const float *sdp = (const float *)(stg + a.dn_rs * rb);
      float *rd = red + slot * red_stride;
      const int j0 = s_act_off[ai], ntok = s_act_off[ai + 1] - j0;
      const int nrows = n > rg ? (n - rg + nrg - 1) / nrg : 0;
      for (int j = 0; j < ntok; ++j) {
        const int slot_id = s_routes[j0 + j];
        Planes pl;
        {
          float v[32];
          if (act) {
            if (a.dn_h_smem) load32_smem(s_h + (int64_t)slot_id * F + col, v);
            else load32<float>(a.h + (int64_t)slot_id * F + col, v);
          } else {
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
  __syncthreads();
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
  }
  if (a.wr) {
    __syncthreads();
    for (int o = tid; o < T * E; o += blockDim.x) {
      const int t = o / E, e = o - t * E;
      float sum = 0.0f;
      for (int r = 0; r < nr; ++r) sum = fmaf(to_f32(s_wr[e * nr + r]), s_xn[t * nr + r], sum);
      a.partials[(size_t)c * T * E + o] = sum;
    }
  }
}

// ---------------------------------------------------------------------------
// host side

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
  g.park = o; o = al16(o + (size_t)(kDec2MaxThreads / 32) * k * 4);
  g.scratch = o; o = al16(o + (size_t)kDec2MaxThreads * 4);
  g.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  g.routes = o; o = al16(o + (size_t)T * KS * 4);
  g.slot_gate = o; o = al16(o + (size_t)T * KS * 4);
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
  g.bar = o; o += (size_t)ns * 16 + 16;
  g.total = al16(o);
  a.gu = g;
  // ---- down
  a.dn_ncg = (F + kChunkCols - 1) / kChunkCols;
  a.dn_nrg = 12 / a.dn_ncg;
  if (a.dn_nrg < 1) a.dn_nrg = 1;
  if (a.dn_ncg * a.dn_nrg > kDec2MaxThreads / 32 - 1) a.dn_nrg = (kDec2MaxThreads / 32 - 1) / a.dn_ncg;
  if (a.dn_nrg < 1) return cudaErrorInvalidValue;
  const int UH = H / 4;
  const int max_nr = 4 * ((UH + n_part - 1) / n_part);
  DnSmem d{};
  o = 0;
  d.act = o; o = al16(o + (size_t)(2 + 2 * (E + S)) * 4);
  d.routes = o; o = al16(o + (size_t)T * KS * 4);
  d.acc = o; o = al16(o + (size_t)T * max_nr * 4);
  d.xn = o; o = al16(o + (size_t)T * max_nr * 4);
  d.wr = o; o = al16(o + (size_t)E * max_nr * 4);
  const size_t fixed_d = o;
  const size_t drow = (size_t)F / 2 + F / 16;
  int rsd = max_nr;
  while ((size_t)rsd * drow > 65536 && rsd > 4) rsd -= 4;
  const size_t red_drow = (size_t)T * a.dn_ncg * 4;
  const size_t hbytes = (size_t)T * KS * F * 4;
  a.dn_h_smem = 0;
  int nsd = 0;
  for (int try_h = 1; try_h >= 0; --try_h) {
    const size_t hb = try_h ? al128(hbytes) : 0;
    if (try_h && hbytes > 98304) continue;
    for (nsd = 16; nsd >= 2; --nsd) {
      const size_t need = al128(fixed_d) + hb + nsd * rsd * drow + nsd * rsd * red_drow + nsd * 16 + 96;
      if (need <= budget) break;
    }
    if (nsd >= 2) { a.dn_h_smem = try_h; break; }
  }
  if (nsd < 2) return cudaErrorInvalidValue;
  // no more stages than the CTA can use
  const int stages_needed = ((E + S) < T * k + S ? (E + S) : T * k + S) * ((max_nr / 4 + rsd / 4 - 1) / (rsd / 4));
  if (nsd > stages_needed && stages_needed >= 2) nsd = stages_needed;
  a.dn_rs = rsd;
  a.dn_ns = nsd;
  o = al128(fixed_d);
  d.h = o; o += a.dn_h_smem ? al128(hbytes) : 0;
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

cudaError_t launch_topk(const Dec2Args &a, cudaStream_t s, bool pdl) {
  const size_t smem = (size_t)(a.T * a.E + 2 * a.T * a.k + 8 * a.k + 256) * 4;
  cudaError_t e = allow_smem(k_topk, smem);
  if (e != cudaSuccess) return e;
  return launch(k_topk, 1, 256, smem, s, pdl, a);
}

cudaError_t launch_gateup(const Dec2Args &a, int x_bf16, int grid, cudaStream_t s, bool pdl) {
  const int threads = (a.gu_ncg * a.gu_nrg + 1) * 32;
  cudaError_t e;
  if (x_bf16) {
    if ((e = allow_smem(k_gateup<__nv_bfloat16>, a.gu.total)) != cudaSuccess) return e;
    return launch(k_gateup<__nv_bfloat16>, grid, threads, a.gu.total, s, pdl, a);
  }
  if ((e = allow_smem(k_gateup<float>, a.gu.total)) != cudaSuccess) return e;
  return launch(k_gateup<float>, grid, threads, a.gu.total, s, pdl, a);
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
