// Device and host helpers shared by the decode kernels (decode2.cu: the
// general GEMV path; decode1.cu: the one-token fused layer kernel): the
// 15-bit activation planes and their dp4a dot products, the warp reduction,
// fixed-point router logits, and launch helpers.
//
// Arithmetic ("从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战",
// matmul_i4_grouped and expert_ffn.h's dot(u,x) - 8 sum(x)): each lane owns 32
// consecutive columns.  Its 32 activations are quantised to 15-bit fixed point
// (scale = max|x| / 16319), split into signed 8-bit high and low planes
// (xq = 128 xh + xl), and dotted with the unsigned nibbles by dp4a; the exact
// integer sum sum_i (u_i - 8) xq_i is scaled by the group scale and the
// activation scale.
#pragma once

#include <mutex>
#include <unordered_map>

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
// activation planes in shared memory, transposed for conflict-free access:
// word w (0..15 planes, 16 = sq, 17 = sx bits) of 32-column block b of vector v
// is at planes[(v * 18 + w) * nbp + b].  Each lane quantises whole blocks in
// registers (the same arithmetic as the per-warp paths); CTAs start at
// different blocks so the grid's reads of the same vectors spread over L2.
__device__ void build_planes_impl(const float *src, int n_vec, int F, const int *list,
                                  uint32_t *planes, int nbp, int warp, int nw) {
  const int nb = F / 32;   // F is a multiple of 64
  const int n_blocks = n_vec * nb;
  if (n_blocks == 0) return;
  const int rot = (int)(((long long)blockIdx.x * 37) % n_blocks);
  for (int i = warp * 32 + (threadIdx.x & 31); i < n_blocks; i += nw * 32) {
    int g = i + rot;
    if (g >= n_blocks) g -= n_blocks;
    const int v = g / nb, b = g - v * nb;
    const int64_t row = list ? list[v] : v;
    float xv[32];
    load32<float>(src + row * F + 32 * b, xv);
    Planes p;
    quantize32(xv, p);
    uint32_t *pv = planes + (size_t)v * 18 * nbp + b;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pv[(size_t)j * nbp] = p.eh[j];
      pv[(size_t)(4 + j) * nbp] = p.el[j];
      pv[(size_t)(8 + j) * nbp] = p.oh[j];
      pv[(size_t)(12 + j) * nbp] = p.ol[j];
    }
    pv[(size_t)16 * nbp] = (uint32_t)p.sq;
    pv[(size_t)17 * nbp] = __float_as_uint(p.sx);
  }
}

// build_planes over a list of source rows: vector p is row list[p] of src.
__device__ void build_planes_list(const float *src, int F, const int *list, int n, uint32_t *planes,
                                  int nbp);

__device__ void build_planes_list(const float *src, int F, const int *list, int n, uint32_t *planes,
                                  int nbp) {
  build_planes_impl(src, n, F, list, planes, nbp, threadIdx.x >> 5, blockDim.x >> 5);
}

// The same planes as build_planes_impl, with four lanes per 32-column block:
// lane j of the group loads columns 8j..8j+7 (two float4) and writes word j of
// each of the four planes; the block's max and sq are combined by shuffles.
// Every quotient, rounding and sum is the one quantize32 takes (max and the
// integer sum do not depend on order), so the planes are bit-identical.  Each
// thread issues the loads of kQ4Batch quarter-blocks before quantising any, so
// one memory round trip covers them.  Threads t = tid0 .. tid0 + nthr - 1
// (nthr a multiple of 32) take part; every lane runs every iteration.
constexpr int kQ4Batch = 12;
__device__ void build_planes_q4(const float *src, int n_vec, int F, uint32_t *planes, int nbp,
                                int tid, int nthr) {
  const int nb = F / 32;
  const int n_tasks = 4 * n_vec * nb;
  const int lane = threadIdx.x & 31, j = lane & 3;
  const int rounds = (n_tasks + nthr * kQ4Batch - 1) / (nthr * kQ4Batch);
  for (int r = 0; r < rounds; ++r) {
    float4 v[kQ4Batch][2];
#pragma unroll
    for (int u = 0; u < kQ4Batch; ++u) {
      const int i = tid + (r * kQ4Batch + u) * nthr;
      if (i < n_tasks) {
        const int g = i >> 2, vv = g / nb, b = g - vv * nb;
        const float4 *p = (const float4 *)(src + (size_t)vv * F + 32 * b + 8 * j);
        v[u][0] = __ldcg(p);
        v[u][1] = __ldcg(p + 1);
      } else {
        v[u][0] = v[u][1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
#pragma unroll
    for (int u = 0; u < kQ4Batch; ++u) {
      const int i = tid + (r * kQ4Batch + u) * nthr;
      const float x[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w,
                          v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
      float m = 0.0f;
      bool bad = false;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        m = fmaxf(m, fabsf(x[q]));
        bad |= (x[q] != x[q]);
      }
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      const unsigned any_bad = __ballot_sync(0xFFFFFFFFu, bad);
      bad = (any_bad >> (lane & ~3)) & 0xFu;
      const float inv = m > 0.0f ? (float)kQ / m : 0.0f;
      uint32_t eh = 0, el = 0, oh = 0, ol = 0;
      int sq = 0;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int qe = (int)fminf(fmaxf(rintf(x[2 * bb] * inv), -(float)kQ), (float)kQ);
        const int qo = (int)fminf(fmaxf(rintf(x[2 * bb + 1] * inv), -(float)kQ), (float)kQ);
        const int he = (qe + 64) >> 7, ho = (qo + 64) >> 7;
        const int le = qe - (he << 7), lo = qo - (ho << 7);
        eh |= (uint32_t)(he & 0xFF) << (8 * bb);
        el |= (uint32_t)(le & 0xFF) << (8 * bb);
        oh |= (uint32_t)(ho & 0xFF) << (8 * bb);
        ol |= (uint32_t)(lo & 0xFF) << (8 * bb);
        sq += qe + qo;
      }
      sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 1);
      sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 2);
      if (i < n_tasks) {
        const int g = i >> 2, vv = g / nb, b = g - vv * nb;
        uint32_t *pv = planes + (size_t)vv * 18 * nbp + b;
        pv[(size_t)j * nbp] = eh;
        pv[(size_t)(4 + j) * nbp] = el;
        pv[(size_t)(8 + j) * nbp] = oh;
        pv[(size_t)(12 + j) * nbp] = ol;
        if (j == 0) {
          pv[(size_t)16 * nbp] = (uint32_t)sq;
          pv[(size_t)17 * nbp] = __float_as_uint(bad ? __int_as_float(0x7FC00000) : m / (float)kQ);
        }
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


// Fixed-point router logits (2^-32 units): a partial p of logit (t, e) is
// added with an integer atomic, so the total does not depend on the order in
// which CTAs arrive.  A non-finite partial, or one of magnitude 1e7 or more,
// marks the logit as NaN instead.
// A fixed-point sum as a float: one rounding of the integer, then the exact
// power-of-two scale.
__device__ __forceinline__ float fx_to_float(long long v) {
  return __ll2float_rn(v) * 0x1p-32f;
}

__host__ __device__ constexpr size_t al16c(size_t v) { return (v + 15) & ~(size_t)15; }

__device__ __forceinline__ void fx_add_to(long long *acc, uint32_t *flag, int o, float p) {
  if (!(fabsf(p) < 1.0e7f)) {
    atomicOr(flag + o, 1u);
    return;
  }
  atomicAdd((unsigned long long *)(acc + o), (unsigned long long)__float2ll_rn(p * 4294967296.0f));
}
__device__ __forceinline__ void fx_add(const Dec2Args &a, int o, float p) {
  fx_add_to(a.fx_acc, a.fx_flag, o, p);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier across the kernel's CTAs, run by one thread per CTA after the
// CTA's own writes are ordered before it (bar.sync).  Sense by generation:
// the last CTA to arrive resets the arrival count and advances the
// generation; the others spin (bounded) until the generation moves.  Both
// words stay consistent between calls.  Returns false if the wait gave up.
__device__ __forceinline__ bool grid_sync(uint32_t *ctrl, unsigned G) {
  const uint32_t lim = ld_acquire(ctrl + kCtrlWaitLimit);
  const long long limit = lim ? (long long)lim : kWaitCycles;
  const uint32_t gen = ld_acquire(ctrl + kCtrlBarGen);
  __threadfence();
  const uint32_t old = atomicAdd(ctrl + kCtrlBarArrive, 1u);
  if (old == G - 1) {
    atomicExch(ctrl + kCtrlBarArrive, 0u);
    __threadfence();
    atomicAdd(ctrl + kCtrlBarGen, 1u);
    return true;
  }
  const long long t0 = clock64();
  while (ld_acquire(ctrl + kCtrlBarGen) == gen) {
    if (clock64() - t0 > limit) return false;
    __nanosleep(64);
  }
  __threadfence();
  return true;
}



// Shared-memory scratch of gu_route (byte offsets from its base).
struct GuRouteSmem {
  size_t logits, sel, bias, topk, idx, gates, vals, flag, total;
};
__host__ __device__ inline GuRouteSmem gu_route_smem(int T, int E, int k) {
  auto a16 = [](size_t v) { return (v + 15) & ~(size_t)15; };
  GuRouteSmem R{};
  size_t o = 0;
  R.logits = o; o = a16(o + (size_t)T * E * 4);
  R.sel = o; o = a16(o + (size_t)T * E * 4);
  R.bias = o; o = a16(o + (size_t)E * 4);
  R.topk = o;
  size_t tk = topk_scratch_bytes(T, E, k);
  if (tk < (size_t)T * k * 4) tk = (size_t)T * k * 4;   // the union's sort scratch
  o = a16(R.topk + tk);
  R.idx = o; o += (size_t)T * k * 4;
  R.gates = o; o += (size_t)T * k * 4;
  R.vals = o; o += (size_t)T * k * 4;
  R.flag = a16(o); o = R.flag + 16;
  R.total = o;
  return R;
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

// The same partial logits, added to the next layer's fixed-point buffer.
template <typename WT>
__device__ void dn_partials_fx(const Dec2Args &a, const WT *s_wr, const float *s_xn) {
  const int T = a.T, H = a.H, E = a.E;
  const int G = gridDim.x, c = blockIdx.x;
  const int UH = H / 4;
  const int nr = 4 * part_lo(c + 1, UH, G) - 4 * part_lo(c, UH, G);
  if (nr <= 0) return;
  for (int o = threadIdx.x; o < T * E; o += blockDim.x) {
    const int t = o / E, e = o - t * E;
    float sum = 0.0f;
    for (int r = 0; r < nr; ++r) sum = fmaf(to_f32(s_wr[e * nr + r]), s_xn[t * nr + r], sum);
    fx_add(a, o, sum);
  }
}

// This CTA's rows [dh0, dh1) of a router matrix, into shared memory.
template <typename WT>
__device__ void load_router_rows(const Dec2Args &a, const WT *wr, WT *s_wr) {
  const int H = a.H, E = a.E;
  const int G = gridDim.x, c = blockIdx.x;
  const int UH = H / 4;
  const int dh0 = 4 * part_lo(c, UH, G), nr = 4 * part_lo(c + 1, UH, G) - dh0;
  // eight loads in flight per thread before any store
  for (int i0 = threadIdx.x; i0 < E * nr; i0 += 8 * blockDim.x) {
    WT v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < E * nr) {
        const int e = i / nr, r = i - e * nr;
        v[u] = __ldg(wr + (size_t)e * H + dh0 + r);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < E * nr) s_wr[i] = v[u];
    }
  }
}

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

}  // namespace coli
