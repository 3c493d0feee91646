// Decode-path expert FFNs over int4-grouped weights: bandwidth-bound GEMVs.
//
// Pages: "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战" (matmul_i4_grouped
// consumes the packed rows directly; the u8 nibble trick dot(q,x) = dot(u,x) -
// 8 sum(x)), "Colibrì 深度解析" §四 (each expert's three matrices adjacent; the
// batch union reads each used expert once) and §十一 (the five steps).
//
// k_gateup: one warp per (used expert, block of rows of gate and up); each
//   lane streams 16 packed bytes (32 columns) per row per 1024-column chunk,
//   converts nibbles to floats in registers and forms h = silu(g) * u * gate
//   (the routing gate is folded into h).
// k_down:   one warp per output row; it walks the used experts in ascending id
//   order and each expert's tokens, so out[t] is summed in a fixed order.
//
// Nibble to float: a byte permute writes nibble u into bits 16..19 under the
// exponent of 0.5, giving f = 0.5 + u/256 exactly; then
//   sum_i (u_i - 8) x_i = 256 sum_i f_i x_i - 136 sum_i x_i,
// one permute and one FMA per element.
#include "coli_internal.cuh"

namespace coli {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 1024;  // columns per warp pass (32 lanes x 32 columns)
constexpr int kGURows = 2;    // rows of gate (and of up) per gate/up item

__device__ __forceinline__ float nib(uint32_t lo_or_hi, int b) {
  return __uint_as_float(__byte_perm(lo_or_hi, 0x3F000000u, 0x7044u | ((unsigned)b << 8)));
}

// sum_i f_i x_i over the 32 nibbles of w (f_i = 0.5 + u_i/256).
__device__ __forceinline__ float dot32(const uint4 w, const float (&x)[32]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = ws[i] & 0x0F0F0F0Fu;
    const uint32_t hi = (ws[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      a0 = fmaf(nib(lo, b), x[8 * i + 2 * b], a0);
      a1 = fmaf(nib(hi, b), x[8 * i + 2 * b + 1], a1);
    }
  }
  return a0 + a1;
}

template <typename XT>
__device__ __forceinline__ void load_x32(const XT *p, float (&x)[32]);

template <>
__device__ __forceinline__ void load_x32<float>(const float *p, float (&x)[32]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = __ldg((const float4 *)p + i);
    x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
  }
}

template <>
__device__ __forceinline__ void load_x32<__nv_bfloat16>(const __nv_bfloat16 *p, float (&x)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 q = __ldg((const uint4 *)p + i);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      x[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ float sum32(const float (&x)[32]) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 4) { s0 += x[i]; s1 += x[i + 1]; s2 += x[i + 2]; s3 += x[i + 3]; }
  return (s0 + s1) + (s2 + s3);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

struct DecodeArgs {
  const void *x;
  int T, H, F, E, S, k;
  const uint8_t *packed;
  const float *scales;
  const uint8_t *ws;
  WsLayout L;
  float *h;
  float *out;
  const float *residual;
  float *layer_out;
  int64_t eb;   // packed bytes per expert
  int64_t es;   // scales per expert
};

template <typename XT, int TB>
__device__ __forceinline__ void gateup_item(const DecodeArgs &a, int e, const int32_t *routes,
                                            int r0, int r1, int f0) {
  const int lane = threadIdx.x & 31;
  const int H = a.H, F = a.F, KS = a.k + a.S;
  const int64_t rb = H / 2, ng = H / kGroup;
  const uint8_t *pg = a.packed + (int64_t)e * a.eb;
  const uint8_t *pu = pg + (int64_t)F * rb;
  const float *sg = a.scales + (int64_t)e * a.es;
  const float *su = sg + (int64_t)F * ng;
  const XT *x = (const XT *)a.x;
  const float *slot_gate = (const float *)(a.ws + a.L.slot_gate);
  for (int p = r0; p < r1; p += TB) {
    int slot[TB], tok[TB];
#pragma unroll
    for (int t = 0; t < TB; ++t) {
      slot[t] = (p + t < r1) ? routes[p + t] : -1;
      tok[t] = slot[t] >= 0 ? slot[t] / KS : 0;
    }
    float ag[kGURows][TB], au[kGURows][TB];
#pragma unroll
    for (int r = 0; r < kGURows; ++r)
#pragma unroll
      for (int t = 0; t < TB; ++t) { ag[r][t] = 0.f; au[r][t] = 0.f; }
    for (int c0 = 0; c0 < H; c0 += kChunk) {
      const int col = c0 + lane * 32;
      if (col < H) {
        uint4 wg[kGURows], wu[kGURows];
        float s_g[kGURows], s_u[kGURows];
#pragma unroll
        for (int r = 0; r < kGURows; ++r) {
          wg[r] = ldg_stream(pg + (int64_t)(f0 + r) * rb + col / 2);
          wu[r] = ldg_stream(pu + (int64_t)(f0 + r) * rb + col / 2);
          s_g[r] = __ldg(sg + (int64_t)(f0 + r) * ng + col / kGroup);
          s_u[r] = __ldg(su + (int64_t)(f0 + r) * ng + col / kGroup);
        }
#pragma unroll
        for (int t = 0; t < TB; ++t) {
          if (slot[t] < 0) continue;
          float xv[32];
          load_x32<XT>(x + (int64_t)tok[t] * H + col, xv);
          const float xs = -136.0f * sum32(xv);
#pragma unroll
          for (int r = 0; r < kGURows; ++r) {
            ag[r][t] = fmaf(s_g[r], fmaf(256.0f, dot32(wg[r], xv), xs), ag[r][t]);
            au[r][t] = fmaf(s_u[r], fmaf(256.0f, dot32(wu[r], xv), xs), au[r][t]);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TB; ++t) {
#pragma unroll
      for (int r = 0; r < kGURows; ++r) {
        const float g = warp_sum(ag[r][t]);
        const float u = warp_sum(au[r][t]);
        if (lane == r && slot[t] >= 0)
          a.h[(int64_t)slot[t] * F + f0 + r] = silu(g) * u * slot_gate[slot[t]];
      }
    }
  }
}

template <typename XT>
__global__ void __launch_bounds__(kThreads) k_gateup(DecodeArgs a) {
  const int32_t *act = (const int32_t *)(a.ws + a.L.act);
  const int n_active = act[0];
  const int32_t *act_expert = act + 1;
  const int32_t *act_off = act + 1 + (a.E + a.S);
  const int32_t *routes = (const int32_t *)(a.ws + a.L.routes);
  const int nrb = a.F / kGURows;
  const int warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * kThreads) >> 5;
  for (int item = warp; item < n_active * nrb; item += nwarps) {
    const int ai = item / nrb, f0 = (item % nrb) * kGURows;
    const int e = act_expert[ai], r0 = act_off[ai], r1 = act_off[ai + 1];
    if (r1 - r0 == 1) gateup_item<XT, 1>(a, e, routes, r0, r1, f0);
    else gateup_item<XT, 4>(a, e, routes, r0, r1, f0);
  }
}

// One warp per output row h0; experts in ascending order, 4 at a time.
template <int TM>
__global__ void __launch_bounds__(kThreads) k_down(DecodeArgs a) {
  const int lane = threadIdx.x & 31;
  const int32_t *act = (const int32_t *)(a.ws + a.L.act);
  const int n_active = act[0];
  const int32_t *act_expert = act + 1;
  const int32_t *act_off = act + 1 + (a.E + a.S);
  const int32_t *routes = (const int32_t *)(a.ws + a.L.routes);
  const int H = a.H, F = a.F, KS = a.k + a.S;
  const int64_t rb = F / 2, ng = F / kGroup;
  const int64_t down_off_b = (int64_t)F * (H / 2) * 2;
  const int64_t down_off_s = (int64_t)F * (H / kGroup) * 2;
  const int warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * kThreads) >> 5;
  constexpr int NB = 4;
  for (int row = warp; row < H; row += nwarps) {
    float acc[TM];
#pragma unroll
    for (int t = 0; t < TM; ++t) acc[t] = 0.f;
    for (int a0 = 0; a0 < n_active; a0 += NB) {
      for (int c0 = 0; c0 < F; c0 += kChunk) {
        const int col = c0 + lane * 32;
        if (col >= F) continue;
        uint4 w[NB];
        float s[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (a0 + b < n_active) {
            const int e = act_expert[a0 + b];
            w[b] = ldg_stream(a.packed + (int64_t)e * a.eb + down_off_b + (int64_t)row * rb + col / 2);
            s[b] = __ldg(a.scales + (int64_t)e * a.es + down_off_s + (int64_t)row * ng + col / kGroup);
          }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (a0 + b >= n_active) break;
          const int r0 = act_off[a0 + b], r1 = act_off[a0 + b + 1];
          for (int p = r0; p < r1; ++p) {
            const int slot = routes[p];
            const int t = slot / KS;
            float hv[32];
            load_x32<float>(a.h + (int64_t)slot * F + col, hv);
            const float hs = -136.0f * sum32(hv);
            const float v = s[b] * fmaf(256.0f, dot32(w[b], hv), hs);
#pragma unroll
            for (int tt = 0; tt < TM; ++tt)
              if (tt == t) acc[tt] += v;
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TM; ++t) {
      if (t >= a.T) break;
      const float v = warp_sum(acc[t]);
      if (lane == 0) {
        const int64_t o = (int64_t)t * H + row;
        if (a.layer_out) a.layer_out[o] = v;
        a.out[o] = a.residual ? a.residual[o] + v : v;
      }
    }
  }
}

template <typename XT>
cudaError_t launch_xt(const DecodeArgs &a, cudaStream_t s) {
  const int sms = num_sms();
  const int max_active = (a.T * a.k < a.E ? a.T * a.k : a.E) + a.S;
  const int gu_items = max_active * (a.F / kGURows);
  int gu_blocks = (gu_items + 7) / 8;
  if (gu_blocks > sms * 8) gu_blocks = sms * 8;
  k_gateup<XT><<<gu_blocks, kThreads, 0, s>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  int d_blocks = (a.H + 7) / 8;
  if (d_blocks > sms * 8) d_blocks = sms * 8;
  if (a.T <= 1) k_down<1><<<d_blocks, kThreads, 0, s>>>(a);
  else if (a.T <= 2) k_down<2><<<d_blocks, kThreads, 0, s>>>(a);
  else if (a.T <= 4) k_down<4><<<d_blocks, kThreads, 0, s>>>(a);
  else if (a.T <= 8) k_down<8><<<d_blocks, kThreads, 0, s>>>(a);
  else k_down<16><<<d_blocks, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_moe_decode(const void *x, int x_dtype, int T, int H, int F, int E, int S,
                              int k, const uint8_t *packed, const float *scales,
                              uint8_t *ws, const WsLayout &L, float *out,
                              const float *residual, float *layer_out, cudaStream_t s) {
  DecodeArgs a;
  a.x = x; a.T = T; a.H = H; a.F = F; a.E = E; a.S = S; a.k = k;
  a.packed = packed; a.scales = scales; a.ws = ws; a.L = L;
  a.h = (float *)(ws + L.h);
  a.out = out; a.residual = residual; a.layer_out = layer_out;
  a.eb = (int64_t)3 * F * (H / 2);
  a.es = (int64_t)3 * F * (H / kGroup);
  if (x_dtype == COLI_BF16) return launch_xt<__nv_bfloat16>(a, s);
  return launch_xt<float>(a, s);
}

}  // namespace coli
