// int4-grouped quantiser (page "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战",
// section 权重转换, quant_int4_grouped): per row and per 64-column group,
// s = max|w| / 7 in f32, q = clip(rint(w / s), -8, 7) with an f32 division and
// round-half-even rint, stored as u = q + 8, even column in the low nibble.
//
// HBM-bound: reads 2 B (bf16) per element and writes 0.5 B + 4 B per 64.
// Bit-exactness with the f32 definition: the quotient w / s is formed as
// w * r with r the approximate reciprocal of s (rcp.approx, at most 1 ulp off);
// for |w / s| <= 7 it lies within 1.7e-6 of the correctly rounded f32 quotient,
// so whenever it is farther than 4e-6 from a half-integer both round to the
// same integer.  The rare element near a half-integer (or any non-finite value,
// or a subnormal s that the approximation flushes) takes the exact IEEE division.
#include "coli_internal.cuh"

namespace coli {
namespace {

__device__ __forceinline__ int quant_one(float w, float s, float r) {
  // s > 0 here
  float a = w * r;
  float d = fabsf(a - floorf(a) - 0.5f);
  float v;
  if (d > 4e-6f && fabsf(a) < 8.0f) {
    v = rintf(a);
  } else {
    v = rintf(__fdiv_rn(w, s));
    if (v != v) return 0;  // NaN weight
  }
  v = fminf(fmaxf(v, -8.0f), 7.0f);
  return (int)v;
}

// The same result with fewer instructions, for the vectorised path: eight
// elements of one group (scale s, r = rcp(s)) into one packed word.  With
// K = 1.5 * 2^23, t = fma(w, r, K) rounds the exact product w r to an integer
// n (ties to even: K is even) held in t's low mantissa bits, so t's low
// nibble is n mod 16 and (n mod 16) ^ 8 = n + 8 = u for n in [-8, 7];
// d = fma(w, r, -n) is the product's distance to n.  For finite weights
// |w r| <= 7 (1 + 2^-20), so n needs no clamp, and the exact quotient w / s
// lies within 1.7e-6 of w r: whenever |d| < 0.5 - 4e-6 both round to n.  If
// any of the eight is closer to a half-integer, or not finite (d is then
// NaN), the word is recomputed element by element with quant_one.
constexpr float kRoundShift = 12582912.0f;   // 1.5 * 2^23

// Approximate reciprocal (PTX rcp.approx: at most 1 ulp of error; subnormal
// input and output flushed to zero).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ uint32_t quant_word(const float *v, float s, float r) {
  uint32_t word = 0;
  bool exact = true;
#pragma unroll
  for (int i = 7; i >= 0; --i) {
    const float t = fmaf(v[i], r, kRoundShift);
    const float n = t - kRoundShift;
    const float d = fmaf(v[i], r, -n);
    word = (word << 4) | (__float_as_uint(t) & 0xFu);
    exact = exact && (fabsf(d) < 0.5f - 4e-6f);
  }
  word ^= 0x88888888u;
  if (!exact) {
    word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= (uint32_t)(quant_one(v[i], s, r) + 8) << (4 * i);
  }
  return word;
}

template <typename T>
struct Load8;

template <>
struct Load8<__nv_bfloat16> {
  // 8 bf16 = 16 bytes
  static __device__ __forceinline__ void run(const __nv_bfloat16 *p, float v[8]) {
    uint4 q = ldg_stream(p);
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

template <>
struct Load8<float> {
  static __device__ __forceinline__ void run(const float *p, float v[8]) {
    uint4 a = ldg_stream(p);
    uint4 b = ldg_stream(p + 4);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
  }
};

// Vectorised path: cols % 64 == 0 and 16-byte aligned w, so group g of the
// flattened matrix is elements [64g, 64g+64), bytes [32g, 32g+32), scale g.
// A team of 4 lanes owns one group; each lane holds 16 consecutive elements
// (two packed words), so the per-group work (max across the team, the scale
// division, the reciprocal, the stores) is shared by 16 elements per lane.
template <typename T, int U>
__global__ void __launch_bounds__(256, 4) k_quant_vec(const T *__restrict__ w, int64_t n_groups,
                                                   uint32_t *__restrict__ packed,
                                                   float *__restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;
  const unsigned team_mask = 0xFu << (lane & 28);
  const int64_t team = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 2;
  const int64_t n_teams = ((int64_t)gridDim.x * blockDim.x) >> 2;
  for (int64_t g0 = team; g0 < n_groups; g0 += n_teams * U) {
    float v[U][16];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + (int64_t)u * n_teams;
      if (g < n_groups) {
        Load8<T>::run(w + g * kGroup + sub * 16, v[u]);
        Load8<T>::run(w + g * kGroup + sub * 16 + 8, v[u] + 8);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + (int64_t)u * n_teams;
      if (g >= n_groups) break;  // uniform across the team
      float m = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[u][i]));
      m = fmaxf(m, __shfl_xor_sync(team_mask, m, 1));
      m = fmaxf(m, __shfl_xor_sync(team_mask, m, 2));
      const float s = __fdiv_rn(m, 7.0f);
      uint2 words = make_uint2(0x88888888u, 0x88888888u);
      if (s != 0.0f) {
        const float r = rcp_approx(s);
        words.x = quant_word(v[u], s, r);
        words.y = quant_word(v[u] + 8, s, r);
      }
      packed[g * 8 + 2 * sub] = words.x;        // packed is only 4-byte aligned
      packed[g * 8 + 2 * sub + 1] = words.y;
      if (sub == 0) scales[g] = s;
    }
  }
}

// General path: any shape and alignment; one thread per (row, group).
template <typename T>
__global__ void k_quant_any(const T *__restrict__ w, int64_t rows, int64_t cols,
                            uint8_t *__restrict__ packed, float *__restrict__ scales) {
  const int64_t ng = (cols + kGroup - 1) / kGroup;
  const int64_t rb = (cols + 1) / 2;
  const int64_t total = rows * ng;
  for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total;
       id += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = id / ng, g = id % ng;
    const int64_t c0 = g * kGroup;
    const int64_t c1 = c0 + kGroup < cols ? c0 + kGroup : cols;
    const T *wr = w + r * cols;
    float m = 0.0f;
    for (int64_t c = c0; c < c1; ++c) m = fmaxf(m, fabsf(to_f32(wr[c])));
    const float s = __fdiv_rn(m, 7.0f);
    const float rc = __frcp_rn(s);
    scales[r * ng + g] = s;
    uint8_t *pr = packed + r * rb;
    for (int64_t c = c0; c < c1; c += 2) {
      const int q0 = s != 0.0f ? quant_one(to_f32(wr[c]), s, rc) : 0;
      uint8_t b = (uint8_t)(q0 + 8);
      if (c + 1 < c1) {
        const int q1 = s != 0.0f ? quant_one(to_f32(wr[c + 1]), s, rc) : 0;
        b |= (uint8_t)((q1 + 8) << 4);
      }
      pr[c >> 1] = b;
    }
  }
}

}  // namespace

cudaError_t launch_quant_i4g(const void *w, int w_dtype, int64_t rows, int64_t cols,
                             uint8_t *packed, float *scales, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorNoDevice;
  const bool aligned = ((uintptr_t)w % 16 == 0) && ((uintptr_t)packed % 4 == 0) &&
                       ((uintptr_t)scales % 4 == 0);
  if (cols % kGroup == 0 && aligned) {
    const int64_t n_groups = rows * (cols / kGroup);
    const int64_t teams_needed = n_groups;
    int64_t blocks = (teams_needed * 4 + 255) / 256;
    const int64_t cap = (int64_t)sms * 4;  // 4 blocks of 256 per SM resident (64 registers)
    if (blocks > cap) blocks = cap;
    if (w_dtype == COLI_BF16)
      k_quant_vec<__nv_bfloat16, 2><<<(unsigned)blocks, 256, 0, s>>>(
          (const __nv_bfloat16 *)w, n_groups, (uint32_t *)packed, scales);
    else
      k_quant_vec<float, 1><<<(unsigned)blocks, 256, 0, s>>>(
          (const float *)w, n_groups, (uint32_t *)packed, scales);
  } else {
    const int64_t total = rows * ((cols + kGroup - 1) / kGroup);
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
    if (w_dtype == COLI_BF16)
      k_quant_any<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>(
          (const __nv_bfloat16 *)w, rows, cols, packed, scales);
    else
      k_quant_any<float><<<(unsigned)blocks, 256, 0, s>>>((const float *)w, rows, cols,
                                                          packed, scales);
  }
  return cudaGetLastError();
}

}  // namespace coli
