// Quantisers of the floating-point containers of the engine's format registry
// (page "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战" §权重转换:
// "2 int4-row", "7 MXFP4", "8 fp8-e4m3-b128"; "Colibrì 深度解析" §十 "从 int4 到
// MXFP4").  MXFP4 and fp8: one thread per row block.
//
// MXFP4 (OCP Microscaling v1.0), blocks of 32 columns: shared exponent
// se = floor(log2 max|w|) - 2 (2 = the largest E2M1 exponent), clamped to
// [-127, 127], stored as the byte se + 127; each element becomes the E2M1 code
// nearest to w / 2^se, ties to the even mantissa, saturating at 6, with w's
// sign in bit 3.
//
// fp8-e4m3-b128, blocks of 128 columns: f32 scale s = max|w| / 448; each
// element becomes the OCP E4M3 code nearest to w / s, ties to the even code,
// saturating at the largest finite value 448.
//
// int4-row ("2 int4-row"): the int4-grouped rule over a whole row, one CTA per
// row (a block-wide max, then a byte per thread and step).
#include <cuda_fp8.h>

#include "coli_internal.cuh"

namespace coli {
namespace {

// E2M1 magnitude code of a >= 0 (< 8) by the midpoints between the values
// 0, .5, 1, 1.5, 2, 3, 4, 6: a midpoint goes to the neighbour with the even
// mantissa (0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4,
// 5 -> 4), and everything above 5 to 6.
__device__ __forceinline__ int e2m1_code(float a) {
  return (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
         (a > 5.0f);
}

template <typename T>
__global__ void k_quant_mx(const T *__restrict__ w, int64_t rows, int64_t cols,
                           uint8_t *__restrict__ packed, uint8_t *__restrict__ scales) {
  const int64_t nb = (cols + kMxBlock - 1) / kMxBlock;
  const int64_t rb = (cols + 1) / 2;
  const int64_t total = rows * nb;
  for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total;
       id += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = id / nb, b = id - r * nb;
    const int64_t c0 = b * kMxBlock;
    const int n = (int)(c0 + kMxBlock < cols ? kMxBlock : cols - c0);
    const T *wr = w + r * cols + c0;
    float v[kMxBlock];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kMxBlock; ++i) {
      v[i] = i < n ? to_f32(wr[i]) : 0.0f;
      m = fmaxf(m, fabsf(v[i]));     // a NaN never raises the max
    }
    int se = -127;
    if (m > 0.0f) {
      int ex;
      frexpf(m, &ex);                // m = f 2^ex, f in [0.5, 1): floor(log2 m) = ex - 1
      se = ex - 1 - 2;
      se = se < -127 ? -127 : (se > 127 ? 127 : se);
    }
    scales[r * nb + b] = (uint8_t)(se + 127);
    uint8_t *pr = packed + r * rb + c0 / 2;
#pragma unroll
    for (int i = 0; i < kMxBlock; i += 2) {
      if (i >= n) break;
      int code[2] = {0, 0};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float x = v[i + j];
        if (i + j < n && m > 0.0f && x == x) {
          const float q = ldexpf(x, -se);          // x / 2^se, exact
          code[j] = e2m1_code(fabsf(q)) | (signbit(q) ? 8 : 0);
        }
      }
      pr[i / 2] = (uint8_t)(code[0] | (code[1] << 4));
    }
  }
}

template <typename T>
__global__ void k_quant_fp8(const T *__restrict__ w, int64_t rows, int64_t cols,
                            uint8_t *__restrict__ packed, float *__restrict__ scales) {
  const int64_t nb = (cols + kFp8Block - 1) / kFp8Block;
  const int64_t total = rows * nb;
  for (int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; id < total;
       id += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = id / nb, b = id - r * nb;
    const int64_t c0 = b * kFp8Block;
    const int n = (int)(c0 + kFp8Block < cols ? kFp8Block : cols - c0);
    const T *wr = w + r * cols + c0;
    float m = 0.0f;
    for (int i = 0; i < n; ++i) m = fmaxf(m, fabsf(to_f32(wr[i])));   // NaN never raises it
    const float s = __fdiv_rn(m, 448.0f);
    scales[r * nb + b] = s;
    uint8_t *pr = packed + r * cols + c0;
    for (int i = 0; i < n; ++i) {
      const float x = to_f32(wr[i]);
      uint8_t code = 0;
      // round to nearest, ties to even, saturating to the largest finite value;
      // the sign is taken from the quotient (a zero result keeps it too)
      if (s != 0.0f && x == x) {
        const float q = __fdiv_rn(x, s);
        code = (uint8_t)(__nv_cvt_float_to_fp8(fabsf(q), __NV_SATFINITE, __NV_E4M3) |
                         (signbit(q) ? 0x80 : 0));
      }
      pr[i] = code;
    }
  }
}

constexpr int kRowThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kRowThreads) k_quant_i4row(const T *__restrict__ w, int64_t rows,
                                                               int64_t cols,
                                                               uint8_t *__restrict__ packed,
                                                               float *__restrict__ scales) {
  __shared__ float s_max[kRowThreads / 32];
  const int64_t rb = (cols + 1) / 2;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T *wr = w + r * cols;
    float m = 0.0f;
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) m = fmaxf(m, fabsf(to_f32(wr[c])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
    __syncthreads();
    m = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, s_max[i]);   // NaN never wins
    __syncthreads();                     // s_max is reused by the next row
    const float s = __fdiv_rn(m, 7.0f);
    if (threadIdx.x == 0) scales[r] = s;
    for (int64_t j = threadIdx.x; j < rb; j += blockDim.x) {
      int u[2] = {8, 0};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t c = 2 * j + h;
        if (c >= cols) break;            // odd column count: the last high nibble stays 0
        int q = 0;
        if (s != 0.0f) {
          const float v = rintf(__fdiv_rn(to_f32(wr[c]), s));
          q = (v != v) ? 0 : (v < -8.0f ? -8 : (v > 7.0f ? 7 : (int)v));
        }
        u[h] = q + 8;
      }
      packed[r * rb + j] = (uint8_t)(u[0] | (u[1] << 4));
    }
  }
}

}  // namespace

cudaError_t launch_quant_i4row(const void *w, int w_dtype, int64_t rows, int64_t cols,
                               uint8_t *packed, float *scales, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorNoDevice;
  const int64_t blocks = rows < (int64_t)sms * 8 ? rows : (int64_t)sms * 8;
  if (w_dtype == COLI_BF16)
    k_quant_i4row<__nv_bfloat16><<<(unsigned)blocks, kRowThreads, 0, s>>>(
        (const __nv_bfloat16 *)w, rows, cols, packed, scales);
  else
    k_quant_i4row<float><<<(unsigned)blocks, kRowThreads, 0, s>>>((const float *)w, rows, cols,
                                                                   packed, scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_fp8b128(const void *w, int w_dtype, int64_t rows, int64_t cols,
                                 uint8_t *packed, float *scales, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorNoDevice;
  const int64_t total = rows * ((cols + kFp8Block - 1) / kFp8Block);
  int64_t blocks = (total + 127) / 128;
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  if (w_dtype == COLI_BF16)
    k_quant_fp8<__nv_bfloat16><<<(unsigned)blocks, 128, 0, s>>>((const __nv_bfloat16 *)w, rows,
                                                                 cols, packed, scales);
  else
    k_quant_fp8<float><<<(unsigned)blocks, 128, 0, s>>>((const float *)w, rows, cols, packed,
                                                         scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_mxfp4(const void *w, int w_dtype, int64_t rows, int64_t cols,
                               uint8_t *packed, uint8_t *scales, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const int sms = num_sms();
  if (sms <= 0) return cudaErrorNoDevice;
  const int64_t total = rows * ((cols + kMxBlock - 1) / kMxBlock);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
  if (w_dtype == COLI_BF16)
    k_quant_mx<__nv_bfloat16><<<(unsigned)blocks, 256, 0, s>>>((const __nv_bfloat16 *)w, rows,
                                                                cols, packed, scales);
  else
    k_quant_mx<float><<<(unsigned)blocks, 256, 0, s>>>((const float *)w, rows, cols, packed,
                                                        scales);
  return cudaGetLastError();
}

}  // namespace coli
