// Batched (prefill) path of the routed-MoE layer: many tokens per call.
//
// Pages: "Colibrì 深度解析" §四 / §十一 (route, group the batch's tokens by
// expert so that each expert's weights are read once, expert FFNs, combine);
// "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战" §权重转换 (the
// int4-grouped format the expert GEMMs dequantise).
//
//   k_x16       activations -> fp16 operand copy
//   k_plogits   router logits on tcgen05 tensor cores (bf16 x and router)
//   k_logits    router logits, tiled f32 SIMT GEMM (the other dtypes)
//   k_ptopk     top-k, gates, NaN flag and route counts (block-parallel top-k)
//   k_gcount / k_gscan / k_gscatter
//               counting sort of the routes by expert (stable in (token, slot)
//               order), expert m-tiles and the GEMM work list
//   k_pgemm<MODE, FMT>
//               token-sorted grouped GEMM on tcgen05 tensor cores: 128-row
//               m-tiles of one expert's routes x 256-column n-tiles, K in
//               steps of 64 (one scale group).  Eight producer warps stage the
//               activation rows with cp.async and dequantise the weight tile
//               (int4-grouped, or MXFP4 E2M1 codes with E8M0 scales) to fp16
//               into 128-byte-swizzled shared memory; one thread
//               issues tcgen05.mma (kind::f16, f32 accumulator in TMEM); four
//               epilogue warps drain TMEM:
//                 gate/up: h = silu(g) * u * gate  -> fp16 [route][F]
//                 down:    y                        -> f32  [route][H]
//   k_pcombine  out[t] = sum_j y[route(t, j)] + sum_s y[shared s, t] (+ residual)
#include <cuda_fp16.h>

#include "coli_internal.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace coli {

namespace {

constexpr int kBM = 128;          // m-tile rows (routes)
constexpr int kBK = 64;           // K per k-tile: one scale group
constexpr int kBN = 256;          // n-tile columns (gate/up: 128 gate + 128 up)
constexpr int kProducerWarps = 8; // two weight-row halves and four activation pieces per thread
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr int kMmaWarp = kProducerWarps;
constexpr int kEpilogueWarps = 4;
constexpr int kEpilogueThreads = 32 * kEpilogueWarps;
constexpr int kGemmThreads = 32 * (kProducerWarps + 1 + kEpilogueWarps);
constexpr int kATileBytes = kBM * kBK * 2;     // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;     // 32 KB
// Raw slot: the k-tile's bytes of every weight row as each thread copied
// them -- [2 rows][chunks][kProducerThreads] 16-byte chunks, a thread's
// chunks covering columns 32 (th % 2) .. + 31 of its rows -- then one 4-byte
// scale word per row half.
constexpr int kRawHalves = 2 * kProducerThreads;
constexpr int kARowPasses = kBM * 8 / kProducerThreads;        // 128-byte rows: 8 threads each
constexpr int kTableBytes = 2 * (kMaxExperts + kMaxShared + 1) * 4;   // item_begin, offsets

// Ring depths per weight container.  A 4-bit row brings 32 bytes per k-tile
// (one 16-byte chunk per thread and row); an fp8 row 64 (two chunks), so its
// raw slots are twice as large and the A and raw rings one stage shallower,
// to stay within one block's shared memory.
template <int FMT>
struct Geo {
  static constexpr int kNA = 5;      // A ring (fp16 activation tiles)
  static constexpr int kNB = 3;      // B ring (dequantised fp16 weight tiles)
  static constexpr int kNR = 4;      // raw ring (weight rows + scales as copied)
  static constexpr int kDist = 3;    // copies run this many k-tiles ahead of the dequantisation
  static constexpr int kChunks = 1;  // 16-byte chunks per thread, row and k-tile
};
template <>
struct Geo<COLI_FMT_FP8> {
  static constexpr int kNA = 4, kNB = 3, kNR = 3, kDist = 2, kChunks = 2;
};
template <int FMT>
struct GeoBytes {
  using G = Geo<FMT>;
  static constexpr int kRawData = kRawHalves * 16 * G::kChunks;   // 8 KB (4-bit), 16 KB (fp8)
  static constexpr int kRaw = kRawData + kRawHalves * 4;          // + 2 KB scale words
  static constexpr int kSmem =
      G::kNA * kATileBytes + G::kNB * kBTileBytes + G::kNR * kRaw + kTableBytes + 2048;
  static_assert(G::kNR > G::kDist, "a raw slot is refilled only after its dequantisation");
  // an A tile is copied kDist ticks before its dequantisation tick and is
  // free again only after the MMA of that k-tile: a shallower ring stalls the
  // producers until their bounded waits give up
  static_assert(G::kNA >= G::kDist + 2, "A ring deep enough for the copy distance");
  static_assert(kSmem <= 232448, "shared memory of one block");
};
static_assert(kProducerThreads == kBN, "a thread pair per B row, two rows per pair");
static_assert(kRawHalves == 2 * kBN && kARowPasses * kProducerThreads == 8 * kBM,
              "copy shares of the producers");

enum GemmMode : int { kModeGateUp = 0, kModeDown = 1 };

__device__ __forceinline__ void set_flag_p(uint32_t *ctrl, uint32_t f) {
  atomicOr(ctrl + kCtrlFlags, f);
}

// Either fp16 of the pair is +-inf (exponent all ones, mantissa zero).
__device__ __forceinline__ bool half2_has_inf(uint32_t w) {
  return (w & 0x7FFFu) == 0x7C00u || (w & 0x7FFF0000u) == 0x7C000000u;
}

// ---------------------------------------------------------------------------
// tcgen05 / TMEM helpers (inline PTX)

__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, M = 128, N from idesc, K = 16.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The mbarrier completes one arrival when all earlier tcgen05 ops of this thread finish.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i gets lane (taddr.lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile stored as rows of 128
// bytes (64 fp16) with the 128-byte swizzle: 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) /* LBO 16 B (unused) */ |
         ((uint64_t)(1024 >> 4) << 32) /* SBO */ | ((uint64_t)1 << 46) /* descriptor version */ |
         ((uint64_t)2 << 61) /* 128-byte swizzle */;
}
// Instruction descriptor, kind::f16: f32 accumulator, fp16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int n, int m) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}
// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void st_shared16(uint32_t dst, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 8 packed bytes (16 int4 values, even column low nibble) -> 8 fp16x2 words of
// (u - 8) * s.  For byte j the pair (2j, 2j+1) is built exactly as fp16
// 1024 + u_even and 1024 + 16 u_odd, mapped to (u - 8) by one fused
// multiply-add (x1, x1/16), then scaled.
__device__ __forceinline__ void dequant8(uint32_t w0, uint32_t w1, __half2 s2, uint32_t (&o)[8]) {
  const __half2 mul = __halves2half2(__float2half_rn(1.0f), __float2half_rn(1.0f / 16.0f));
  const __half2 add = __halves2half2(__float2half_rn(-1032.0f), __float2half_rn(-72.0f));
  const uint32_t ws[2] = {w0, w1};
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t t = __byte_perm(ws[i], 0, 0x4040u | (j * 0x0101u));
      const uint32_t m = (t & 0x00F0000Fu) | 0x64006400u;
      __half2 h = *reinterpret_cast<const __half2 *>(&m);
      h = __hfma2(h, mul, add);
      h = __hmul2(h, s2);
      o[4 * i + j] = *reinterpret_cast<const uint32_t *>(&h);
    }
}

// 8 packed bytes of MXFP4 (16 E2M1 codes, even column low nibble) -> 8 fp16x2
// words of e2m1(code) * X.  The eight E2M1 magnitudes are exact fp16 numbers
// whose low bytes are zero: a byte permute of the 3-bit magnitude codes picks
// their high bytes from a table, the code's sign bit goes to the fp16 sign,
// and the power-of-two scale X (as fp16) multiplies exactly while the product
// stays in the fp16 range.
__device__ __forceinline__ void dequant8_mx(uint32_t w0, uint32_t w1, __half2 s2, uint32_t (&o)[8]) {
  constexpr uint32_t kMagLo = 0x3E3C3800u;   // fp16 high bytes of 0, 0.5, 1, 1.5
  constexpr uint32_t kMagHi = 0x46444240u;   //                    2, 3, 4, 6
  const uint32_t ws[2] = {w0, w1};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w = ws[i];
    const uint32_t m = w & 0x77777777u;
    const uint32_t r0 = __byte_perm(kMagLo, kMagHi, m);         // columns 0..3 of the word
    const uint32_t r1 = __byte_perm(kMagLo, kMagHi, m >> 16);   // columns 4..7
    uint32_t h[4];
    h[0] = __byte_perm(r0, 0, 0x1404) | ((w << 12) & 0x8000u) | ((w << 24) & 0x80000000u);
    h[1] = __byte_perm(r0, 0, 0x3424) | ((w << 4) & 0x8000u) | ((w << 16) & 0x80000000u);
    h[2] = __byte_perm(r1, 0, 0x1404) | ((w >> 4) & 0x8000u) | ((w << 8) & 0x80000000u);
    h[3] = __byte_perm(r1, 0, 0x3424) | ((w >> 12) & 0x8000u) | (w & 0x80000000u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 v = *reinterpret_cast<const __half2 *>(&h[j]);
      v = __hmul2(v, s2);
      o[4 * i + j] = *reinterpret_cast<const uint32_t *>(&v);
    }
  }
}

// 16 fp8 E4M3 codes (one per byte, column order) -> 8 fp16x2 words of
// e4m3(code) * X.  Moving a code's exponent and mantissa bits (6..0) to fp16
// bits 13..7 and its sign to bit 15 gives exactly e4m3(code) * 2^-8: the
// exponent biases differ by 8 (15 - 7), and E4M3 subnormals (exponent 0,
// m 2^-9) land on fp16 subnormals of the same mantissa.  The caller passes
// X = s * 256 as fp16.
__device__ __forceinline__ void dequant16_fp8(uint4 w, __half2 s2, uint32_t (&o)[8]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      // codes 2j, 2j + 1 of the word into bytes 1 and 3
      const uint32_t t = __byte_perm(ws[i], 0, j ? 0x3424u : 0x1404u);
      const uint32_t h = (t & 0x80008000u) | ((t >> 1) & 0x3F803F80u);
      __half2 v = *reinterpret_cast<const __half2 *>(&h);
      v = __hmul2(v, s2);
      o[2 * i + j] = *reinterpret_cast<const uint32_t *>(&v);
    }
}

// The E8M0 scale byte e as an fp16 pair: 2^(e - 127) (255: NaN).
__device__ __forceinline__ __half2 e8m0_half2(uint32_t e) {
  const float x = e == 255u ? __int_as_float(0x7FC00000) : ldexpf(1.0f, (int)e - 127);
  return __float2half2_rn(x);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// A GEMM work item: expert e, n-tile ni, and the rows [p0, p0 + rows) of its
// m-tile in route order.  Items are ordered (expert, n-tile, m-tile);
// begin[] (shared memory) holds the experts' m-tile prefix, off[] their
// first route position.
struct Item {
  int e, ni, p0, rows;
};
__device__ __forceinline__ Item decode_item(const int *begin, const int *off, int n_groups, int w,
                                            int n_ntiles) {
  int lo = 0, hi = n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (begin[mid] * n_ntiles <= w) lo = mid; else hi = mid;
  }
  Item it;
  it.e = lo;
  const int nm = begin[lo + 1] - begin[lo];
  const int local = w - begin[lo] * n_ntiles;
  it.ni = local / nm;
  const int mi = local - it.ni * nm;
  it.p0 = off[lo] + mi * kBM;
  const int left = off[lo + 1] - it.p0;
  it.rows = left < kBM ? left : kBM;
  return it;
}

}  // namespace

// ---------------------------------------------------------------------------
// Activations to fp16 (exact for bf16 inputs inside the fp16 range), 8
// elements (one 16-byte store) per thread and step; n is a multiple of 8.

__device__ __forceinline__ void load8(const __nv_bfloat16 *src, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(src);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    v[2 * j] = __uint_as_float(w[j] << 16);
    v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load8(const float *src, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(src);
  const float4 b = *reinterpret_cast<const float4 *>(src + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename XT>
__global__ void k_x16(const XT *x, __half *x16, int64_t n, uint32_t *ctrl) {
  bool inf = false;
  for (int64_t i = 8 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x); i < n;
       i += 8 * (int64_t)gridDim.x * blockDim.x) {
    float v[8];
    load8(x + i, v);
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
      o[j] = *reinterpret_cast<const uint32_t *>(&h);
      inf |= half2_has_inf(o[j]);
    }
    *reinterpret_cast<uint4 *>(x16 + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (inf) set_flag_p(ctrl, COLI_FLAG_RANGE);
}

// ---------------------------------------------------------------------------
// Router logits [T][E] = x [T][H] . Wr [E][H]^T, f32 accumulation.  64 x 64
// tiles, K in steps of 32 through shared memory (stored k-major, so each
// thread reads its 4 x 4 operands as two float4); 256 threads x (4 x 4), each
// output a sequential fmaf chain over k.  Thread (r, q) fetches 8 consecutive
// k of row r for the next step into registers while the current one computes.

template <typename XT, typename WT>
__global__ void __launch_bounds__(256) k_logits(const XT *x, const WT *wr, float *logits, int T,
                                                int H, int E) {
  __shared__ __align__(16) float sx[32][68];
  __shared__ __align__(16) float sw[32][68];
  const int t0 = blockIdx.y * 64, e0 = blockIdx.x * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int lr = threadIdx.x & 63, lq = threadIdx.x >> 6;     // fetch: row lr, k 8 lq .. + 7
  const bool x_ok = t0 + lr < T, w_ok = e0 + lr < E;
  const XT *xs = x + (size_t)(x_ok ? t0 + lr : 0) * H + 8 * lq;
  const WT *ws = wr + (size_t)(w_ok ? e0 + lr : 0) * H + 8 * lq;
  float rx[8], rw[8];
  auto fetch = [&](int k0) {
    if (x_ok) load8(xs + k0, rx);
    else
#pragma unroll
      for (int j = 0; j < 8; ++j) rx[j] = 0.0f;
    if (w_ok) load8(ws + k0, rw);
    else
#pragma unroll
      for (int j = 0; j < 8; ++j) rw[j] = 0.0f;
  };
  float acc[4][4] = {};
  fetch(0);
  for (int k0 = 0; k0 < H; k0 += 32) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sx[8 * lq + j][lr] = rx[j];
      sw[8 * lq + j][lr] = rw[j];
    }
    __syncthreads();
    if (k0 + 32 < H) fetch(k0 + 32);
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      const float4 a4 = *reinterpret_cast<const float4 *>(&sx[kk][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4 *>(&sw[kk][tx * 4]);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w};
      const float b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = t0 + ty * 4 + i, e = e0 + tx * 4 + j;
      if (t < T && e < E) logits[(size_t)t * E + e] = acc[i][j];
    }
}

// ---------------------------------------------------------------------------
// Router logits on the tensor cores when x and the router are both bf16:
// logits [T][E] = x [T][H] . Wr [E][H]^T with tcgen05.mma kind::f16 (bf16
// operands, exact products, f32 accumulation in TMEM).  One CTA per 128-token
// x 256-expert tile, K in steps of 64 (128-byte rows, the grouped GEMM's
// swizzled layout).  Eight producer warps copy both operand tiles with
// cp.async (kLgStages stages, kLgDist tiles ahead); one thread issues the
// MMAs; four warps write the f32 logits.  Rows past T and experts past E are
// not copied and never stored.  The sum order differs from k_logits' fmaf
// chain only by rounding; token inputs keep a gap between ranked logits.

constexpr int kLgStages = 4, kLgDist = 3;
constexpr int kLgATile = kBM * kBK * 2;             // 16 KB
constexpr int kLgBTile = kBN * kBK * 2;             // 32 KB
constexpr int kLgSmem = kLgStages * (kLgATile + kLgBTile) + 1024 + 256;
static_assert(kLgStages > kLgDist, "a stage is refilled only after the MMA that read it");
static_assert(kLgSmem <= 232448, "shared memory of one block");

__host__ __device__ constexpr uint32_t idesc_bf16(int n, int m) {
  return idesc_f16(n, m) | (1u << 7) | (1u << 10);   // A and B formats: BF16
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    k_plogits(const __nv_bfloat16 *__restrict__ x, const __nv_bfloat16 *__restrict__ wr,
              float *__restrict__ logits, int T, int H, int E, uint32_t *ctrl) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *a_ring = smem;                                     // stages x 16 KB
  uint8_t *b_ring = a_ring + kLgStages * kLgATile;            // stages x 32 KB
  uint64_t *full = (uint64_t *)(b_ring + kLgStages * kLgBTile);
  uint64_t *empty = full + kLgStages;
  uint64_t *acc_full = empty + kLgStages;
  uint64_t *mma_done = acc_full + 1;
  uint32_t *s_taddr = (uint32_t *)(mma_done + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
  const int nk = H / kBK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLgStages; ++s) {
      mbar_init(&full[s], kProducerThreads);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_taddr, kBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependents_launch();
  grid_dependency_wait();
  const uint32_t tbase = *s_taddr;
  const uint32_t lim_word = __ldcg(ctrl + kCtrlWaitLimit);
  const long long lim = lim_word ? (long long)lim_word : kWaitCycles;

  if (warp < kProducerWarps) {
    // 8 threads per 128-byte row: A rows th/8 + 32 j (4 passes), B rows th/8 + 32 j (8)
    const int th = threadIdx.x, chunk = th & 7, row0 = th >> 3;
    bool ok = true;
    for (int t = 0; t < nk + kLgDist && ok; ++t) {
      if (t < nk) {
        const int st = t % kLgStages;
        if (!mbar_wait(&empty[st], ((t / kLgStages) & 1) ^ 1, lim)) { ok = false; break; }
        const uint32_t a_dst = smem_u32(a_ring + st * kLgATile);
        const uint32_t b_dst = smem_u32(b_ring + st * kLgBTile);
        const int k0 = t * kBK + 8 * chunk;
#pragma unroll
        for (int j = 0; j < kBM / 32; ++j) {
          const int r = row0 + 32 * j;
          if (m0 + r < T) cp16(a_dst + sw128_off(r, chunk), x + (size_t)(m0 + r) * H + k0);
        }
#pragma unroll
        for (int j = 0; j < kBN / 32; ++j) {
          const int r = row0 + 32 * j;
          if (n0 + r < E) cp16(b_dst + sw128_off(r, chunk), wr + (size_t)(n0 + r) * H + k0);
        }
      }
      cp_commit();
      const int c = t - kLgDist;
      if (c < 0) continue;
      cp_wait<kLgDist>();          // this thread's copies of tile c have landed
      fence_proxy_async();         // generic-proxy writes -> tensor core reads
      mbar_arrive(&full[c % kLgStages]);
    }
    cp_wait<0>();
    if (!ok) set_flag_p(ctrl, COLI_FLAG_TIMEOUT);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kBN, kBM);
      bool ok = true;
      for (int c = 0; c < nk; ++c) {
        const int st = c % kLgStages;
        if (!mbar_wait(&full[st], (c / kLgStages) & 1, lim)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(a_ring + st * kLgATile);
        const uint32_t b0 = smem_u32(b_ring + st * kLgBTile);
#pragma unroll
        for (int k16 = 0; k16 < kBK / 16; ++k16)
          tc_mma(tbase, sw128_desc(a0 + 32 * k16), sw128_desc(b0 + 32 * k16), idesc,
                 (c | k16) != 0);
        tc_commit(&empty[st]);
      }
      if (ok) tc_commit(acc_full);
      else set_flag_p(ctrl, COLI_FLAG_TIMEOUT);
      // every MMA issued has completed before TMEM is freed
      tc_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) set_flag_p(ctrl, COLI_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else {
    // epilogue: TMEM lane quarter (warp % 4) holds tile rows 32 (warp % 4) + lane
    const int q = warp & 3;
    const int r = 32 * q + lane;
    if (mbar_wait(acc_full, 0, lim)) {
      tc_fence_after();
      const uint32_t trow = tbase + ((uint32_t)(32 * q) << 16);
      for (int cc = 0; cc < kBN; cc += 32) {
        uint32_t v[32];
        tmem_ld32(trow + cc, v);
        tmem_ld_wait();
        if (m0 + r < T) {
          float *dst = logits + (size_t)(m0 + r) * E + n0 + cc;
          if (n0 + cc + 32 <= E && (E & 3) == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              ((float4 *)dst)[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                               __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          } else {
            for (int j = 0; j < 32; ++j)
              if (n0 + cc + j < E) dst[j] = __uint_as_float(v[j]);
          }
        }
      }
    } else {
      set_flag_p(ctrl, COLI_FLAG_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, kBN);
}

// ---------------------------------------------------------------------------
// Top-k of kPTopkTokens tokens per block (the decode path's block top-k).

constexpr int kPTopkTokens = 8;

__global__ void __launch_bounds__(256) k_ptopk(PrefillArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int T = p.T, E = p.E, k = p.k;
  const int t0 = blockIdx.x * kPTopkTokens;
  const int TB = (T - t0 < kPTopkTokens) ? T - t0 : kPTopkTokens;
  const size_t lg_bytes = ((size_t)kPTopkTokens * E * 4 + 15) & ~(size_t)15;
  float *lg = (float *)smem;                                      // [kPTopkTokens][E]
  float *sel = (float *)(smem + lg_bytes);                        // [kPTopkTokens][E]
  uint8_t *s_tk = smem + 2 * lg_bytes;                            // top-k scratch
  int *s_idx = (int *)(s_tk + ((topk_scratch_bytes(kPTopkTokens, E, k) + 15) & ~(size_t)15));
  float *s_gates = (float *)(s_idx + kPTopkTokens * k);
  float *s_vals = s_gates + kPTopkTokens * k;
  int *s_flag = (int *)(s_vals + kPTopkTokens * k);
  for (int i = threadIdx.x; i < TB * E; i += blockDim.x) lg[i] = p.logits[(size_t)t0 * E + i];
  __syncthreads();
  const bool sig = p.router_fn == COLI_ROUTER_SIGMOID_BIAS;
  if (sig) sigmoid_keys(lg, sel, p.router_bias, TB, E);
  const bool nan = select_topk(sig ? sel : lg, TB, E, k, s_idx, s_gates, s_vals, s_tk, s_flag);
  if (sig) sigmoid_gates(lg, s_idx, TB, E, k, s_gates);
  if (threadIdx.x == 0 && nan) set_flag_p(p.ctrl, COLI_FLAG_NAN_LOGITS);
  for (int i = threadIdx.x; i < TB * k; i += blockDim.x) {
    p.idx[(size_t)t0 * k + i] = s_idx[i];
    p.gates[(size_t)t0 * k + i] = s_gates[i];
    if (p.route_counts) atomicAdd(p.route_counts + COLI_CHK(s_idx[i], p.E, p.ctrl), 1u);
  }
}

// ---------------------------------------------------------------------------
// Counting sort of the T*k routes by expert.  Block b owns tokens
// [b * kGroupTokens, ...): k_gcount histograms them, k_gscan turns the
// histograms into per-(block, expert) start positions and lays out the expert
// m-tiles and GEMM work items, k_gscatter places every route in (token, slot)
// order within its block.  Shared expert s serves all T tokens at positions
// T*k + s*T + t.

__global__ void __launch_bounds__(256) k_gcount(PrefillArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  int *hist = (int *)smem;
  const int E = p.E, k = p.k;
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kGroupTokens;
  const int t1 = (t0 + kGroupTokens < p.T) ? t0 + kGroupTokens : p.T;
  for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) atomicAdd(hist + p.idx[i], 1);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += blockDim.x) p.hist[(size_t)blockIdx.x * E + i] = hist[i];
}

// One block: expert offsets (routed experts, then the shared ones), the
// per-(block, expert) start positions (in place of the histograms), m-tile
// counts and the work-item prefix of the GEMMs.
__global__ void __launch_bounds__(1024) k_gscan(PrefillArgs p, int n_blocks) {
  __shared__ int s_cnt[kMaxExperts + kMaxShared + 1];
  __shared__ int s_items[kMaxExperts + kMaxShared + 1];
  const int E = p.E, S = p.S, T = p.T, G = E + S;
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    int n = T;
    if (e < E) {
      n = 0;
      for (int b = 0; b < n_blocks; ++b) {
        const int c = p.hist[(size_t)b * E + e];
        p.hist[(size_t)b * E + e] = n;       // start of block b within expert e
        n += c;
      }
    }
    s_cnt[e] = n;
    s_items[e] = (n + kBM - 1) / kBM;        // m-tiles of expert e
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, it = 0;
    for (int e = 0; e < G; ++e) {
      p.offsets[e] = off;
      p.item_begin[e] = it;
      off += s_cnt[e];
      it += s_items[e];
    }
    p.offsets[G] = off;
    p.item_begin[G] = it;           // m-tiles in total; the GEMMs scale by their n-tiles
    p.ctrl[kCtrlPrefillMTiles] = (uint32_t)it;
  }
}

__global__ void __launch_bounds__(256) k_gscatter(PrefillArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int E = p.E, k = p.k, T = p.T;
  int *base = (int *)smem;                  // [E] next position of each expert in this block
  const int t0 = blockIdx.x * kGroupTokens;
  const int t1 = (t0 + kGroupTokens < T) ? t0 + kGroupTokens : T;
  const int n = (t1 - t0) * k;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    base[e] = p.offsets[e] + p.hist[(size_t)blockIdx.x * E + e];
  __syncthreads();
  // The block's routes in (token, slot) order, blockDim.x at a time: a route's
  // place is its expert's next position plus the number of earlier routes of
  // the same expert, counted inside the warp by a match and across warps by
  // letting the warps take their experts' positions one after another.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, n_warps = blockDim.x >> 5;
  const unsigned lower = (1u << lane) - 1u;
  for (int c0 = 0; c0 < n; c0 += blockDim.x) {
    const int i = c0 + threadIdx.x;
    const int g = t0 * k + i;
    const int e = i < n ? p.idx[g] : -1;
    const unsigned same = __match_any_sync(~0u, e);
    const int leader = __ffs(same) - 1;
    int first = 0;
    for (int w = 0; w < n_warps; ++w) {
      if (warp == w && lane == leader && e >= 0) {
        first = base[e];
        base[e] = first + __popc(same);
      }
      __syncthreads();
    }
    first = __shfl_sync(~0u, first, leader);
    if (e >= 0) {
      const int pos = COLI_CHK(first + __popc(same & lower), T * (k + p.S), p.ctrl);
      p.route_tok[pos] = g / k;
      p.route_gate[pos] = p.gates[g];
      p.inv[g] = pos;
    }
  }
  // shared experts: every token, in order
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.S * T; i += gridDim.x * blockDim.x) {
    const int pos = T * k + i;
    p.route_tok[pos] = i % T;
    p.route_gate[pos] = 1.0f;
  }
}

// ---------------------------------------------------------------------------
// The grouped GEMM.

// FMT: COLI_FMT_I4G (one f32 scale per row and k-tile), COLI_FMT_I4ROW (one
// f32 scale per row), COLI_FMT_MXFP4 (one E8M0 byte per row and 32 columns: a
// thread's half of the k-tile has exactly one; the copy brings the aligned
// 4-byte word that holds it) or COLI_FMT_FP8 (one f32 scale per row and two
// k-tiles).
template <int MODE, int FMT>
__global__ void __launch_bounds__(kGemmThreads, 1) k_pgemm(PrefillArgs p) {
  using G = Geo<FMT>;
  constexpr int kNA = G::kNA, kNB = G::kNB, kNR = G::kNR, kDist = G::kDist, kCh = G::kChunks;
  constexpr int kRawData = GeoBytes<FMT>::kRawData, kRawBytes = GeoBytes<FMT>::kRaw;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *a_ring = smem;                                  // kNA x 16 KB (fp16, swizzled)
  uint8_t *b_ring = a_ring + kNA * kATileBytes;            // kNB x 32 KB (fp16, swizzled)
  uint8_t *r_ring = b_ring + kNB * kBTileBytes;            // kNR x raw nibble halves + scales
  uint64_t *full = (uint64_t *)(r_ring + kNR * kRawBytes);
  uint64_t *a_empty = full + kNB;
  uint64_t *b_empty = a_empty + kNA;
  uint64_t *tm_full = b_empty + kNB;                       // [2]
  uint64_t *tm_empty = tm_full + 2;                        // [2]
  uint64_t *mma_done = tm_empty + 2;                       // the MMA thread's last commit
  uint32_t *s_taddr = (uint32_t *)(mma_done + 1);
  int *s_abort = (int *)(s_taddr + 1);
  int *s_begin = s_abort + 4;                              // [n_groups + 1]
  int *s_off = s_begin + (kMaxExperts + kMaxShared + 1);   // [n_groups + 1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, F = p.F;
  const int K = MODE == kModeGateUp ? H : F;
  const int nk = K / kBK;
  const int n_ntiles = MODE == kModeGateUp ? F / (kBN / 2) : H / kBN;
  const int P_routes = p.T * (p.k + p.S);    // rows of h16 / y, entries of route_tok
  (void)P_routes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNB; ++s) {
      mbar_init(&full[s], kProducerThreads);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < kNA; ++s) mbar_init(&a_empty[s], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tm_full[b], 1);
      mbar_init(&tm_empty[b], kEpilogueThreads);
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(s_taddr, 2 * kBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dependents_launch();
  grid_dependency_wait();
  for (int i = threadIdx.x; i <= p.n_groups; i += blockDim.x) {
    s_begin[i] = __ldcg(p.item_begin + i);
    s_off[i] = __ldcg(p.offsets + i);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_taddr;
  const int n_items = s_begin[p.n_groups] * n_ntiles;
  const int my_items = n_items > (int)blockIdx.x ? (n_items - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int n_ticks = my_items * nk;         // this CTA's k-tiles over all its items
  const uint32_t lim_word = __ldcg(p.ctrl + kCtrlWaitLimit);
  const long long lim = lim_word ? (long long)lim_word : kWaitCycles;   // pipeline waits

  if (warp < kProducerWarps) {
    // ---- producers: tick t issues the copies of k-tile t (A rows, raw B
    // rows) and dequantises k-tile t - kDist into the B ring.  Copies are laid
    // out so that each warp instruction reads whole lines: for A, 8 threads
    // per 128-byte activation row (rows th/8 + 32 j); for B, a thread pair per
    // 32-byte weight sector (rows th/2 and th/2 + 128, half th % 2).  A thread
    // dequantises only the halves it copied itself, so its own cp.async wait
    // is the only one it needs.  A rows past the item's last route are left
    // as they are: they reach only accumulator rows that are never stored.
    const int th = threadIdx.x;
    const int a_chunk = th & 7, a_row0 = th >> 3;
    const int b_half = th & 1, b_row0 = th >> 1;
    Item it{};
    const __half *a_src[kARowPasses];
    bool a_ok[kARowPasses];
    const uint8_t *b_src[2];
    const uint8_t *b_sc[2];          // the row's scales (bytes)
    bool ok = true;
    int item = 0, kt = 0;                  // k-tile t = item * nk + kt
    for (int t = 0; t < n_ticks + kDist && ok; ++t) {
      if (t < n_ticks) {
        if (kt == 0) {
          it = decode_item(s_begin, s_off, p.n_groups, blockIdx.x + item * gridDim.x, n_ntiles);
          it.e = COLI_CHK(it.e, p.n_groups, p.ctrl);
#pragma unroll
          for (int j = 0; j < kARowPasses; ++j) {
            const int r = a_row0 + 32 * j;
            a_ok[j] = r < it.rows;
            a_src[j] = nullptr;
            if (a_ok[j])
              a_src[j] = MODE == kModeGateUp
                             ? p.x16 + (int64_t)COLI_CHK(p.route_tok[COLI_CHK(it.p0 + r, P_routes, p.ctrl)],
                                                         p.T, p.ctrl) * H
                             : p.h16 + (int64_t)COLI_CHK(it.p0 + r, P_routes, p.ctrl) * F;
          }
          const uint8_t *pk;
          const uint8_t *sc;
          if (FMT != COLI_FMT_I4G) {
            pk = p.packed + (int64_t)it.e * p.eb;
            sc = (const uint8_t *)p.scales + (int64_t)it.e * p.es;
          } else {
            const float *scf;
            expert_record(p.tier, p.packed, p.scales, p.eb, p.es, it.e, &pk, &scf);
            sc = (const uint8_t *)scf;
          }
          // bytes of one row (K columns) and of its scales, for the
          // gate/up (K = H) and down (K = F) matrices
          const int64_t rh = FMT == COLI_FMT_FP8 ? H : H / 2;
          const int64_t rf = FMT == COLI_FMT_FP8 ? F : F / 2;
          const int64_t sh = FMT == COLI_FMT_MXFP4 ? H / kMxBlock
                             : FMT == COLI_FMT_FP8 ? 4 * (H / kFp8Block)
                             : FMT == COLI_FMT_I4ROW ? 4 : 4 * (H / kGroup);
          const int64_t sf = FMT == COLI_FMT_MXFP4 ? F / kMxBlock
                             : FMT == COLI_FMT_FP8 ? 4 * (F / kFp8Block)
                             : FMT == COLI_FMT_I4ROW ? 4 : 4 * (F / kGroup);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (MODE == kModeGateUp) {
              // B rows 0..127 are gate rows, 128..255 the up rows of the same f
              const int f = it.ni * (kBN / 2) + b_row0;
              const int64_t mat = j;
              b_src[j] = pk + mat * (int64_t)F * rh + (int64_t)f * rh;
              b_sc[j] = sc + mat * (int64_t)F * sh + (int64_t)f * sh;
            } else {
              const int hr = it.ni * kBN + b_row0 + 128 * j;
              b_src[j] = pk + 2 * (int64_t)F * rh + (int64_t)hr * rf;
              b_sc[j] = sc + (int64_t)2 * F * sh + (int64_t)hr * sf;
            }
          }
        }
        const int sa = t % kNA;
        if (!mbar_wait(&a_empty[sa], ((t / kNA) & 1) ^ 1, lim)) { ok = false; break; }
        const uint32_t a_dst = smem_u32(a_ring + sa * kATileBytes);
        const int k0 = kt * kBK;
#pragma unroll
        for (int j = 0; j < kARowPasses; ++j)
          if (a_ok[j]) cp16(a_dst + sw128_off(a_row0 + 32 * j, a_chunk), a_src[j] + k0 + 8 * a_chunk);
        uint8_t *raw = r_ring + (t % kNR) * kRawBytes;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int ch = 0; ch < kCh; ++ch)
            cp16(smem_u32(raw + ((j * kCh + ch) * kProducerThreads + th) * 16),
                 b_src[j] + (k0 + 32 * b_half) * kCh / 2 + 16 * ch);
          // int4-grouped: the k-tile's f32 scale; MXFP4: the word holding its
          // two E8M0 bytes; fp8: the f32 scale of the 128 columns holding the
          // k-tile; int4-row: the row's scale
          cp4(smem_u32(raw + kRawData + (j * kProducerThreads + th) * 4),
              b_sc[j] + (FMT == COLI_FMT_I4G ? kt * 4 : FMT == COLI_FMT_I4ROW ? 0 : (kt >> 1) * 4));
        }
        if (++kt == nk) { kt = 0; ++item; }
      }
      cp_commit();
      const int c = t - kDist;
      if (c < 0) continue;
      cp_wait<kDist>();            // groups of ticks <= c have landed (this thread's copies)
      const int sb = c % kNB;
      if (!mbar_wait(&b_empty[sb], ((c / kNB) & 1) ^ 1, lim)) { ok = false; break; }
      const uint8_t *raw = r_ring + (c % kNR) * kRawBytes;
      const uint32_t b_dst = smem_u32(b_ring + sb * kBTileBytes);
      const int kt_c = c % nk;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int slot = j * kProducerThreads + th;
        const uint32_t sw = *(const uint32_t *)(raw + kRawData + slot * 4);
        const __half2 s2 = FMT == COLI_FMT_MXFP4
                               ? e8m0_half2((sw >> (8 * (2 * (kt_c & 1) + b_half))) & 0xFFu)
                           : FMT == COLI_FMT_FP8 ? __float2half2_rn(__uint_as_float(sw) * 256.0f)
                                                 : __float2half2_rn(__uint_as_float(sw));
        const int row = b_row0 + 128 * j;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          // columns 32 b_half + 16 q .. + 15: 16-byte chunks 4 b_half + 2 q, + 1
          uint32_t o[8];
          if (FMT == COLI_FMT_FP8) {
            const uint4 w = *(const uint4 *)(raw + ((j * kCh + q) * kProducerThreads + th) * 16);
            dequant16_fp8(w, s2, o);
          } else {
            const uint4 w = *(const uint4 *)(raw + slot * 16);
            const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
            if (FMT == COLI_FMT_MXFP4) dequant8_mx(wd[2 * q], wd[2 * q + 1], s2, o);
            else dequant8(wd[2 * q], wd[2 * q + 1], s2, o);
          }
          st_shared16(b_dst + sw128_off(row, 4 * b_half + 2 * q), o[0], o[1], o[2], o[3]);
          st_shared16(b_dst + sw128_off(row, 4 * b_half + 2 * q + 1), o[4], o[5], o[6], o[7]);
        }
      }
      fence_proxy_async();         // A (landed copies) and B of k-tile c -> tensor core reads
      mbar_arrive(&full[sb]);
    }
    cp_wait<0>();
    if (!ok) {
      set_flag_p(p.ctrl, COLI_FLAG_TIMEOUT);
      *(volatile int *)s_abort = 1;
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer (one lane)
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kBN, kBM);
      for (int c = 0; c < n_ticks; ++c) {
        const int item = c / nk, kt = c % nk, buf = item & 1;
        const uint32_t acc = tbase + (uint32_t)(buf * kBN);
        const int sb = c % kNB, sa = c % kNA;
        if ((kt == 0 && !mbar_wait(&tm_empty[buf], ((item >> 1) & 1) ^ 1, lim)) ||
            !mbar_wait(&full[sb], (c / kNB) & 1, lim)) {
          set_flag_p(p.ctrl, COLI_FLAG_TIMEOUT);
          break;
        }
        if (*(volatile int *)s_abort) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(a_ring + sa * kATileBytes);
        const uint32_t b0 = smem_u32(b_ring + sb * kBTileBytes);
#pragma unroll
        for (int k16 = 0; k16 < kBK / 16; ++k16)
          tc_mma(acc, sw128_desc(a0 + 32 * k16), sw128_desc(b0 + 32 * k16), idesc,
                 (kt | k16) != 0);
        tc_commit(&a_empty[sa]);
        tc_commit(&b_empty[sb]);
        if (kt == nk - 1) tc_commit(&tm_full[buf]);
      }
      // Whether the loop ran to its end or gave up, wait until every MMA this
      // thread issued has completed, so that none is in flight when TMEM is
      // freed (an abandoned item's accumulator is never read).
      tc_commit(mma_done);
      if (!mbar_wait(mma_done, 0)) set_flag_p(p.ctrl, COLI_FLAG_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---- epilogue warps: TMEM lane quarter (warp % 4) holds rows 32 (warp % 4) + lane
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    for (int i = 0; i < my_items; ++i) {
      const int buf = i & 1;
      if (!mbar_wait(&tm_full[buf], (i >> 1) & 1, lim)) {
        set_flag_p(p.ctrl, COLI_FLAG_TIMEOUT);
        break;
      }
      tc_fence_after();
      const Item it = decode_item(s_begin, s_off, p.n_groups, blockIdx.x + i * gridDim.x, n_ntiles);
      const int r = 32 * q + lane;
      // (a checked build also drops a row outside the route arrays)
      const bool r_ok = r < it.rows && COLI_CHK(it.p0 + r, P_routes, p.ctrl) == it.p0 + r;
      const uint32_t trow = tbase + lane_off + (uint32_t)(buf * kBN);
      if (MODE == kModeGateUp) {
        const float gate = r_ok ? p.route_gate[it.p0 + r] : 0.0f;
        __half *dst = p.h16 + (int64_t)(it.p0 + r) * F + it.ni * (kBN / 2);
        bool inf = false;
        for (int cc = 0; cc < kBN / 2; cc += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(trow + cc, g);
          tmem_ld32(trow + kBN / 2 + cc, u);
          tmem_ld_wait();
          uint32_t o[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]) * gate;
            const float h1 =
                silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]) * gate;
            const __half2 hh = __floats2half2_rn(h0, h1);
            o[j] = *reinterpret_cast<const uint32_t *>(&hh);
            inf |= half2_has_inf(o[j]);
          }
          if (r_ok) {
            uint4 *d4 = (uint4 *)(dst + cc);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              d4[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
        }
        if (r_ok && inf) set_flag_p(p.ctrl, COLI_FLAG_RANGE);
      } else {
        float *dst = p.y + (int64_t)(it.p0 + r) * H + it.ni * kBN;
        for (int cc = 0; cc < kBN; cc += 32) {
          uint32_t v[32];
          tmem_ld32(trow + cc, v);
          tmem_ld_wait();
          if (r_ok) {
            float4 *d4 = (float4 *)(dst + cc);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              d4[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                  __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tm_empty[buf]);
    }
  }
  // every MMA has completed (the MMA thread's final commit)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, 2 * kBN);
}

// ---------------------------------------------------------------------------
// Combine: out[t] = sum_j y[inv(t, j)] + sum_s y[T k + s T + t] (+ residual),
// fixed order; layer_out receives the MoE output without the residual.

__global__ void k_pcombine(PrefillArgs p) {
  const int T = p.T, H = p.H, k = p.k, S = p.S;
  const int H4 = H / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)T * H4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H4), c = (int)(i - (int64_t)t * H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float4 v = ((const float4 *)(p.y + (int64_t)COLI_CHK(p.inv[t * k + j], T * k, p.ctrl) * H))[c];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    for (int s = 0; s < S; ++s) {
      const float4 v = ((const float4 *)(p.y + (int64_t)(T * k + s * T + t) * H))[c];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (p.layer_out) ((float4 *)(p.layer_out + (int64_t)t * H))[c] = acc;
    if (p.residual) {
      const float4 r = ((const float4 *)(p.residual + (int64_t)t * H))[c];
      acc.x += r.x; acc.y += r.y; acc.z += r.z; acc.w += r.w;
    }
    ((float4 *)(p.out + (int64_t)t * H))[c] = acc;
  }
}

// ---------------------------------------------------------------------------
// host side

namespace {
template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
}  // namespace

PrefillLayout prefill_layout(int T, int H, int F, int E, int S, int k) {
  auto a256 = [](size_t v) { return (v + 255) & ~(size_t)255; };
  PrefillLayout L{};
  const size_t P = (size_t)T * (k + S);
  const size_t nb = ((size_t)T + kGroupTokens - 1) / kGroupTokens;
  size_t o = kWsFixedBytes;         // control words and the decode path's fixed region first
  L.x16 = o;        o = a256(o + (size_t)T * H * 2);
  L.logits = o;     o = a256(o + (size_t)T * E * 4);
  L.idx = o;        o = a256(o + (size_t)T * k * 4);
  L.gates = o;      o = a256(o + (size_t)T * k * 4);
  L.hist = o;       o = a256(o + nb * E * 4);
  L.offsets = o;    o = a256(o + (size_t)(E + S + 1) * 4);
  L.item_begin = o; o = a256(o + (size_t)(E + S + 1) * 4);
  L.route_tok = o;  o = a256(o + P * 4);
  L.route_gate = o; o = a256(o + P * 4);
  L.inv = o;        o = a256(o + (size_t)T * k * 4);
  L.h16 = o;        o = a256(o + P * F * 2);
  L.y = o;          o = a256(o + P * H * 4);
  L.total = o;
  return L;
}

bool prefill_supported(int H, int F) {
  // K of both GEMMs in whole stages, n-tiles whole
  return H % kBN == 0 && F % (kBN / 2) == 0 && H % kBK == 0 && F % kBK == 0;
}

namespace {
// The gate/up and down GEMMs of one layer over weights in container FMT.
template <int FMT>
cudaError_t launch_gemms(const PrefillArgs &p, int nsm, cudaStream_t s) {
  constexpr int smem = GeoBytes<FMT>::kSmem;
  auto gemm_gu = k_pgemm<kModeGateUp, FMT>;
  auto gemm_dn = k_pgemm<kModeDown, FMT>;
  cudaError_t e;
  if ((e = set_smem(gemm_gu, smem)) != cudaSuccess) return e;
  if ((e = set_smem(gemm_dn, smem)) != cudaSuccess) return e;
  size_t slot = 0;
  if ((e = record_profile(COLI_KERNEL_PREFILL_GATEUP, s, false, &slot)) != cudaSuccess) return e;
  gemm_gu<<<nsm, kGemmThreads, smem, s>>>(p);
  if ((e = record_profile(COLI_KERNEL_PREFILL_GATEUP, s, true, &slot)) != cudaSuccess) return e;
  if ((e = record_profile(COLI_KERNEL_PREFILL_DOWN, s, false, &slot)) != cudaSuccess) return e;
  gemm_dn<<<nsm, kGemmThreads, smem, s>>>(p);
  return record_profile(COLI_KERNEL_PREFILL_DOWN, s, true, &slot);
}
}  // namespace

cudaError_t launch_prefill(const PrefillArgs &p, int x_dtype, int wr_dtype, cudaStream_t s) {
  cudaError_t e;
  const int T = p.T, H = p.H, E = p.E, k = p.k;
  const int nsm = num_sms();
  if (nsm <= 0) return cudaErrorNoDevice;
  // activations -> fp16
  const int64_t nx = (int64_t)T * H;
  const int gx = (int)((nx / 8 + 255) / 256 < 4 * nsm ? (nx / 8 + 255) / 256 : 4 * nsm);
  if (x_dtype == COLI_BF16)
    k_x16<__nv_bfloat16><<<gx, 256, 0, s>>>((const __nv_bfloat16 *)p.x, p.x16, nx, p.ctrl);
  else k_x16<float><<<gx, 256, 0, s>>>((const float *)p.x, p.x16, nx, p.ctrl);
  // router logits: tensor cores when both operands are bf16 (exact products),
  // else the f32 SIMT GEMM
  const dim3 gl((E + 63) / 64, (T + 63) / 64);
#define COLI_LOGITS(XT, WT) \
  k_logits<XT, WT><<<gl, 256, 0, s>>>((const XT *)p.x, (const WT *)p.wr, p.logits, T, H, E)
  if (x_dtype == COLI_BF16 && wr_dtype == COLI_BF16) {
    if ((e = set_smem(k_plogits, kLgSmem)) != cudaSuccess) return e;
    const dim3 gp((T + kBM - 1) / kBM, (E + kBN - 1) / kBN);
    k_plogits<<<gp, kGemmThreads, kLgSmem, s>>>((const __nv_bfloat16 *)p.x,
                                                (const __nv_bfloat16 *)p.wr, p.logits, T, H, E,
                                                p.ctrl);
  } else if (x_dtype == COLI_BF16) COLI_LOGITS(__nv_bfloat16, float);
  else if (wr_dtype == COLI_BF16) COLI_LOGITS(float, __nv_bfloat16);
  else COLI_LOGITS(float, float);
#undef COLI_LOGITS
  // top-k
  const size_t tk_smem = 2 * (((size_t)kPTopkTokens * E * 4 + 15) & ~(size_t)15) +
                         ((topk_scratch_bytes(kPTopkTokens, E, k) + 15) & ~(size_t)15) +
                         (size_t)kPTopkTokens * k * 12 + 16;
  if ((e = set_smem(k_ptopk, tk_smem)) != cudaSuccess) return e;
  k_ptopk<<<(T + kPTopkTokens - 1) / kPTopkTokens, 256, tk_smem, s>>>(p);
  // grouping
  const int nb = (T + kGroupTokens - 1) / kGroupTokens;
  k_gcount<<<nb, 256, (size_t)E * 4, s>>>(p);
  k_gscan<<<1, 1024, 0, s>>>(p, nb);
  k_gscatter<<<nb, 256, (size_t)E * 4, s>>>(p);
  // GEMMs
  if (p.fmt == COLI_FMT_MXFP4) e = launch_gemms<COLI_FMT_MXFP4>(p, nsm, s);
  else if (p.fmt == COLI_FMT_FP8) e = launch_gemms<COLI_FMT_FP8>(p, nsm, s);
  else if (p.fmt == COLI_FMT_I4ROW) e = launch_gemms<COLI_FMT_I4ROW>(p, nsm, s);
  else e = launch_gemms<COLI_FMT_I4G>(p, nsm, s);
  if (e != cudaSuccess) return e;
  // combine
  const int64_t nc = (int64_t)T * (H / 4);
  const int gc = (int)((nc + 255) / 256 < 8 * nsm ? (nc + 255) / 256 : 8 * nsm);
  k_pcombine<<<gc, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace coli
