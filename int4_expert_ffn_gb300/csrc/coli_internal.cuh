// Internal declarations shared by the CUDA translation units of libcoli.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "coli.h"

namespace coli {

constexpr int kGroup = 64;          // columns per scale
constexpr int kDecodeMaxT = 16;     // tokens per call served by the GEMV path
constexpr int kMaxTopK = 64;
constexpr int kMaxExperts = 1024;
constexpr int kMaxShared = 8;

// Control words at the head of every workspace.
enum CtrlWord : int {
  kCtrlFlags = 0,      // COLI_FLAG_* bits (sticky until coli_moe_check clears)
  kCtrlRouterTicket = 1,
  kCtrlWords = 64,     // 256 bytes
};

// Byte offsets of the scratch arrays inside a workspace (all 256-aligned).
struct WsLayout {
  size_t ctrl;       // uint32[kCtrlWords]
  size_t logits;     // f32 [T][E]
  size_t idx;        // i32 [T][k]
  size_t gates;      // f32 [T][k]
  size_t act;        // i32: n_active, act_expert[E+S], act_off[E+S+1]
  size_t routes;     // i32 [T*(k+S)] slot ids grouped by active expert
  size_t slot_gate;  // f32 [T*(k+S)]
  size_t h;          // f32 [T*(k+S)][F]
  size_t total;
};

WsLayout ws_layout(int T, int H, int F, int E, int S, int k);

// Router + top-k + union (router.cu).  x_dtype / w_dtype are coli_dtype.
// Writes logits, idx, gates, union lists into ws; optional user copies.
cudaError_t launch_router_topk(const void *x, int x_dtype, const void *wr, int w_dtype,
                               int T, int H, int E, int S, int k, uint8_t *ws,
                               const WsLayout &L, int32_t *idx_out, float *gates_out,
                               uint32_t *counts, bool build_union, cudaStream_t s);

// Expert FFN over the union lists (moe_decode.cu).
cudaError_t launch_moe_decode(const void *x, int x_dtype, int T, int H, int F, int E, int S,
                              int k, const uint8_t *packed, const float *scales,
                              uint8_t *ws, const WsLayout &L, float *out,
                              const float *residual, float *layer_out, cudaStream_t s);

// Quantiser (quant.cu).
cudaError_t launch_quant_i4g(const void *w, int w_dtype, int64_t rows, int64_t cols,
                             uint8_t *packed, float *scales, cudaStream_t s);

int num_sms();

// ---------------------------------------------------------------------------
// device helpers

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  // 16-byte load that bypasses L1 allocation (weights are read once)
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace coli
