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
// Buffers that every CTA of a kernel reads (layer input, h, router partials)
// are written in this many copies, each read by 1/kReplicas of the CTAs, so
// that no single L2 slice serves the whole grid.
constexpr int kReplicas = 8;

// Control words at the head of every workspace.
enum CtrlWord : int {
  kCtrlFlags = 0,      // COLI_FLAG_* bits (sticky until coli_moe_check clears)
  kCtrlRouterTicket = 1,
  kCtrlBarrier = 2,    // grid barrier counter of the persistent stack kernel
  kCtrlExit = 3,       // its exit ticket (resets the barrier counter)
  kCtrlWords = 64,     // 256 bytes
};

// Byte offsets of the scratch arrays inside a workspace (all 256-aligned).
struct WsLayout {
  size_t ctrl;       // uint32[kCtrlWords]
  size_t partials;   // f32 [kReplicas][n_part][T][E] router partial logits (copy r at r*part_stride)
  size_t idx;        // i32 [T][k]
  size_t gates;      // f32 [T][k]
  size_t act;        // i32: n_active, act_expert[E+S], act_off[E+S+1]
  size_t routes;     // i32 [T*(k+S)] slot ids grouped by used expert
  size_t slot_gate;  // f32 [T*(k+S)]
  size_t h;          // f32 [kReplicas][T*(k+S)][F]
  size_t xrep;       // f32 [kReplicas][T][H]
  size_t total;
  int n_part;
  size_t part_stride, h_stride, x_stride;   // replica strides (floats)
};

WsLayout ws_layout(int T, int H, int F, int E, int S, int k);

constexpr int kDec2MaxThreads = 512;

// Shared-memory plan of k_gateup (byte offsets into dynamic smem).
struct GuSmem {
  size_t act, routes, slot_gate, red, xpl, total;
};
// Shared-memory plan of k_down.
struct DnSmem {
  size_t act, routes, acc, xn, wr, planes, total;
};

// Arguments of the decode kernels (one layer, T <= kDecodeMaxT tokens).
struct Dec2Args {
  int T, H, F, E, S, k;
  const void *x;            // layer input [T][H], f32 or bf16
  const void *wr;           // k_route: this layer's router; k_down: next layer's (or null)
  const float *residual;    // k_down: added to the layer output (or null)
  const uint8_t *packed;    // this layer's expert records
  const float *scales;
  int64_t eb, es;           // packed bytes / scales per expert
  float *partials;          // [n_part][T][E] router partial logits
  int n_part;
  int n_rep;                // replicas of the buffers every CTA reads
  float *xrep;              // [n_rep][T][H] f32 layer input (or null)
  size_t x_stride;
  size_t h_stride;          // h replica stride (floats)
  int32_t *g_idx;
  float *g_gates;
  int32_t *g_act, *g_routes;
  float *g_slot_gate;
  float *h;                 // [n_rep][T*(k+S)][F]
  uint32_t *ctrl;
  uint32_t *route_counts;   // route counts [E] of the layer this kernel routes (or null)
  uint32_t *next_counts;    // k_down: route counts of the next layer (or null)
  float *out;               // k_down output [T][H]
  float *layer_out;         // or null
  int32_t *idx_out;         // k_topk user outputs (or null)
  float *gates_out;
  int build_union;          // k_topk also builds and publishes the union lists
  int stage_partials;       // routing stages the partials in shared memory
  int gu_ncg, gu_nrg, gu_xpl;
  int dn_ncg, dn_nrg, dn_slots;
  GuSmem gu;
  DnSmem dn;
};

// Shared-memory plan of the persistent stack kernel: union lists, router rows,
// then one area reused by the routing, gate/up and down phases.
struct StkSmem {
  size_t act, routes, slot_gate, wr, area;
  size_t gu_red, gu_xpl, dn_acc, dn_xn, dn_planes;   // offsets inside the area
  size_t total;
};

struct StackArgs {
  int n_layers;
  const void *router;       // [n_layers][E][H]
  size_t wr_stride;         // bytes per layer
  size_t pk_stride, sc_stride;
  uint32_t *counts;         // [n_layers][E] or null
  float *layer_out;         // [n_layers][T][H] or null
  float *x_out;             // [T][H]
  size_t part_stride;       // floats between the partials' copies
  StkSmem sm;
};

cudaError_t plan_decode(Dec2Args &a, int n_part);
cudaError_t plan_stack(Dec2Args &a, StackArgs &st);
cudaError_t launch_stack(const Dec2Args &a, const StackArgs &st, int x_bf16, int wr_bf16,
                         cudaStream_t s);
cudaError_t launch_route_partials(const Dec2Args &a, int x_bf16, int w_bf16, cudaStream_t s,
                                  bool pdl);
cudaError_t launch_gateup(const Dec2Args &a, int grid, cudaStream_t s, bool pdl);
cudaError_t launch_down(const Dec2Args &a, int wr_bf16, cudaStream_t s, bool pdl);

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
