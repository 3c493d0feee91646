// Internal declarations shared by the CUDA translation units of libcoli.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda_fp16.h>

#include "coli.h"

namespace coli {

constexpr int kGroup = 64;          // columns per scale
constexpr int kMxBlock = 32;        // MXFP4: columns per E8M0 scale
constexpr int kFp8Block = 128;      // fp8-e4m3-b128: columns per f32 scale
constexpr int kDecodeMaxT = 16;     // tokens per call served by the GEMV path
constexpr int kMaxTopK = 64;
constexpr int kMaxExperts = 1024;
constexpr int kMaxShared = 8;
// Largest SM count the workspace layout provides for (GB300: 152).
constexpr int kMaxParts = 256;
// Router logits accumulated as fixed-point integers (deterministic in any
// order) by the CTAs that form their partials.  In the layer forward every
// CTA of the next gate/up kernel routes from them (two buffers, by layer
// parity; the down kernel of a layer clears the buffer its gate/up read);
// the router-only call routes in the last CTA of the partials' kernel.
constexpr int kFxMaxTE = 2048;          // tokens x experts routed this way (else a ticket)
// The fixed-point buffers sit at one offset for every shape, right after the
// control words, and every call leaves them zero; no other array of any
// layout overlaps them, so a workspace zero-filled once stays valid across
// calls of different shapes.
constexpr size_t kFxOffset = 256;
constexpr size_t kFxBufBytes = (size_t)kFxMaxTE * 8 + (size_t)kFxMaxTE * 4;
constexpr size_t kFxRegionBytes = 2 * kFxBufBytes;
constexpr size_t kWsFixedBytes = kFxOffset + ((kFxRegionBytes + 255) & ~(size_t)255);
// Buffers that every CTA of a kernel reads (layer input, h)
// are written in this many copies, each read by 1/kReplicas of the CTAs, so
// that no single L2 slice serves the whole grid.
constexpr int kReplicas = 8;

// Control words at the head of every workspace.
enum CtrlWord : int {
  kCtrlFlags = 0,      // COLI_FLAG_* bits (sticky until coli_moe_check clears)
  kCtrlRouterTicket = 1,
  kCtrlPrefillMTiles = 2,  // m-tiles of the current batched call (written by the grouping)
  kCtrlBarArrive = 3,  // grid barrier of the one-token layer kernel: arrivals of this use
  kCtrlBarGen = 4,     //   and its generation (left as they are between calls)
  kCtrlWaitLimit = 5,  // 0: default bounded waits; else the spin limit in clock cycles of
                       //   the grid barriers (one-token layer kernel, first-layer router
                       //   in k_gateup) and of the grouped GEMMs' pipeline waits (a test
                       //   hook that makes the waits run out)
  kCtrlWords = 64,     // 256 bytes
};
static_assert(kCtrlWords * 4 <= kFxOffset, "control words precede the fixed-point region");

// Byte offsets of the scratch arrays inside a workspace (all 256-aligned).
struct WsLayout {
  size_t ctrl;       // uint32[kCtrlWords]
  size_t partials;   // f32 [n_part][T][E] router partial logits
  size_t fx;         // i64 [T][E] fixed-point logits, then u32 [T][E] flags
  size_t idx;        // i32 [T][k]
  size_t gates;      // f32 [T][k]
  size_t act;        // i32: n_active, act_expert[E+S], act_off[E+S+1]
  size_t routes;     // i32 [T*(k+S)] slot ids grouped by used expert
  size_t slot_gate;  // f32 [T*(k+S)]
  size_t h;          // f32 [kReplicas][T*(k+S)][F]
  size_t xrep;       // f32 [kReplicas][T][H]
  size_t y;          // f32 [T*(k+S)][H] (T > 1 only)
  size_t total;
  int n_part;                  // kMaxParts: partials rows the layout holds
  size_t h_stride, x_stride;   // replica strides (floats)
};

WsLayout ws_layout(int T, int H, int F, int E, int S, int k);

constexpr int kDec2MaxThreads = 512;
constexpr int kDnMaxThreads = 640;      // k_down: up to 20 warps

// Shared-memory plan of k_gateup (byte offsets into dynamic smem).
struct GuSmem {
  size_t act, routes, slot_gate, tok, xpl, ring, red, total;
};
// Shared-memory plan of k_down.
struct DnSmem {
  size_t act, routes, acc, xn, wr, ring, red, total;
};
// Shared-memory plan of k_down_multi.
struct DmSmem {
  size_t act, routes, u, planes, acc, ring, total;
};
// Shared-memory plan of the one-token layer kernel k_layer1 (decode1.cu).
struct L1Smem {
  size_t bar, lst, red, xn, wr, hacc, u, ring, total;
};

// Tiered expert store of one layer (coli_moe_forward_tiered): experts whose
// slot_of entry is >= 0 live in that slot of the HBM pool; the others are read
// from the layer's own store (pinned host memory, device-accessible).  All
// null: every expert in the layer's store.
struct TierMap {
  const int32_t *slot_of;       // [E + S]
  const uint8_t *pool_packed;   // [n_slots] expert records
  const float *pool_scales;
};

// Expert e's record: its HBM slot when the tier map holds it, else its place
// in the layer's store.
__device__ __forceinline__ void expert_record(const TierMap &t, const uint8_t *packed,
                                              const float *scales, int64_t eb, int64_t es, int e,
                                              const uint8_t **pk, const float **sc) {
  const int slot = t.slot_of ? __ldg(t.slot_of + e) : -1;
  if (slot >= 0) {
    *pk = t.pool_packed + (int64_t)slot * eb;
    *sc = t.pool_scales + (int64_t)slot * es;
  } else {
    *pk = packed + (int64_t)e * eb;
    *sc = scales + (int64_t)e * es;
  }
}

// Diagnostic build (-DCOLI_CHECK): an index that a kernel derives from data
// (expert ids from routing, slot and route lists, token ids from the grouping)
// is checked against the extent of the buffer it indexes; one outside sets
// COLI_FLAG_BOUNDS and is replaced by 0, so the access stays inside the buffer.
// Without the flag the check compiles away.
#ifdef COLI_CHECK
__device__ __forceinline__ int64_t chk_idx(int64_t i, int64_t n, uint32_t *ctrl) {
  if (i >= 0 && i < n) return i;
  atomicOr(ctrl, COLI_FLAG_BOUNDS);     // the flag word is control word 0
  return 0;
}
#define COLI_CHK(i, n, ctrl) ((int)::coli::chk_idx((int64_t)(i), (int64_t)(n), (ctrl)))
#else
#define COLI_CHK(i, n, ctrl) ((int)(i))
#endif

// Arguments of the decode kernels (one layer, T <= kDecodeMaxT tokens).
struct Dec2Args {
  TierMap tier;
  int T, H, F, E, S, k;
  int layer;                // index of the layer in the stack (phase tracing only)
  int fx;                   // router partials as fixed-point sums (T*E <= kFxMaxTE)
  long long *fx_acc;        // [T][E] partials are added here
  uint32_t *fx_flag;        // [T][E] non-finite or out-of-range partial seen
  int router_fn;            // coli_router_fn of the layer being routed
  const float *router_bias; // its selection bias [E] (sigmoid router) or null
  int route_gu;             // every gate/up CTA routes its layer from fx_rd_*
  int gu_route_fits;        // the routing scratch fits in k_gateup's pipeline ring
  int gu_router;            // one token, first layer of the call: the k_gateup CTAs form
                            // the logits themselves (each the whole logits of its own
                            // experts, as floats over fx_rd_acc, then a grid barrier)
                            // instead of a k_route launch
  int gu_rt_off;            // byte offset of that router scratch in k_gateup's ring
  int x_bf16;               // x (the call's input) is bf16, else f32
  const long long *fx_rd_acc;   // k_gateup: this layer's fixed-point logits
  const uint32_t *fx_rd_flag;
  long long *fx_clr_acc;    // k_down: buffer its gate/up read, cleared here
  uint32_t *fx_clr_flag;
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
  int gu_ncg;               // 1024-column chunks of a gate/up row
  int gu_nw;                // warps of k_gateup
  int gu_slots;             // depth of each warp's cp.async pipeline (2..4)
  int gu_slot_bytes;        // bytes of one pipeline slot (weights + scales)
  int gu_rows;              // rows whose partial sums fit in shared memory at once
  int gu_xpl;               // x planes held in shared memory
  int dn_ncg;               // 1024-column chunks of a down row
  int dn_nw;                // warps of k_down
  int dn_slots_pipe;        // depth of each warp's cp.async pipeline
  int dn_slot_bytes;
  int wr_bf16;              // the router (and its rows in k_down's shared memory) is bf16
  int chain;                // a next layer follows (k_down forms its router partials)
  int dm_nw;                // warps of k_down_multi
  int dm_slots_pipe;        // depth of each warp's cp.async pipeline
  int dm_cap;               // h rows whose planes fit in k_down_multi's shared memory
  float *y;                 // [T*(k+S)][H] per-slot down outputs (several tokens)
  GuSmem gu;
  DnSmem dn;
  DmSmem dm;
  // one-token layer kernel (decode1.cu): l1_nc warps of l1_spw bulk-copy slots
  // each (l1_ns in all) of l1_slot bytes; gate/up stages of
  // l1_rg gate + l1_rg up rows, down stages of l1_dr rows; x (f32) and its
  // planes at bytes l1_xs_off / l1_xpl_off of the kernel's U region; at most
  // l1_nblk h blocks per CTA
  int l1_ns, l1_nc, l1_spw, l1_rg, l1_slot, l1_dr, l1_xs_off, l1_xpl_off, l1_nblk;
  L1Smem l1;
};


// Batched (prefill) path: arguments of its kernels for one layer.
constexpr int kPrefillMinT = 64;      // calls with at least this many tokens take it
constexpr int kGroupTokens = 256;     // tokens per block of the counting sort
struct PrefillArgs {
  TierMap tier;
  int fmt;                  // COLI_FMT_I4G, _I4ROW, _MXFP4 or _FP8 (all but I4G: es counts bytes)
  int T, H, F, E, S, k;
  int router_fn;            // coli_router_fn
  const float *router_bias; // [E] (sigmoid router) or null
  const void *x;            // [T][H] x_dtype
  const void *wr;           // [E][H] router dtype
  const uint8_t *packed;    // expert records of this layer
  const float *scales;
  int64_t eb, es;
  const float *residual;    // added to out (or null)
  float *out;               // [T][H]
  float *layer_out;         // [T][H] MoE output without the residual (or null)
  uint32_t *route_counts;   // [E] (or null)
  uint32_t *ctrl;
  __half *x16;              // [T][H]
  float *logits;            // [T][E]
  int32_t *idx;             // [T][k]
  float *gates;             // [T][k]
  int32_t *hist;            // [blocks][E]
  int32_t *offsets;         // [E+S+1] first route position of each expert
  int32_t *item_begin;      // [E+S+1] m-tile prefix
  int n_groups;             // E + S
  int32_t *route_tok;       // [T(k+S)] token of each route position
  float *route_gate;        // [T(k+S)] its gate (1 for shared experts)
  int32_t *inv;             // [T k] route position of (t, j)
  __half *h16;              // [T(k+S)][F]
  float *y;                 // [T(k+S)][H]
};
struct PrefillLayout {
  size_t x16, logits, idx, gates, hist, offsets, item_begin, route_tok, route_gate, inv, h16, y,
      total;
};
PrefillLayout prefill_layout(int T, int H, int F, int E, int S, int k);
bool prefill_supported(int H, int F);
cudaError_t launch_prefill(const PrefillArgs &p, int x_dtype, int wr_dtype, cudaStream_t s);

// Fill the kernels' launch plan (warps per phase, shared-memory layouts).
cudaError_t plan_decode(Dec2Args &a, int n_part);
cudaError_t launch_route_partials(const Dec2Args &a, int x_bf16, int w_bf16, cudaStream_t s,
                                  bool pdl);
cudaError_t launch_gateup(const Dec2Args &a, int grid, cudaStream_t s, bool pdl);
cudaError_t launch_down(const Dec2Args &a, int wr_bf16, cudaStream_t s, bool pdl);
cudaError_t launch_down_multi(const Dec2Args &a, cudaStream_t s, bool pdl);
// One-token layers (decode1.cu): plan_layer1 returns true when the fused
// kernel handles this shape (and fills its plan); launch_layer1 runs one layer.
bool plan_layer1(Dec2Args &a);
cudaError_t launch_layer1(const Dec2Args &a, cudaStream_t s, bool pdl);

// Quantisers (quant.cu, quant_fmt.cu).
cudaError_t launch_quant_i4g(const void *w, int w_dtype, int64_t rows, int64_t cols,
                             uint8_t *packed, float *scales, cudaStream_t s);
cudaError_t launch_quant_mxfp4(const void *w, int w_dtype, int64_t rows, int64_t cols,
                               uint8_t *packed, uint8_t *scales, cudaStream_t s);
cudaError_t launch_quant_fp8b128(const void *w, int w_dtype, int64_t rows, int64_t cols,
                                 uint8_t *packed, float *scales, cudaStream_t s);
cudaError_t launch_quant_i4row(const void *w, int w_dtype, int64_t rows, int64_t cols,
                               uint8_t *packed, float *scales, cudaStream_t s);

int num_sms();
// The layer forward over a tiered expert store (coli_api.cu); `packed` and
// `scales` are device-accessible addresses of the full store.
int moe_forward_tiered(const coli_moe_desc *d, int top_k, const void *x, const void *router_w,
                       const uint8_t *packed, const float *scales, const TierMap &tier,
                       float *out, uint32_t *route_counts, void *workspace, size_t ws_bytes,
                       cudaStream_t stream);
// Records the caller's profiling event before (is_after false: claims a slot)
// or after a launch of `kernel` if coli_profile_events selected it.
cudaError_t record_profile(int kernel, cudaStream_t s, bool is_after, size_t *slot);
// COLI_OK for cudaSuccess; else records the error's message for
// coli_last_error() and returns COLI_ECUDA.
int cuda_status(cudaError_t e);
const char *last_error();

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
