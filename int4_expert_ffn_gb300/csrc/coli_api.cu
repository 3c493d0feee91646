// C ABI entry points of libcoli: host-side validation, workspace layout and
// dispatch.  Declarations and the meaning of every argument are in coli.h.
#include <limits.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "coli_internal.cuh"

namespace coli {

static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

WsLayout ws_layout(int T, int H, int F, int E, int S, int k) {
  WsLayout L{};
  size_t o = 0;
  const size_t KS = (size_t)k + S;
  // the row-split kernels run one CTA per SM; their f32 router partials (only
  // when the logits do not fit the fixed-point buffers) are sized for the
  // largest SM count the library accepts, so the layout does not depend on
  // the device
  L.n_part = kMaxParts;
  // replica strides: whole 256-byte units plus one, so replicas start at
  // different offsets modulo any power of two
  L.h_stride = (align256((size_t)T * KS * F * 4) + 256) / 4;
  L.x_stride = (align256((size_t)T * H * 4) + 256) / 4;
  L.ctrl = o;
  L.fx = kFxOffset;
  o = kWsFixedBytes;
  L.partials = o;
  if ((size_t)T * E > (size_t)kFxMaxTE) o = align256(o + (size_t)kMaxParts * T * E * 4);
  L.idx = o;       o = align256(o + (size_t)T * k * sizeof(int32_t));
  L.gates = o;     o = align256(o + (size_t)T * k * sizeof(float));
  L.act = o;       o = align256(o + (size_t)(2 * (E + S) + 2) * sizeof(int32_t));
  L.routes = o;    o = align256(o + (size_t)T * KS * sizeof(int32_t));
  L.slot_gate = o; o = align256(o + (size_t)T * KS * sizeof(float));
  L.h = o;         o = align256(o + kReplicas * L.h_stride * 4);
  L.xrep = o;      o = align256(o + kReplicas * L.x_stride * 4);
  L.y = o;         o = align256(o + (T > 1 ? (size_t)T * KS * H * 4 : 0));
  L.total = o;
  return L;
}

// SM count of the current device, queried once per device.  0 when there is
// no usable device (the callers turn that into an error; there is no default).
int num_sms() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    return 0;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Message of the last CUDA error that a call on this thread returned as COLI_ECUDA.
static thread_local const char *t_last_error = "no error";

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return COLI_OK;
  t_last_error = cudaGetErrorString(e);
  return COLI_ECUDA;
}

const char *last_error() { return t_last_error; }

}  // namespace coli

using namespace coli;

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int check_desc(const coli_moe_desc *d, int top_k) {
  if (!d) return COLI_EINVAL;
  if (d->hidden < 64 || d->hidden > 16384 || d->hidden % kGroup) return COLI_EINVAL;
  if (d->ffn < 64 || d->ffn > 16384 || d->ffn % kGroup) return COLI_EINVAL;
  if (d->n_experts < 1 || d->n_experts > kMaxExperts) return COLI_EINVAL;
  if (d->n_shared < 0 || d->n_shared > kMaxShared) return COLI_EINVAL;
  if (d->n_tokens < 0) return COLI_EINVAL;
  if (top_k < 1 || top_k > d->n_experts || top_k > kMaxTopK) return COLI_EINVAL;
  if ((d->x_dtype != COLI_F32 && d->x_dtype != COLI_BF16) ||
      (d->router_dtype != COLI_F32 && d->router_dtype != COLI_BF16))
    return COLI_EINVAL;
  if (d->router_fn != COLI_ROUTER_SOFTMAX && d->router_fn != COLI_ROUTER_SIGMOID_BIAS)
    return COLI_EINVAL;
  if (d->router_fn == COLI_ROUTER_SIGMOID_BIAS && ((uintptr_t)d->router_bias & 3u))
    return COLI_EALIGN;
  if (d->weight_fmt != 0 && d->weight_fmt != COLI_FMT_I4G && d->weight_fmt != COLI_FMT_MXFP4 &&
      d->weight_fmt != COLI_FMT_FP8 && d->weight_fmt != COLI_FMT_I4ROW)
    return COLI_EINVAL;
  return COLI_OK;
}

int weight_fmt(const coli_moe_desc *d) { return d->weight_fmt == 0 ? COLI_FMT_I4G : d->weight_fmt; }


// Tokens per internal pass of the GEMV path; larger calls run in passes.
int pass_tokens(int T) { return T < kDecodeMaxT ? T : kDecodeMaxT; }

// Calls with many tokens take the batched path (grouped tensor-core GEMMs)
// when its tile shapes divide the layer.
// The other containers (int4-row, MXFP4, fp8) take it at every token count.
bool use_prefill(const coli_moe_desc *d) {
  if (weight_fmt(d) != COLI_FMT_I4G) return true;
  return d->n_tokens >= kPrefillMinT && prefill_supported(d->hidden, d->ffn);
}

// A format the layer's shape cannot run in.
int fmt_unsupported(const coli_moe_desc *d) {
  return weight_fmt(d) != COLI_FMT_I4G && !prefill_supported(d->hidden, d->ffn);
}

int map_err(cudaError_t e) { return coli::cuda_status(e); }

// Diagnostic event recording around the gate/up kernel (coli_profile_events).
struct ProfileState {
  std::mutex mu;
  int kernel = -1;
  std::vector<cudaEvent_t> before, after;
  size_t next = 0;
};
ProfileState &profile() {
  static ProfileState p;
  return p;
}

}  // namespace

cudaError_t coli::record_profile(int kernel, cudaStream_t s, bool is_after, size_t *slot) {
  ProfileState &p = profile();
  std::lock_guard<std::mutex> lock(p.mu);
  if (!is_after) {
    if (kernel != p.kernel || p.next >= p.before.size()) { *slot = (size_t)-1; return cudaSuccess; }
    *slot = p.next++;
  }
  if (*slot == (size_t)-1) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0;
  cudaEvent_t ev = is_after ? p.after[*slot] : p.before[*slot];
  return cudaEventRecordWithFlags(ev, s, flags);
}

namespace {

// Launch one kernel of the layer forward, bracketed by the caller's profiling
// events when coli_profile_events selected it.
template <class Launch>
cudaError_t profiled(int kernel, cudaStream_t s, Launch launch) {
  size_t slot = 0;
  cudaError_t e = coli::record_profile(kernel, s, false, &slot);
  if (e == cudaSuccess) e = launch();
  if (e == cudaSuccess) e = coli::record_profile(kernel, s, true, &slot);
  return e;
}

size_t xsize(coli_dtype t) { return t == COLI_BF16 ? 2 : 4; }

// CTAs of the row-split kernels on the current device (one per SM), or a
// status: COLI_ECUDA without a usable device, COLI_EUNSUPPORTED above the SM
// count the workspace layout provides for.
int device_parts(int *parts) {
  const int G = num_sms();
  if (G <= 0) return coli::cuda_status(cudaErrorNoDevice);
  if (G > kMaxParts) return COLI_EUNSUPPORTED;
  *parts = G;
  return COLI_OK;
}

Dec2Args make_args(const coli_moe_desc *d, int k, int tn, uint8_t *ws, const WsLayout &L,
                   int parts, const TierMap *tier = nullptr) {
  Dec2Args a{};
  if (tier) a.tier = *tier;
  a.T = tn;
  a.H = d->hidden;
  a.F = d->ffn;
  a.E = d->n_experts;
  a.S = d->n_shared;
  a.k = k;
  a.eb = coli_expert_packed_bytes(a.H, a.F);
  a.es = coli_expert_scale_count(a.H, a.F);
  a.n_part = parts;
  a.n_rep = kReplicas;
  a.partials = (float *)(ws + L.partials);
  a.h_stride = L.h_stride;
  a.xrep = (float *)(ws + L.xrep);
  a.x_stride = L.x_stride;
  a.g_idx = (int32_t *)(ws + L.idx);
  a.g_gates = (float *)(ws + L.gates);
  a.g_act = (int32_t *)(ws + L.act);
  a.g_routes = (int32_t *)(ws + L.routes);
  a.g_slot_gate = (float *)(ws + L.slot_gate);
  a.h = (float *)(ws + L.h);
  a.y = (float *)(ws + L.y);
  a.ctrl = (uint32_t *)(ws + L.ctrl);
  a.wr_bf16 = d->router_dtype == COLI_BF16;
  a.router_fn = d->router_fn;
  a.router_bias = d->router_fn == COLI_ROUTER_SIGMOID_BIAS ? d->router_bias : nullptr;
  a.fx = tn * a.E <= kFxMaxTE;
  a.fx_acc = (long long *)(ws + L.fx);
  a.fx_flag = (uint32_t *)(ws + L.fx + (size_t)tn * a.E * 8);
  return a;
}

// Fixed-point buffer b (0 or 1) of a workspace.
void fx_buffer(const Dec2Args &a, uint8_t *ws, const WsLayout &L, int b, long long **acc,
               uint32_t **flag) {
  uint8_t *base = ws + L.fx + (size_t)b * kFxBufBytes;
  *acc = (long long *)base;
  *flag = (uint32_t *)(base + (size_t)a.T * a.E * 8);
}

}  // namespace

extern "C" {

const char *coli_last_error(void) { return coli::last_error(); }

const char *coli_status_str(int status) {
  switch (status) {
    case COLI_OK: return "ok";
    case COLI_EINVAL: return "invalid argument";
    case COLI_EALIGN: return "pointer not 16-byte aligned";
    case COLI_ECUDA: return "CUDA error";
    case COLI_ETIMEOUT: return "device-side wait timed out";
    case COLI_ENOMEM: return "workspace too small";
    case COLI_EUNSUPPORTED: return "unsupported configuration";
    case COLI_EIO: return "file I/O failed";
    case COLI_EREFUSED: return "usage history of another model or format";
    case COLI_ERANGE: return "operand outside the fp16 range of the batched path";
    case COLI_EBOUNDS: return "index outside its buffer (checked build)";
    default: return "unknown status";
  }
}

int64_t coli_packed_row_bytes(int64_t cols) { return cols < 0 ? 0 : (cols + 1) / 2; }
int64_t coli_scales_per_row(int64_t cols) { return cols < 0 ? 0 : (cols + kGroup - 1) / kGroup; }
int64_t coli_expert_packed_bytes(int64_t H, int64_t F) {
  return 2 * F * coli_packed_row_bytes(H) + H * coli_packed_row_bytes(F);
}
int64_t coli_expert_scale_count(int64_t H, int64_t F) {
  return 2 * F * coli_scales_per_row(H) + H * coli_scales_per_row(F);
}

int64_t coli_fmt_row_bytes(int32_t fmt, int64_t cols) {
  if (cols < 0) return 0;
  if (fmt == 0 || fmt == COLI_FMT_I4G || fmt == COLI_FMT_MXFP4 || fmt == COLI_FMT_I4ROW)
    return (cols + 1) / 2;
  if (fmt == COLI_FMT_FP8) return cols;
  return 0;
}
int64_t coli_fmt_scale_bytes(int32_t fmt, int64_t cols) {
  if (cols < 0) return 0;
  if (fmt == 0 || fmt == COLI_FMT_I4G) return 4 * coli_scales_per_row(cols);
  if (fmt == COLI_FMT_MXFP4) return (cols + kMxBlock - 1) / kMxBlock;
  if (fmt == COLI_FMT_FP8) return 4 * ((cols + kFp8Block - 1) / kFp8Block);
  if (fmt == COLI_FMT_I4ROW) return 4;
  return 0;
}
int64_t coli_fmt_expert_bytes(int32_t fmt, int64_t H, int64_t F) {
  return 2 * F * coli_fmt_row_bytes(fmt, H) + H * coli_fmt_row_bytes(fmt, F);
}
int64_t coli_fmt_expert_scale_bytes(int32_t fmt, int64_t H, int64_t F) {
  return 2 * F * coli_fmt_scale_bytes(fmt, H) + H * coli_fmt_scale_bytes(fmt, F);
}

int coli_quant_i4g(const void *w, coli_dtype w_dtype, int64_t rows, int64_t cols,
                   uint8_t *packed, float *scales, cudaStream_t stream) {
  if (rows < 0 || cols < 1) return COLI_EINVAL;
  if (w_dtype != COLI_F32 && w_dtype != COLI_BF16) return COLI_EINVAL;
  if (rows > 0 && (!w || !packed || !scales)) return COLI_EINVAL;
  if (rows > 0 && cols > INT64_MAX / rows) return COLI_EINVAL;
  return map_err(launch_quant_i4g(w, w_dtype, rows, cols, packed, scales, stream));
}

size_t coli_router_workspace_size(const coli_moe_desc *d, int top_k) {
  return coli_moe_workspace_size(d, top_k);
}

int coli_quant_mxfp4(const void *w, coli_dtype w_dtype, int64_t rows, int64_t cols,
                     uint8_t *packed, uint8_t *scales, cudaStream_t stream) {
  if (rows < 0 || cols < 1) return COLI_EINVAL;
  if (w_dtype != COLI_F32 && w_dtype != COLI_BF16) return COLI_EINVAL;
  if (rows > 0 && (!w || !packed || !scales)) return COLI_EINVAL;
  if (rows > 0 && cols > INT64_MAX / rows) return COLI_EINVAL;
  return map_err(launch_quant_mxfp4(w, w_dtype, rows, cols, packed, scales, stream));
}

int coli_quant_i4row(const void *w, coli_dtype w_dtype, int64_t rows, int64_t cols,
                     uint8_t *packed, float *scales, cudaStream_t stream) {
  if (rows < 0 || cols < 1) return COLI_EINVAL;
  if (w_dtype != COLI_F32 && w_dtype != COLI_BF16) return COLI_EINVAL;
  if (rows > 0 && (!w || !packed || !scales)) return COLI_EINVAL;
  if (rows > 0 && cols > INT64_MAX / rows) return COLI_EINVAL;
  return map_err(launch_quant_i4row(w, w_dtype, rows, cols, packed, scales, stream));
}

int coli_quant_fp8b128(const void *w, coli_dtype w_dtype, int64_t rows, int64_t cols,
                       uint8_t *packed, float *scales, cudaStream_t stream) {
  if (rows < 0 || cols < 1) return COLI_EINVAL;
  if (w_dtype != COLI_F32 && w_dtype != COLI_BF16) return COLI_EINVAL;
  if (rows > 0 && (!w || !packed || !scales)) return COLI_EINVAL;
  if (rows > 0 && cols > INT64_MAX / rows) return COLI_EINVAL;
  return map_err(launch_quant_fp8b128(w, w_dtype, rows, cols, packed, scales, stream));
}

size_t coli_moe_workspace_size(const coli_moe_desc *d, int top_k) {
  if (check_desc(d, top_k) != COLI_OK || fmt_unsupported(d)) return 0;
  if (use_prefill(d))
    return prefill_layout(d->n_tokens, d->hidden, d->ffn, d->n_experts, d->n_shared, top_k).total;
  const int T = pass_tokens(d->n_tokens);
  return ws_layout(T > 0 ? T : 1, d->hidden, d->ffn, d->n_experts, d->n_shared, top_k).total;
}

int coli_router_topk(const coli_moe_desc *d, int top_k, const void *x, const void *router_w,
                     int32_t *idx, float *gates, uint32_t *route_counts, void *workspace,
                     size_t ws_bytes, cudaStream_t stream) {
  int st = check_desc(d, top_k);
  if (st) return st;
  const int T = d->n_tokens;
  if (T == 0) return COLI_OK;
  if (!x || !router_w || !idx || !gates || !workspace) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(router_w) || ((uintptr_t)workspace & 255u)) return COLI_EALIGN;
  if (ws_bytes < coli_router_workspace_size(d, top_k)) return COLI_ENOMEM;
  int parts = 0;
  if ((st = device_parts(&parts)) != COLI_OK) return st;
  const int H = d->hidden, E = d->n_experts, k = top_k;
  const int TP = pass_tokens(T);
  const WsLayout L = ws_layout(TP, H, d->ffn, E, d->n_shared, k);
  uint8_t *ws = (uint8_t *)workspace;
  for (int t0 = 0; t0 < T; t0 += TP) {
    const int tn = T - t0 < TP ? T - t0 : TP;
    Dec2Args a = make_args(d, k, tn, ws, L, parts);
    a.x = (const char *)x + (size_t)t0 * H * xsize(d->x_dtype);
    a.wr = router_w;
    a.route_counts = route_counts;
    a.idx_out = idx + (size_t)t0 * k;
    a.gates_out = gates + (size_t)t0 * k;
    a.build_union = 0;
    a.xrep = nullptr;
    cudaError_t e = launch_route_partials(a, d->x_dtype == COLI_BF16,
                                          d->router_dtype == COLI_BF16, stream, true);
    if (e != cudaSuccess) return map_err(e);
  }
  return COLI_OK;
}

// One token pass (<= kDecodeMaxT tokens) through n_layers layers.  Layer l reads
// x (l = 0, dtype x_dtype) or out (l > 0, f32); with a residual the output of
// layer l is x_l + MoE_l(x_l), else MoE_l(x_l) (single layer only).
static int moe_pass(const coli_moe_desc *d, int k, int n_layers, int tn, const void *x,
                    coli_dtype x_dtype, const void *router_w, const uint8_t *packed,
                    const float *scales, float *out, bool residual, float *layer_out,
                    uint32_t *route_counts, void *workspace, const WsLayout &L,
                    cudaStream_t stream, const TierMap *tier) {
  const int H = d->hidden, F = d->ffn, E = d->n_experts, S = d->n_shared;
  const size_t wr_stride = (size_t)E * H * xsize(d->router_dtype);
  const size_t pk_stride = (size_t)(E + S) * coli_expert_packed_bytes(H, F);
  const size_t sc_stride = (size_t)(E + S) * coli_expert_scale_count(H, F);
  const size_t T_H = (size_t)d->n_tokens * H;
  int parts = 0;
  const int st = device_parts(&parts);
  if (st != COLI_OK) return st;
  Dec2Args a = make_args(d, k, tn, (uint8_t *)workspace, L, parts, tier);
  a.chain = n_layers > 1;
  // one token at shapes of whole 1024-column chunks: one fused kernel per
  // layer (decode1.cu); otherwise the gate/up and down GEMV kernels
  const bool fused = plan_layer1(a);
  if (!fused && plan_decode(a, parts) != cudaSuccess) return COLI_EUNSUPPORTED;
  const int wr_bf16 = d->router_dtype == COLI_BF16;
  cudaError_t e = cudaSuccess;
  a.build_union = 1;
  // with fixed-point logits every gate/up CTA (every fused-kernel CTA) routes
  // its own layer
  a.route_gu = fused || (a.fx && a.gu_route_fits);
  // one token on the GEMV kernels: the first layer's gate/up CTAs form its
  // logits themselves (no router-partials launch before them)
  const bool gu_router = !fused && tn == 1 && a.route_gu && a.gu_rt_off >= 0;
  a.x_bf16 = x_dtype == COLI_BF16;
  const float *bias0 = d->router_fn == COLI_ROUTER_SIGMOID_BIAS ? d->router_bias : nullptr;
  uint8_t *ws = (uint8_t *)workspace;
  for (int l = 0; l < n_layers && e == cudaSuccess; ++l) {
    const void *xin = (l == 0) ? x : (const void *)out;
    a.x = xin;
    a.layer = l;
    a.packed = packed + l * pk_stride;
    a.scales = scales + l * sc_stride;
    // counts of layer l: added by whichever kernel routes it (the gate/up CTAs
    // with fixed-point logits, else the last CTA of the partials' kernel)
    a.route_counts = route_counts ? route_counts + (size_t)l * E : nullptr;
    if (a.route_gu) {
      // layer l's logits in buffer l % 2 (read by its gate/up, cleared by its
      // down kernel); the down kernel adds layer l + 1's into the other
      long long *rd_acc;
      uint32_t *rd_flag;
      fx_buffer(a, ws, L, l & 1, &rd_acc, &rd_flag);
      a.fx_rd_acc = rd_acc;
      a.fx_rd_flag = rd_flag;
      a.fx_clr_acc = rd_acc;
      a.fx_clr_flag = rd_flag;
      fx_buffer(a, ws, L, l == 0 ? 0 : (l + 1) & 1, &a.fx_acc, &a.fx_flag);
    }
    // the bias of the layer each launch routes: layer l for k_route (l = 0)
    // and k_gateup, layer l + 1 for the last CTA of k_down (without fixed point)
    a.router_bias = bias0 ? bias0 + (size_t)l * E : nullptr;
    if (l == 0) {
      // router partials of layer 0 (a launch of their own, or in its gate/up CTAs)
      a.wr = router_w;
      if (!gu_router) {
        e = profiled(COLI_KERNEL_ROUTE, stream, [&] {
          return launch_route_partials(a, x_dtype == COLI_BF16, wr_bf16, stream, true);
        });
        if (e != cudaSuccess) break;
      }
      if (a.route_gu) fx_buffer(a, ws, L, 1, &a.fx_acc, &a.fx_flag);
    }
    a.gu_router = (l == 0 && gu_router) ? 1 : 0;
    if (fused) {
      // routing, gate/up, down, combine and the next layer's router partials
      const bool next = l + 1 < n_layers;
      a.wr = next ? (const void *)((const char *)router_w + (l + 1) * wr_stride) : nullptr;
      a.residual = residual ? (const float *)xin : nullptr;
      a.out = out;
      a.layer_out = layer_out ? layer_out + (size_t)l * T_H : nullptr;
      e = profiled(COLI_KERNEL_LAYER, stream, [&] { return launch_layer1(a, stream, true); });
      continue;
    }
    e = profiled(COLI_KERNEL_GATEUP, stream, [&] { return launch_gateup(a, parts, stream, true); });
    if (e != cudaSuccess) break;
    // down also forms the next layer's router partials (and, without fixed-point
    // logits, routes it in its last CTA)
    const bool next = l + 1 < n_layers;
    a.wr = next ? (const void *)((const char *)router_w + (l + 1) * wr_stride) : nullptr;
    a.next_counts = (next && route_counts) ? route_counts + (size_t)(l + 1) * E : nullptr;
    a.residual = residual ? (const float *)xin : nullptr;
    if (bias0 && !a.route_gu) a.router_bias = bias0 + (size_t)(l + 1) * E;
    a.out = out;
    a.layer_out = layer_out ? layer_out + (size_t)l * T_H : nullptr;
    // several tokens: the expert GEMVs (k_down_multi), then the combine (k_down)
    e = profiled(COLI_KERNEL_DOWN, stream, [&] {
      if (a.T > 1) {
        const cudaError_t em = launch_down_multi(a, stream, true);
        if (em != cudaSuccess) return em;
      }
      return launch_down(a, wr_bf16, stream, true);
    });
  }
  return map_err(e);
}

// The batched path: every layer in one pass over all T tokens.
static int prefill_run(const coli_moe_desc *d, int k, int n_layers, const void *x,
                       const void *router_w, const uint8_t *packed, const float *scales,
                       float *out, bool residual, float *layer_out, uint32_t *route_counts,
                       void *workspace, cudaStream_t stream, const TierMap *tier) {
  const int T = d->n_tokens, H = d->hidden, F = d->ffn, E = d->n_experts, S = d->n_shared;
  const PrefillLayout L = prefill_layout(T, H, F, E, S, k);
  uint8_t *ws = (uint8_t *)workspace;
  const int fmt = weight_fmt(d);
  const size_t wr_stride = (size_t)E * H * xsize(d->router_dtype);
  const size_t pk_stride = (size_t)(E + S) * coli_fmt_expert_bytes(fmt, H, F);
  const size_t sc_bytes = (size_t)(E + S) * coli_fmt_expert_scale_bytes(fmt, H, F);
  for (int l = 0; l < n_layers; ++l) {
    PrefillArgs a{};
    if (tier) a.tier = *tier;
    a.T = T; a.H = H; a.F = F; a.E = E; a.S = S; a.k = k;
    a.router_fn = d->router_fn;
    a.router_bias = (d->router_fn == COLI_ROUTER_SIGMOID_BIAS && d->router_bias)
                        ? d->router_bias + (size_t)l * E : nullptr;
    a.x = l == 0 ? x : (const void *)out;
    a.wr = (const char *)router_w + l * wr_stride;
    a.fmt = fmt;
    a.packed = packed + l * pk_stride;
    a.scales = (const float *)((const uint8_t *)scales + l * sc_bytes);
    a.eb = coli_fmt_expert_bytes(fmt, H, F);
    a.es = fmt == COLI_FMT_I4G ? coli_expert_scale_count(H, F)
                               : coli_fmt_expert_scale_bytes(fmt, H, F);
    a.residual = residual ? (l == 0 ? (const float *)x : out) : nullptr;
    a.out = out;
    a.layer_out = layer_out ? layer_out + (size_t)l * T * H : nullptr;
    a.route_counts = route_counts ? route_counts + (size_t)l * E : nullptr;
    a.ctrl = (uint32_t *)ws;
    a.x16 = (__half *)(ws + L.x16);
    a.logits = (float *)(ws + L.logits);
    a.idx = (int32_t *)(ws + L.idx);
    a.gates = (float *)(ws + L.gates);
    a.hist = (int32_t *)(ws + L.hist);
    a.offsets = (int32_t *)(ws + L.offsets);
    a.item_begin = (int32_t *)(ws + L.item_begin);
    a.n_groups = E + S;
    a.route_tok = (int32_t *)(ws + L.route_tok);
    a.route_gate = (float *)(ws + L.route_gate);
    a.inv = (int32_t *)(ws + L.inv);
    a.h16 = (__half *)(ws + L.h16);
    a.y = (float *)(ws + L.y);
    const int xdt = l == 0 ? d->x_dtype : COLI_F32;
    const cudaError_t e = launch_prefill(a, xdt, d->router_dtype, stream);
    if (e != cudaSuccess) return map_err(e);
  }
  return COLI_OK;
}

static int moe_run(const coli_moe_desc *d, int k, int n_layers, const void *x, const void *router_w,
                   const uint8_t *packed, const float *scales, float *out, bool residual,
                   float *layer_out, uint32_t *route_counts, void *workspace, cudaStream_t stream,
                   const TierMap *tier = nullptr) {
  if (use_prefill(d))
    return prefill_run(d, k, n_layers, x, router_w, packed, scales, out, residual, layer_out,
                       route_counts, workspace, stream, tier);
  const int T = d->n_tokens, H = d->hidden;
  const int TP = pass_tokens(T);
  const WsLayout L = ws_layout(TP, H, d->ffn, d->n_experts, d->n_shared, k);
  for (int t0 = 0; t0 < T; t0 += TP) {
    const int tn = T - t0 < TP ? T - t0 : TP;
    const size_t xo = (size_t)t0 * H;
    const void *xp = (const char *)x + xo * xsize(d->x_dtype);
    const int st = moe_pass(d, k, n_layers, tn, xp, d->x_dtype, router_w, packed, scales,
                            out + xo, residual, layer_out ? layer_out + xo : nullptr,
                            route_counts, workspace, L, stream, tier);
    if (st != COLI_OK) return st;
  }
  return COLI_OK;
}

}  // extern "C"

// The layer forward over a tiered expert store (tier.cu validates the map).
int coli::moe_forward_tiered(const coli_moe_desc *d, int top_k, const void *x,
                             const void *router_w, const uint8_t *packed, const float *scales,
                             const TierMap &tier, float *out, uint32_t *route_counts,
                             void *workspace, size_t ws_bytes, cudaStream_t stream) {
  int st = check_desc(d, top_k);
  if (st) return st;
  if (weight_fmt(d) != COLI_FMT_I4G) return COLI_EUNSUPPORTED;
  if (d->n_tokens == 0) return COLI_OK;
  if (!x || !router_w || !packed || !scales || !out || !workspace) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(packed) || !aligned16(scales) ||
      !aligned16(out) || ((uintptr_t)workspace & 255u))
    return COLI_EALIGN;
  if (ws_bytes < coli_moe_workspace_size(d, top_k)) return COLI_ENOMEM;
  return moe_run(d, top_k, 1, x, router_w, packed, scales, out, false, nullptr, route_counts,
                 workspace, stream, &tier);
}

extern "C" {

int coli_moe_forward(const coli_moe_desc *d, int top_k, const void *x, const void *router_w,
                     const uint8_t *packed_experts, const void *scales_v, float *out,
                     uint32_t *route_counts, void *workspace, size_t ws_bytes,
                     cudaStream_t stream) {
  const float *scales = (const float *)scales_v;   // E8M0 bytes for an MXFP4 layer
  int st = check_desc(d, top_k);
  if (st) return st;
  if (fmt_unsupported(d)) return COLI_EUNSUPPORTED;
  if (d->n_tokens == 0) return COLI_OK;
  if (!x || !router_w || !packed_experts || !scales || !out || !workspace) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(packed_experts) ||
      !aligned16(scales) || !aligned16(out) || ((uintptr_t)workspace & 255u))
    return COLI_EALIGN;
  if (ws_bytes < coli_moe_workspace_size(d, top_k)) return COLI_ENOMEM;
  return moe_run(d, top_k, 1, x, router_w, packed_experts, scales, out, false, nullptr,
                 route_counts, workspace, stream);
}

int coli_moe_stack_forward(const coli_moe_desc *d, int top_k, int n_layers, const void *x,
                           const void *router_w, const uint8_t *packed_experts,
                           const void *scales_v, float *x_out, float *layer_out,
                           uint32_t *route_counts, void *workspace, size_t ws_bytes,
                           cudaStream_t stream) {
  const float *scales = (const float *)scales_v;   // E8M0 bytes for an MXFP4 layer
  int st = check_desc(d, top_k);
  if (st) return st;
  if (fmt_unsupported(d)) return COLI_EUNSUPPORTED;
  if (n_layers < 1) return COLI_EINVAL;
  if (d->n_tokens == 0) return COLI_OK;
  if (!x || !router_w || !packed_experts || !scales || !x_out || !workspace)
    return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(packed_experts) ||
      !aligned16(scales) || !aligned16(x_out) || (layer_out && !aligned16(layer_out)) ||
      ((uintptr_t)workspace & 255u))
    return COLI_EALIGN;
  if (ws_bytes < coli_moe_workspace_size(d, top_k)) return COLI_ENOMEM;
  // The residual stream is f32: the stack takes an f32 input.
  if (d->x_dtype != COLI_F32) return COLI_EUNSUPPORTED;
  return moe_run(d, top_k, n_layers, x, router_w, packed_experts, scales, x_out, true, layer_out,
                 route_counts, workspace, stream);
}

int coli_profile_events(int kernel, const cudaEvent_t *before, const cudaEvent_t *after,
                        int n) {
  if (n < 0 || (n > 0 && (!before || !after))) return COLI_EINVAL;
  if (kernel < COLI_KERNEL_ROUTE || kernel > COLI_KERNEL_LAYER) return COLI_EINVAL;
  ProfileState &p = profile();
  std::lock_guard<std::mutex> lock(p.mu);
  const int done = (int)p.next;
  p.kernel = n > 0 ? kernel : -1;
  p.before.assign(before, before + n);
  p.after.assign(after, after + n);
  p.next = 0;
  return done;
}

int coli_moe_check(void *workspace, int clear, uint32_t *flags, cudaStream_t stream) {
  if (!workspace || !flags) return COLI_EINVAL;
  uint32_t v = 0;
  uint32_t *dev = (uint32_t *)workspace + kCtrlFlags;
  cudaError_t e = cudaMemcpyAsync(&v, dev, sizeof(v), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && clear && v) e = cudaMemsetAsync(dev, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return map_err(e);
  *flags = v;
  if (v & COLI_FLAG_TIMEOUT) return COLI_ETIMEOUT;
  if (v & COLI_FLAG_BOUNDS) return COLI_EBOUNDS;
  return (v & COLI_FLAG_RANGE) ? COLI_ERANGE : COLI_OK;
}

}  // extern "C"
