// coli_moe_forward_noalloc: the routed-MoE layer forward for callers that
// cannot allocate device memory -- hosts that own the whole device-memory budget
// up front, or latency-critical loops that must never reach cudaMalloc (which
// can synchronise the device).  Its scratch is a fixed array in the library's
// own device image instead of a caller-provided workspace.
#include <mutex>

#include "coli_internal.cuh"

namespace {

// Scratch for one call.  Every GPU that loads the library holds these bytes
// until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;
static_assert(coli::kWsFixedBytes <= kNoAllocScratchBytes, "fixed region fits the scratch");

static __device__ __align__(256) uint8_t g_coli_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a stand-in, so the address is looked up once per device
// with that device current, and cached (a device reset invalidates it: see
// coli.h).
int scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return coli::cuda_status(e);
  if (dev < 0 || dev >= kMaxDevices) return COLI_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_coli_scratch);
    if (e != cudaSuccess || !p) return coli::cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return COLI_OK;
}

}  // namespace

extern "C" int coli_moe_forward_noalloc(const coli_moe_desc *d, int top_k, const void *x,
                                        const void *router_w, const uint8_t *packed_experts,
                                        const void *scales, float *out,
                                        uint32_t *route_counts, cudaStream_t stream) {
  const size_t need = coli_moe_workspace_size(d, top_k);
  if (need == 0) return COLI_EINVAL;
  if (need > kNoAllocScratchBytes) return COLI_ENOMEM;
  if (d->n_tokens == 0) return COLI_OK;
  void *ws = nullptr;
  int st = scratch_address(&ws);
  if (st != COLI_OK) return st;
  // The array keeps whatever the previous call left.  The control words (flags,
  // completion ticket) and the fixed-point router buffers must start at zero; a
  // successful call leaves them zero, but one that failed part-way may not, and
  // no caller can reach this array to clear it, so every call clears them.
  const cudaError_t e = cudaMemsetAsync(ws, 0, coli::kWsFixedBytes, stream);
  if (e != cudaSuccess) return coli::cuda_status(e);
  return coli_moe_forward(d, top_k, x, router_w, packed_experts, scales, out, route_counts, ws,
                          kNoAllocScratchBytes, stream);
}
