// Phase tracing of the decode kernels.  Compiled in only with -DCOLI_TRACE
// (a separate diagnostic build); otherwise every trace point is empty.
// Thread 0 of every CTA folds %globaltimer (ns) at each point into the
// earliest and latest value seen for [layer][point]; coli_trace_reset()
// clears the tables and coli_trace_read() copies them out.
#pragma once

#include <stdint.h>

namespace coli {

constexpr int kTraceLayers = 64, kTracePoints = 24;

#ifdef COLI_TRACE
// Defined here; only the decode translation unit includes this header.
static __device__ unsigned long long g_trace_lo[kTraceLayers][kTracePoints];
static __device__ unsigned long long g_trace_hi[kTraceLayers][kTracePoints];
__device__ __forceinline__ void trace_point(int layer, int pt) {
  if (threadIdx.x != 0 || layer < 0 || layer >= kTraceLayers) return;
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  atomicMin(&g_trace_lo[layer][pt], t);
  atomicMax(&g_trace_hi[layer][pt], t);
}
#define COLI_TRACE_POINT(layer, pt) ::coli::trace_point((layer), (pt))
#else
#define COLI_TRACE_POINT(layer, pt) do {} while (0)
#endif

// Trace points (second index).
enum TracePoint : int {
  kTpGuEntry = 0, kTpGuDepWait, kTpGuLists, kTpGuPlanes, kTpGuFirstLoads, kTpGuCompute, kTpGuEnd,
  kTpDnEntry, kTpDnDepWait, kTpDnLists, kTpDnPlanes, kTpDnCompute, kTpDnCombine,
  kTpDnPartials, kTpRouteStart, kTpEnd,
  kTpRtLogits, kTpRtTopk, kTpRtPublish, kTpRtUnion,
};

}  // namespace coli
