// Phase tracing of the decode kernels.  Compiled in only with -DCOLI_TRACE
// (a separate diagnostic build); otherwise every trace point is empty.
// Thread 0 of every CTA stores %globaltimer (ns) at each point into its own
// [layer][point][cta] entry (plain stores: no contended atomics that would
// slow the traced CTA); coli_trace_reset() clears the table and
// coli_trace_read() / coli_trace_read_raw() copy it out.
#pragma once

#include <stdint.h>

namespace coli {

constexpr int kTraceLayers = 64, kTracePoints = 25, kTraceCtas = 160;

#ifdef COLI_TRACE
// Defined here; only the decode translation unit includes this header.
static __device__ unsigned long long g_trace[kTraceLayers][kTracePoints][kTraceCtas];
__device__ __forceinline__ void trace_point(int layer, int pt) {
  if (threadIdx.x != 0 || layer < 0 || layer >= kTraceLayers || pt < 0 || pt >= kTracePoints ||
      blockIdx.x >= kTraceCtas)
    return;
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  g_trace[layer][pt][blockIdx.x] = t;
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
  kTpRtLogits, kTpRtTopk, kTpRtPublish, kTpRtUnion, kTpDnPlaneStart, kTpDnPlaneBuilt,
  kTpGuSplit, kTpGuNeed, kTpGuRouter,
};

}  // namespace coli
