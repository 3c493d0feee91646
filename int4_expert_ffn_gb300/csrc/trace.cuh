// Phase tracing of the decode kernels.  Compiled in only with -DCOLI_TRACE
// (a separate diagnostic build); otherwise every trace point is empty.
// Each point stores %globaltimer (ns) at [kernel][cta][point]; stage points
// of one chosen CTA go to a second table.  Read back with coli_trace_read().
#pragma once

#include <stdint.h>

namespace coli {

constexpr int kTraceCtas = 256, kTracePoints = 16, kTraceStages = 32, kTraceCta = 7;

#ifdef COLI_TRACE
// Defined here; only the decode translation unit includes this header.
static __device__ unsigned long long g_trace[2][kTraceCtas][kTracePoints];
static __device__ unsigned long long g_trace_stage[2][kTraceStages];
static __device__ unsigned long long g_trace_issue[2][kTraceStages];
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
#define COLI_TRACE_POINT(kern, pt)                                                        \
  do {                                                                                    \
    if (blockIdx.x < ::coli::kTraceCtas) ::coli::g_trace[kern][blockIdx.x][pt] = ::coli::trace_now(); \
  } while (0)
#define COLI_TRACE_ISSUE(kern, s)                                                         \
  do {                                                                                    \
    if (blockIdx.x == ::coli::kTraceCta && (s) < ::coli::kTraceStages)                    \
      ::coli::g_trace_issue[kern][s] = ::coli::trace_now();                               \
  } while (0)
#define COLI_TRACE_STAGE(kern, s)                                                         \
  do {                                                                                    \
    if (blockIdx.x == ::coli::kTraceCta && (s) < ::coli::kTraceStages)                    \
      ::coli::g_trace_stage[kern][s] = ::coli::trace_now();                               \
  } while (0)
#else
#define COLI_TRACE_POINT(kern, pt) do {} while (0)
#define COLI_TRACE_ISSUE(kern, s) do {} while (0)
#define COLI_TRACE_STAGE(kern, s) do {} while (0)
#endif

}  // namespace coli
