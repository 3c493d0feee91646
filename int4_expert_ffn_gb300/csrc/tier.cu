// Tiered expert store: the layer forward over an HBM slot pool plus the full
// store in pinned host memory, the LFRU admission policy tick, and the
// uploads it decides.
//
// Pages: "Colibrì 深度解析" §四 (三层存储层级: VRAM / RAM / NVMe, one forward for
// every tier, so placement changes speed and never the result; the three
// matrices of an expert adjacent, read in one go), §十一 (place, overlap,
// learn), §三 (LFRU: frequency first, recency breaks close calls; promotion
// with 25% + 4 hysteresis, widened before the margin is added).
//
// On GB300 the host store is read by the GPU itself over NVLink-C2C: the
// expert GEMVs take each expert's record from its pool slot or from host
// memory (expert_record), so missing experts stream while resident ones
// compute, in the same kernels.  The policy tick runs in one CTA; uploads are
// plain copies from the host store by a grid of CTAs.
#include "coli_internal.cuh"

namespace coli {

namespace {

constexpr int kTierThreads = 1024;

__device__ __forceinline__ uint32_t lfru_recent(uint32_t clock, uint32_t last) {
  const uint32_t age = clock - last;
  return age < 255u ? 255u - age : 0u;
}
__device__ __forceinline__ uint64_t lfru_score(uint32_t heat, uint32_t last, uint32_t clock) {
  return ((uint64_t)heat << 8) | lfru_recent(clock, last);
}
__device__ __forceinline__ bool should_promote(uint32_t hot, uint32_t cold) {
  const uint64_t threshold = (uint64_t)cold + ((uint64_t)cold >> 2) + 4u;
  return (uint64_t)hot > threshold;
}

// Block-wide argmin / argmax helpers over (key, index): the smallest key,
// ties to the smaller index (argmin); the largest key, ties to the smaller
// index (argmax).
struct KeyIdx {
  uint64_t key;
  int idx;
};
__device__ __forceinline__ bool better_min(const KeyIdx &a, const KeyIdx &b) {
  return a.key < b.key || (a.key == b.key && a.idx < b.idx);
}
__device__ __forceinline__ bool better_max(const KeyIdx &a, const KeyIdx &b) {
  return a.key > b.key || (a.key == b.key && a.idx < b.idx);
}
template <bool kMin>
__device__ KeyIdx block_best(KeyIdx v, KeyIdx *s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    KeyIdx o;
    o.key = __shfl_xor_sync(0xFFFFFFFFu, v.key, off);
    o.idx = __shfl_xor_sync(0xFFFFFFFFu, v.idx, off);
    if (kMin ? better_min(o, v) : better_max(o, v)) v = o;
  }
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < nw ? s_red[lane] : KeyIdx{kMin ? ~0ull : 0ull, 0x7FFFFFFF};
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      KeyIdx o;
      o.key = __shfl_xor_sync(0xFFFFFFFFu, v.key, off);
      o.idx = __shfl_xor_sync(0xFFFFFFFFu, v.idx, off);
      if (kMin ? better_min(o, v) : better_max(o, v)) v = o;
    }
    if (lane == 0) s_red[0] = v;
  }
  __syncthreads();
  const KeyIdx r = s_red[0];
  __syncthreads();
  return r;
}

// One policy tick (one CTA).
__global__ void __launch_bounds__(kTierThreads) k_tier_update(const uint32_t *counts, int E,
                                                              coli_tier t) {
  __shared__ KeyIdx s_red[32];
  __shared__ uint32_t s_clock;
  __shared__ int s_n, s_target, s_cand;
  __shared__ uint32_t s_cold;
  extern __shared__ uint8_t s_dyn[];
  uint8_t *s_admitted = s_dyn;                      // [E] admitted this tick
  if (threadIdx.x == 0) {
    s_clock = *t.clock + 1u;
    *t.clock = s_clock;
    s_n = 0;
  }
  __syncthreads();
  const uint32_t clock = s_clock;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const uint32_t c = counts[e];
    const uint32_t h = t.heat[e];
    const uint64_t nh = (uint64_t)(h - (h >> 3)) + c;
    t.heat[e] = nh > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)nh;
    if (c) t.last[e] = clock;
    s_admitted[e] = 0;
  }
  __syncthreads();
  // candidates one at a time, best first: used this tick, not resident, not
  // yet considered; at most max_uploads moves
  while (s_n < t.max_uploads) {
    KeyIdx best{0ull, 0x7FFFFFFF};
    bool any = false;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      if (!counts[e] || t.slot_of[e] >= 0 || s_admitted[e]) continue;
      const KeyIdx v{lfru_score(t.heat[e], t.last[e], clock), e};
      if (!any || better_max(v, best)) best = v;
      any = true;
    }
    if (!any) best = KeyIdx{0ull, 0x7FFFFFFF};
    // candidates have score >= 256 (used this tick), so key 0 means none
    const KeyIdx cand = block_best<false>(best, s_red);
    if (cand.idx == 0x7FFFFFFF || cand.key == 0ull) break;
    // target: the lowest free slot, else the resident routed expert of lowest score
    KeyIdx freeb{0ull, 0x7FFFFFFF};
    KeyIdx victim{~0ull, 0x7FFFFFFF};
    for (int sl = threadIdx.x; sl < t.n_slots; sl += blockDim.x) {
      const int owner = t.slot_owner[sl];
      if (owner < 0) {
        if (sl < freeb.idx) freeb = KeyIdx{0ull, sl};
      } else if (owner < E && !s_admitted[owner]) {
        const KeyIdx v{lfru_score(t.heat[owner], t.last[owner], clock), sl};
        if (better_min(v, victim)) victim = v;
      }
    }
    const KeyIdx fr = block_best<true>(KeyIdx{freeb.idx == 0x7FFFFFFF ? ~0ull : 0ull, freeb.idx},
                                       s_red);
    const KeyIdx vi = block_best<true>(victim, s_red);
    if (threadIdx.x == 0) {
      s_target = -1;
      s_cand = cand.idx;
      if (fr.key == 0ull && fr.idx != 0x7FFFFFFF) {
        s_target = fr.idx;
        s_cold = 0u;
      } else if (vi.idx != 0x7FFFFFFF) {
        s_target = vi.idx;
        s_cold = t.heat[t.slot_owner[vi.idx]];
      }
      if (s_target >= 0 && should_promote(t.heat[s_cand], s_cold)) {
        const int old = t.slot_owner[s_target];
        if (old >= 0) t.slot_of[old] = -1;
        t.slot_owner[s_target] = s_cand;
        t.slot_of[s_cand] = s_target;
        t.uploads[1 + 2 * s_n] = (uint32_t)s_cand;
        t.uploads[2 + 2 * s_n] = (uint32_t)s_target;
        ++s_n;
      }
      s_admitted[s_cand] = 1;    // considered: not again this tick
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) t.uploads[0] = (uint32_t)s_n;
}

// Copy the records of the listed (expert, slot) pairs from the store into the
// pool, 16 bytes per thread and step.  list: count, then pairs; n_fixed >= 0
// overrides the count with a list of that many slots whose expert is
// slot_owner[slot] (initial placement: every slot in order).
__global__ void k_tier_copy(const uint8_t *store_packed, const float *store_scales, coli_tier t,
                            int64_t eb, int64_t es, int n_fixed) {
  const int n = n_fixed >= 0 ? n_fixed : (int)t.uploads[0];
  const int64_t pw = eb / 16, sw = es * 4 / 16;
  for (int i = 0; i < n; ++i) {
    int e, sl;
    if (n_fixed >= 0) {
      sl = i;
      e = t.slot_owner[sl];
      if (e < 0) continue;
    } else {
      e = (int)t.uploads[1 + 2 * i];
      sl = (int)t.uploads[2 + 2 * i];
    }
    const uint4 *sp = (const uint4 *)(store_packed + (int64_t)e * eb);
    uint4 *dp = (uint4 *)(t.pool_packed + (int64_t)sl * eb);
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < pw;
         j += (int64_t)gridDim.x * blockDim.x)
      dp[j] = sp[j];
    const uint4 *ss = (const uint4 *)(store_scales + (int64_t)e * es);
    uint4 *ds = (uint4 *)(t.pool_scales + (int64_t)sl * es);
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < sw;
         j += (int64_t)gridDim.x * blockDim.x)
      ds[j] = ss[j];
  }
}

// Device-accessible address of pinned host memory, or null.
const void *host_device_ptr(const void *p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  return at.devicePointer;
}

bool tier_ok(const coli_moe_desc *d, const coli_tier *t) {
  if (!d || !t || t->n_slots < 0 || t->max_uploads < 0) return false;
  if (t->n_slots > 0 && (!t->slot_owner || !t->pool_packed || !t->pool_scales)) return false;
  if (!t->slot_of) return false;
  if (((uintptr_t)t->pool_packed | (uintptr_t)t->pool_scales) & 15u) return false;
  return true;
}

}  // namespace

}  // namespace coli

using namespace coli;

extern "C" {

int coli_moe_forward_tiered(const coli_moe_desc *d, int top_k, const void *x,
                            const void *router_w, const uint8_t *host_packed,
                            const float *host_scales, const coli_tier *tier, float *out,
                            uint32_t *route_counts, void *workspace, size_t ws_bytes,
                            cudaStream_t stream) {
  if (!tier_ok(d, tier)) return COLI_EINVAL;
  if (!host_packed || !host_scales) return COLI_EINVAL;
  const uint8_t *pk = (const uint8_t *)host_device_ptr(host_packed);
  const float *sc = (const float *)host_device_ptr(host_scales);
  if (!pk || !sc) return COLI_EINVAL;
  TierMap m;
  m.slot_of = tier->slot_of;
  m.pool_packed = tier->pool_packed;
  m.pool_scales = tier->pool_scales;
  return moe_forward_tiered(d, top_k, x, router_w, pk, sc, m, out, route_counts, workspace,
                            ws_bytes, stream);
}

int coli_tier_place(const coli_moe_desc *d, const uint8_t *host_packed, const float *host_scales,
                    const coli_tier *tier, cudaStream_t stream) {
  if (!tier_ok(d, tier) || !host_packed || !host_scales) return COLI_EINVAL;
  if (d->hidden < 64 || d->ffn < 64 || d->hidden % kGroup || d->ffn % kGroup) return COLI_EINVAL;
  const uint8_t *pk = (const uint8_t *)host_device_ptr(host_packed);
  const float *sc = (const float *)host_device_ptr(host_scales);
  if (!pk || !sc) return COLI_EINVAL;
  if (tier->n_slots == 0) return COLI_OK;
  const int sms = num_sms();
  if (sms <= 0) return cuda_status(cudaErrorNoDevice);
  const int64_t eb = coli_expert_packed_bytes(d->hidden, d->ffn);
  const int64_t es = coli_expert_scale_count(d->hidden, d->ffn);
  k_tier_copy<<<sms * 2, 512, 0, stream>>>(pk, sc, *tier, eb, es, tier->n_slots);
  return cuda_status(cudaGetLastError());
}

int coli_tier_update(const coli_moe_desc *d, const uint32_t *call_counts,
                     const uint8_t *host_packed, const float *host_scales, const coli_tier *tier,
                     cudaStream_t stream) {
  if (!tier_ok(d, tier) || !call_counts || !host_packed || !host_scales) return COLI_EINVAL;
  if (!tier->heat || !tier->last || !tier->clock || !tier->uploads) return COLI_EINVAL;
  if (d->n_experts < 1 || d->n_experts > kMaxExperts) return COLI_EINVAL;
  if (d->hidden < 64 || d->ffn < 64 || d->hidden % kGroup || d->ffn % kGroup) return COLI_EINVAL;
  const uint8_t *pk = (const uint8_t *)host_device_ptr(host_packed);
  const float *sc = (const float *)host_device_ptr(host_scales);
  if (!pk || !sc) return COLI_EINVAL;
  const int sms = num_sms();
  if (sms <= 0) return cuda_status(cudaErrorNoDevice);
  k_tier_update<<<1, kTierThreads, d->n_experts, stream>>>(call_counts, d->n_experts, *tier);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  if (tier->max_uploads == 0) return COLI_OK;
  const int64_t eb = coli_expert_packed_bytes(d->hidden, d->ffn);
  const int64_t es = coli_expert_scale_count(d->hidden, d->ffn);
  k_tier_copy<<<sms * 2, 512, 0, stream>>>(pk, sc, *tier, eb, es, -1);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"
