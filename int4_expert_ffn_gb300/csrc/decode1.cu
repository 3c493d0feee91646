// One-token decode layer of the routed-MoE forward over int4-grouped experts,
// fused into a single kernel per layer (k_layer1).
//
// Pages: "Colibrì 深度解析" §十一 (route -> union -> compute; at one token the
// union is the token's k experts), §四 (an expert's three matrices adjacent),
// "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战" (matmul_i4_grouped
// consumes the packed rows directly), "colibrì 路由遥测全解析" (route counts,
// normalised gates).
//
// At one token a layer moves ~(k + S) experts' packed rows once (194 MB for
// the GLM-like shape) and does almost no arithmetic per byte, so it is a
// streaming problem.  One CTA per SM of l1_nc warps.  Every warp streams its
// own stages (s = warp, warp + l1_nc, ...) through its own l1_spw
// shared-memory slots with 1-D bulk copies (cp.async.bulk, completion counted
// on the slot's mbarrier): after computing a stage it copies the stage l1_spw
// later into the freed slot, so l1_spw - 1 stages stay in flight while it
// computes.  (One issuing thread per CTA cannot keep HBM busy: a thread's
// wait-and-issue loop sustains only about three bulk copies per microsecond,
// so every warp issues its own.)
//   - Gate/up stages: l1_rg gate rows + l1_rg up rows of one expert (full
//     width) and their scales.  The rows are cut into h blocks of 32 rows of
//     one expert; CTA c owns blocks c, c + G, ... (the lowest CTAs' first
//     blocks are shared-expert ones, known before routing, so their copies
//     are issued before the kernel waits for its predecessor).  The warp that
//     completes a block quantises its 32 h values into activation planes and
//     publishes them to every replica of the h-plane buffer.
//   - Down stages: l1_dr rows [dh0, dh1) of one used expert's down matrix;
//     every CTA owns the same output rows of every used expert and adds the
//     experts in a fixed order (rank order, then the shared experts).  A
//     warp's first down stages are copied while it still computes gate/up.
//   - Between the two phases the warps pass a grid barrier (every CTA's h
//     planes must be published; one CTA per SM, all co-resident; bounded, a
//     timeout sets COLI_FLAG_TIMEOUT); then one bulk copy brings all h planes
//     of the CTA's replica into shared memory.  The token's x also arrives by
//     one bulk copy: ordinary loads queue behind the weight stream.
// The dot products are those of the GEMV path (15-bit activation planes,
// dp4a against the unsigned nibbles, exact int32 sums, f32 scaling).
#include "coli_internal.cuh"
#include "decode_common.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace coli {

namespace {

// Phase trace of k_layer1, compiled in only with -DCOLI_TRACE (a diagnostic
// build): one %globaltimer stamp per (layer, point, CTA) for the first
// kT1Layers layers of a call, read by coli_trace1_read_raw.
#ifdef COLI_TRACE
constexpr int kT1Layers = 4, kT1Points = 12, kT1Ctas = 160;
static __device__ unsigned long long g_trace1[kT1Layers][kT1Points][kT1Ctas];
__device__ __forceinline__ void t1_point(int layer, int pt) {
  if (blockIdx.x >= kT1Ctas || layer < 0 || layer >= kT1Layers) return;
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  g_trace1[layer][pt][blockIdx.x] = t;
}
#define T1(pt, who) do { if (threadIdx.x == (who)) t1_point(a.layer, pt); } while (0)
#else
#define T1(pt, who) do {} while (0)
#endif

constexpr int kL1Consumers = 8;                    // warps, at most
constexpr int kL1Threads = 32 * kL1Consumers;
constexpr int kL1MinWarps = 4;
constexpr double kL1MaxBytesPerSm = 512.0 * 1024.0;
constexpr int kL1MaxStages = 16;



// Where the CTA's stages come from.  Gate/up work is cut into h blocks: 32
// consecutive rows (gate and up) of one used expert, the rows whose h values
// form one 32-column block of that expert's activation planes.  The blocks
// are numbered shared experts first, then the routed ones by rank; CTA c owns
// blocks c, c + G, c + 2G, ... (so the first block of the lowest CTAs is a
// shared one, known before routing), each cut into 32 / l1_rg stages.
struct L1Work {
  int nblk;         // h blocks owned
  int spb;          // stages per block
  int n_gu;         // gate/up stages = nblk * spb
  int dh0, nr;      // output rows [dh0, dh0 + nr)
  int spe;          // down stages per used expert
  int n_st;         // all stages
};

__device__ __forceinline__ L1Work l1_work(const Dec2Args &a) {
  L1Work w;
  const int G = gridDim.x, c = blockIdx.x;
  const int btot = (a.k + a.S) * (a.F / 32);
  w.nblk = c < btot ? (btot - 1 - c) / G + 1 : 0;
  w.spb = 32 / a.l1_rg;
  w.n_gu = w.nblk * w.spb;
  const int UH = a.H / 4;
  w.dh0 = 4 * part_lo(c, UH, G);
  w.nr = 4 * part_lo(c + 1, UH, G) - w.dh0;
  w.spe = (w.nr + a.l1_dr - 1) / a.l1_dr;
  w.n_st = w.n_gu + (a.k + a.S) * w.spe;
  return w;
}

// Gate/up stage s (< n_gu): expert, first row f, h slot ai (0..k-1 routed
// rank, k..k+S-1 shared), local block lb and the block's index b within the
// expert's planes.
struct GuUnit {
  int e, f, ai, lb, b;
};
__device__ __forceinline__ bool gu_block_shared(const Dec2Args &a, int lb) {
  return (int)blockIdx.x + lb * (int)gridDim.x < a.S * (a.F / 32);
}
__device__ __forceinline__ GuUnit gu_unit(const Dec2Args &a, const L1Work &w, const int *s_idx,
                                          int s) {
  const int bpe = a.F / 32;
  GuUnit u;
  u.lb = s / w.spb;
  const int sub = s - u.lb * w.spb;
  const int B = (int)blockIdx.x + u.lb * (int)gridDim.x;
  const int bs = a.S * bpe;
  if (B < bs) {
    u.ai = a.k + B / bpe;
    u.e = a.E + B / bpe;
    u.b = B - (B / bpe) * bpe;
  } else {
    const int x = B - bs;
    u.ai = x / bpe;
    u.e = COLI_CHK(s_idx[u.ai], a.E, a.ctrl);
    u.b = x - u.ai * bpe;
  }
  u.f = 32 * u.b + sub * a.l1_rg;
  return u;
}

// The copies of stage s into a slot (one thread).
__device__ __forceinline__ void l1_issue(const Dec2Args &a, const L1Work &w, const int *s_idx,
                                         uint8_t *ring, uint64_t *full, int slot, int s) {
  uint8_t *dst = ring + (size_t)slot * a.l1_slot;
  uint64_t *bar = full + slot;
  if (s < w.n_gu) {
    const GuUnit u = gu_unit(a, w, s_idx, s);
    const int64_t rb = a.H / 2, ngr = a.H / kGroup, R = a.l1_rg;
    const uint8_t *pg = a.packed + (int64_t)u.e * a.eb + (int64_t)u.f * rb;
    const float *sg = a.scales + (int64_t)u.e * a.es + (int64_t)u.f * ngr;
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * R * rb + 2 * R * ngr * 4));
    bulk_g2s(dst, pg, (uint32_t)(R * rb), bar);                                  // gate rows
    bulk_g2s(dst + R * rb, pg + (int64_t)a.F * rb, (uint32_t)(R * rb), bar);     // up rows
    bulk_g2s(dst + 2 * R * rb, sg, (uint32_t)(R * ngr * 4), bar);
    bulk_g2s(dst + 2 * R * rb + R * ngr * 4, sg + (int64_t)a.F * ngr, (uint32_t)(R * ngr * 4), bar);
  } else {
    const int d = s - w.n_gu, ai = d / w.spe;
    const int r0 = (d - ai * w.spe) * a.l1_dr;
    const int nq = w.nr - r0 < a.l1_dr ? w.nr - r0 : a.l1_dr;
    const int e = ai < a.k ? COLI_CHK(s_idx[ai], a.E, a.ctrl) : a.E + (ai - a.k);
    const int64_t rb = a.F / 2, ngr = a.F / kGroup;
    const int64_t row = w.dh0 + r0;
    const uint8_t *pd = a.packed + (int64_t)e * a.eb + (int64_t)a.F * a.H + row * rb;
    const float *sd = a.scales + (int64_t)e * a.es + (int64_t)2 * a.F * (a.H / kGroup) + row * ngr;
    mbar_arrive_expect_tx(bar, (uint32_t)(nq * rb + nq * ngr * 4));
    bulk_g2s(dst, pd, (uint32_t)(nq * rb), bar);
    bulk_g2s(dst + (int64_t)a.l1_dr * rb, sd, (uint32_t)(nq * ngr * 4), bar);
  }
}

// Routing of the layer's one token from the fixed-point logits, by every CTA
// alike (same integers, same result): top-k, gates (softmax renormalised, or
// the sigmoid router's), into s_idx / s_gate.  CTA 0 publishes the route
// counts, the NaN flag and idx/gates.  `scratch` holds gu_route_smem(1,E,k).
__device__ void l1_route(const Dec2Args &a, uint8_t *scratch, int *s_idx, float *s_gate) {
  const int E = a.E, k = a.k;
  const GuRouteSmem R = gu_route_smem(1, E, k);
  float *s_logits = (float *)(scratch + R.logits);
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const long long v = __ldcg(a.fx_rd_acc + i);
    const uint32_t f = __ldcg(a.fx_rd_flag + i);
    s_logits[i] = f ? __int_as_float(0x7FC00000) : fx_to_float(v);
  }
  __syncthreads();
  const bool sig = a.router_fn == COLI_ROUTER_SIGMOID_BIAS;
  float *s_keys = s_logits;
  if (sig) {
    s_keys = (float *)(scratch + R.sel);
    sigmoid_keys(s_logits, s_keys, a.router_bias ? (const float *)(scratch + R.bias) : nullptr,
                 1, E);
  }
  const bool nan = select_topk(s_keys, 1, E, k, s_idx, s_gate, (float *)(scratch + R.vals),
                               scratch + R.topk, (int *)(scratch + R.flag));
  if (sig) sigmoid_gates(s_logits, s_idx, 1, E, k, s_gate);
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0 && nan) set_flag(a.ctrl, COLI_FLAG_NAN_LOGITS);
    for (int i = threadIdx.x; i < k; i += blockDim.x) {
      a.g_idx[i] = s_idx[i];
      a.g_gates[i] = s_gate[i];
      if (a.route_counts) atomicAdd(a.route_counts + COLI_CHK(s_idx[i], a.E, a.ctrl), 1u);
    }
  }
  __syncthreads();
}

// Consumer: one gate/up stage (RG gate rows + RG up rows of the expert, full
// width) against the x planes; h = silu(g) * u * gate of its RG rows goes to
// the stage's h block accumulator in shared memory (hb[row within block]).
template <int RG>
__device__ __forceinline__ void l1_gateup_stage(const Dec2Args &a, const uint8_t *st,
                                                const uint32_t *xpl, float *hb, int f_in_block,
                                                float gate) {
  const int lane = threadIdx.x & 31;
  const int H = a.H, rb = H / 2, ngr = H / kGroup, ncg = H / kChunkCols, nbp = H / 32;
  const float *sc = (const float *)(st + 2 * RG * rb);
  float v[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) v[q] = 0.0f;
  for (int j = 0; j < ncg; ++j) {
    Planes p;
    load_planes(xpl, 0, 32 * j + lane, nbp, p);
#pragma unroll
    for (int q = 0; q < 2 * RG; ++q) {
      const uint4 wv = *(const uint4 *)(st + q * rb + 512 * j + 16 * lane);
      v[q] = fmaf(sc[q * ngr + 16 * j + (lane >> 1)], dot32(wv, p), v[q]);
    }
  }
  // lane 4 vi ends with value vi: gate row r is value r, up row r is value RG + r
  const float tot = reduce8(v);
  const float ut = __shfl_sync(0xFFFFFFFFu, tot, (lane & (4 * RG - 4)) + 4 * RG);
  if (lane < 4 * RG && (lane & 3) == 0) hb[f_in_block + (lane >> 2)] = silu(tot) * ut * gate;
}

// Publish h block lb (32 values in shared memory, complete) as its activation
// planes: quantised by lane 0 exactly as the GEMV path quantises activations,
// then its 18 words written by 18 lanes to every replica of the h-plane buffer
// ([replica][k + S][18][F / 32] words, replica stride h_stride floats).
__device__ __forceinline__ void l1_publish_block(const Dec2Args &a, const float *hb,
                                                 uint32_t *stage18, int ai, int b) {
  const int lane = threadIdx.x & 31, nbp = a.F / 32;
  if (lane == 0) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = hb[i];
    Planes p;
    quantize32(v, p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      stage18[i] = p.eh[i];
      stage18[4 + i] = p.el[i];
      stage18[8 + i] = p.oh[i];
      stage18[12 + i] = p.ol[i];
    }
    stage18[16] = (uint32_t)p.sq;
    stage18[17] = __float_as_uint(p.sx);
  }
  __syncwarp();
  if (lane < 18) {
    const uint32_t word = stage18[lane];
    uint32_t *base = (uint32_t *)a.h + ((size_t)ai * 18 + lane) * nbp + b;
    for (int r = 0; r < a.n_rep; ++r) base[(size_t)r * a.h_stride] = word;
    fence_proxy_async_global();   // read back by other CTAs' bulk copies
  }
  __syncwarp();
}

// Consumer: one down stage (nq rows of used expert ai) against the h planes;
// leaves each row's sum in red[ai][row].
__device__ __forceinline__ void l1_down_stage(const Dec2Args &a, const L1Work &w, const uint8_t *st,
                                              const uint32_t *hpl, float *red, int s) {
  const int lane = threadIdx.x & 31;
  const int F = a.F, rb = F / 2, ngr = F / kGroup, ncg = F / kChunkCols, nbp = F / 32;
  const int d = s - w.n_gu, ai = d / w.spe;
  const int r0 = (d - ai * w.spe) * a.l1_dr;
  const int nq = w.nr - r0 < a.l1_dr ? w.nr - r0 : a.l1_dr;
  const float *sc = (const float *)(st + (size_t)a.l1_dr * rb);
  for (int g = 0; g < nq; g += 8) {
    const int nrow = nq - g < 8 ? nq - g : 8;     // 8, or 4 at a ragged end
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = 0.0f;
    for (int j = 0; j < ncg; ++j) {
      Planes p;
      load_planes(hpl, ai, 32 * j + lane, nbp, p);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (q < nrow) {
          const uint4 wv = *(const uint4 *)(st + (size_t)(g + q) * rb + 512 * j + 16 * lane);
          v[q] = fmaf(sc[(g + q) * ngr + 16 * j + (lane >> 1)], dot32(wv, p), v[q]);
        }
      }
    }
    const float tot = reduce8(v);   // lane 4 q: row q
    const int q = lane >> 2;
    if ((lane & 3) == 0 && q < nrow) red[ai * w.nr + r0 + g + q] = tot;
  }
}

// The next layer's router-row slice ([E][nr] values of type WT, this CTA's
// columns dh0 .. dh0 + nr) into shared memory by cp.async, 8 bytes per copy,
// so the kernel does not wait for it at its start; the partials at the end
// wait for the group.  dh0 and nr are multiples of 4 and the rows whole
// multiples of 1024 values, so with an 8-byte aligned base every piece is
// aligned.  Returns false (nothing issued) for a misaligned base.
template <typename WT>
__device__ __forceinline__ bool l1_router_rows_async(const Dec2Args &a, const WT *wr, WT *s_wr) {
  if (((uintptr_t)wr & 7) != 0) return false;
  const int H = a.H, E = a.E, G = gridDim.x, c = blockIdx.x, UH = H / 4;
  const int dh0 = 4 * part_lo(c, UH, G), nr = 4 * part_lo(c + 1, UH, G) - dh0;
  constexpr int kPer = 8 / (int)sizeof(WT);     // values per 8-byte piece
  const int ppr = nr / kPer;                    // pieces per row
  for (int i = threadIdx.x; i < E * ppr; i += blockDim.x) {
    const int e = i / ppr, q = i - e * ppr;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(
                     smem_u32(s_wr + (size_t)e * nr + q * kPer)),
                 "l"(wr + (size_t)e * H + dh0 + q * kPer)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  return true;
}

template <typename WT>
__global__ void __launch_bounds__(kL1Threads, 1) k_layer1(Dec2Args a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const L1Smem &L = a.l1;
  uint64_t *full = (uint64_t *)(smem + L.bar);
  uint64_t *xbar = full + kL1MaxStages;      // the token's x in shared memory
  uint64_t *hbar = xbar + 1;                 // every CTA's h planes in shared memory
  int *s_idx = (int *)(smem + L.lst);
  float *s_gate = (float *)(s_idx + kMaxTopK);
  float *red = (float *)(smem + L.red);
  float *s_xn = (float *)(smem + L.xn);
  WT *s_wr = (WT *)(smem + L.wr);
  float *s_hacc = (float *)(smem + L.hacc);                 // [nblk][32] h blocks being built
  int *s_hcnt = (int *)(s_hacc + (size_t)a.l1_nblk * 32);   // stages done per block
  uint32_t *s_pub = (uint32_t *)(s_hcnt + a.l1_nblk);       // [kL1Consumers][18]
  uint8_t *U = smem + L.u;
  uint8_t *ring = smem + L.ring;
  float *s_x = (float *)(U + a.l1_xs_off);
  uint32_t *xpl = (uint32_t *)(U + a.l1_xpl_off);
  uint32_t *hpl = (uint32_t *)U;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NC = a.l1_nc, SPW = a.l1_spw;
  const L1Work w = l1_work(a);
  // this warp's stages: warp, warp + NC, ...; its t-th stage goes to slot
  // warp * SPW + t % SPW (use t / SPW of that slot)
  const int my_gu = w.n_gu > warp ? (w.n_gu - warp + NC - 1) / NC : 0;
  const int my_st = w.n_st > warp ? (w.n_st - warp + NC - 1) / NC : 0;
  auto slot_of = [&](int t) { return warp * SPW + t % SPW; };

  T1(0, 0);
  if (tid == 0) {
    for (int i = 0; i < NC * SPW; ++i) mbar_init(full + i, 1);
    mbar_init(xbar, 1);
    mbar_init(hbar, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < w.nblk; i += blockDim.x) s_hcnt[i] = 0;
  __syncthreads();
  // Before the dependency wait: only data no kernel of this stream writes --
  // a warp's first stage when it belongs to a shared-expert block (one per
  // warp, so that the token's x, copied after the wait, is not queued behind
  // much), the next layer's router rows, the sigmoid router's bias.
  int issued = 0;                                   // this warp's stages issued so far
  if (lane == 0 && my_gu > 0 && gu_block_shared(a, warp / w.spb)) {
    l1_issue(a, w, s_idx, ring, full, slot_of(0), warp);
    issued = 1;
  }
  if (a.wr && !l1_router_rows_async<WT>(a, (const WT *)a.wr, s_wr))
    load_router_rows<WT>(a, (const WT *)a.wr, s_wr);
  if (a.router_fn == COLI_ROUTER_SIGMOID_BIAS && a.router_bias) {
    float *s_bias = (float *)(U + gu_route_smem(1, a.E, a.k).bias);
    for (int i = tid; i < a.E; i += blockDim.x) s_bias[i] = __ldg(a.router_bias + i);
  }
  T1(1, 0);
  grid_dependents_launch();
  grid_dependency_wait();
  T1(2, 0);
  // the token's x (this CTA's replica) by one bulk copy, while the block routes
  if (tid == 0) {
    fence_proxy_async_global();   // x was written by the previous kernel's generic stores
    mbar_arrive_expect_tx(xbar, (uint32_t)(a.H * 4));
    bulk_g2s(s_x, a.xrep + (size_t)(blockIdx.x % a.n_rep) * a.x_stride, (uint32_t)(a.H * 4), xbar);
  }
  l1_route(a, U, s_idx, s_gate);                 // ends with __syncthreads
  T1(3, 0);
  // every warp's remaining first stages (routed experts are known now)
  if (lane == 0)
    for (; issued < SPW && issued < my_st; ++issued)
      l1_issue(a, w, s_idx, ring, full, slot_of(issued), warp + issued * NC);
  // x planes from shared memory: one 32-column block per thread
  if (!mbar_wait(xbar, 0) && tid == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
  for (int b = tid; b < a.H / 32; b += blockDim.x) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 q = *(const float4 *)(s_x + 32 * b + 4 * i);
      v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
    }
    Planes p;
    quantize32(v, p);
    uint32_t *pv = xpl + b;
    const int nbp = a.H / 32;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pv[(size_t)i * nbp] = p.eh[i];
      pv[(size_t)(4 + i) * nbp] = p.el[i];
      pv[(size_t)(8 + i) * nbp] = p.oh[i];
      pv[(size_t)(12 + i) * nbp] = p.ol[i];
    }
    pv[(size_t)16 * nbp] = (uint32_t)p.sq;
    pv[(size_t)17 * nbp] = __float_as_uint(p.sx);
  }
  // U is written by the bulk copy of the h planes later: order these generic
  // writes (routing scratch, x planes) before it
  fence_proxy_async();
  __syncthreads();
  T1(4, 0);

  // wait for this warp's t-th stage; after computing it, copy stage t + SPW
  // into the freed slot
  auto take = [&](int t) -> const uint8_t * {
    const int slot = slot_of(t);
    if (!mbar_wait(full + slot, (t / SPW) & 1) && lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
    return ring + (size_t)slot * a.l1_slot;
  };
  auto refill = [&](int t) {
    __syncwarp();
    if (lane == 0 && t + SPW < my_st) l1_issue(a, w, s_idx, ring, full, slot_of(t), warp + (t + SPW) * NC);
  };
  int t = 0;
  for (; t < my_gu; ++t) {
    const int s = warp + t * NC;
    const uint8_t *st = take(t);
    const GuUnit u = gu_unit(a, w, s_idx, s);
    const float g = u.ai < a.k ? s_gate[u.ai] : 1.0f;
    float *hb = s_hacc + (size_t)u.lb * 32;
    if (a.l1_rg == 4) l1_gateup_stage<4>(a, st, xpl, hb, u.f - 32 * u.b, g);
    else if (a.l1_rg == 2) l1_gateup_stage<2>(a, st, xpl, hb, u.f - 32 * u.b, g);
    else l1_gateup_stage<1>(a, st, xpl, hb, u.f - 32 * u.b, g);
    refill(t);
    // the warp that completes a block's last stage publishes its planes
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = atomicAdd(s_hcnt + u.lb, 1) == w.spb - 1;
    }
    if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
      __threadfence_block();
      l1_publish_block(a, hb, s_pub + warp * 18, u.ai, u.b);
    }
  }
  T1(5, 0);
  // every CTA's h planes complete before any CTA reads them
  __syncthreads();
  if (tid == 0) {
    if (!grid_sync(a.ctrl, gridDim.x)) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
    fence_proxy_async_global();
    // all k + S slots' planes of this CTA's replica into U, by one bulk copy
    const uint32_t bytes = (uint32_t)((a.k + a.S) * 18 * (a.F / 32) * 4);
    mbar_arrive_expect_tx(hbar, bytes);
    bulk_g2s(hpl, a.h + (size_t)(blockIdx.x % a.n_rep) * a.h_stride, bytes, hbar);
  }
  T1(6, 0);
  // every CTA has routed: clear this CTA's share of the logits it read
  {
    const int TE = a.E, G = gridDim.x, c = blockIdx.x;
    const int i0 = part_lo(c, TE, G), i1 = part_lo(c + 1, TE, G);
    for (int i = i0 + tid; i < i1; i += blockDim.x) {
      a.fx_clr_acc[i] = 0;
      a.fx_clr_flag[i] = 0u;
    }
  }
  if (!mbar_wait(hbar, 0) && lane == 0) set_flag(a.ctrl, COLI_FLAG_TIMEOUT);
  T1(7, 0);
  for (; t < my_st; ++t) {
    const uint8_t *st = take(t);
    l1_down_stage(a, w, st, hpl, red, warp + t * NC);
    refill(t);
  }
  T1(8, 0);
  __syncthreads();
  T1(9, 0);
  // combine: each row adds the used experts in a fixed order (rank order,
  // then the shared experts); residual, outputs, next layer's input replicas
  const int KS = a.k + a.S;
  for (int r = tid; r < w.nr; r += blockDim.x) {
    float sum = 0.0f;
    for (int x = 0; x < KS; ++x) sum += red[x * w.nr + r];
    const int64_t o = w.dh0 + r;
    if (a.layer_out) a.layer_out[o] = sum;
    const float xn = a.residual ? a.residual[o] + sum : sum;
    a.out[o] = xn;
    s_xn[r] = xn;
    if (a.xrep)
      for (int rr = 0; rr < a.n_rep; ++rr) a.xrep[rr * a.x_stride + o] = xn;
  }
  // this thread's router-row pieces (if any) have landed; the barrier makes
  // every thread's visible
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  T1(10, 0);
  if (a.wr) dn_partials_fx<WT>(a, s_wr, s_xn);
  T1(11, 0);
}

}  // namespace

#ifdef COLI_TRACE
extern "C" int coli_trace1_reset() {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_trace1) != cudaSuccess) return -1;
  return cudaMemset(p, 0, sizeof(g_trace1)) == cudaSuccess ? 0 : -1;
}
// [layer][point][cta] timestamps in ns (0: not reached).
extern "C" int coli_trace1_read_raw(void *buf) {
  return cudaMemcpyFromSymbol(buf, g_trace1, sizeof(g_trace1)) == cudaSuccess ? 0 : -1;
}
#endif

// Plan of the fused one-token layer kernel; false when the shape is outside
// what it handles (the GEMV kernel pair takes it).
bool plan_layer1(Dec2Args &a) {
  // its bulk copies read HBM only: a tiered store (experts partly in host
  // memory) takes the GEMV kernels
  if (a.T != 1 || !a.fx || a.n_rep != 8 || a.tier.slot_of) return false;
  if (a.H % kChunkCols || a.F % kChunkCols) return false;
  // Taken where a layer's used experts are a small share per SM (the
  // latency-bound regime: one launch instead of two, no kernel boundary
  // between gate/up and down).  Wide layers stream well enough in the GEMV
  // kernel pair, which measured faster there: 1.92 k vs 1.65 k tokens/s on the
  // GLM-like layers (1.26 MB per SM), against 2.96 k vs 2.58 k on the
  // OLMoE-like stack (0.19 MB per SM).
  if ((double)(a.k + a.S) * (double)(a.eb + 4 * a.es) / a.n_part > kL1MaxBytesPerSm) return false;
  const int G = a.n_part, KS = a.k + a.S;
  const size_t budget = (size_t)max_smem() - 1024;
  const int max_nr = 4 * ((a.H / 4 + G - 1) / G);
  const size_t gu_row = (size_t)(a.H / 2) + (size_t)(a.H / kGroup) * 4;
  const size_t dn_row = (size_t)(a.F / 2) + (size_t)(a.F / kGroup) * 4;
  L1Smem m{};
  size_t o = 0;
  m.bar = o; o += (size_t)(kL1MaxStages + 2) * 8;
  m.lst = o; o = al16(o + (size_t)2 * kMaxTopK * 4);
  m.red = o; o = al16(o + (size_t)KS * max_nr * 4);
  m.xn = o; o = al16(o + (size_t)max_nr * 4);
  m.wr = o; o = al16(o + (a.chain ? (size_t)a.E * max_nr * (a.wr_bf16 ? 2 : 4) : 0));
  // h blocks: accumulators, stage counters, each consumer warp's 18-word staging
  const int btot = KS * (a.F / 32);
  const int nblk = (btot + G - 1) / G;
  m.hacc = o; o = al16(o + (size_t)nblk * 32 * 4 + (size_t)nblk * 4 + (size_t)kL1Consumers * 18 * 4);
  // U: the routing scratch, x (f32) and its planes side by side; later the h
  // planes of every used expert
  const size_t route = al128(gu_route_smem(1, a.E, a.k).total);
  const size_t xs = al128((size_t)a.H * 4);
  const size_t xpl = (size_t)18 * (a.H / 32) * 4;
  const size_t hpl = (size_t)KS * 18 * (a.F / 32) * 4;
  const size_t u = route + xs + xpl > hpl ? route + xs + xpl : hpl;
  m.u = o; o = al128(o + u);
  m.ring = o;
  if (o >= budget) return false;
  // stages of rg gate + rg up rows (rg = 4 before rg = 2), two slots per
  // warp, 4..8 warps (measured on GB300: more warps beat deeper per-warp
  // rings -- a warp's dp4a chains need other warps to hide their latency --
  // and smaller stages lose to the per-copy cost)
  int best_rg = 0, best_ns = 0, best_nc = 0, best_spw = 0;
  size_t best_slot = 0;
  for (int rg = 4; rg >= 2 && !best_rg; rg /= 2) {
    const size_t slot0 = (size_t)2 * rg * gu_row;
    const size_t slot = slot0 > 4 * dn_row ? slot0 : 4 * dn_row;
    int ns = (int)((budget - o) / slot);
    if (ns > kL1MaxStages) ns = kL1MaxStages;
    const int nc = ns / 2 > kL1Consumers ? kL1Consumers : ns / 2;
    if (nc < kL1MinWarps) continue;
    best_rg = rg; best_ns = nc * 2; best_nc = nc; best_spw = 2; best_slot = slot;
  }
  if (!best_rg) return false;
  int dr = 4 * (int)(best_slot / (4 * dn_row));
  const int dr_cap = (max_nr + 3) & ~3;
  if (dr > dr_cap) dr = dr_cap;
  m.total = al16(o + (size_t)best_ns * best_slot);
  a.l1 = m;
  a.l1_ns = best_ns;
  a.l1_nc = best_nc;
  a.l1_spw = best_spw;
  a.l1_rg = best_rg;
  a.l1_slot = (int)best_slot;
  a.l1_dr = dr;
  a.l1_xs_off = (int)route;
  a.l1_xpl_off = (int)(route + xs);
  a.l1_nblk = nblk;
  return true;
}

cudaError_t launch_layer1(const Dec2Args &a, cudaStream_t s, bool pdl) {
  cudaError_t e;
  if (a.wr_bf16) {
    if ((e = allow_smem(k_layer1<__nv_bfloat16>, a.l1.total)) != cudaSuccess) return e;
    return launch(k_layer1<__nv_bfloat16>, a.n_part, 32 * a.l1_nc, a.l1.total, s, pdl, a);
  }
  if ((e = allow_smem(k_layer1<float>, a.l1.total)) != cudaSuccess) return e;
  return launch(k_layer1<float>, a.n_part, 32 * a.l1_nc, a.l1.total, s, pdl, a);
}

}  // namespace coli
