/*
 * coli.h -- C ABI of the GB300 (sm_103a) routed-MoE forward over int4-grouped
 * expert weights.
 *
 * What it computes (pages about the "colibri" pure-C MoE engine):
 *   [P1] "Colibrì 深度解析:用 12 万行纯 C 把 744B MoE 塞进 25GB 笔记本"
 *   [P2] "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战"
 *   [P4] "colibrì 路由遥测全解析.coli_usage专家历史、ROUTE_TRACE追踪流与route_trace.h统一格式"
 *
 * Weight format ([P2] §权重转换, quant_int4_grouped / matmul_i4_grouped):
 * a matrix W[O][I] is stored as
 *   packed  uint8 [O][ceil(I/2)]   element (o,i) is nibble u = q + 8 of byte
 *                                  i/2, low nibble for even i, high for odd i
 *   scales  f32   [O][ceil(I/64)]  one scale per 64 consecutive columns
 * and W[o][i] = scales[o][i/64] * (u - 8).
 *
 * Expert record ([P1] §四: an expert's three matrices sit next to each other):
 *   packed_experts = for e in 0 .. E+S-1:  gate[F][H/2] | up[F][H/2] | down[H][F/2]
 *   scales         = for e in 0 .. E+S-1:  gate[F][H/64] | up[F][H/64] | down[H][F/64]
 * experts 0..E-1 are routed, E..E+S-1 are the S shared experts.
 *
 * Conventions of every entry point:
 *   - all array arguments are DEVICE pointers owned by the caller; the library
 *     allocates no memory on any call (scratch lives in the caller's workspace);
 *   - work is enqueued on `stream` and is asynchronous; COLI_OK means the
 *     arguments were valid and the launches were accepted;
 *   - arguments are validated on the host before anything is launched; a
 *     rejected call has no side effect;
 *   - device-side conditions (NaN router logits) are recorded as flag bits
 *     in the workspace and read back with coli_moe_check().
 */
#ifndef COLI_H
#define COLI_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    COLI_OK = 0,
    COLI_EINVAL = -1,        /* null pointer, bad size or dtype */
    COLI_EALIGN = -2,        /* a pointer is not 16-byte aligned */
    COLI_ECUDA = -3,         /* a CUDA launch or query failed */
    COLI_ETIMEOUT = -4,      /* a bounded device-side wait gave up */
    COLI_ENOMEM = -5,        /* the caller's workspace is too small */
    COLI_EUNSUPPORTED = -6,  /* valid, but outside what this build handles */
    COLI_EIO = -7,           /* a file could not be opened, written or renamed */
    COLI_EREFUSED = -8,      /* a usage history belongs to another model or format */
    COLI_ERANGE = -9,        /* an operand left the fp16 range of the batched path */
    COLI_EBOUNDS = -10       /* checked build: an index outside its buffer (COLI_FLAG_BOUNDS) */
} coli_status;

typedef enum { COLI_F32 = 0, COLI_BF16 = 1 } coli_dtype;

/* Device-side flag bits (coli_moe_check). */
#define COLI_FLAG_NAN_LOGITS 0x1u   /* a token had a NaN router logit */
#define COLI_FLAG_TIMEOUT    0x2u   /* a bounded wait gave up */
#define COLI_FLAG_RANGE      0x4u   /* batched path: a value of x or of h = silu(g) u gate
                                       rounded to +-inf in its fp16 operand copy (|v| above
                                       65504); that call's output is not to be used */
#define COLI_FLAG_BOUNDS     0x8u   /* diagnostic build only (-DCOLI_CHECK): an index a kernel
                                       derived from data (expert ids, slot and route lists,
                                       token ids) fell outside its buffer; the access was
                                       redirected to element 0 and the output is not to be used */

/*
 * Routing function ([P1] §十一 "route"; GLM layers: "per-layer n_group=1
 * sigmoid + noaux_tc").
 *   COLI_ROUTER_SOFTMAX       rank the logits; gates = softmax over all E
 *                             renormalised over the k picked.
 *   COLI_ROUTER_SIGMOID_BIAS  scores s_e = 1 / (1 + e^-l_e); rank s_e + b_e,
 *                             b = router_bias, a per-expert bias that only
 *                             selects (noaux_tc with one group: plain top-k
 *                             over all experts); gates = the picked s
 *                             normalised to sum 1 (no further scaling).
 * Both: equal keys -> lower expert id; NaN ranks below every number; a
 * picked NaN gets gate 0; an all-NaN token takes experts 0..k-1 with gates
 * 1/k and sets COLI_FLAG_NAN_LOGITS.
 */
typedef enum { COLI_ROUTER_SOFTMAX = 0, COLI_ROUTER_SIGMOID_BIAS = 1 } coli_router_fn;

/* Shape of one MoE layer call. */
typedef struct {
    int32_t hidden;        /* H: multiple of 64, 64 .. 16384 */
    int32_t ffn;           /* F: multiple of 64, 64 .. 16384 */
    int32_t n_experts;     /* E routed experts, 1 .. 1024 */
    int32_t n_shared;      /* S shared experts, 0 .. 8 */
    int32_t n_tokens;      /* T tokens in this call, >= 0 (0 is a no-op) */
    coli_dtype x_dtype;    /* activations x: COLI_F32 or COLI_BF16 */
    coli_dtype router_dtype; /* router weights: COLI_F32 or COLI_BF16 */
    int32_t router_fn;     /* coli_router_fn; 0 (softmax) when zero-initialised */
    const float *router_bias; /* COLI_ROUTER_SIGMOID_BIAS: device f32 [E] per layer
                                 ([n_layers][E] for the stack), 4-byte aligned,
                                 read-only; NULL = zero bias.  Ignored otherwise. */
    int32_t weight_fmt;    /* coli_weight_fmt of the expert records; 0 = int4-grouped */
} coli_moe_desc;

/*
 * Expert weight containers (the engine's format registry, [P2] §权重转换:
 * "2 int4-row", "4 int4-grouped", "7 MXFP4", "8 fp8-e4m3-b128"; [P1] §十 "从 int4 到
 * MXFP4").
 *   COLI_FMT_I4ROW  int4-row: the int4-grouped rule with one group per row --
 *                   nibbles as above, one f32 scale per row:
 *                     packed uint8 [O][ceil(I/2)], scales f32 [O]
 *                   and W[o][i] = s[o] * (u - 8).  Runs like MXFP4 (below).
 *   COLI_FMT_I4G    int4-grouped, the format above: nibbles + f32 scale per 64
 *   COLI_FMT_MXFP4  OCP Microscaling MXFP4: blocks of 32 columns share one
 *                   E8M0 scale byte e (X = 2^(e - 127)); each element is an
 *                   FP4 E2M1 code (sign bit 3; magnitudes 0, .5, 1, 1.5, 2, 3,
 *                   4, 6), packed two per byte, even column in the low nibble:
 *                     packed uint8 [O][ceil(I/2)], scales uint8 [O][ceil(I/32)]
 *                   and W[o][i] = X[o][i/32] * e2m1(code).  The expert record
 *                   and its scales keep the gate | up | down order; `scales`
 *                   arguments then point to these bytes.  MXFP4 layers run on
 *                   the tensor-core grouped GEMM at every token count, and
 *                   need hidden % 256 == 0 and ffn % 128 == 0; the decoded
 *                   weights must lie in the fp16 range (as the activations).
 *   COLI_FMT_FP8    fp8-e4m3-b128 (the registry's "8 fp8-e4m3-b128"): blocks
 *                   of 128 columns share one f32 scale s; each element is one
 *                   OCP FP8 E4M3 byte (sign bit 7, 4 exponent bits with bias
 *                   7, 3 mantissa bits; exponent 0 subnormal; 0x7F / 0xFF
 *                   NaN, never written by coli_quant_fp8b128):
 *                     packed uint8 [O][I], scales f32 [O][ceil(I/128)]
 *                   and W[o][i] = s[o][i/128] * e4m3(code).  Record order and
 *                   shape rules as for MXFP4 (the grouped GEMM at every token
 *                   count).  The kernels decode e4m3(code) * 2^-8 and multiply
 *                   by s * 256 rounded to fp16, so blocks need s * 256 inside
 *                   the fp16 normal range (max|w| between about 1.1e-4 and
 *                   1.1e5) for full precision; a NaN code decodes as +-480 s.
 */
typedef enum {
    COLI_FMT_I4ROW = 2, COLI_FMT_I4G = 4, COLI_FMT_MXFP4 = 7, COLI_FMT_FP8 = 8
} coli_weight_fmt;

const char *coli_status_str(int status);

/* Message of the last CUDA error that a call made on this host thread
 * returned as COLI_ECUDA ("no error" before any).  Static storage; never NULL. */
const char *coli_last_error(void);

/* Size helpers of the packed format (bytes / element counts). */
int64_t coli_packed_row_bytes(int64_t cols);            /* ceil(cols/2) */
int64_t coli_scales_per_row(int64_t cols);              /* ceil(cols/64) */
int64_t coli_expert_packed_bytes(int64_t H, int64_t F); /* 2 F ceil(H/2) + H ceil(F/2) */
int64_t coli_expert_scale_count(int64_t H, int64_t F);  /* 2 F ceil(H/64) + H ceil(F/64) */
/* The same for a chosen container: bytes of a packed row, of a row's scales,
 * of an expert record and of its scales (0 for an unknown format). */
int64_t coli_fmt_row_bytes(int32_t fmt, int64_t cols);
int64_t coli_fmt_scale_bytes(int32_t fmt, int64_t cols);
int64_t coli_fmt_expert_bytes(int32_t fmt, int64_t H, int64_t F);
int64_t coli_fmt_expert_scale_bytes(int32_t fmt, int64_t H, int64_t F);

/*
 * coli_quant_i4g -- quantise W[rows][cols] into the int4-grouped format
 * ([P2] §权重转换, quant_int4_grouped).  Per row and per group of 64 columns:
 *   s = max|w| / 7            (f32 division, round to nearest even)
 *   q = clip(rint(w / s), -8, 7)  (f32 division; rint rounds half to even)
 *   u = q + 8; byte j of a row = u[2j] | u[2j+1] << 4
 * A group whose max is 0 stores s = 0 and u = 8; a NaN weight stores u = 8;
 * with an odd column count the high nibble of the last byte is 0.
 *   w        [rows][cols] row-major, dtype w_dtype (COLI_BF16 or COLI_F32)
 *   packed   [rows][ceil(cols/2)]  written
 *   scales   [rows][ceil(cols/64)] written
 * rows >= 0, cols >= 1.  Any alignment is accepted; 16-byte aligned pointers
 * with cols % 64 == 0 take the vectorised path.  Result is bit-identical to
 * the definition above for every finite input.
 */
int coli_quant_i4g(const void *w, coli_dtype w_dtype, int64_t rows, int64_t cols,
                   uint8_t *packed, float *scales, cudaStream_t stream);

/*
 * coli_quant_mxfp4 -- quantise W[rows][cols] into MXFP4 (COLI_FMT_MXFP4, OCP
 * Microscaling v1.0).  Per row and block of 32 columns: shared exponent
 * se = floor(log2 max|w|) - 2, clamped to [-127, 127]; scale byte se + 127;
 * code of each w = the E2M1 value nearest to w / 2^se, ties to the even
 * mantissa, saturating at 6, with w's sign.  An all-zero block stores scale
 * byte 0 and codes 0; a NaN weight is ignored by the max and stored as +0.
 *   w       [rows][cols] row-major, dtype w_dtype (COLI_BF16 or COLI_F32)
 *   packed  [rows][ceil(cols/2)] written;  scales [rows][ceil(cols/32)] written
 * rows >= 0, cols >= 1, any alignment.  Bit-identical to the definition.
 */
int coli_quant_mxfp4(const void *w, coli_dtype w_dtype, int64_t rows, int64_t cols,
                     uint8_t *packed, uint8_t *scales, cudaStream_t stream);

/*
 * coli_quant_i4row -- quantise W[rows][cols] into int4-row (COLI_FMT_I4ROW):
 * per row s = max|w| / 7 (f32 division), q = clip(rint(w / s), -8, 7) (f32
 * division, ties to even), u = q + 8, byte j = u[2j] | u[2j+1] << 4.  An
 * all-zero row stores s = 0 and u = 8; a NaN weight is ignored by the max and
 * stored as u = 8; with an odd column count the last high nibble is 0.
 *   w       [rows][cols] row-major, dtype w_dtype (COLI_BF16 or COLI_F32)
 *   packed  [rows][ceil(cols/2)] written;  scales f32 [rows] written
 * rows >= 0, cols >= 1, any alignment.  Bit-identical to the definition.
 */
int coli_quant_i4row(const void *w, coli_dtype w_dtype, int64_t rows, int64_t cols,
                     uint8_t *packed, float *scales, cudaStream_t stream);

/*
 * coli_quant_fp8b128 -- quantise W[rows][cols] into fp8-e4m3-b128
 * (COLI_FMT_FP8).  Per row and block of 128 columns: s = max|w| / 448 (f32
 * division; 448 = the largest finite E4M3 value); code of each w = the E4M3
 * value nearest to w / s (f32 division), ties to the even code, saturating at
 * +-448 (finite), with w's sign.  An all-zero block stores s = 0 and codes 0;
 * a NaN weight is ignored by the max and stored as +0.
 *   w       [rows][cols] row-major, dtype w_dtype (COLI_BF16 or COLI_F32)
 *   packed  [rows][cols] written;  scales f32 [rows][ceil(cols/128)] written
 * rows >= 0, cols >= 1, any alignment.  Bit-identical to the definition.
 */
int coli_quant_fp8b128(const void *w, coli_dtype w_dtype, int64_t rows, int64_t cols,
                       uint8_t *packed, float *scales, cudaStream_t stream);

/*
 * Workspace: every routed call needs caller-owned device scratch of at least
 * the returned size, 256-byte aligned.  It must be zero-filled once before its
 * first use (cudaMemset); each call leaves it ready for the next.  Calls that
 * share one workspace must be ordered (same stream or events).
 */
size_t coli_router_workspace_size(const coli_moe_desc *d, int top_k);
size_t coli_moe_workspace_size(const coli_moe_desc *d, int top_k);

/*
 * coli_router_topk -- router GEMV, top-k selection and route counts
 * ([P1] §十一 "route"; [P4] §追踪流: gates are the normalised values the
 * layer applies; §从新引擎接入: one count per routing decision).
 *   logits[t][e] = sum_h router_w[e][h] x[t][h]      (f32 accumulation)
 *   idx[t][0..k-1]  the k largest logits, descending; equal logits -> lower e;
 *                   NaN ranks below every number
 *   gates[t][j]     softmax over all E renormalised over the k picked
 *                   = exp(l_j - l_0) / sum_{j'<k} exp(l_j' - l_0);
 *                   a picked NaN logit gets gate 0; if every logit of a
 *                   token is NaN, idx = 0..k-1 and gates = 1/k
 *                   ([P4] §测试与 CI, the rt_router_pick fallback), and
 *                   COLI_FLAG_NAN_LOGITS is set in the workspace
 *                   (with d->router_fn = COLI_ROUTER_SIGMOID_BIAS: ranked by
 *                   sigmoid(l) + router_bias, gates the picked sigmoid(l)
 *                   normalised, as described at coli_router_fn)
 *   route_counts[e] += number of (t, j) with idx[t][j] == e  (may be NULL;
 *                   never zeroed by the library: counts accumulate)
 *   x [T][H] (d->x_dtype), router_w [E][H] (d->router_dtype),
 *   idx int32 [T][k], gates f32 [T][k].   1 <= top_k <= min(E, 64).
 */
int coli_router_topk(const coli_moe_desc *d, int top_k, const void *x,
                     const void *router_w, int32_t *idx, float *gates,
                     uint32_t *route_counts, void *workspace, size_t ws_bytes,
                     cudaStream_t stream);

/*
 * coli_moe_forward -- one routed-MoE layer ([P1] §十一: route, union of the
 * batch's experts, expert FFNs, combine).
 *   out[t] = sum_j gates[t][j] * E_{idx[t][j]}(x[t]) + sum_s E_{E+s}(x[t])
 *   E_e(x) = Wd_e (silu(Wg_e x) * (Wu_e x)),  silu(z) = z / (1 + e^-z)
 * with routing as in coli_router_topk (route_counts updated the same way; the
 * shared experts are not counted).  Each expert used by the batch is read
 * once (batch union).  The per-token sum runs in a fixed order, so results
 * are deterministic.
 *   x [T][H] (d->x_dtype), router_w [E][H], packed_experts / scales in the
 *   expert record layout above (f32 scales, or the E8M0 bytes of an MXFP4
 *   layer: d->weight_fmt), out f32 [T][H].
 */
int coli_moe_forward(const coli_moe_desc *d, int top_k, const void *x,
                     const void *router_w, const uint8_t *packed_experts,
                     const void *scales, float *out, uint32_t *route_counts,
                     void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * coli_moe_forward_noalloc -- coli_moe_forward without a workspace argument,
 * for callers that cannot allocate device memory: hosts that hand the whole
 * device-memory budget out up front, or latency-critical loops that must
 * never reach cudaMalloc (it can synchronise the device).  The pages have no
 * counterpart of this entry point; it only changes where the scratch lives.
 *   Scratch: a 4 MiB array in the library's device image, which every GPU
 *   that loads the library holds until the process exits.  Calls whose
 *   coli_moe_workspace_size(d, top_k) exceeds 4 MiB return COLI_ENOMEM and
 *   launch nothing.  The array's device address is looked up on the first
 *   call on each device (with that device current), so make that first call
 *   before any stream capture.
 *   The cached address belongs to the device's current context: after
 *   cudaDeviceReset (or anything else that destroys and re-creates the
 *   primary context) this entry point must not be called again in the
 *   process.
 *   All calls share the one array: calls that overlap on the GPU (different
 *   streams, or several host threads) race and give wrong results; order them.
 *   Each call first clears the array's control words and fixed-point router
 *   buffers (a call that failed part-way may have left them non-zero), so the
 *   NaN-logit flag of coli_moe_check is not available through this entry point.
 *   Batched calls (n_tokens >= 64 with hidden % 256 == 0) run here too when
 *   their workspace fits in the 4 MiB.
 *   Allocates nothing (no cudaMalloc, no allocating library routine); the
 *   caller still provides x, the weights, out and route_counts.
 */
int coli_moe_forward_noalloc(const coli_moe_desc *d, int top_k, const void *x,
                             const void *router_w, const uint8_t *packed_experts,
                             const void *scales, float *out, uint32_t *route_counts,
                             cudaStream_t stream);

/*
 * Tiered expert store ([P1] §四 "三层存储层级": each expert is read from the
 * tier that holds it -- VRAM, RAM, NVMe -- and placement changes speed, never
 * the result; §十一 place / overlap / learn; §三 LFRU admission).  On GB300
 * the two tiers are an HBM pool of expert slots and the full store in pinned
 * host memory, which the GPU reads directly over NVLink-C2C: a layer streams
 * its resident experts from HBM and its missing ones from host memory in the
 * same kernels, and a policy step then uploads experts that have earned a
 * slot.  Every array is device memory unless said otherwise.
 *   slot_of      int32 [E + S]   slot of each expert, or -1 (not resident)
 *   slot_owner   int32 [n_slots] expert in each slot, or -1 (free)
 *   pool_packed  uint8 [n_slots][coli_expert_packed_bytes(H, F)] resident records
 *   pool_scales  f32   [n_slots][coli_expert_scale_count(H, F)]
 *   heat         uint32 [E]  route counts with exponential decay (LFRU frequency)
 *   last         uint32 [E]  tick of each expert's last route (LFRU recency)
 *   clock        uint32 [1]  policy ticks so far
 *   uploads      uint32 [1 + 2 * max_uploads]  written by coli_tier_update:
 *                the number of uploads of its tick, then (expert, slot) pairs
 * Zero heat, last and clock before the first use; slot_of and slot_owner must
 * describe the same placement (coli_tier_place fills the slots they name).
 * Shared experts (E .. E+S-1) may be placed in slots; the policy never evicts
 * them and never admits them.  Int4-grouped layers only (COLI_EUNSUPPORTED
 * for another d->weight_fmt).
 */
typedef struct {
    int32_t n_slots;
    int32_t max_uploads;
    int32_t *slot_of;
    int32_t *slot_owner;
    uint8_t *pool_packed;
    float *pool_scales;
    uint32_t *heat;
    uint32_t *last;
    uint32_t *clock;
    uint32_t *uploads;
} coli_tier;

/*
 * coli_moe_forward_tiered -- coli_moe_forward with each expert read from its
 * slot of the HBM pool when resident, else from host_packed / host_scales:
 * the full store (every expert, the expert record layout above) in pinned,
 * device-accessible host memory (cudaHostAlloc / cudaHostRegister; host
 * pointers).  Results are bit-identical to coli_moe_forward on the same
 * experts.  COLI_EINVAL if the store is not pinned host memory.
 */
int coli_moe_forward_tiered(const coli_moe_desc *d, int top_k, const void *x,
                            const void *router_w, const uint8_t *host_packed,
                            const float *host_scales, const coli_tier *tier, float *out,
                            uint32_t *route_counts, void *workspace, size_t ws_bytes,
                            cudaStream_t stream);

/*
 * coli_tier_place -- copy every expert named in slot_owner from the host
 * store into its slot (initial placement).  Asynchronous on `stream`.
 */
int coli_tier_place(const coli_moe_desc *d, const uint8_t *host_packed, const float *host_scales,
                    const coli_tier *tier, cudaStream_t stream);

/*
 * coli_tier_update -- one LFRU policy tick after a layer call, then the
 * uploads it decides, copied from the host store into the pool ([P1] §三).
 * call_counts [E] (device uint32): route counts of that call alone.
 *   clock += 1
 *   heat[e] = heat[e] - (heat[e] >> 3) + call_counts[e]   (saturating)
 *   last[e] = clock for every e with call_counts[e] > 0
 *   score(e) = heat[e] * 256 + recent(e), recent = 255 - (clock - last[e]) if
 *              that is positive, else 0: frequency first, recency only breaks
 *              close calls (a route is worth more than any recency)
 *   candidates: routed experts used in the call and not resident, by
 *   decreasing score (equal scores: lower id first).  For each, the target
 *   slot is the lowest free slot (cold heat 0) or else the resident routed
 *   expert of lowest score (equal: lowest slot), and the candidate moves in
 *   if heat[c] > cold + cold / 4 + 4 (in 64 bits: a saturated counter never
 *   wraps the threshold).  At most max_uploads moves per tick; their (expert,
 *   slot) pairs go to uploads.  Experts admitted this tick are not evicted in
 *   the same tick.
 * Asynchronous on `stream`; the policy runs on the GPU (no host sync).
 */
int coli_tier_update(const coli_moe_desc *d, const uint32_t *call_counts,
                     const uint8_t *host_packed, const float *host_scales, const coli_tier *tier,
                     cudaStream_t stream);

/*
 * coli_moe_stack_forward -- n_layers MoE layers chained through a residual
 * stream (decode stack without attention or norms):
 *   x_0 = x;  x_{l+1} = x_l + MoE_l(x_l);  x_out = x_{n_layers}
 * Layer l uses router_w + l*E*H elements, packed_experts + l*(E+S)*
 * coli_expert_packed_bytes(H,F), scales + l*(E+S)*coli_expert_scale_count(H,F),
 * route_counts + l*E, and (sigmoid router) router_bias + l*E.  x is d->x_dtype; x_out f32 [T][H]; layer_out (may be
 * NULL) receives MoE_l(x_l) as f32 [n_layers][T][H].  Same workspace size as
 * coli_moe_forward.
 */
int coli_moe_stack_forward(const coli_moe_desc *d, int top_k, int n_layers,
                           const void *x, const void *router_w,
                           const uint8_t *packed_experts, const void *scales,
                           float *x_out, float *layer_out, uint32_t *route_counts,
                           void *workspace, size_t ws_bytes, cudaStream_t stream);

/* Kernels of the layer forward that coli_profile_events can bracket. */
#define COLI_KERNEL_ROUTE  0   /* router partials of a pass's first layer */
#define COLI_KERNEL_GATEUP 1   /* gate/up expert GEMVs + SwiGLU */
#define COLI_KERNEL_DOWN   2   /* down expert GEMVs + combine (+ next routing) */
#define COLI_KERNEL_PREFILL_GATEUP 3  /* batched path: gate/up grouped GEMM + SwiGLU */
#define COLI_KERNEL_PREFILL_DOWN   4  /* batched path: down grouped GEMM */
#define COLI_KERNEL_LAYER  5   /* one-token layer kernel (routing, gate/up, down,
                                  combine in one launch; taken at one token when
                                  hidden and ffn are multiples of 1024) */

/*
 * coli_profile_events -- diagnostic, not on the compute path: record the
 * caller's CUDA events before[i] / after[i] on the launch stream around the
 * next n launches of one kernel of the layer forward (COLI_KERNEL_*), so a
 * caller can time that kernel inside a larger region.  Works while the stream
 * is captured into a CUDA graph (the records become event-record nodes).  The
 * records order the bracketed kernel after all earlier work of its stream, so
 * they remove the overlap of its launch with the kernel before it.
 * before/after are host arrays of n cudaEvent_t (the library copies them);
 * n = 0 turns recording off.  Process-wide state: not for concurrent callers.
 * Returns the number of launches bracketed under the previous setting (>= 0),
 * or COLI_EINVAL.
 */
int coli_profile_events(int kernel, const cudaEvent_t *before, const cudaEvent_t *after,
                        int n);

/*
 * coli_moe_check -- read (and optionally clear) the device-side flag word of a
 * workspace.  Synchronises `stream`.  *flags receives COLI_FLAG_* bits.
 * Returns COLI_ETIMEOUT if COLI_FLAG_TIMEOUT is set, else COLI_EBOUNDS if
 * COLI_FLAG_BOUNDS is set, else COLI_ERANGE if COLI_FLAG_RANGE is set, else
 * COLI_OK (COLI_FLAG_NAN_LOGITS alone is a handled condition: the rule above
 * defines that token's routing).
 */
int coli_moe_check(void *workspace, int clear, uint32_t *flags, cudaStream_t stream);

/*
 * Route-count history file (".coli_usage", [P4] §历史文件): the per-(layer,
 * expert) route counts of coli_moe_forward / coli_moe_stack_forward kept
 * across runs.  Host-side; every pointer here is a host pointer.
 *
 * Format: text, one record of exactly three decimal fields per line,
 *   -1 n_layers n_experts          geometry
 *   -2 1 engine_id                 format version, then the writer's identity
 *   layer expert count             one per nonzero count, layer-major order
 * engine_id is the 32-bit FNV-1a hash of the engine's name (the third field,
 * so a reader that takes the second field as a signed int never sees it).
 * Records whose first field is negative are headers: a reader that only
 * knows "layer expert count" skips them.  A history with no nonzero count is
 * written as an empty (0-byte) file, without headers.
 */

/* 32-bit FNV-1a hash of a NUL-terminated name (the engine_id field). */
uint32_t coli_usage_engine_id(const char *engine);

/*
 * coli_usage_save -- write counts [n_layers][n_experts] (uint32, host) to
 * `path`: through "<path>.tmp" and rename(), so a reader never sees a partial
 * file.  decay in (0, 1) first scales every count c > 0 to
 * max(1, round(c * decay)) (older routes weigh less; an expert routed once
 * stays); any other decay (1.0 included) leaves the counts as they are.
 * Errors: COLI_EINVAL (null arguments, non-positive sizes, or a path so long
 * that the temporary name would be truncated: refused before any file is
 * touched), COLI_EIO.
 */
int coli_usage_save(const char *path, const uint32_t *counts, int32_t n_layers, int32_t n_experts,
                    const char *engine, float decay);

/*
 * coli_usage_load -- add the records of `path` into counts [n_layers][n_experts]
 * (uint32, host; not cleared) and set *n_records (may be NULL) to the number of
 * records added.  An empty file adds nothing.  Records outside the geometry are
 * discarded and not counted; header kinds other than -1 and -2 are skipped;
 * files without headers (the older layout) are taken as they are.
 * Refused with COLI_EREFUSED, adding nothing:
 *   - a -1 record whose geometry differs, a -2 record of a later format
 *     version, or a dense binary history (first four bytes "IKU1") -- always;
 *   - a -2 record written by another engine -- unless `trusted` is nonzero
 *     (the caller named this file on purpose).
 * Errors: COLI_EINVAL, COLI_EIO (the file cannot be opened).
 */
int coli_usage_load(const char *path, uint32_t *counts, int32_t n_layers, int32_t n_experts,
                    const char *engine, int trusted, int64_t *n_records);

#ifdef __cplusplus
}
#endif
#endif /* COLI_H */
