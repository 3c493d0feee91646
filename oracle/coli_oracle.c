/*
 * coli_oracle.c -- plain, slow, obviously-correct CPU oracle of the routed-MoE
 * layer forward over int4-grouped expert weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library (the CUDA path) includes,
 * links or calls this file; only the tests, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code with the CUDA path.
 *
 * Sources (pages about the "colibri" pure-C MoE engine):
 *   [P1] "Colibrì 深度解析:用 12 万行纯 C 把 744B MoE 塞进 25GB 笔记本"
 *   [P2] "从源码开始colibri纯C引擎的编译、权重转换与.bin直映射实战"
 *   [P4] "colibrì 路由遥测全解析.coli_usage专家历史、ROUTE_TRACE追踪流与route_trace.h统一格式"
 *
 * Precision: the quantiser works in f32 because the format fixes those bits
 * (the converter divides float32 weights by a float32 scale and rounds with
 * np.rint, which the engine mirrors with lrintf: [P2] §权重转换).  Everything
 * else accumulates in double.  Expert ranking is decided on logits rounded to
 * f32, the precision the GPU router decides in; gates are computed in double.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - scale rule s = max|w| / 7 per group (f32 division), elided on [P2];
 *   - an all-zero group stores s = 0 and q = 0 (nibble 8);
 *   - a NaN weight is ignored by the max and stored as q = 0;
 *   - odd column count: the high nibble of the last byte is 0;
 *   - routing = softmax over E, top-k (ties to the lower id), renormalise;
 *   - the GLM router ("per-layer n_group=1 sigmoid + noaux_tc", [P1] §十一):
 *     scores s = 1 / (1 + e^-l); experts ranked by s + b with b a per-expert
 *     bias used only for the choice (one group: plain top-k over all
 *     experts); gates = the picked s over their sum, no further scale;
 *   - NaN logits rank below every number; if all are NaN the slots take
 *     experts 0..k-1 with gates 1/k ([P4] §测试与 CI, rt_router_pick);
 *   - activation SwiGLU, silu(z) = z / (1 + e^-z); the shared expert is added
 *     with weight 1 and is not counted.
 *
 * Build: cc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math); a
 * second build adds -fopenmp, which only spreads independent rows / tokens
 * over threads (every sum keeps its order, so both builds give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_GROUP 64

/* ---------------------------------------------------------------------- */
/* Format geometry: uint8[rows][ceil(cols/2)] nibbles, f32[rows][ceil(cols/64)]. */

int64_t orc_packed_row_bytes(int64_t cols) { return (cols + 1) / 2; }
int64_t orc_scales_per_row(int64_t cols) { return (cols + ORC_GROUP - 1) / ORC_GROUP; }

/* ---------------------------------------------------------------------- */
/* quant_int4_grouped ([P2] §权重转换): per row, per group of 64 columns along
 * the row, s = max|w| / 7; q = clip(rint(w / s), -8, 7); stored unsigned as
 * q + 8; even column -> low nibble, odd column -> high nibble. */
void orc_quant_i4g(const float *w, int64_t rows, int64_t cols,
                   uint8_t *packed, float *scales)
{
    const int64_t rb = orc_packed_row_bytes(cols);
    const int64_t ng = orc_scales_per_row(cols);
    /* rows are independent; the OpenMP build of this file (the benchmark's
     * multi-core leg, large test cases) splits them over threads */
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float *wr = w + r * cols;
        uint8_t *pr = packed + r * rb;
        memset(pr, 0, (size_t)rb);
        for (int64_t g = 0; g < ng; ++g) {
            const int64_t c0 = g * ORC_GROUP;
            const int64_t c1 = (c0 + ORC_GROUP < cols) ? c0 + ORC_GROUP : cols;
            float m = 0.0f;
            for (int64_t c = c0; c < c1; ++c) {
                float a = fabsf(wr[c]);
                if (a > m) m = a;              /* NaN never compares greater */
            }
            const float s = m / 7.0f;          /* IEEE f32 division */
            scales[r * ng + g] = s;
            for (int64_t c = c0; c < c1; ++c) {
                int q;
                if (s == 0.0f) {
                    q = 0;
                } else {
                    float v = rintf(wr[c] / s); /* f32 divide, round half to even */
                    if (v != v) q = 0;           /* NaN weight */
                    else if (v < -8.0f) q = -8;
                    else if (v > 7.0f) q = 7;
                    else q = (int)v;
                }
                const uint8_t u = (uint8_t)(q + 8);
                if ((c & 1) == 0) pr[c >> 1] |= u;
                else pr[c >> 1] |= (uint8_t)(u << 4);
            }
        }
    }
}

/* The engine consumes the packed rows directly (matmul_i4_grouped, [P2]):
 * element (r, c) is s[r][c/64] * (u - 8). */
static double orc_elem(const uint8_t *packed, const float *scales,
                       int64_t rb, int64_t ng, int64_t r, int64_t c)
{
    const uint8_t b = packed[r * rb + (c >> 1)];
    const int u = (c & 1) ? (b >> 4) : (b & 0x0F);
    return (double)scales[r * ng + c / ORC_GROUP] * (double)(u - 8);
}

void orc_dequant_i4g(const uint8_t *packed, const float *scales,
                     int64_t rows, int64_t cols, double *w)
{
    const int64_t rb = orc_packed_row_bytes(cols);
    const int64_t ng = orc_scales_per_row(cols);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            w[r * cols + c] = orc_elem(packed, scales, rb, ng, r, c);
}

/* y[r] = sum_c W[r][c] x[c] with W the dequantised matrix. */
void orc_matvec_i4g(const uint8_t *packed, const float *scales,
                    int64_t rows, int64_t cols, const double *x, double *y)
{
    const int64_t rb = orc_packed_row_bytes(cols);
    const int64_t ng = orc_scales_per_row(cols);
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < cols; ++c)
            acc += orc_elem(packed, scales, rb, ng, r, c) * x[c];
        y[r] = acc;
    }
}

/* ---------------------------------------------------------------------- */
/* Router GEMV: logits[t][e] = sum_h Wr[e][h] x[t][h]. */
void orc_router_logits(const double *x, const double *wr, int64_t T, int64_t H,
                       int64_t E, double *logits)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h) acc += wr[e * H + h] * x[t * H + h];
            logits[t * E + e] = acc;
        }
}

/* Ranking key: the f32 logit; NaN below every number; equal keys -> lower id. */
static int orc_ranks_before(float a, int64_t ia, float b, int64_t ib)
{
    const int na = (a != a), nb = (b != b);
    if (na != nb) return nb;        /* the number ranks before the NaN */
    if (!na && a != b) return a > b;
    return ia < ib;
}

/* Top-k with renormalised softmax gates for one token.
 * Softmax over all E followed by renormalisation over the k picked equals
 * exp(l_j - l_0) / sum_{j'<k} exp(l_j' - l_0), l_0 the top logit.
 * Returns 1 if any logit of the token is NaN, else 0. */
int orc_topk(const double *logits, int64_t E, int k, int32_t *idx, double *gates)
{
    int64_t *ord = (int64_t *)malloc((size_t)E * sizeof(int64_t));
    float *key = (float *)malloc((size_t)E * sizeof(float));
    int any_nan = 0;
    for (int64_t e = 0; e < E; ++e) {
        ord[e] = e;
        key[e] = (float)logits[e];
        if (logits[e] != logits[e]) any_nan = 1;
    }
    /* insertion sort: slow, stable, plain */
    for (int64_t i = 1; i < E; ++i) {
        int64_t v = ord[i], j = i - 1;
        while (j >= 0 && orc_ranks_before(key[v], v, key[ord[j]], ord[j])) {
            ord[j + 1] = ord[j];
            --j;
        }
        ord[j + 1] = v;
    }
    for (int j = 0; j < k; ++j) idx[j] = (int32_t)ord[j];
    const double l0 = logits[ord[0]];
    if (l0 != l0) {                  /* every logit NaN */
        for (int j = 0; j < k; ++j) gates[j] = 1.0 / (double)k;
    } else {
        double den = 0.0;
        for (int j = 0; j < k; ++j) {
            const double lj = logits[ord[j]];
            gates[j] = (lj != lj) ? 0.0 : exp(lj - l0);
            den += gates[j];
        }
        for (int j = 0; j < k; ++j) gates[j] /= den;
    }
    free(ord);
    free(key);
    return any_nan;
}

/* Top-k of the GLM router for one token ([P1] §十一: "per-layer n_group=1
 * sigmoid + noaux_tc"): s_e = 1 / (1 + exp(-l_e)); the k experts with the
 * largest s_e + bias_e (bias may be NULL = 0) in the orc_topk order, the keys
 * ranked in f32 like the logits above; gates[j] = s_{idx[j]} / sum_j' s_{idx[j']}.
 * NaN rules as orc_topk: a NaN key ranks last, a picked NaN score gets gate 0,
 * an all-NaN token takes experts 0..k-1 with gates 1/k.  Returns 1 if any
 * logit of the token is NaN. */
int orc_topk_sigmoid(const double *logits, const double *bias, int64_t E, int k,
                     int32_t *idx, double *gates)
{
    int64_t *ord = (int64_t *)malloc((size_t)E * sizeof(int64_t));
    float *key = (float *)malloc((size_t)E * sizeof(float));
    double *sc = (double *)malloc((size_t)E * sizeof(double));
    int any_nan = 0;
    for (int64_t e = 0; e < E; ++e) {
        ord[e] = e;
        sc[e] = 1.0 / (1.0 + exp(-logits[e]));
        key[e] = (float)(sc[e] + (bias ? bias[e] : 0.0));
        if (logits[e] != logits[e]) any_nan = 1;
    }
    for (int64_t i = 1; i < E; ++i) {
        int64_t v = ord[i], j = i - 1;
        while (j >= 0 && orc_ranks_before(key[v], v, key[ord[j]], ord[j])) {
            ord[j + 1] = ord[j];
            --j;
        }
        ord[j + 1] = v;
    }
    for (int j = 0; j < k; ++j) idx[j] = (int32_t)ord[j];
    if (sc[ord[0]] != sc[ord[0]]) {    /* every logit NaN */
        for (int j = 0; j < k; ++j) gates[j] = 1.0 / (double)k;
    } else {
        double den = 0.0;
        for (int j = 0; j < k; ++j) {
            const double s = sc[ord[j]];
            gates[j] = (s != s) ? 0.0 : s;
            den += gates[j];
        }
        for (int j = 0; j < k; ++j) gates[j] /= den;
    }
    free(ord);
    free(key);
    free(sc);
    return any_nan;
}

/* ---------------------------------------------------------------------- */
/* Expert record: gate[F][H] | up[F][H] | down[H][F], each matrix in the
 * packed format, stored adjacently ([P1] §四: the three matrices of an expert
 * are stored next to each other and read in one go). */

int64_t orc_expert_packed_bytes(int64_t H, int64_t F)
{
    return 2 * F * orc_packed_row_bytes(H) + H * orc_packed_row_bytes(F);
}

int64_t orc_expert_scales(int64_t H, int64_t F)
{
    return 2 * F * orc_scales_per_row(H) + H * orc_scales_per_row(F);
}

static double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* y = Wd (silu(Wg x) * (Wu x)) */
void orc_expert(const uint8_t *pe, const float *se, int64_t H, int64_t F,
                const double *x, double *y)
{
    const uint8_t *pg = pe;
    const uint8_t *pu = pg + F * orc_packed_row_bytes(H);
    const uint8_t *pd = pu + F * orc_packed_row_bytes(H);
    const float *sg = se;
    const float *su = sg + F * orc_scales_per_row(H);
    const float *sd = su + F * orc_scales_per_row(H);
    double *g = (double *)malloc((size_t)F * sizeof(double));
    double *u = (double *)malloc((size_t)F * sizeof(double));
    orc_matvec_i4g(pg, sg, F, H, x, g);
    orc_matvec_i4g(pu, su, F, H, x, u);
    for (int64_t f = 0; f < F; ++f) g[f] = orc_silu(g[f]) * u[f];
    orc_matvec_i4g(pd, sd, H, F, g, y);
    free(g);
    free(u);
}

/* One routed-MoE layer for T tokens ([P1] §十一 route -> union -> compute;
 * [P4] route counts, one per routing decision).
 *   x       [T][H]              layer input
 *   wr      [E][H]              router weights
 *   packed  experts 0..E+S-1    S = n_shared shared experts after the routed
 *   out     [T][H]              sum_j gates[t][j] E_idx(x) + sum_s E_shared(x)
 *   idx     [T][k], gates [T][k]
 *   counts  [E]                 += 1 per (token, slot); may be NULL
 * Returns the number of tokens that saw a NaN logit. */
int orc_moe_forward_router(const double *x, int64_t T, int64_t H, int64_t F, int64_t E,
                           int64_t n_shared, const double *wr, int router_fn,
                           const double *bias, const uint8_t *packed, const float *scales,
                           int k, double *out, int32_t *idx, double *gates, uint32_t *counts);

int orc_moe_forward(const double *x, int64_t T, int64_t H, int64_t F, int64_t E,
                    int64_t n_shared, const double *wr, const uint8_t *packed,
                    const float *scales, int k, double *out, int32_t *idx,
                    double *gates, uint32_t *counts)
{
    return orc_moe_forward_router(x, T, H, F, E, n_shared, wr, 0, NULL, packed, scales, k,
                                  out, idx, gates, counts);
}

/* The same layer with the routing function chosen: router_fn 0 = softmax
 * (orc_topk), 1 = sigmoid scores with a selection bias (orc_topk_sigmoid,
 * bias [E] or NULL). */
int orc_moe_forward_router(const double *x, int64_t T, int64_t H, int64_t F, int64_t E,
                           int64_t n_shared, const double *wr, int router_fn,
                           const double *bias, const uint8_t *packed, const float *scales,
                           int k, double *out, int32_t *idx, double *gates, uint32_t *counts)
{
    const int64_t eb = orc_expert_packed_bytes(H, F);
    const int64_t es = orc_expert_scales(H, F);
    double *logits = (double *)malloc((size_t)(T * E) * sizeof(double));
    int nan_tokens = 0;
    orc_router_logits(x, wr, T, H, E, logits);
    for (int64_t t = 0; t < T; ++t) {
        nan_tokens += router_fn == 1
            ? orc_topk_sigmoid(logits + t * E, bias, E, k, idx + t * k, gates + t * k)
            : orc_topk(logits + t * E, E, k, idx + t * k, gates + t * k);
        if (counts)
            for (int j = 0; j < k; ++j) counts[idx[t * k + j]] += 1u;
    }
    /* tokens are independent once routed (the OpenMP build runs them on
     * several threads; each token's sum keeps the same order) */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double *y = (double *)malloc((size_t)H * sizeof(double));
        double *o = out + t * H;
        for (int64_t h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            const int64_t e = idx[t * k + j];
            orc_expert(packed + e * eb, scales + e * es, H, F, x + t * H, y);
            for (int64_t h = 0; h < H; ++h) o[h] += gates[t * k + j] * y[h];
        }
        for (int64_t s = 0; s < n_shared; ++s) {
            const int64_t e = E + s;
            orc_expert(packed + e * eb, scales + e * es, H, F, x + t * H, y);
            for (int64_t h = 0; h < H; ++h) o[h] += y[h];
        }
        free(y);
    }
    free(logits);
    return nan_tokens;
}

/* ---------------------------------------------------------------------- */
/* Other container formats of the engine's registry ([P2] §权重转换 lists
 * "7 MXFP4" and "8 fp8-e4m3-b128"; [P1] §十 "从 int4 到 MXFP4").  The pages
 * name them only; their definitions are the public ones:
 *
 * MXFP4 (OCP Microscaling Formats v1.0): blocks of 32 consecutive elements
 * of a row share one E8M0 scale X = 2^(e - 127) (a biased exponent byte);
 * each element is FP4 E2M1 (1 sign, 2 exponent, 1 mantissa bit, bias 1):
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Conversion of a block: shared
 * exponent = floor(log2(max|v|)) - 2 (2 = the largest E2M1 exponent), then
 * each v / X rounded to nearest E2M1, ties to the even mantissa, saturating
 * at 6.  Storage, as the int4 container: codes packed two per byte, even
 * column in the low nibble; scales one byte per 32 columns.
 * Readings (design notes): an all-zero block stores e = 0 and codes 0; a NaN
 * element is ignored by the max and stored as +0; the shared exponent is
 * clamped to [-127, 127]; the sign of a value that rounds to zero is kept. */

#define ORC_MX_BLOCK 32

int64_t orc_mx_row_bytes(int64_t cols) { return (cols + 1) / 2; }
int64_t orc_mx_scales_per_row(int64_t cols) { return (cols + ORC_MX_BLOCK - 1) / ORC_MX_BLOCK; }

/* E2M1 magnitude of a 3-bit code (exponent bits 2..1, mantissa bit 0). */
double orc_e2m1_magnitude(int m)
{
    const int ex = (m >> 1) & 3, man = m & 1;
    if (ex == 0) return man ? 0.5 : 0.0;                 /* subnormal: m * 2^(1-1) / 2 */
    return (1.0 + 0.5 * man) * ldexp(1.0, ex - 1);       /* (1 + m/2) 2^(e - bias) */
}

double orc_e2m1_value(int code)
{
    const double v = orc_e2m1_magnitude(code & 7);
    return (code & 8) ? -v : v;
}

/* Nearest E2M1 magnitude code of a >= 0 (f32), ties to the even mantissa,
 * saturating at 6: every magnitude is compared, plainly. */
static int orc_e2m1_round(float a)
{
    int best = 0;
    for (int m = 1; m < 8; ++m) {
        const double d_best = fabs((double)a - orc_e2m1_magnitude(best));
        const double d = fabs((double)a - orc_e2m1_magnitude(m));
        if (d < d_best || (d == d_best && (m & 1) == 0 && (best & 1) == 1)) best = m;
    }
    return best;
}

void orc_quant_mxfp4(const float *w, int64_t rows, int64_t cols, uint8_t *packed, uint8_t *scales)
{
    const int64_t rb = orc_mx_row_bytes(cols);
    const int64_t nb = orc_mx_scales_per_row(cols);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float *wr = w + r * cols;
        uint8_t *pr = packed + r * rb;
        memset(pr, 0, (size_t)rb);
        for (int64_t b = 0; b < nb; ++b) {
            const int64_t c0 = b * ORC_MX_BLOCK;
            const int64_t c1 = (c0 + ORC_MX_BLOCK < cols) ? c0 + ORC_MX_BLOCK : cols;
            float m = 0.0f;
            for (int64_t c = c0; c < c1; ++c) {
                const float a = fabsf(wr[c]);
                if (a > m) m = a;                       /* NaN never compares greater */
            }
            int se = -127;
            if (m > 0.0f) {
                int ex;
                frexpf(m, &ex);                         /* m = f 2^ex, f in [0.5, 1) */
                se = (ex - 1) - 2;                      /* floor(log2 m) - emax(E2M1) */
                if (se < -127) se = -127;
                if (se > 127) se = 127;
            }
            scales[r * nb + b] = (uint8_t)(se + 127);
            for (int64_t c = c0; c < c1; ++c) {
                int code = 0;
                if (m > 0.0f && wr[c] == wr[c]) {
                    const float q = ldexpf(wr[c], -se);  /* v / X, exact */
                    code = orc_e2m1_round(fabsf(q)) | (signbit(q) ? 8 : 0);
                }
                if ((c & 1) == 0) pr[c >> 1] |= (uint8_t)code;
                else pr[c >> 1] |= (uint8_t)(code << 4);
            }
        }
    }
}

/* Dequantised element: X * value(code). */
static double orc_mx_elem(const uint8_t *packed, const uint8_t *scales, int64_t rb, int64_t nb,
                          int64_t r, int64_t c)
{
    const uint8_t byte = packed[r * rb + (c >> 1)];
    const int code = (c & 1) ? (byte >> 4) : (byte & 0x0F);
    const int e = scales[r * nb + c / ORC_MX_BLOCK];
    return ldexp(orc_e2m1_value(code), e - 127);
}

void orc_dequant_mxfp4(const uint8_t *packed, const uint8_t *scales, int64_t rows, int64_t cols,
                       double *w)
{
    const int64_t rb = orc_mx_row_bytes(cols), nb = orc_mx_scales_per_row(cols);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) w[r * cols + c] = orc_mx_elem(packed, scales, rb, nb, r, c);
}

/* ---------------------------------------------------------------------- */
/* The layer over a chosen container: fmt 4 = int4-grouped (the functions
 * above), 7 = MXFP4, 2 = int4-row and 8 = fp8-e4m3-b128 (below).  Expert record: gate | up | down, each in the format;
 * `scales` points to f32 scales (fmt 2, 4, 8) or E8M0 bytes (fmt 7), expert
 * after expert in the same order. */

int64_t orc_fp8_row_bytes(int64_t cols);
int64_t orc_fp8_scales_per_row(int64_t cols);
void orc_matvec_fp8b128(const uint8_t *packed, const float *scales, int64_t rows, int64_t cols,
                        const double *x, double *y);
void orc_matvec_i4row(const uint8_t *packed, const float *scales, int64_t rows, int64_t cols,
                      const double *x, double *y);

int64_t orc_fmt_row_bytes(int fmt, int64_t cols)
{
    if (fmt == 2) return orc_packed_row_bytes(cols);
    if (fmt == 8) return orc_fp8_row_bytes(cols);
    return fmt == 7 ? orc_mx_row_bytes(cols) : orc_packed_row_bytes(cols);
}
/* Bytes of one row's scales. */
int64_t orc_fmt_scale_bytes(int fmt, int64_t cols)
{
    if (fmt == 2) return 4;
    if (fmt == 8) return 4 * orc_fp8_scales_per_row(cols);
    return fmt == 7 ? orc_mx_scales_per_row(cols) : 4 * orc_scales_per_row(cols);
}
int64_t orc_fmt_expert_bytes(int fmt, int64_t H, int64_t F)
{
    return 2 * F * orc_fmt_row_bytes(fmt, H) + H * orc_fmt_row_bytes(fmt, F);
}
int64_t orc_fmt_expert_scale_bytes(int fmt, int64_t H, int64_t F)
{
    return 2 * F * orc_fmt_scale_bytes(fmt, H) + H * orc_fmt_scale_bytes(fmt, F);
}

static void orc_matvec_fmt(int fmt, const uint8_t *packed, const uint8_t *scales, int64_t rows,
                           int64_t cols, const double *x, double *y)
{
    if (fmt == 8) {
        orc_matvec_fp8b128(packed, (const float *)scales, rows, cols, x, y);
        return;
    }
    if (fmt == 2) {
        orc_matvec_i4row(packed, (const float *)scales, rows, cols, x, y);
        return;
    }
    if (fmt != 7) {
        orc_matvec_i4g(packed, (const float *)scales, rows, cols, x, y);
        return;
    }
    const int64_t rb = orc_mx_row_bytes(cols), nb = orc_mx_scales_per_row(cols);
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < cols; ++c) acc += orc_mx_elem(packed, scales, rb, nb, r, c) * x[c];
        y[r] = acc;
    }
}

/* y = Wd (silu(Wg x) * (Wu x)) over the chosen container. */
void orc_expert_fmt(int fmt, const uint8_t *pe, const uint8_t *se, int64_t H, int64_t F,
                    const double *x, double *y)
{
    const uint8_t *pg = pe, *pu = pg + F * orc_fmt_row_bytes(fmt, H);
    const uint8_t *pd = pu + F * orc_fmt_row_bytes(fmt, H);
    const uint8_t *sg = se, *su = sg + F * orc_fmt_scale_bytes(fmt, H);
    const uint8_t *sd = su + F * orc_fmt_scale_bytes(fmt, H);
    double *g = (double *)malloc((size_t)F * sizeof(double));
    double *u = (double *)malloc((size_t)F * sizeof(double));
    orc_matvec_fmt(fmt, pg, sg, F, H, x, g);
    orc_matvec_fmt(fmt, pu, su, F, H, x, u);
    for (int64_t f = 0; f < F; ++f) g[f] = orc_silu(g[f]) * u[f];
    orc_matvec_fmt(fmt, pd, sd, H, F, g, y);
    free(g);
    free(u);
}

/* orc_moe_forward_router over the chosen container (same routing, order and
 * accumulation; only the weights' decoding differs). */
int orc_moe_forward_fmt(int fmt, const double *x, int64_t T, int64_t H, int64_t F, int64_t E,
                        int64_t n_shared, const double *wr, int router_fn, const double *bias,
                        const uint8_t *packed, const uint8_t *scales, int k, double *out,
                        int32_t *idx, double *gates, uint32_t *counts)
{
    const int64_t eb = orc_fmt_expert_bytes(fmt, H, F);
    const int64_t es = orc_fmt_expert_scale_bytes(fmt, H, F);
    double *logits = (double *)malloc((size_t)(T * E) * sizeof(double));
    int nan_tokens = 0;
    orc_router_logits(x, wr, T, H, E, logits);
    for (int64_t t = 0; t < T; ++t) {
        nan_tokens += router_fn == 1
            ? orc_topk_sigmoid(logits + t * E, bias, E, k, idx + t * k, gates + t * k)
            : orc_topk(logits + t * E, E, k, idx + t * k, gates + t * k);
        if (counts)
            for (int j = 0; j < k; ++j) counts[idx[t * k + j]] += 1u;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double *y = (double *)malloc((size_t)H * sizeof(double));
        double *o = out + t * H;
        for (int64_t h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            const int64_t e = idx[t * k + j];
            orc_expert_fmt(fmt, packed + e * eb, scales + e * es, H, F, x + t * H, y);
            for (int64_t h = 0; h < H; ++h) o[h] += gates[t * k + j] * y[h];
        }
        for (int64_t s = 0; s < n_shared; ++s) {
            const int64_t e = E + s;
            orc_expert_fmt(fmt, packed + e * eb, scales + e * es, H, F, x + t * H, y);
            for (int64_t h = 0; h < H; ++h) o[h] += y[h];
        }
        free(y);
    }
    free(logits);
    return nan_tokens;
}

/* ---------------------------------------------------------------------- */
/* fp8-e4m3-b128 ([P2] §权重转换, "8 fp8-e4m3-b128" of the format registry).
 * The page gives the name only; the reading (design notes): rows quantised in
 * blocks of 128 consecutive columns, one f32 scale per block, s = max|w| / 448
 * (448 = the largest finite E4M3 value; f32 division), each element the
 * E4M3 code nearest to w / s (f32 division), ties to the even code, finite
 * saturation at +-448.  E4M3 (OCP 8-bit floating point): 1 sign, 4 exponent
 * (bias 7), 3 mantissa bits; exponent 0 is subnormal (m 2^-9); no infinity;
 * exponent 15 with mantissa 7 is NaN.  Storage: one code per byte, row after
 * row; scales f32 [rows][ceil(cols/128)].  An all-zero block stores s = 0 and
 * codes 0; a NaN weight is ignored by the max and stored as +0. */

#define ORC_FP8_BLOCK 128

int64_t orc_fp8_row_bytes(int64_t cols) { return cols; }
int64_t orc_fp8_scales_per_row(int64_t cols) { return (cols + ORC_FP8_BLOCK - 1) / ORC_FP8_BLOCK; }

/* Value of an E4M3 code, from the definition. */
double orc_e4m3_value(int code)
{
    const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);                 /* m / 8 * 2^(1 - 7) */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest finite E4M3 code of a (f32), ties to the even code, saturating:
 * every non-negative finite code compared, plainly. */
static int orc_e4m3_round(float a)
{
    const double x = fabs((double)a);
    int best = 0;
    for (int c = 1; c <= 0x7E; ++c) {
        const double d_best = fabs(x - orc_e4m3_value(best));
        const double d = fabs(x - orc_e4m3_value(c));
        if (d < d_best || (d == d_best && (c & 1) == 0 && (best & 1) == 1)) best = c;
    }
    return best | (signbit(a) ? 0x80 : 0);
}

void orc_quant_fp8b128(const float *w, int64_t rows, int64_t cols, uint8_t *packed, float *scales)
{
    const int64_t nb = orc_fp8_scales_per_row(cols);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float *wr = w + r * cols;
        for (int64_t b = 0; b < nb; ++b) {
            const int64_t c0 = b * ORC_FP8_BLOCK;
            const int64_t c1 = (c0 + ORC_FP8_BLOCK < cols) ? c0 + ORC_FP8_BLOCK : cols;
            float m = 0.0f;
            for (int64_t c = c0; c < c1; ++c) {
                const float a = fabsf(wr[c]);
                if (a > m) m = a;
            }
            const float s = m / 448.0f;                      /* IEEE f32 division */
            scales[r * nb + b] = s;
            for (int64_t c = c0; c < c1; ++c)
                packed[r * cols + c] =
                    (uint8_t)((s == 0.0f || wr[c] != wr[c]) ? 0 : orc_e4m3_round(wr[c] / s));
        }
    }
}

static double orc_fp8_elem(const uint8_t *packed, const float *scales, int64_t cols, int64_t nb,
                           int64_t r, int64_t c)
{
    return (double)scales[r * nb + c / ORC_FP8_BLOCK] * orc_e4m3_value(packed[r * cols + c]);
}

void orc_dequant_fp8b128(const uint8_t *packed, const float *scales, int64_t rows, int64_t cols,
                         double *w)
{
    const int64_t nb = orc_fp8_scales_per_row(cols);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) w[r * cols + c] = orc_fp8_elem(packed, scales, cols, nb, r, c);
}

void orc_matvec_fp8b128(const uint8_t *packed, const float *scales, int64_t rows, int64_t cols,
                        const double *x, double *y)
{
    const int64_t nb = orc_fp8_scales_per_row(cols);
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < cols; ++c) acc += orc_fp8_elem(packed, scales, cols, nb, r, c) * x[c];
        y[r] = acc;
    }
}

/* ---------------------------------------------------------------------- */
/* int4-row ([P2] §权重转换, "2 int4-row" of the format registry).  The page
 * gives the name only; the reading (design notes): the int4-grouped rule with
 * one group per row -- per row s = max|w| / 7 (f32 division), q =
 * clip(rint(w / s), -8, 7) (f32 division, ties to even), stored as u = q + 8,
 * two per byte, even column in the low nibble; scales f32 [rows].  An all-zero
 * row stores s = 0 and u = 8; a NaN weight is ignored by the max and stored as
 * u = 8; with an odd column count the last high nibble is 0. */

void orc_quant_i4row(const float *w, int64_t rows, int64_t cols, uint8_t *packed, float *scales)
{
    const int64_t rb = orc_packed_row_bytes(cols);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const float *wr = w + r * cols;
        uint8_t *pr = packed + r * rb;
        memset(pr, 0, (size_t)rb);
        float m = 0.0f;
        for (int64_t c = 0; c < cols; ++c) {
            const float a = fabsf(wr[c]);
            if (a > m) m = a;
        }
        const float s = m / 7.0f;
        scales[r] = s;
        for (int64_t c = 0; c < cols; ++c) {
            int q = 0;
            if (s != 0.0f) {
                const float v = rintf(wr[c] / s);
                q = (v != v) ? 0 : (v < -8.0f ? -8 : (v > 7.0f ? 7 : (int)v));
            }
            const uint8_t u = (uint8_t)(q + 8);
            pr[c >> 1] |= (c & 1) ? (uint8_t)(u << 4) : u;
        }
    }
}

static double orc_i4row_elem(const uint8_t *packed, const float *scales, int64_t rb, int64_t r,
                             int64_t c)
{
    const uint8_t b = packed[r * rb + (c >> 1)];
    const int u = (c & 1) ? (b >> 4) : (b & 0x0F);
    return (double)scales[r] * (double)(u - 8);
}

void orc_dequant_i4row(const uint8_t *packed, const float *scales, int64_t rows, int64_t cols,
                       double *w)
{
    const int64_t rb = orc_packed_row_bytes(cols);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) w[r * cols + c] = orc_i4row_elem(packed, scales, rb, r, c);
}

void orc_matvec_i4row(const uint8_t *packed, const float *scales, int64_t rows, int64_t cols,
                      const double *x, double *y)
{
    const int64_t rb = orc_packed_row_bytes(cols);
    for (int64_t r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int64_t c = 0; c < cols; ++c) acc += orc_i4row_elem(packed, scales, rb, r, c) * x[c];
        y[r] = acc;
    }
}
