/*
 * Plain CPU oracle for the weight-only FP4 mixture-of-experts layer (QMoE, W4A16).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the CUDA
 * path.  Every result is computed the slow, obvious way in double precision;
 * the only roundings are the ones the method itself defines (to bf16).
 *
 * Sources (page title, section):
 *  - "MoE and QMoE - CUDA Operator Documentation" (ONNX Runtime moe_qmoe doc):
 *      §1 pipeline (router top-k softmax -> permute -> GEMM1 -> activation ->
 *      GEMM2 -> un-permute -> weighted sum), §6.5 MXFP4 storage [E,K,N/2] and the
 *      dequantisation W = fp4(W) * ue8m0(scale) * global_scale, §8 SwiGLU,
 *      §9b NVFP4 (E4M3 block-16 scales, per-expert fp32 global scale),
 *      §9b.3 the E2M1 code layout (sign in bit 3, eight magnitudes in bits 2:0),
 *      §13 the reference computation "dequantize, then input @ W^T".
 *  - "[CUDA] Coalesce QMoE MXFP4/NVFP4 weight dequantization" (PR #31349):
 *      packed weights [E, K, N/2] (n-packed), output [E, N, K], block scale
 *      index [e][n][k / block], global scale per expert.
 *  - "[CUDA] Cut the MoE routing prologue/epilogue cost for small-batch decode"
 *      (PR #31156): top-k with a stable tie-break, renormalised top-k weights,
 *      stable ranking of (token, expert) assignments by expert.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - nibble order: the low nibble of a byte holds the even n (the INT4 layout in
 *    §6.1 of the operator doc, and "nibble j of the word is logical element j"
 *    in PR #31159);
 *  - E8M0 bias 127, code 255 = NaN; E4M3FN: no infinities, S.1111.111 = NaN;
 *  - dequantised value = one round-to-nearest-even to bf16 of the exact product
 *    e2m1 * block_scale * global_scale (exact in double: <= 30 significant bits);
 *  - a NULL global scale means 1.0;
 *  - top-k order: logit descending, then expert index ascending; selection is
 *    made on the fp32 logits (softmax is monotone); -0.0 == +0.0;
 *  - routing weights: softmax over all E experts, then (normalize != 0) divided
 *    by their sum over the k selected experts;
 *  - with router_weights (input 14 of the operator schema, §2.3: "DeepSeek-
 *    style routing", router_probs selects, router_weights gives the mixing
 *    weights gathered at the selected experts): weight j = router_weights[t][id_j]
 *    as given, then the same renormalisation over the k when normalize != 0;
 *  - expanded index i = t*k + j; rows of one expert keep ascending i;
 *  - FC1 columns: swiglu_fusion=1 interleaves them, 2m = gate and 2m+1 =
 *    linear; swiglu_fusion=2 concatenates them, m = gate and I+m = linear
 *    (the fc1 (gate) / fc3 (value) concatenation of the SwiGLU fusion
 *    section); swiglu_fusion=0 is read as 1, the pages' backward-compatibility
 *    remap for QMoE;
 *  - the FC1 activation a is rounded to bf16, y and the weighted sum stay wide,
 *    the layer output is rounded to bf16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

/* Formats, as the boundary numbers them: 0 = NVFP4 (E4M3 scale per 16 k),
 * 1 = MXFP4 (E8M0 scale per 32 k). */
#define ORACLE_NVFP4 0
#define ORACLE_MXFP4 1

/* ---- element codecs --------------------------------------------------- */

/* E2M1 (FP4): bit 3 = sign, bits 2:0 index the eight magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Operator doc §9b.3. */
double oracle_e2m1(unsigned code) {
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[code & 7u];
    return (code & 8u) ? -v : v;
}

/* Float8 E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is
 * subnormal; S.1111.111 is NaN; there is no infinity.  Operator doc §6.4/§9b. */
double oracle_e4m3fn(unsigned byte) {
    unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
    double v;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -v : v;
}

/* E8M0 (ue8m0): an unsigned power-of-two exponent with bias 127; 0xFF is NaN.
 * Operator doc §6.5. */
double oracle_e8m0(unsigned byte) {
    if ((byte & 0xFFu) == 0xFFu) return NAN;
    return ldexp(1.0, (int)(byte & 0xFFu) - 127);
}

/* bf16 bits -> double (exact). */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round a double to bf16 (8 significant bits, fp32 exponent range, subnormals
 * kept) with round-to-nearest, ties-to-even.  NaN -> 0x7FC0. */
uint16_t oracle_bf16_rne(double v) {
    uint16_t sign;
    double a, m, r;
    int e, q;
    float f;
    uint32_t bits;
    if (isnan(v)) return 0x7FC0u;
    sign = signbit(v) ? 0x8000u : 0u;
    a = fabs(v);
    if (a == 0.0) return sign;
    if (a >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    frexp(a, &e);            /* a in [2^(e-1), 2^e) */
    q = e - 8;               /* spacing of 8-significant-bit numbers there */
    if (q < -133) q = -133;  /* bf16 subnormal spacing */
    m = nearbyint(ldexp(a, -q)); /* default rounding mode: nearest, ties to even */
    r = ldexp(m, q);
    if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    f = (float)r;            /* exact: r has <= 8 significant bits */
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* ---- dequantisation ----------------------------------------------------- */

static int block_size(int fmt) { return fmt == ORACLE_NVFP4 ? 16 : 32; }

static double scale_decode(int fmt, unsigned byte) {
    return fmt == ORACLE_NVFP4 ? oracle_e4m3fn(byte) : oracle_e8m0(byte);
}

/* One dequantised weight Wd[e][n][k] as the exact bf16 value, from packed
 * [E, K, N/2] codes, block scales [E, N, K/bs] and the per-expert global
 * scale (NULL -> 1.0).  PR #31349 (index map), operator doc §6.5/§9b. */
double oracle_dequant_element(const uint8_t *packed, const uint8_t *scales,
                              const float *gscale, int N, int K, int fmt,
                              int e, int n, int k) {
    int bs = block_size(fmt);
    size_t pidx = ((size_t)e * (size_t)K + (size_t)k) * (size_t)(N / 2) + (size_t)(n / 2);
    unsigned nib = (packed[pidx] >> (4 * (n & 1))) & 15u;
    size_t sidx = ((size_t)e * (size_t)N + (size_t)n) * (size_t)(K / bs) + (size_t)(k / bs);
    double g = gscale ? (double)gscale[e] : 1.0;
    double w = oracle_e2m1(nib) * scale_decode(fmt, scales[sidx]) * g;
    return oracle_bf16_to_double(oracle_bf16_rne(w));
}

/* Full dequantisation [E, K, N/2] -> bf16 bits [E, N, K]. */
int oracle_dequant(const uint8_t *packed, const uint8_t *scales, const float *gscale,
                   int E, int N, int K, int fmt, uint16_t *out) {
    int e, n, k, bs;
    if (!packed || !scales || !out || E < 0 || N < 0 || K < 0) return ORACLE_BAD_ARG;
    if (fmt != ORACLE_NVFP4 && fmt != ORACLE_MXFP4) return ORACLE_BAD_ARG;
    bs = block_size(fmt);
    if ((N & 1) || (K % bs)) return ORACLE_BAD_ARG;
#pragma omp parallel for private(n, k) schedule(static)
    for (e = 0; e < E; ++e)
        for (n = 0; n < N; ++n)
            for (k = 0; k < K; ++k) {
                double w = oracle_dequant_element(packed, scales, gscale, N, K, fmt, e, n, k);
                out[((size_t)e * N + n) * (size_t)K + k] = oracle_bf16_rne(w);
            }
    return ORACLE_OK;
}

/* Block scales [E][N][nb] -> the k-major layout [E][nb][N] the forward path
 * also accepts: out[e][b][n] = in[e][n][b], every byte copied unchanged.  (A
 * storage order of this library, not of the pages; the pages index scales as
 * [e][n][k / block], PR #31349.) */
int oracle_scales_kmajor(const uint8_t *in, int E, int N, int nb, uint8_t *out) {
    if (!in || !out || E < 1 || N < 1 || nb < 1) return 1;
    for (int e = 0; e < E; ++e)
        for (int b = 0; b < nb; ++b)
            for (int n = 0; n < N; ++n)
                out[((size_t)e * nb + b) * N + n] = in[((size_t)e * N + n) * nb + b];
    return 0;
}

/* ---- routing ------------------------------------------------------------- */

typedef struct { float logit; int idx; } key_t_;

/* Larger logit first; equal logits (including -0.0 == +0.0): lower index first. */
static int key_cmp(const void *pa, const void *pb) {
    const key_t_ *a = (const key_t_ *)pa, *b = (const key_t_ *)pb;
    if (a->logit > b->logit) return -1;
    if (a->logit < b->logit) return 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

/* Top-k softmax routing and the permute-by-expert maps.
 *   ids[T*k], weights[T*k]: per token, the k experts in selection order and
 *       their routing weights (softmax over all E, renormalised over the k if
 *       normalize != 0); with router_weights [T, E] (may be NULL) the weights
 *       are router_weights[t][ids[t*k+j]] instead, renormalised the same way;
 *   offsets[E+1]: first permuted row of each expert, offsets[E] = T*k;
 *   expanded_to_perm[T*k]: permuted row of expanded index i = t*k + j;
 *   perm_to_expanded[T*k]: its inverse.
 * Any of the map outputs may be NULL. */
int oracle_route_mixed(const float *logits, const float *router_weights, int T, int E, int k, int normalize,
                       int32_t *ids, double *weights, int32_t *offsets,
                       int32_t *perm_to_expanded, int32_t *expanded_to_perm) {
    int t, j, e, i, R = T * k;
    key_t_ *keys;
    int32_t *count, *seen;
    if (!logits || !ids || T < 0 || E <= 0 || k <= 0 || k > E) return ORACLE_BAD_ARG;
    keys = (key_t_ *)malloc(sizeof(key_t_) * (size_t)E);
    if (!keys) return ORACLE_BAD_ARG;
    for (t = 0; t < T; ++t) {
        const float *row = logits + (size_t)t * E;
        double mx = -INFINITY, den = 0.0, sel = 0.0;
        for (e = 0; e < E; ++e) { keys[e].logit = row[e]; keys[e].idx = e; }
        qsort(keys, (size_t)E, sizeof(key_t_), key_cmp);
        for (e = 0; e < E; ++e) if ((double)row[e] > mx) mx = (double)row[e];
        for (e = 0; e < E; ++e) den += exp((double)row[e] - mx);
        for (j = 0; j < k; ++j) {
            ids[t * k + j] = keys[j].idx;
            if (weights)
                weights[t * k + j] = router_weights ? (double)router_weights[(size_t)t * E + keys[j].idx]
                                                    : exp((double)row[keys[j].idx] - mx) / den;
        }
        if (weights && normalize) {
            for (j = 0; j < k; ++j) sel += weights[t * k + j];
            for (j = 0; j < k; ++j) weights[t * k + j] /= sel;
        }
    }
    free(keys);
    if (!offsets && !perm_to_expanded && !expanded_to_perm) return ORACLE_OK;
    count = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    seen = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    if (!count || !seen) { free(count); free(seen); return ORACLE_BAD_ARG; }
    for (i = 0; i < R; ++i) count[ids[i]] += 1;
    {
        int32_t run = 0;
        for (e = 0; e < E; ++e) {
            if (offsets) offsets[e] = run;
            seen[e] = run; /* next free permuted row of expert e */
            run += count[e];
        }
        if (offsets) offsets[E] = run;
    }
    for (i = 0; i < R; ++i) {
        int32_t p = seen[ids[i]]++;
        if (expanded_to_perm) expanded_to_perm[i] = p;
        if (perm_to_expanded) perm_to_expanded[p] = i;
    }
    free(count);
    free(seen);
    return ORACLE_OK;
}

int oracle_route(const float *logits, int T, int E, int k, int normalize,
                 int32_t *ids, double *weights, int32_t *offsets,
                 int32_t *perm_to_expanded, int32_t *expanded_to_perm) {
    return oracle_route_mixed(logits, NULL, T, E, k, normalize, ids, weights, offsets, perm_to_expanded,
                              expanded_to_perm);
}

/* ---- activation ---------------------------------------------------------- */

/* SwiGLU, operator doc §8:
 *   G = min(gate, limit); L = clamp(value, -limit, limit);
 *   out = G * sigmoid(alpha * G) * (L + beta). */
double oracle_swiglu(double gate, double value, double alpha, double beta, double limit) {
    double G = gate > limit ? limit : gate;
    double L = value > limit ? limit : (value < -limit ? -limit : value);
    return G * (1.0 / (1.0 + exp(-alpha * G))) * (L + beta);
}

/* ---- one expert ----------------------------------------------------------- */

/* FC1 pre-activation of one token row against expert e:
 *   h[n] = sum_k x[k] * Wd1[e][n][k], n < 2I, with Wd1 the dequantised
 *   [E, 2I, H] matrix of fc1 (packed [E, H, I]).  Exact products, double sum. */
int oracle_expert_fc1(const uint16_t *x_row, int e, const uint8_t *w1, const uint8_t *s1,
                      const float *g1, int fmt, int H, int I, double *h) {
    int n, kk, N = 2 * I;
    for (n = 0; n < N; ++n) {
        double acc = 0.0;
        for (kk = 0; kk < H; ++kk)
            acc += oracle_bf16_to_double(x_row[kk]) *
                   oracle_dequant_element(w1, s1, g1, N, H, fmt, e, n, kk);
        h[n] = acc;
    }
    return ORACLE_OK;
}

/* FC2 of one activation row a[I] (bf16 values held as doubles):
 *   y[n] = sum_m a[m] * Wd2[e][n][m], n < H (packed [E, I, H/2]). */
int oracle_expert_fc2(const double *a, int e, const uint8_t *w2, const uint8_t *s2,
                      const float *g2, int fmt, int H, int I, double *y) {
    int n, m;
    for (n = 0; n < H; ++n) {
        double acc = 0.0;
        for (m = 0; m < I; ++m)
            acc += a[m] * oracle_dequant_element(w2, s2, g2, H, I, fmt, e, n, m);
        y[n] = acc;
    }
    return ORACLE_OK;
}

/* y = FFN_e(x): FC1, SwiGLU on the (gate, linear) pairs of the FC1 columns
 * (interleaved for swiglu_fusion 0 and 1, concatenated for 2) with the result
 * rounded to bf16, then FC2. */
int oracle_expert_ffn(const uint16_t *x_row, int e,
                      const uint8_t *w1, const uint8_t *s1, const float *g1,
                      const uint8_t *w2, const uint8_t *s2, const float *g2,
                      int fmt, int H, int I, double alpha, double beta, double limit,
                      int fusion, double *y) {
    int m;
    double *h, *a;
    if (fusion < 0 || fusion > 2) return ORACLE_BAD_ARG;
    h = (double *)malloc(sizeof(double) * 2 * (size_t)I);
    a = (double *)malloc(sizeof(double) * (size_t)I);
    if (!h || !a) { free(h); free(a); return ORACLE_BAD_ARG; }
    oracle_expert_fc1(x_row, e, w1, s1, g1, fmt, H, I, h);
    for (m = 0; m < I; ++m) {
        const double gate = fusion == 2 ? h[m] : h[2 * m];
        const double lin = fusion == 2 ? h[I + m] : h[2 * m + 1];
        a[m] = oracle_bf16_to_double(oracle_bf16_rne(oracle_swiglu(gate, lin, alpha, beta, limit)));
    }
    oracle_expert_fc2(a, e, w2, s2, g2, fmt, H, I, y);
    free(h);
    free(a);
    return ORACLE_OK;
}

/* ---- the layer ---------------------------------------------------------- */

/* The whole layer for the tokens listed in `tokens` (NULL: all T tokens, in
 * order): out[r][h] = bf16( sum_j w[t][j] * FFN_{id[t][j]}(x[t])[h] ) for the
 * r-th listed token t.  Routing uses the full logits row of each token; the
 * mixing weights come from router_weights when it is not NULL.
 * `nthreads` > 0 caps the OpenMP threads used over the (token, j) pairs. */
int oracle_moe_forward(const uint16_t *x, const float *logits, const float *router_weights,
                       const uint8_t *w1, const uint8_t *s1, const float *g1,
                       const uint8_t *w2, const uint8_t *s2, const float *g2,
                       int fmt, int T, int H, int I, int E, int k, int normalize,
                       double alpha, double beta, double limit, int fusion,
                       const int32_t *tokens, int ntok, uint16_t *out, int nthreads) {
    int r, npairs, pidx, status = ORACLE_OK;
    int32_t *ids;
    double *wts, *y;
    if (!x || !logits || !w1 || !s1 || !w2 || !s2 || !out) return ORACLE_BAD_ARG;
    if (fmt != ORACLE_NVFP4 && fmt != ORACLE_MXFP4) return ORACLE_BAD_ARG;
    if (fusion < 0 || fusion > 2) return ORACLE_BAD_ARG;
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || k > E) return ORACLE_BAD_ARG;
    if (H % block_size(fmt) || I % block_size(fmt) || (H & 1)) return ORACLE_BAD_ARG;
    if (!tokens) ntok = T;
    if (ntok < 0) return ORACLE_BAD_ARG;
    for (r = 0; tokens && r < ntok; ++r)
        if (tokens[r] < 0 || tokens[r] >= T) return ORACLE_BAD_ARG;
    ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k + 1);
    wts = (double *)malloc(sizeof(double) * (size_t)T * k + 1);
    npairs = ntok * k;
    y = (double *)malloc(sizeof(double) * (size_t)npairs * H + 1);
    if (!ids || !wts || !y) { free(ids); free(wts); free(y); return ORACLE_BAD_ARG; }
    oracle_route_mixed(logits, router_weights, T, E, k, normalize, ids, wts, NULL, NULL, NULL);
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (pidx = 0; pidx < npairs; ++pidx) {
        int rr = pidx / k, j = pidx % k;
        int t = tokens ? tokens[rr] : rr;
        oracle_expert_ffn(x + (size_t)t * H, ids[t * k + j], w1, s1, g1, w2, s2, g2,
                          fmt, H, I, alpha, beta, limit, fusion, y + (size_t)pidx * H);
    }
    for (r = 0; r < ntok; ++r) {
        int t = tokens ? tokens[r] : r, j, hh;
        for (hh = 0; hh < H; ++hh) {
            double acc = 0.0;
            for (j = 0; j < k; ++j) acc += wts[t * k + j] * y[((size_t)r * k + j) * H + hh];
            out[(size_t)r * H + hh] = oracle_bf16_rne(acc);
        }
    }
    free(ids);
    free(wts);
    free(y);
    return status;
}
