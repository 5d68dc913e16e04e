/*
 * CPU oracle for the NVFP4-weight mixture-of-experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow statement of what
 * the layer computes.  It is used by the tests, by smoke() and by the bench's
 * cpu_baseline leg; the product path (the CUDA library) never calls, links or
 * includes it, and it shares no code, header or table with that path.
 *
 * Sources, cited by page title and section:
 *   [P3-Scope]  "[Kernel][SM70] Improve Qwen3.8 no-MTP concurrency",
 *               section "Scope and related PRs": native NVFP4 weights with
 *               FP16 activations; raw E4M3 scale storage; router, expert
 *               dispatch, W13/SwiGLU fusion, W2/reduction fusion, shared gate;
 *               one integer plan shared by grouped W13 and grouped W2.
 *   [P3-Test]   same page, "Test Plan" item 2 and "Test Result": native E4M3
 *               encoding, subnormal, signed-zero and NaN cases; all-singleton,
 *               repeated and invalid experts.
 *   [P1-QSA]    "[Perf][SM70] Optimize Qwen3.8 Flash Next prefill", section
 *               "SM70 QSA indexer hotspot update": the 8192-token, top-10
 *               NVFP4 MoE (W13 then W2).
 *   [P2-QPN2]   "[SM70][Draft] Extend Qwen3.8 DFlash2 concurrency paths",
 *               sections "Purpose" and "Test Result": the QPN2 NVFP4 dense
 *               projection over a few rows (eight-row tiles, M <= 32),
 *               compared against FP32.
 * The pages do not print the bit layout.  The format followed here is the
 * standard NVFP4 one: E2M1 elements, one E4M3 ("fn": no infinities, 0x7F and
 * 0xFF are NaN) block scale per 16 consecutive K elements of a row, and one
 * FP32 global scale per tensor.  Each reading taken where the pages are
 * silent is marked "READING".
 *
 * Precision: every step that decides an integer (a quantised code, a top-k
 * selection) is done in FP32, the precision of the method; dot products and
 * the combine that produce real-valued outputs are accumulated in FP64.
 * Build with -ffp-contract=off and without fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_ST_INVALID_ID 0x1u
#define ORACLE_ST_NONFINITE 0x2u

/* ------------------------------------------------------------------------ */
/* FP16 <-> double (IEEE binary16, round to nearest even).                   */
/* ------------------------------------------------------------------------ */

double oracle_f16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int ex = (b >> 10) & 31;
    int man = b & 1023;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + man), ex - 25);
    return sign ? -v : v;
}

uint16_t oracle_f16_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return 0x7E00u;
    double a = fabs(v);
    /* 65520 is the midpoint between 65504 (odd mantissa) and 65536: ties go up. */
    if (a >= 65520.0)
        return sign | 0x7C00u;
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: spacing 2^-24; rint rounds half to even */
        double q = rint(a * ldexp(1.0, 24));
        return sign | (uint16_t)q; /* q == 1024 is the smallest normal */
    }
    int e;
    frexp(a, &e);
    int be = e - 1; /* a in [2^be, 2^(be+1)) */
    double q = rint(a / ldexp(1.0, be - 10)); /* in [1024, 2048] */
    if (q == 2048.0) {
        q = 1024.0;
        be += 1;
    }
    if (be > 15)
        return sign | 0x7C00u;
    return sign | (uint16_t)((be + 15) << 10) | (uint16_t)(q - 1024.0);
}

/* ------------------------------------------------------------------------ */
/* E2M1 and E4M3 codecs.                                                      */
/* ------------------------------------------------------------------------ */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value m * 0.5.  Magnitudes by code:
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Code 8 is -0. */
double oracle_e2m1_value(int code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* E4M3 (fn): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.
 * Exponent field 0 is subnormal: m * 2^-9.  0x7F / 0xFF are NaN; there is no
 * infinity; the largest finite magnitude is 0x7E = 448. */
double oracle_e4m3_value(int code)
{
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even E2M1 encoding with saturation to +-6.  The decision
 * thresholds are the midpoints between neighbouring magnitudes; a value
 * exactly on a midpoint goes to the neighbour whose mantissa bit is 0.
 * The sign of x is kept, so negative values that round to zero give -0. */
int oracle_e2m1_encode(float x)
{
    double a = fabs((double)x);
    int c;
    if (a <= 0.25)
        c = 0;
    else if (a < 0.75)
        c = 1;
    else if (a <= 1.25)
        c = 2;
    else if (a < 1.75)
        c = 3;
    else if (a <= 2.5)
        c = 4;
    else if (a < 3.5)
        c = 5;
    else if (a <= 5.0)
        c = 6;
    else
        c = 7;
    return signbit(x) ? (c | 8) : c;
}

/* Round-to-nearest-even E4M3 (fn) encoding, saturating to +-448 ("satfinite").
 * NaN maps to 0x7F (never produced by the quantiser, which rejects
 * non-finite input). */
int oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    int sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    int be = e - 1; /* binade exponent */
    if (be < -6)
        be = -6; /* subnormals share the spacing of the lowest binade */
    double spacing = ldexp(1.0, be - 3);
    double r = rint(a / spacing); /* exact division by a power of two */
    double v = r * spacing;       /* the rounded magnitude, exact */
    if (v == 0.0)
        return sign;
    if (v >= 448.0)
        return sign | 0x7E;
    frexp(v, &e);
    be = e - 1;
    int code;
    if (be < -6)
        code = (int)(v / ldexp(1.0, -9)); /* subnormal: m * 2^-9 */
    else
        code = ((be + 7) << 3) | (int)((v / ldexp(1.0, be) - 1.0) * 8.0);
    return sign | code;
}

/* The dequantised weight E2M1(q) * E4M3(s) as an FP16 bit pattern.  Every
 * product of a finite E4M3 value and an E2M1 value is exactly representable
 * in FP16 (largest 6 * 448 = 2688, smallest nonzero 0.5 * 2^-9 = 2^-10), so
 * this is exact; the sign of a zero product is the XOR of the signs. */
uint16_t oracle_dequant_f16(int q, int s)
{
    return oracle_f16_from_double(oracle_e2m1_value(q) * oracle_e4m3_value(s));
}

/* ------------------------------------------------------------------------ */
/* Quantiser: FP32 matrices -> NVFP4 (canonical layout).                       */
/* ------------------------------------------------------------------------ */

/*
 * w : n_mats x rows x k FP32, row-major.
 * q : n_mats x rows x (k/2) bytes; byte i of a row holds element 2i in its
 *     low nibble and element 2i+1 in its high nibble (READING: the pages do
 *     not give the nibble order).
 * s : n_mats x rows x (k/16) E4M3 bytes, one per 16 consecutive elements.
 * g : n_mats FP32 global scales.
 * Returns a status word (ORACLE_ST_NONFINITE if any input is NaN or inf).
 *
 * Steps (READING of "E4M3 scale = amax/6 after global scale", with the
 * global scale chosen so the largest magnitude maps to 6 * 448); every step
 * is one correctly rounded FP32 operation:
 *   g  = amax(tensor) / 2688            (g = 1 when the tensor is all zero)
 *   s  = E4M3_rne_sat((amax(block) / g) / 6)
 *   d  = value(s) * g
 *   q  = E2M1_rne_sat(x / d)            (q = +-0 keeping the sign when d == 0)
 */
uint32_t oracle_quantize(const float *w, int64_t n_mats, int64_t rows, int64_t k,
                         uint8_t *q, uint8_t *s, float *g)
{
    uint32_t status = 0;
    int64_t nb = k / 16;
    for (int64_t m = 0; m < n_mats; ++m) {
        const float *wm = w + m * rows * k;
        float amax = 0.0f;
        for (int64_t i = 0; i < rows * k; ++i) {
            float v = wm[i];
            if (!isfinite(v)) {
                status |= ORACLE_ST_NONFINITE;
                continue;
            }
            float a = fabsf(v);
            if (a > amax)
                amax = a;
        }
        volatile float gm = amax / 2688.0f;
        if (amax == 0.0f)
            gm = 1.0f;
        g[m] = gm;
        for (int64_t r = 0; r < rows; ++r) {
            const float *wr = wm + r * k;
            uint8_t *qr = q + (m * rows + r) * (k / 2);
            uint8_t *sr = s + (m * rows + r) * nb;
            for (int64_t b = 0; b < nb; ++b) {
                float bmax = 0.0f;
                for (int j = 0; j < 16; ++j) {
                    float v = wr[b * 16 + j];
                    float a = isfinite(v) ? fabsf(v) : 0.0f;
                    if (a > bmax)
                        bmax = a;
                }
                volatile float t = bmax / gm;
                volatile float sb = t / 6.0f;
                int sc = oracle_e4m3_encode(sb);
                sr[b] = (uint8_t)sc;
                volatile float d = (float)oracle_e4m3_value(sc) * gm;
                for (int j = 0; j < 16; j += 2) {
                    int c[2];
                    for (int u = 0; u < 2; ++u) {
                        float v = wr[b * 16 + j + u];
                        if (!isfinite(v))
                            v = 0.0f;
                        if (d == 0.0f) {
                            c[u] = signbit(v) ? 8 : 0;
                        } else {
                            volatile float z = v / d;
                            c[u] = oracle_e2m1_encode(z);
                        }
                    }
                    qr[(b * 16 + j) / 2] = (uint8_t)(c[0] | (c[1] << 4));
                }
            }
        }
    }
    return status;
}

/* Dequantise canonical NVFP4 rows to FP16 bit patterns (exact). */
void oracle_dequant(const uint8_t *q, const uint8_t *s, int64_t rows, int64_t k,
                    uint16_t *out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < k; ++c) {
            uint8_t byte = q[r * (k / 2) + c / 2];
            int code = (c & 1) ? (byte >> 4) : (byte & 15);
            out[r * k + c] = oracle_dequant_f16(code, s[r * (k / 16) + c / 16]);
        }
}

/* ------------------------------------------------------------------------ */
/* Router: FP32 logits, top-k, renormalised softmax weights; shared gate.     */
/* ------------------------------------------------------------------------ */

/*
 * x      : M x H FP16 bits (row-major).
 * wr     : H x E FP16 bits (row-major: expert index fastest).
 * bias   : E FP32 or NULL.
 * logits : M x E FP32 out: sum over h = 0..H-1 in ascending order of
 *          float(x) * float(wr) in FP32 (each product is exact in FP32),
 *          then + bias (READING: the bias is part of the logit and so enters
 *          both the selection and the weights).
 * ids    : M x k int32 out, the k largest logits in descending order; equal
 *          logits are ordered by ascending expert id.
 * w      : M x k FP32 out, exp(l_j - l_max) / sum over the k selected.  This
 *          equals the full softmax renormalised over the selected k.
 * [P3-Scope] lists the router; [P1-QSA] gives top-10.
 */
void oracle_router(const uint16_t *x, const uint16_t *wr, const float *bias,
                   int64_t M, int64_t H, int64_t E, int64_t k, float *logits,
                   int32_t *ids, float *w)
{
    /* tokens are independent; each logit is summed in ascending h order.
     * Built without fast-math and with -ffp-contract=off, so every product
     * and sum below is one IEEE FP32 operation in program order. */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < M; ++t) {
        float *lt = logits + t * E;
        float *xf = (float *)malloc(sizeof(float) * H);
        for (int64_t h = 0; h < H; ++h)
            xf[h] = (float)oracle_f16_to_double(x[t * H + h]);
        for (int64_t e = 0; e < E; ++e) {
            float acc = 0.0f;
            for (int64_t h = 0; h < H; ++h) {
                float p = xf[h] * (float)oracle_f16_to_double(wr[h * E + e]);
                acc = acc + p;
            }
            lt[e] = bias ? acc + bias[e] : acc;
        }
        free(xf);
        /* selection: repeatedly take the largest remaining logit, the lowest
         * id winning ties (a stable descending sort, truncated to k) */
        unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
        for (int64_t j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || lt[e] > lt[best])
                    best = e;
            }
            taken[best] = 1;
            ids[t * k + j] = (int32_t)best;
        }
        free(taken);
        double lmax = lt[ids[t * k]];
        double den = 0.0;
        for (int64_t j = 0; j < k; ++j)
            den += exp((double)lt[ids[t * k + j]] - lmax);
        for (int64_t j = 0; j < k; ++j)
            w[t * k + j] = (float)(exp((double)lt[ids[t * k + j]] - lmax) / den);
    }
}

/* Shared-expert gate [P3-Scope] "shared gate": gamma_t = sigmoid(x_t . w_g). */
void oracle_shared_gate(const uint16_t *x, const uint16_t *wg, int64_t M, int64_t H,
                        float *gamma)
{
    for (int64_t t = 0; t < M; ++t) {
        double z = 0.0;
        for (int64_t h = 0; h < H; ++h)
            z += oracle_f16_to_double(x[t * H + h]) * oracle_f16_to_double(wg[h]);
        gamma[t] = (float)(1.0 / (1.0 + exp(-z)));
    }
}

/* ------------------------------------------------------------------------ */
/* Plan: the integer routing plan shared by W13 and W2 [P3-Scope].            */
/* ------------------------------------------------------------------------ */

/*
 * ids    : n_pairs expert ids; pair p is token p / k, slot p % k.
 * counts : n_exp out, valid pairs per expert.
 * offsets: n_exp + 1 out, exclusive prefix sum of counts.
 * perm   : n_valid out; the pairs sorted by expert, pairs of one expert in
 *          ascending pair id (a stable sort).  perm[position] = pair id.
 * inv    : n_pairs out; inv[pair id] = position, or -1 for a pair whose id is
 *          outside [0, n_exp) (READING: such pairs are dropped and flagged).
 * tiles  : out, up to max_tiles triples (expert, first row, rows): each
 *          expert's segment cut into pieces of at most bn rows, experts in
 *          ascending order.  Returns the tile count in *n_tiles.
 * Returns a status word (ORACLE_ST_INVALID_ID if any id was invalid).
 */
uint32_t oracle_plan(const int32_t *ids, int64_t n_pairs, int64_t n_exp, int64_t bn,
                     int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv,
                     int32_t *tiles, int64_t max_tiles, int64_t *n_tiles)
{
    uint32_t status = 0;
    for (int64_t e = 0; e < n_exp; ++e)
        counts[e] = 0;
    for (int64_t p = 0; p < n_pairs; ++p) {
        int32_t e = ids[p];
        if (e < 0 || e >= n_exp)
            status |= ORACLE_ST_INVALID_ID;
        else
            counts[e] += 1;
    }
    offsets[0] = 0;
    for (int64_t e = 0; e < n_exp; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    /* stable placement: walk pairs in ascending id, append to their expert */
    int32_t *fill = (int32_t *)calloc((size_t)(n_exp > 0 ? n_exp : 1), sizeof(int32_t));
    for (int64_t p = 0; p < n_pairs; ++p) {
        int32_t e = ids[p];
        if (e < 0 || e >= n_exp) {
            inv[p] = -1;
            continue;
        }
        int32_t pos = offsets[e] + fill[e]++;
        perm[pos] = (int32_t)p;
        inv[p] = pos;
    }
    free(fill);
    int64_t nt = 0;
    for (int64_t e = 0; e < n_exp; ++e)
        for (int32_t r0 = 0; r0 < counts[e]; r0 += (int32_t)bn) {
            if (nt < max_tiles) {
                tiles[nt * 3 + 0] = (int32_t)e;
                tiles[nt * 3 + 1] = r0;
                tiles[nt * 3 + 2] = (counts[e] - r0 < bn) ? counts[e] - r0 : (int32_t)bn;
            }
            ++nt;
        }
    *n_tiles = nt;
    return status;
}

/* ------------------------------------------------------------------------ */
/* Expert MLP and combine.                                                    */
/* ------------------------------------------------------------------------ */

static double e2m1_tab[16];
static double e4m3_tab[256];
static int tabs_ready = 0;

static void init_tabs(void)
{
    if (tabs_ready)
        return;
    for (int c = 0; c < 16; ++c)
        e2m1_tab[c] = oracle_e2m1_value(c);
    for (int c = 0; c < 256; ++c)
        e4m3_tab[c] = oracle_e4m3_value(c);
    tabs_ready = 1;
}

/* Dequantised weight (row r, column c) of a canonical NVFP4 matrix whose rows
 * have k elements, as a double (exact). */
static double wval(const uint8_t *q, const uint8_t *s, int64_t k, int64_t r, int64_t c)
{
    uint8_t byte = q[r * (k / 2) + c / 2];
    int code = (c & 1) ? (byte >> 4) : (byte & 15);
    return e2m1_tab[code] * e4m3_tab[s[r * (k / 16) + c / 16]];
}

/*
 * One expert MLP for one token [P3-Scope] "W13/SwiGLU fusion",
 * "W2/reduction fusion":
 *   G_i = g13 * sum_K x_K W13[i][K],  U_i = g13 * sum_K x_K W13[I+i][K]
 *   h_i = fp16( silu(G_i) * U_i ),     silu(z) = z / (1 + exp(-z))
 *   o_n = g2 * sum_i h_i W2[n][i]
 * W13 rows 0..I-1 are the gate projection and rows I..2I-1 the up projection
 * (READING of the name W13 = w1 (gate) stacked over w3 (up)); the one global
 * scale g13 covers both halves (READING: one tensor per expert and matrix).
 * Rounding h to FP16 is a READING: the second GEMM consumes FP16 operands.
 * With h_exact the other reading is taken instead: h stays unrounded (a
 * double), as if the two GEMMs were fused with no narrowing between them.
 */
static void expert_mlp(const double *xt, int64_t H, int64_t I, const uint8_t *q13,
                       const uint8_t *s13, float g13, const uint8_t *q2,
                       const uint8_t *s2, float g2, int h_exact, double *h, double *o)
{
    for (int64_t i = 0; i < I; ++i) {
        double G = 0.0, U = 0.0;
        for (int64_t c = 0; c < H; ++c) {
            G += xt[c] * wval(q13, s13, H, i, c);
            U += xt[c] * wval(q13, s13, H, I + i, c);
        }
        G *= (double)g13;
        U *= (double)g13;
        double a = G / (1.0 + exp(-G)) * U;
        h[i] = h_exact ? a : oracle_f16_to_double(oracle_f16_from_double(a));
    }
    for (int64_t n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i)
            acc += h[i] * wval(q2, s2, I, n, i);
        o[n] = acc * (double)g2;
    }
}

/*
 * The layer forward for the tokens in `tokens` (all M tokens when tokens is
 * NULL; then n_tok must equal M).  Outputs y[n_tok][H] as FP16 bits, row j of
 * y belonging to token tokens[j].
 *
 *   y_t = fp16( sum_{j=0..k-1} w[t,j] * o_{t,j}  +  gamma_t * s_t )
 *
 * summed in slot order j = 0..k-1, then the shared term (READING: the pages
 * do not fix the combine order), with one rounding to FP16.  o_{t,j} is the
 * MLP of expert ids[t,j]; a pair with an id outside [0, E) contributes 0
 * (READING, see oracle_plan).  The shared term is present when sq13 is not
 * NULL; gamma may then be NULL only if the caller wants gamma = 1.
 *
 * Weights are canonical NVFP4: q13 [E][2I][H/2], s13 [E][2I][H/16], g13 [E];
 * q2 [E][H][I/2], s2 [E][H][I/16], g2 [E]; shared expert the same without E.
 * h_out (optional): the h of each pair, [n_tok][k][I] as double (FP16-rounded
 * unless h_exact).
 */
uint32_t oracle_forward(int64_t M, int64_t H, int64_t E, int64_t k, int64_t I,
                        const uint16_t *x, const int32_t *ids, const float *w,
                        const uint8_t *q13, const uint8_t *s13, const float *g13,
                        const uint8_t *q2, const uint8_t *s2, const float *g2,
                        const uint8_t *sq13, const uint8_t *ss13, const float *sg13,
                        const uint8_t *sq2, const uint8_t *ss2, const float *sg2,
                        const float *gamma, const int64_t *tokens, int64_t n_tok,
                        int h_exact, uint16_t *y, double *h_out)
{
    init_tabs();
    uint32_t status = 0;
    const int64_t b13 = 2 * I * (H / 2), c13 = 2 * I * (H / 16);
    const int64_t b2 = H * (I / 2), c2 = H * (I / 16);
    for (int64_t jt = 0; jt < n_tok; ++jt) {
        int64_t t = tokens ? tokens[jt] : jt;
        for (int64_t j = 0; j < k; ++j) {
            int32_t e = ids[t * k + j];
            if (e < 0 || e >= E)
                status |= ORACLE_ST_INVALID_ID;
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t jt = 0; jt < n_tok; ++jt) {
        int64_t t = tokens ? tokens[jt] : jt;
        double *xt = (double *)malloc(sizeof(double) * H);
        double *h = (double *)malloc(sizeof(double) * I);
        double *o = (double *)malloc(sizeof(double) * H);
        double *acc = (double *)calloc((size_t)H, sizeof(double));
        for (int64_t c = 0; c < H; ++c)
            xt[c] = oracle_f16_to_double(x[t * H + c]);
        for (int64_t j = 0; j < k; ++j) {
            int32_t e = ids[t * k + j];
            if (e < 0 || e >= E) {
                if (h_out)
                    for (int64_t i = 0; i < I; ++i)
                        h_out[(jt * k + j) * I + i] = 0.0;
                continue;
            }
            expert_mlp(xt, H, I, q13 + e * b13, s13 + e * c13, g13[e], q2 + e * b2,
                       s2 + e * c2, g2[e], h_exact, h, o);
            if (h_out)
                for (int64_t i = 0; i < I; ++i)
                    h_out[(jt * k + j) * I + i] = h[i];
            for (int64_t n = 0; n < H; ++n)
                acc[n] += (double)w[t * k + j] * o[n];
        }
        if (sq13) {
            expert_mlp(xt, H, I, sq13, ss13, sg13[0], sq2, ss2, sg2[0], h_exact, h, o);
            double gm = gamma ? (double)gamma[t] : 1.0;
            for (int64_t n = 0; n < H; ++n)
                acc[n] += gm * o[n];
        }
        for (int64_t n = 0; n < H; ++n)
            y[jt * H + n] = oracle_f16_from_double(acc[n]);
        free(xt);
        free(h);
        free(o);
        free(acc);
    }
    return status;
}

/*
 * Dense NVFP4 projection of a few FP16 rows [P2-QPN2]:
 *   y[m][n] = fp16( g * sum_K x[m][K] * w16[n][K] )
 * accumulated in FP64 and rounded to FP16 once (READING: the pages print no
 * formula for QPN2; this is the layer's own projection step, the same as the
 * expert MLP's second GEMM, without routing).  Canonical NVFP4 weights:
 * q [N][K/2], s [N][K/16], one FP32 global scale g.  x [M][K] and y [M][N]
 * are FP16 bits.  Each row is computed on its own, so a row's output does not
 * depend on the other rows of the call.
 */
void oracle_dense(int64_t M, int64_t N, int64_t K, const uint16_t *x, const uint8_t *q,
                  const uint8_t *s, float g, uint16_t *y)
{
    init_tabs();
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t c = 0; c < K; ++c)
                acc += oracle_f16_to_double(x[m * K + c]) * wval(q, s, K, n, c);
            y[m * N + n] = oracle_f16_from_double(acc * (double)g);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Prepared-scale storage ("[Kernel][SM70] Improve Qwen3.8 no-MTP           */
/* concurrency", sections "Purpose" and "Scope and related PRs": the        */
/* prepared arm stores effective decode scales instead of raw E4M3 bytes;   */
/* "Test Result": raw and prepared outputs are bitwise equal).              */
/* ------------------------------------------------------------------------ */

/*
 * out[i] = the FP16 bit pattern of E4M3(s[i]), for i < n, in the same order
 * (READING: the prepared scale is the raw scale's value widened to the FP16
 * operand type of the GEMM, exact since every finite E4M3 value is an FP16
 * value; the global scale stays on the FP32 accumulator).  NaN codes give the
 * FP16 NaN 0x7E00 and set ORACLE_ST_NONFINITE.
 */
uint32_t oracle_prepare_scales(const uint8_t *s, int64_t n, uint16_t *out)
{
    uint32_t status = 0;
    for (int64_t i = 0; i < n; ++i) {
        double v = oracle_e4m3_value(s[i]);
        if (isnan(v)) {
            out[i] = 0x7E00;
            status |= ORACLE_ST_NONFINITE;
        } else {
            out[i] = oracle_f16_from_double(v);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Channel-FP8 weights (QPN8: "[SM70][Draft] Extend Qwen3.8 DFlash2         */
/* concurrency paths", section "Follow-up: exact channel-FP8 QPN8           */
/* concurrency paths and endpoint evidence").                               */
/* ------------------------------------------------------------------------ */

/*
 * w  : rows x k FP32, row-major (row = output channel).
 * q  : rows x k E4M3 codes, row-major (canonical: one byte per element).
 * cs : rows FP32 channel scales.
 * READING: the pages name FP8 weights with one scale per output channel but
 * print no recipe; the plainest one, with every step one correctly rounded
 * FP32 operation, is
 *   cs_r = amax(row r) / 448          (cs_r = 1 when the row is all zero)
 *   q    = E4M3_rne_satfinite(x / cs_r)
 * so that the row's largest magnitude maps to the largest E4M3 value.  NaN or
 * infinite input sets ORACLE_ST_NONFINITE and is quantised as zero.
 */
uint32_t oracle_fp8_quantize(const float *w, int64_t rows, int64_t k, uint8_t *q, float *cs)
{
    uint32_t status = 0;
    for (int64_t r = 0; r < rows; ++r) {
        const float *wr = w + r * k;
        float amax = 0.0f;
        for (int64_t i = 0; i < k; ++i) {
            if (!isfinite(wr[i])) {
                status |= ORACLE_ST_NONFINITE;
                continue;
            }
            float a = fabsf(wr[i]);
            if (a > amax)
                amax = a;
        }
        volatile float c = amax / 448.0f;
        if (amax == 0.0f)
            c = 1.0f;
        cs[r] = c;
        for (int64_t i = 0; i < k; ++i) {
            float v = isfinite(wr[i]) ? wr[i] : 0.0f;
            volatile float z = v / c;
            q[r * k + i] = (uint8_t)oracle_e4m3_encode(z);
        }
    }
    return status;
}

/*
 * Dense channel-FP8 projection of a few FP16 rows:
 *   y[m][n] = fp16( cs[n] * sum_K x[m][K] * E4M3(q[n][K]) )
 * accumulated in FP64, one rounding to FP16.  READING: the channel scale
 * multiplies the accumulated dot product (the pages only say that where the
 * scale is applied changes the FP32 result; any exact placement gives the
 * same real value, which is what the oracle computes).  x [M][K] and y
 * [M][N] are FP16 bits, q [N][K] canonical, cs [N].  Rows are independent.
 */
void oracle_fp8_dense(int64_t M, int64_t N, int64_t K, const uint16_t *x, const uint8_t *q,
                      const float *cs, uint16_t *y)
{
    init_tabs();
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int64_t c = 0; c < K; ++c)
                acc += oracle_f16_to_double(x[m * K + c]) * e4m3_tab[q[n * K + c]];
            y[m * N + n] = oracle_f16_from_double(acc * (double)cs[n]);
        }
    }
}

int oracle_abi_version(void) { return 1; }
