/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for the dropless
 * Mixture-of-Experts layer hot path.
 *
 * TEST INFRASTRUCTURE. This file is the correctness reference that the GPU
 * kernels are checked against. Only the test suite, the package smoke check
 * and the benchmark's CPU-baseline leg load it (through oracle/__init__.py).
 * The library never includes, links or calls anything here, and nothing here
 * includes or calls the library: the two share no code.
 *
 * Every floating-point step is evaluated in double precision; results are
 * rounded once, to the output format, at the end (round-to-nearest-even).
 * Loops follow the definitions one to one: no blocking, no fusion, no
 * reordering beyond what a definition states.
 *
 * Sources (web pages on the subject; cited by title and section):
 *   [SPARSER]  "Sparser MoE end-to-end" (harryzhou2000 blog):
 *              sections "The workload changes the bottleneck",
 *              "Preserve a compact route", "Remove work that has no selected route".
 *   [TEJAX]    "Dropless MoE acceleration in JAX with NVIDIA Transformer Engine"
 *              (news.bpdata.com): sections "Dropless vs capacity-based MoE",
 *              "Transformer Engine building blocks for dropless MoE in JAX" (and
 *              its MoE-layer figure), "Optimization 1: Grouped GEMM",
 *              "Optimization 2: Expert parallelism to fuse Dispatch and Combine".
 *   [WITTY]    "NVIDIA says its JAX stack makes dropless MoE training 10x faster"
 *              (wittywires.com): section "What to watch".
 *   [CLARITY]  "NVIDIA's unoptimized DeepSeek-V3 baseline spends 84% of kernel
 *              time moving tokens between GPUs" (theclarity.today).
 * Where the pages leave a step open, the reading taken is stated beside the
 * code (and listed with the other readings in the design notes).
 *
 * Parity status: every exported function is pinned by the CPU tests
 * (tests/test_oracle_*.py) against brute force, library routines, closed
 * forms or invariants.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 -> double: bf16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a finite |a| > 0 to a binary format with `p` significand bits
 * (including the implicit one) and minimum normal exponent `emin`; values
 * below 2^emin use the fixed subnormal quantum 2^(emin - p + 1).
 * Round-to-nearest, ties-to-even (nearbyint under the default rounding mode).
 * Division and multiplication by powers of two are exact here.
 */
static double round_to_format(double a, int p, int emin)
{
    int e;
    frexp(a, &e);            /* a in [2^(e-1), 2^e) */
    int ex = e - 1;
    if (ex < emin)
        ex = emin;
    double quantum = ldexp(1.0, ex - (p - 1));
    return nearbyint(a / quantum) * quantum;
}

/* double -> bfloat16, round to nearest even, overflow to infinity. */
uint16_t oracle_double_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return 0x7FC0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    double q = round_to_format(a, 8, -126);
    if (q >= 0x1p128)
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)q;      /* exact: q has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/*
 * E4M3 (the "FN" variant used by MXFP8): 1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448.
 */
double oracle_e4m3_decode(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 0xF, M = c & 7;
    double v;
    if (E == 15 && M == 7)
        v = NAN;
    else if (E == 0)
        v = ldexp((double)M, -9);          /* subnormal: M * 2^-9 */
    else
        v = ldexp(1.0 + M / 8.0, E - 7);
    return s ? -v : v;
}

/* double -> E4M3, round to nearest even, saturating to +-448 ("satfinite").
 * The sign of zero is kept. */
uint8_t oracle_e4m3_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    double a = fabs(v);
    if (a == 0.0 || isnan(a))
        return sign;
    double q = isinf(a) ? 448.0 : round_to_format(a, 4, -6);
    if (q > 448.0)
        q = 448.0;
    if (q == 0.0)
        return sign;
    int e;
    frexp(q, &e);
    int ex = e - 1;
    if (ex < -6)                              /* subnormal code 1..7 */
        return (uint8_t)(sign | (uint8_t)(q / ldexp(1.0, -9)));
    int mant = (int)((q / ldexp(1.0, ex) - 1.0) * 8.0);
    return (uint8_t)(sign | (uint8_t)(((ex + 7) << 3) | mant));
}

/*
 * Shared E8M0 block exponent of one MXFP8 block ([TEJAX] "Transformer Engine
 * building blocks": MXFP8 with 1x32 E8M0 block scales). Reading taken: the
 * Microscaling convention -- exponent = floor(log2(amax)) - 8, where 8 is the
 * exponent of E4M3's largest power of two (448 = 1.75 * 2^8); the stored byte
 * is exponent + 127 clamped to [0, 254]; an all-zero block gets byte 127 (2^0).
 */
int oracle_e8m0_scale_byte(double amax)
{
    if (amax == 0.0)
        return 127;
    int e;
    frexp(amax, &e);                 /* floor(log2(amax)) = e - 1 */
    int b = (e - 1) - 8 + 127;
    if (b < 0)
        b = 0;
    if (b > 254)
        b = 254;
    return b;
}

/* Quantise n = 32 consecutive values (stride `stride` apart) to one MXFP8
 * block: writes 32 E4M3 codes (same stride) and returns the scale byte. */
static int quant_block(const double *x, long stride, int n, uint8_t *q, long qstride)
{
    double amax = 0.0;
    for (int i = 0; i < n; i++) {
        double a = fabs(x[i * stride]);
        if (a > amax)
            amax = a;
    }
    int sb = oracle_e8m0_scale_byte(amax);
    double inv = ldexp(1.0, 127 - sb);   /* x / 2^(sb-127) */
    for (int i = 0; i < n; i++)
        q[i * qstride] = oracle_e4m3_encode(x[i * stride] * inv);
    return sb;
}

/* Row-wise 1x32 MXFP8 quantisation of a bf16 matrix [rows, cols]
 * (cols % 32 == 0). Payload q[rows, cols]; scales s[rows, cols/32]. */
void oracle_quant_rows_bf16(const uint16_t *x, long rows, long cols, uint8_t *q, uint8_t *s)
{
    double buf[32];
    for (long r = 0; r < rows; r++)
        for (long b = 0; b < cols / 32; b++) {
            for (int i = 0; i < 32; i++)
                buf[i] = oracle_bf16_to_double(x[r * cols + b * 32 + i]);
            s[r * (cols / 32) + b] = (uint8_t)quant_block(buf, 1, 32, q + r * cols + b * 32, 1);
        }
}

/* ------------------------------------------------------------------------ */
/* NVFP4                                                                     */
/* ------------------------------------------------------------------------ */

/*
 * NVFP4 ([TEJAX] "Measured training impact with JAX + Transformer Engine" and
 * [WITTY] "What to watch" name it as a planned addition; neither defines it).
 * Reading taken: NVIDIA's published NVFP4 format --
 *   elements  E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit):
 *             magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6;
 *   blocks    16 consecutive elements along a row share one E4M3 decode scale;
 *   tensor    one fp32 encode scale S = 448 * 6 / amax(tensor) (S = 1 when the
 *             tensor is all zero, at most FLT_MAX), so that the block scales
 *             use E4M3's range;
 *   decode    x = e2m1(q) * e4m3(sb) / S.
 * The encoder's decisions are taken in fp32 (each operation one IEEE rounding):
 *   sb = E4M3(rne, saturating)( (amax_block / 6) * S )
 *   q  = E2M1(rne, saturating to 6, sign kept)( x * (S / e4m3(sb)) ), 0 when the
 *        decoded block scale is 0.
 * Packing: element 2i in the low nibble of byte i, element 2i+1 in the high one.
 */
double oracle_e2m1_decode(uint8_t code)
{
    const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* The values of the 16 E2M1 codes (oracle_e2m1_decode of each), for loops over many elements. */
static void e2m1_values(double val[16])
{
    for (int c = 0; c < 16; c++)
        val[c] = oracle_e2m1_decode((uint8_t)c);
}

/* Nearest E2M1 code to v (ties to the even mantissa bit), saturating to +-6, sign kept;
 * val holds the code values (e2m1_values). */
static uint8_t e2m1_encode_with(const double val[16], double v)
{
    const uint8_t sign = signbit(v) ? 8 : 0;
    const double a = fmin(fabs(v), 6.0);      /* saturating: beyond 6 is 6 */
    int best = 0;
    double db = fabs(val[0] - a);
    for (int c = 1; c < 8; c++) {
        const double dc = fabs(val[c] - a);
        if (dc < db || (dc == db && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            db = dc;
        }
    }
    return (uint8_t)(sign | best);
}

/* Nearest E2M1 code (ties to the even mantissa bit), saturating to +-6, sign kept. */
uint8_t oracle_e2m1_encode(double v)
{
    double val[16];
    e2m1_values(val);
    return e2m1_encode_with(val, v);
}

/* The tensor's fp32 encode scale from its amax. */
float oracle_nvfp4_encode_scale(float amax)
{
    if (!(amax > 0.0f))
        return 1.0f;
    volatile float s = 2688.0f / amax;           /* 448 * 6 */
    return s > FLT_MAX ? FLT_MAX : s;
}

/*
 * Row-wise NVFP4 of a bf16 matrix x[rows, cols] (cols % 16 == 0) with the
 * tensor encode scale S (oracle_nvfp4_encode_scale of the amax the caller
 * chooses, normally that of x): q[rows, cols/2] packed E2M1, s[rows, cols/16]
 * E4M3 decode scales.
 */
void oracle_quant_rows_nvfp4(const uint16_t *x, long rows, long cols, float S, uint8_t *q, uint8_t *s)
{
    double val[16];
    e2m1_values(val);
    for (long r = 0; r < rows; r++)
        for (long b = 0; b < cols / 16; b++) {
            const uint16_t *blk = x + r * cols + b * 16;
            float amax = 0.0f;
            for (int i = 0; i < 16; i++) {
                const float v = (float)fabs(oracle_bf16_to_double(blk[i]));
                if (v > amax)
                    amax = v;
            }
            volatile float t = amax / 6.0f;
            volatile float sbf = t * S;
            const uint8_t sb = oracle_e4m3_encode((double)sbf);
            const float ds = (float)oracle_e4m3_decode(sb);
            s[r * (cols / 16) + b] = sb;
            volatile float rs = ds > 0.0f ? S / ds : 0.0f;
            for (int i = 0; i < 16; i++) {
                volatile float v = (float)oracle_bf16_to_double(blk[i]) * rs;
                const uint8_t c = ds > 0.0f ? e2m1_encode_with(val, (double)v) : 0;
                uint8_t *byte = q + r * (cols / 2) + b * 8 + i / 2;
                if (i % 2 == 0)
                    *byte = (uint8_t)((*byte & 0xF0) | c);
                else
                    *byte = (uint8_t)((*byte & 0x0F) | (c << 4));
            }
        }
}

/* Decode an NVFP4 matrix (packed q[rows, cols/2], scales s[rows, cols/16], encode scale S). */
void oracle_nvfp4_decode(const uint8_t *q, const uint8_t *s, long rows, long cols, float S, double *out)
{
    double val[16];
    e2m1_values(val);
    for (long r = 0; r < rows; r++)
        for (long b = 0; b < cols / 16; b++) {
            const double scale = oracle_e4m3_decode(s[r * (cols / 16) + b]);
            for (long c = 16 * b; c < 16 * b + 16; c++) {
                const uint8_t byte = q[r * (cols / 2) + c / 2];
                const uint8_t code = (c % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
                out[r * cols + c] = val[code] * scale / (double)S;
            }
        }
}

/* Dequantise one MXFP8 element. */
static double mx_value(uint8_t code, uint8_t sbyte)
{
    return ldexp(oracle_e4m3_decode(code), (int)sbyte - 127);
}

/*
 * Group-aware column-wise MXFP8 quantisation of a bf16 matrix x[R_cap, cols]
 * whose rows [off[e], off[e+1]) form group e ([TEJAX] "group-aware MXFP8
 * quantization"). Blocks are 32 consecutive rows of one column and never
 * cross a group boundary: they start at each group's first row; a group's
 * last block may be partial and then takes its amax over its valid rows only.
 * Scale layout: block b of group e is scale row (e + off[e] / 32 + b) of
 * s[E + R_cap/32 + 1, cols] -- a padded layout that needs no scan (rows of
 * the block index space that no block uses are left untouched). Payload
 * rows >= off[E] are not written.
 */
void oracle_quant_cols_grouped_bf16(const uint16_t *x, long cols, const int32_t *off, int E,
                                    uint8_t *q, uint8_t *s)
{
    double buf[32];
    uint8_t qb[32];
    for (int e = 0; e < E; e++) {
        long r0 = off[e], r1 = off[e + 1];
        for (long b = 0; r0 + 32 * b < r1; b++) {
            long rs = r0 + 32 * b;
            int n = (int)((r1 - rs) < 32 ? (r1 - rs) : 32);
            long srow = e + r0 / 32 + b;
            for (long c = 0; c < cols; c++) {
                for (int i = 0; i < n; i++)
                    buf[i] = oracle_bf16_to_double(x[(rs + i) * cols + c]);
                s[srow * cols + c] = (uint8_t)quant_block(buf, 1, n, qb, 1);
                for (int i = 0; i < n; i++)
                    q[(rs + i) * cols + c] = qb[i];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Router: softmax scores + top-K on raw logits                              */
/* ------------------------------------------------------------------------ */

typedef struct {
    float v;
    int idx;
} scored;

/* Descending logit; equal logits (IEEE compare, so -0 == +0): lower index first. */
static int cmp_scored(const void *pa, const void *pb)
{
    const scored *a = pa, *b = pb;
    if (a->v > b->v)
        return -1;
    if (a->v < b->v)
        return 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

/*
 * Router top-K ([SPARSER] "Preserve a compact route": selected expert ids
 * carried as a dense [T, K] list; [TEJAX] "Optimization 2": the router kernels
 * assign tokens before permutation).
 * Readings taken: (1) selection is on the raw logits, ties go to the lower
 * expert index, ids are stored in selection order (descending logit);
 * (2) probs[t,k] is the softmax over all E logits of the row, taken at the
 * selected id; with renorm != 0 the denominator is the sum over the K
 * selected experts only.
 * ids is int32 [T,K]; probs is float [T,K] (each rounded once from double).
 */
void oracle_route_topk(const float *logits, int T, int E, int K, int renorm,
                       int32_t *ids, float *probs)
{
    scored *row = (scored *)malloc(sizeof(scored) * (size_t)E);
    for (int t = 0; t < T; t++) {
        const float *l = logits + (size_t)t * E;
        for (int e = 0; e < E; e++) {
            row[e].v = l[e];
            row[e].idx = e;
        }
        qsort(row, (size_t)E, sizeof(scored), cmp_scored);
        double m = (double)row[0].v;          /* row maximum */
        double denom = 0.0;
        if (renorm) {
            for (int k = 0; k < K; k++)
                denom += exp((double)row[k].v - m);
        } else {
            for (int e = 0; e < E; e++)
                denom += exp((double)l[e] - m);
        }
        for (int k = 0; k < K; k++) {
            ids[(size_t)t * K + k] = row[k].idx;
            probs[(size_t)t * K + k] = (float)(exp((double)row[k].v - m) / denom);
        }
    }
    free(row);
}

/*
 * Sigmoid-score routing with a per-expert selection bias. The pages name the
 * router's "score transformation" and the "bias statistics" that compact
 * routes must preserve ([SPARSER] "The workload changes the bottleneck",
 * "Preserve a compact route") without defining either. Reading taken: the
 * DeepSeek-style score function and bias-steered selection --
 *   score     s_e = 1 / (1 + exp(-l_e))     (double, rounded once to fp32)
 *   key       k_e = s_e + b_e               (fp32 addition; b = 0 when absent)
 *   ids       the K largest keys, in descending key order, lower index first
 *             on equal keys (IEEE compare)
 *   probs     s at the selected ids, or with renorm s / (sum of the K selected
 *             s) (double, rounded to fp32).
 * The bias steers only the selection; the bias statistics are the per-expert
 * counts of valid routes (oracle_permute's group_sizes).
 */
static float sigmoid_f32(float l)
{
    return (float)(1.0 / (1.0 + exp(-(double)l)));
}

void oracle_route_sigmoid_topk(const float *logits, const float *bias, int T, int E, int K, int renorm,
                               int32_t *ids, float *probs)
{
    scored *row = (scored *)malloc(sizeof(scored) * (size_t)E);
    float *sc = (float *)malloc(sizeof(float) * (size_t)E);
    for (int t = 0; t < T; t++) {
        const float *l = logits + (size_t)t * E;
        for (int e = 0; e < E; e++) {
            sc[e] = sigmoid_f32(l[e]);
            volatile float key = sc[e] + (bias ? bias[e] : 0.0f);   /* one fp32 rounding */
            row[e].v = key;
            row[e].idx = e;
        }
        qsort(row, (size_t)E, sizeof(scored), cmp_scored);
        double denom = 0.0;
        for (int k = 0; k < K; k++)
            denom += (double)sc[row[k].idx];
        for (int k = 0; k < K; k++) {
            ids[(size_t)t * K + k] = row[k].idx;
            const double s = (double)sc[row[k].idx];
            probs[(size_t)t * K + k] = (float)(renorm ? s / denom : s);
        }
    }
    free(sc);
    free(row);
}

/*
 * Backward of oracle_route_sigmoid_topk's probabilities with respect to the
 * logits, selection held fixed (the derivative of the forward's formulas; the
 * pages name a router backward, [SPARSER] "The workload changes the
 * bottleneck", without giving it). Row t: S = the distinct valid ids, g[k] =
 * dprobs[t,k], G_e = sum of g[k] over k with ids[t,k] = e, s_e = sigmoid(l_e)
 * in double.
 *   without renorm:  dlogits[t,e] = G_e s_e (1 - s_e)                  (e in S)
 *   with renorm:     Z = sum over S of s_e, p_e = s_e / Z,
 *                    c = sum over valid k of g[k] p_{ids[t,k]},
 *                    dlogits[t,e] = s_e (1 - s_e) (G_e - c) / Z         (e in S)
 * and 0 for e outside S. The bias has no gradient path.
 */
void oracle_route_sigmoid_backward(const float *logits, const int32_t *ids, const float *dprobs,
                                   int T, int E, int K, int renorm, double *dlogits)
{
    double *G = (double *)malloc(sizeof(double) * (size_t)E);
    char *sel = (char *)malloc((size_t)E);
    for (int t = 0; t < T; t++) {
        const float *l = logits + (size_t)t * E;
        for (int e = 0; e < E; e++) {
            G[e] = 0.0;
            sel[e] = 0;
        }
        for (int k = 0; k < K; k++) {
            int e = ids[(size_t)t * K + k];
            if (e < 0 || e >= E)
                continue;
            sel[e] = 1;
            G[e] += (double)dprobs[(size_t)t * K + k];
        }
        double Z = 0.0;
        for (int e = 0; e < E; e++)
            if (sel[e])
                Z += 1.0 / (1.0 + exp(-(double)l[e]));
        double c = 0.0;
        for (int k = 0; k < K; k++) {
            int e = ids[(size_t)t * K + k];
            if (e < 0 || e >= E)
                continue;
            c += (double)dprobs[(size_t)t * K + k] * (1.0 / (1.0 + exp(-(double)l[e]))) / Z;
        }
        for (int e = 0; e < E; e++) {
            double d = 0.0;
            if (sel[e]) {
                const double s = 1.0 / (1.0 + exp(-(double)l[e]));
                d = renorm ? s * (1.0 - s) * (G[e] - c) / Z : G[e] * s * (1.0 - s);
            }
            dlogits[(size_t)t * E + e] = d;
        }
    }
    free(G);
    free(sel);
}

/* ------------------------------------------------------------------------ */
/* Permute (dispatch into expert-contiguous order)                           */
/* ------------------------------------------------------------------------ */

/*
 * Dropless permutation ([TEJAX] "Dropless vs capacity-based MoE": every
 * routed token is processed, no drop, no pad; figure: dispatch groups tokens
 * by expert, combine restores token order; [SPARSER] "Preserve a compact
 * route": -1 marks an invalid route, which is skipped).
 * Readings taken: a route (t,k) is valid iff 0 <= ids[t,k] < E (anything else,
 * -1 included, is skipped); within a group, rows are ordered by ascending
 * flattened route index t*K + k.
 * Outputs: group_sizes[E], group_offsets[E+1] (exclusive scan, offsets[E] = R),
 * row_map[T,K] (destination row or -1), perm_src[R] (source token of each
 * destination row), x_perm[R, H] (bitwise copies of x rows; x_perm may be NULL).
 * Returns R, the number of valid routes.
 */
long oracle_permute(const uint16_t *x, int T, int H, const int32_t *ids, int K, int E,
                    uint16_t *x_perm, int32_t *group_sizes, int32_t *group_offsets,
                    int32_t *row_map, int32_t *perm_src)
{
    for (int e = 0; e < E; e++)
        group_sizes[e] = 0;
    for (long i = 0; i < (long)T * K; i++)
        if (ids[i] >= 0 && ids[i] < E)
            group_sizes[ids[i]]++;
    group_offsets[0] = 0;
    for (int e = 0; e < E; e++)
        group_offsets[e + 1] = group_offsets[e] + group_sizes[e];
    int32_t *cursor = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (long i = 0; i < (long)T * K; i++) {
        int e = ids[i];
        if (e < 0 || e >= E) {
            row_map[i] = -1;
            continue;
        }
        long r = group_offsets[e] + cursor[e]++;
        long t = i / K;
        row_map[i] = (int32_t)r;
        perm_src[r] = (int32_t)t;
        if (x_perm)
            memcpy(x_perm + r * H, x + t * H, sizeof(uint16_t) * (size_t)H);
    }
    free(cursor);
    return group_offsets[E];
}

/* ------------------------------------------------------------------------ */
/* Unpermute / combine                                                      */
/* ------------------------------------------------------------------------ */

/*
 * Probability-weighted combine back to token order ([TEJAX] figure and
 * "Optimization 2": results are routed back and accumulated; [SPARSER]
 * "Remove work that has no selected route": combine with probabilities).
 * y[t,:] = bf16( sum over k ascending with row_map[t,k] >= 0 of
 *                probs[t,k] * y_perm[row_map[t,k], :] ), accumulated in double.
 * A token with no valid route gets zeros.
 */
void oracle_combine(const uint16_t *y_perm, const int32_t *row_map, const float *probs,
                    int T, int K, int H, uint16_t *y)
{
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    for (int t = 0; t < T; t++) {
        for (int j = 0; j < H; j++)
            acc[j] = 0.0;
        for (int k = 0; k < K; k++) {
            long r = row_map[(size_t)t * K + k];
            if (r < 0)
                continue;
            double p = (double)probs[(size_t)t * K + k];
            for (int j = 0; j < H; j++)
                acc[j] += p * oracle_bf16_to_double(y_perm[r * H + j]);
        }
        for (int j = 0; j < H; j++)
            y[(size_t)t * H + j] = oracle_double_to_bf16(acc[j]);
    }
    free(acc);
}

/* ------------------------------------------------------------------------ */
/* Backward of the router, the combine and the permute                       */
/* ------------------------------------------------------------------------ */

/*
 * Router backward. [SPARSER] "The workload changes the bottleneck" lists a
 * router backward among the Transformer Engine kernels and "Preserve a compact
 * route" extends the router work to forward and backward kernels; neither
 * defines it. Reading taken: the gradient of the forward's probabilities with
 * respect to the logits, the selection held fixed (top-K is piecewise
 * constant). For row t, with S the selected experts (ids[t,k] in [0, E); -1
 * and other ids are skipped), g[k] = dprobs[t,k] and G_e = sum of g[k] over
 * the k with ids[t,k] = e:
 *   softmax over all E:   p_e = exp(l_e - m) / sum_j exp(l_j - m),
 *                         dlogits[t,e] = p_e * (G_e - sum_{valid k} g[k] p_{ids[t,k]});
 *   renormalised over S:  q_e = exp(l_e - m) / sum_{j in S} exp(l_j - m) for e in S,
 *                         dlogits[t,e] = q_e * (G_e - sum_{valid k} g[k] q_{ids[t,k]}) on S,
 *                         0 off S.
 * (Each is J^T g for the softmax Jacobian d p_i / d l_j = p_i (delta_ij - p_j).)
 * m is the row maximum, as in the forward. dlogits is [T, E] doubles.
 */
void oracle_route_backward(const float *logits, const int32_t *ids, const float *dprobs,
                           int T, int E, int K, int renorm, double *dlogits)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    double *G = (double *)malloc(sizeof(double) * (size_t)E);
    char *sel = (char *)malloc((size_t)E);
    for (int t = 0; t < T; t++) {
        const float *l = logits + (size_t)t * E;
        for (int e = 0; e < E; e++) {
            G[e] = 0.0;
            sel[e] = 0;
        }
        for (int k = 0; k < K; k++) {
            int e = ids[(size_t)t * K + k];
            if (e < 0 || e >= E)
                continue;
            sel[e] = 1;
            G[e] += (double)dprobs[(size_t)t * K + k];
        }
        double m = (double)l[0];
        for (int e = 1; e < E; e++)
            if ((double)l[e] > m)
                m = (double)l[e];
        double denom = 0.0;
        for (int e = 0; e < E; e++)
            if (!renorm || sel[e])
                denom += exp((double)l[e] - m);
        for (int e = 0; e < E; e++)
            p[e] = (!renorm || sel[e]) ? exp((double)l[e] - m) / denom : 0.0;
        double s = 0.0;
        for (int k = 0; k < K; k++) {
            int e = ids[(size_t)t * K + k];
            if (e < 0 || e >= E)
                continue;
            s += (double)dprobs[(size_t)t * K + k] * p[e];
        }
        for (int e = 0; e < E; e++)
            dlogits[(size_t)t * E + e] = (renorm && !sel[e]) ? 0.0 : p[e] * (G[e] - s);
    }
    free(p);
    free(G);
    free(sel);
}

/*
 * Combine backward: the adjoint of oracle_combine. The pages give the forward
 * ([TEJAX] "Optimization 2": results routed back and accumulated in token
 * order; [SPARSER] "Remove work that has no selected route": combine with
 * probabilities); reading taken for the backward: the chain rule through
 * y[t] = sum_k p[t,k] y_perm[row_map[t,k]]:
 *   dy_perm[row_map[t,k]] = p[t,k] * dy[t]         (rounded once to bf16),
 *   dprobs[t,k] = sum_j dy[t,j] * y_perm[row_map[t,k], j]   (double),
 * for every valid route; an invalid route (row_map < 0) gets dprobs 0 and no
 * row. Rows of dy_perm that no route maps to are left as they are.
 */
void oracle_combine_backward(const uint16_t *dy, const uint16_t *y_perm, const int32_t *row_map,
                             const float *probs, int T, int K, int H, uint16_t *dy_perm,
                             double *dprobs)
{
    for (int t = 0; t < T; t++) {
        for (int k = 0; k < K; k++) {
            long r = row_map[(size_t)t * K + k];
            double d = 0.0;
            if (r >= 0) {
                double p = (double)probs[(size_t)t * K + k];
                for (int j = 0; j < H; j++) {
                    double g = oracle_bf16_to_double(dy[(size_t)t * H + j]);
                    d += g * oracle_bf16_to_double(y_perm[r * H + j]);
                    dy_perm[r * H + j] = oracle_double_to_bf16(p * g);
                }
            }
            dprobs[(size_t)t * K + k] = d;
        }
    }
}

/*
 * Permute backward: the adjoint of the permute's row copies (x_perm[row] =
 * x[t] for every valid route of t), i.e. dx[t] = sum over the valid k of
 * dx_perm[row_map[t,k]], accumulated in ascending k and rounded once to bf16
 * (the combine with every weight 1). Tokens without a valid route get 0.
 */
void oracle_permute_backward(const uint16_t *dx_perm, const int32_t *row_map, int T, int K, int H,
                             uint16_t *dx)
{
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    for (int t = 0; t < T; t++) {
        for (int j = 0; j < H; j++)
            acc[j] = 0.0;
        for (int k = 0; k < K; k++) {
            long r = row_map[(size_t)t * K + k];
            if (r < 0)
                continue;
            for (int j = 0; j < H; j++)
                acc[j] += oracle_bf16_to_double(dx_perm[r * H + j]);
        }
        for (int j = 0; j < H; j++)
            dx[(size_t)t * H + j] = oracle_double_to_bf16(acc[j]);
    }
    free(acc);
}

/* ------------------------------------------------------------------------ */
/* Grouped SwiGLU expert MLP                                                 */
/* ------------------------------------------------------------------------ */

/*
 * A 2-D operand view. Element (r, c) of a [rows, cols] row-major matrix of
 * kind MAT_BF16 (uint16 bits), MAT_F64 (double) or MAT_MXFP8 (E4M3 codes plus
 * E8M0 scales; blocks of 32 run along rows when blk_rows, i.e. scale
 * [rows/32, cols], else along columns, i.e. scale [rows, cols/32]).
 */
enum { MAT_BF16 = 0, MAT_F64 = 1, MAT_MXFP8 = 2 };

typedef struct {
    int kind;
    const void *v;
    const uint8_t *s;
    long rows, cols;
    int blk_rows;
} mat;

/* Row r of the matrix as doubles. */
static void mat_row(const mat *m, long r, double *out)
{
    long c;
    switch (m->kind) {
    case MAT_BF16: {
        const uint16_t *p = (const uint16_t *)m->v + r * m->cols;
        for (c = 0; c < m->cols; c++)
            out[c] = oracle_bf16_to_double(p[c]);
        break;
    }
    case MAT_F64:
        memcpy(out, (const double *)m->v + r * m->cols, sizeof(double) * (size_t)m->cols);
        break;
    default: {
        const uint8_t *p = (const uint8_t *)m->v + r * m->cols;
        for (c = 0; c < m->cols; c++) {
            uint8_t sb = m->blk_rows ? m->s[(r / 32) * m->cols + c] : m->s[r * (m->cols / 32) + c / 32];
            out[c] = mx_value(p[c], sb);
        }
    }
    }
}

/* Expert e's slice of a stacked [E, rows, cols] weight view. */
static mat expert_slice(const mat *w, int e)
{
    mat m = *w;
    long n = w->rows * w->cols;
    size_t esz = (w->kind == MAT_BF16) ? 2 : (w->kind == MAT_F64) ? 8 : 1;
    m.v = (const char *)w->v + (size_t)e * (size_t)n * esz;
    if (w->kind == MAT_MXFP8)
        m.s = w->s + (size_t)e * (size_t)(n / 32);
    return m;
}

static int expert_of_row(const int32_t *off, int E, long r)
{
    int lo = 0, hi = E - 1;            /* last e with off[e] <= r < off[e+1] */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (off[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    while (lo < E - 1 && off[lo + 1] <= r)
        lo++;
    return lo;
}

static double silu(double a) { return a / (1.0 + exp(-a)); }

/* The SwiGLU step of one element: h = silu(a) * b. */
static double swiglu_value(double a, double b) { return silu(a) * b; }

/* Its derivatives at (a, b) applied to dh (the chain rule of the line above):
 *   da = dh * b * silu'(a),  silu'(a) = s(a) (1 + a (1 - s(a))),  s = logistic
 *   db = dh * silu(a) */
static void swiglu_grad(double dh, double a, double b, double *da, double *db)
{
    double sg = 1.0 / (1.0 + exp(-a));
    *da = dh * b * (sg * (1.0 + a * (1.0 - sg)));
    *db = dh * silu(a);
}

/* Rounding applied to the intermediate h before the second GEMM. */
enum { H_NONE = 0, H_BF16 = 1, H_MXFP8 = 2 };

/*
 * Grouped SwiGLU MLP on the listed rows of the permuted activations
 * ([TEJAX] "Optimization 1: Grouped GEMM": every expert with its actual token
 * count, only valid regions computed; figure: the grouped MLP is two grouped
 * GEMMs on variable-length groups). For a row r of group e:
 *   a[f] = sum_h x[r,h] W1[e][h,f],  b[f] = sum_h x[r,h] W3[e][h,f]
 *   h[f] = silu(a[f]) * b[f],        silu(a) = a / (1 + exp(-a))
 *   y[r,j] = sum_f round_h(h)[f] W2[e][f,j]
 * Readings taken: silu gates the W1 product and W3 is the linear branch;
 * round_h is none (h_mode 0), bf16 (1) or MXFP8 1x32 along F (2), applied to
 * the unrounded h. Operand kinds: x [R_cap, H], W1/W3 [E][H, F], W2 [E][F, H]
 * (weights in MXFP8 carry blocks along their contraction dimension).
 * Outputs for row list entry i: y_bf16[i, H] (if not NULL), y_f64[i, H] (if not
 * NULL, unrounded), h_bf16[i, F] (if not NULL), h_q[i, F] + h_s[i, F/32]
 * (MXFP8 mode, if not NULL), h_f64[i, F] (if not NULL, unrounded),
 * a_f64[i, F] and b_f64[i, F] (if not NULL: the two pre-activations).
 */
void oracle_swiglu_rows(int x_kind, const void *x_v, const uint8_t *x_s,
                        int w_kind, const void *w1_v, const uint8_t *w1_s,
                        const void *w3_v, const uint8_t *w3_s,
                        const void *w2_v, const uint8_t *w2_s,
                        const int32_t *group_offsets, int E, int H, int F, long R_cap,
                        const int32_t *rows, long nrows, int h_mode,
                        uint16_t *y_bf16, double *y_f64, uint16_t *h_bf16,
                        uint8_t *h_q, uint8_t *h_s, double *h_f64,
                        double *a_f64, double *b_f64)
{
    mat X = {x_kind, x_v, x_s, R_cap, H, 0};
    mat W1 = {w_kind, w1_v, w1_s, H, F, 1};
    mat W3 = {w_kind, w3_v, w3_s, H, F, 1};
    mat W2 = {w_kind, w2_v, w2_s, F, H, 1};
    double *xr = malloc(sizeof(double) * H), *a = malloc(sizeof(double) * F);
    double *b = malloc(sizeof(double) * F), *hv = malloc(sizeof(double) * F);
    double *wr = malloc(sizeof(double) * (F > H ? F : H)), *wr3 = malloc(sizeof(double) * F);
    double *y = malloc(sizeof(double) * H);
    uint8_t *qb = malloc((size_t)F), *sbuf = malloc((size_t)F / 32 + 1);
    for (long i = 0; i < nrows; i++) {
        long r = rows[i];
        int e = expert_of_row(group_offsets, E, r);
        mat w1 = expert_slice(&W1, e), w3 = expert_slice(&W3, e), w2 = expert_slice(&W2, e);
        mat_row(&X, r, xr);
        for (int f = 0; f < F; f++)
            a[f] = b[f] = 0.0;
        for (int h = 0; h < H; h++) {
            mat_row(&w1, h, wr);
            mat_row(&w3, h, wr3);
            for (int f = 0; f < F; f++) {
                a[f] += xr[h] * wr[f];
                b[f] += xr[h] * wr3[f];
            }
        }
        for (int f = 0; f < F; f++)
            hv[f] = swiglu_value(a[f], b[f]);
        if (a_f64)
            memcpy(a_f64 + i * F, a, sizeof(double) * F);
        if (b_f64)
            memcpy(b_f64 + i * F, b, sizeof(double) * F);
        if (h_f64)
            memcpy(h_f64 + i * F, hv, sizeof(double) * F);
        if (h_mode == H_BF16) {
            for (int f = 0; f < F; f++) {
                uint16_t hb = oracle_double_to_bf16(hv[f]);
                if (h_bf16)
                    h_bf16[i * F + f] = hb;
                hv[f] = oracle_bf16_to_double(hb);
            }
        } else if (h_mode == H_MXFP8) {
            for (int blk = 0; blk < F / 32; blk++)
                sbuf[blk] = (uint8_t)quant_block(hv + 32 * blk, 1, 32, qb + 32 * blk, 1);
            for (int f = 0; f < F; f++)
                hv[f] = mx_value(qb[f], sbuf[f / 32]);
            if (h_q)
                memcpy(h_q + i * F, qb, (size_t)F);
            if (h_s)
                memcpy(h_s + i * (F / 32), sbuf, (size_t)F / 32);
        }
        for (int j = 0; j < H; j++)
            y[j] = 0.0;
        for (int f = 0; f < F; f++) {
            mat_row(&w2, f, wr);
            for (int j = 0; j < H; j++)
                y[j] += hv[f] * wr[j];
        }
        for (int j = 0; j < H; j++) {
            if (y_bf16)
                y_bf16[i * H + j] = oracle_double_to_bf16(y[j]);
            if (y_f64)
                y_f64[i * H + j] = y[j];
        }
    }
    free(xr); free(a); free(b); free(hv); free(wr); free(wr3); free(y); free(qb); free(sbuf);
}

/*
 * Backward of the grouped SwiGLU MLP, activation gradient (dgrad), for the
 * listed rows. Given the forward pre-activations a, b of each row (as the
 * forward computed them, see oracle_swiglu_rows' a_f64 / b_f64 outputs):
 *   dh[f] = sum_j dy[r,j] W2[e][f,j]
 *   da[f] = dh[f] * b[f] * silu'(a[f]),   silu'(a) = s(a) (1 + a (1 - s(a))), s = logistic
 *   db[f] = dh[f] * silu(a[f])
 *   dx[r,h] = sum_f da[f] W1[e][h,f] + db[f] W3[e][h,f]
 * Operand views: dy [R_cap, H], a and b [R_cap, F] (bf16 or f64), weights as in
 * the forward; for MXFP8 weights w_blk_rows says along which dimension of the
 * stored [H,F] / [F,H] matrices the 32-blocks run (the backward contracts
 * W2 over its columns and W1, W3 over their columns, so a caller quantising for
 * the backward passes column blocks, w_blk_rows = 0).
 * dab_mode says how da, db are rounded before the second product (the dx GEMM
 * reads them as an operand): 0 = not at all, 1 = to bf16, 2 = to bf16 and then
 * MXFP8 1x32 along F (blocks never mix da and db). Reading taken: the backward
 * stores da, db as a bf16 operand (and quantises that operand for MXFP8).
 * Outputs per listed row (each optional): dx_bf16 / dx_f64 [H], da_f64 / db_f64 [F]
 * (unrounded).
 */
void oracle_swiglu_dgrad_rows(int dy_kind, const void *dy_v, const uint8_t *dy_s,
                              int ab_kind, const void *a_v, const void *b_v,
                              int w_kind, int w_blk_rows,
                              const void *w1_v, const uint8_t *w1_s,
                              const void *w3_v, const uint8_t *w3_s,
                              const void *w2_v, const uint8_t *w2_s,
                              const int32_t *group_offsets, int E, int H, int F, long R_cap,
                              const int32_t *rows, long nrows, int dab_mode,
                              uint16_t *dx_bf16, double *dx_f64, double *da_f64, double *db_f64)
{
    mat DY = {dy_kind, dy_v, dy_s, R_cap, H, 0};
    mat A = {ab_kind, a_v, NULL, R_cap, F, 0};
    mat B = {ab_kind, b_v, NULL, R_cap, F, 0};
    mat W1 = {w_kind, w1_v, w1_s, H, F, w_blk_rows};
    mat W3 = {w_kind, w3_v, w3_s, H, F, w_blk_rows};
    mat W2 = {w_kind, w2_v, w2_s, F, H, w_blk_rows};
    double *dyr = malloc(sizeof(double) * H);
    double *a = malloc(sizeof(double) * F), *b = malloc(sizeof(double) * F);
    double *dh = malloc(sizeof(double) * F), *da = malloc(sizeof(double) * F);
    double *db = malloc(sizeof(double) * F), *dx = malloc(sizeof(double) * H);
    double *wr = malloc(sizeof(double) * (F > H ? F : H)), *wr3 = malloc(sizeof(double) * F);
    for (long i = 0; i < nrows; i++) {
        long r = rows[i];
        int e = expert_of_row(group_offsets, E, r);
        mat w1 = expert_slice(&W1, e), w3 = expert_slice(&W3, e), w2 = expert_slice(&W2, e);
        mat_row(&DY, r, dyr);
        mat_row(&A, r, a);
        mat_row(&B, r, b);
        for (int f = 0; f < F; f++) {
            mat_row(&w2, f, wr);
            double acc = 0.0;
            for (int j = 0; j < H; j++)
                acc += dyr[j] * wr[j];
            dh[f] = acc;
        }
        for (int f = 0; f < F; f++)
            swiglu_grad(dh[f], a[f], b[f], &da[f], &db[f]);
        if (da_f64)
            memcpy(da_f64 + i * F, da, sizeof(double) * F);
        if (db_f64)
            memcpy(db_f64 + i * F, db, sizeof(double) * F);
        if (dab_mode >= 1) {
            for (int f = 0; f < F; f++) {
                da[f] = oracle_bf16_to_double(oracle_double_to_bf16(da[f]));
                db[f] = oracle_bf16_to_double(oracle_double_to_bf16(db[f]));
            }
        }
        if (dab_mode == 2) {
            double *v[2] = {da, db};
            for (int w = 0; w < 2; w++)
                for (int blk = 0; blk < F / 32; blk++) {
                    uint8_t q[32];
                    int sb = quant_block(v[w] + 32 * blk, 1, 32, q, 1);
                    for (int j = 0; j < 32; j++)
                        v[w][32 * blk + j] = mx_value(q[j], (uint8_t)sb);
                }
        }
        for (int h = 0; h < H; h++) {
            mat_row(&w1, h, wr);
            mat_row(&w3, h, wr3);
            double acc = 0.0;
            for (int f = 0; f < F; f++)
                acc += da[f] * wr[f] + db[f] * wr3[f];
            dx[h] = acc;
        }
        for (int h = 0; h < H; h++) {
            if (dx_bf16)
                dx_bf16[i * H + h] = oracle_double_to_bf16(dx[h]);
            if (dx_f64)
                dx_f64[i * H + h] = dx[h];
        }
    }
    free(dyr); free(a); free(b); free(dh); free(da); free(db); free(dx);
    free(wr); free(wr3);
}

/*
 * Weight gradient (wgrad) of one expert, contraction over the rows of its
 * group (a ragged contraction length m_e = off[e+1] - off[e]):
 *   dW[c1, c2] = sum_{r in group e} A[r, c1] * B[r, c2]
 * for the listed output columns c2 only (all c1). With A = h, B = dy this is
 * dW2[e]; with A = x, B = da (or db) it is dW1[e] (or dW3[e]).
 * A [R_cap, n1] and B [R_cap, n2] are operand views (MXFP8 views carry
 * group-aware column-wise scales, see oracle_quant_cols_grouped_bf16).
 * Output dw_f64[n1, ncols] (column i of the output is c2 = cols[i]).
 */
void oracle_wgrad_expert(int a_kind, const void *a_v, const uint8_t *a_s, long n1,
                         int b_kind, const void *b_v, const uint8_t *b_s, long n2,
                         const int32_t *group_offsets, int E, int e, long R_cap,
                         const int32_t *cols, long ncols, double *dw_f64)
{
    long r0 = group_offsets[e], r1 = group_offsets[e + 1];
    double *ar = malloc(sizeof(double) * n1), *br = malloc(sizeof(double) * n2);
    for (long i = 0; i < n1 * ncols; i++)
        dw_f64[i] = 0.0;
    for (long r = r0; r < r1; r++) {
        /* group-aware column-wise MXFP8 views: scale row for r is
         * e + off[e]/32 + (r - off[e])/32 (see oracle_quant_cols_grouped_bf16) */
        long srow = e + r0 / 32 + (r - r0) / 32;
        if (a_kind == MAT_MXFP8) {
            for (long c = 0; c < n1; c++)
                ar[c] = mx_value(((const uint8_t *)a_v)[r * n1 + c], a_s[srow * n1 + c]);
        } else {
            mat A = {a_kind, a_v, NULL, R_cap, n1, 0};
            mat_row(&A, r, ar);
        }
        if (b_kind == MAT_MXFP8) {
            for (long c = 0; c < n2; c++)
                br[c] = mx_value(((const uint8_t *)b_v)[r * n2 + c], b_s[srow * n2 + c]);
        } else {
            mat B = {b_kind, b_v, NULL, R_cap, n2, 0};
            mat_row(&B, r, br);
        }
        for (long c1 = 0; c1 < n1; c1++)
            for (long i = 0; i < ncols; i++)
                dw_f64[c1 * ncols + i] += ar[c1] * br[cols[i]];
    }
    free(ar);
    free(br);
    (void)E;
}

/* Expert of a permuted row (exported for the tests' sampling helpers). */
int oracle_expert_of_row(const int32_t *group_offsets, int E, long r)
{
    return expert_of_row(group_offsets, E, r);
}

/* ------------------------------------------------------------------------ */
/* Element-wise array forms (for checks that take whole experts at once)     */
/* ------------------------------------------------------------------------ */

/* out[i] = bf16 bits of v[i] (oracle_double_to_bf16 per element). */
void oracle_double_to_bf16_n(const double *v, long n, uint16_t *out)
{
    for (long i = 0; i < n; i++)
        out[i] = oracle_double_to_bf16(v[i]);
}

/* h[i] = silu(a[i]) * b[i] (the SwiGLU step of oracle_swiglu_rows). */
void oracle_swiglu_n(const double *a, const double *b, long n, double *h)
{
    for (long i = 0; i < n; i++)
        h[i] = swiglu_value(a[i], b[i]);
}

/* da[i], db[i] from dh[i], a[i], b[i] (the SwiGLU backward step of
 * oracle_swiglu_dgrad_rows). */
void oracle_swiglu_grad_n(const double *dh, const double *a, const double *b, long n,
                          double *da, double *db)
{
    for (long i = 0; i < n; i++)
        swiglu_grad(dh[i], a[i], b[i], &da[i], &db[i]);
}

/* Row-wise 1x32 MXFP8 quantisation of a double matrix [rows, cols] (cols % 32 == 0):
 * the rule of oracle_quant_rows_bf16 applied to unrounded values (MXFP8 h is quantised
 * from its unrounded value). */
void oracle_quant_rows_f64(const double *x, long rows, long cols, uint8_t *q, uint8_t *s)
{
    for (long r = 0; r < rows; r++)
        for (long b = 0; b < cols / 32; b++)
            s[r * (cols / 32) + b] =
                (uint8_t)quant_block(x + r * cols + b * 32, 1, 32, q + r * cols + b * 32, 1);
}

/* ------------------------------------------------------------------------ */
/* Expert parallelism: the receiving side's expert of each received row      */
/* ------------------------------------------------------------------------ */

/*
 * Expert-parallel dispatch ([TEJAX] "Optimization 2: Expert parallelism to
 * fuse Dispatch and Combine"; [SPARSER] "Remove work that has no selected
 * route": only the selected routes travel, each destination receives the rows
 * of its own experts). With G ranks and E_loc experts per rank, rank g owning
 * experts g*E_loc .. g*E_loc + E_loc - 1, every source rank sends the rows of
 * its expert-contiguous permuted order that belong to the destination's
 * experts; the destination receives them source rank by source rank, and
 * within a source expert by expert, in the source's order.
 * counts[s][j] = rows received from source s for local expert j. Received row
 * r belongs to local expert j of the segment (s, j) that contains it (the
 * segments laid end to end in that order); rows past the last segment, up to
 * R_cap, get -1 (no route).
 */
void oracle_ep_recv_expert_ids(const int32_t *counts, int G, int E_loc, long R_cap, int32_t *ids)
{
    long r = 0;
    for (int s = 0; s < G; s++)
        for (int j = 0; j < E_loc; j++)
            for (long i = 0; i < counts[(long)s * E_loc + j] && r < R_cap; i++)
                ids[r++] = j;
    for (; r < R_cap; r++)
        ids[r] = -1;
}
