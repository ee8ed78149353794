/*
 * oracle.c -- plain, slow, fp64 CPU reference for the block-quantized decode
 * matvec y = W.x (NVFP4 and Q8_0 weights) and its top-k routed MoE variant.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library's product path may include,
 * link, load or call this file. Only the test suite, the package smoke check
 * and the benchmark's CPU-baseline leg use it. It shares no code, header,
 * table or constant with the CUDA kernels.
 *
 * Sources of what is computed:
 *  - "Vemloir/LumenLLM" README, Quantization bullet: weights stored natively
 *    in NVFP4, a 4-bit floating point format with block scales; Kernels bullet:
 *    decode runs warp-shuffle GEMVs.
 *  - "robertbfuentes7-cloud/bw24" README, feature list: NVFP4 (W4) decode path
 *    (block-scaled FP4 matvec); MoE bullet: expert-major batching of routed
 *    tokens with experts decoded once; speculative bullet: K+1 tokens verified
 *    in one batched target forward (N = K+1 columns).
 *  - "avifenesh/memra" README, Decode kernels bullet: NVFP4 / Q4_0 / Q8_0
 *    matvecs; "robertbfuentes7-cloud/bw24" README, GGUF bullet: files mix
 *    BF16, Q8_0, Q4_0, Q4_1 and the K-quants.
 *  - "Vemloir/LumenLLM" README, Quantization bullet: FP8 (E4M3) weights
 *    beside NVFP4; "avifenesh/memra" README, Loaders bullet: FP8 checkpoints
 *    quantised in blocks of 128 (one scale per 128 x 128 tile of the weight,
 *    the scale multiplying the E4M3 value).
 *  The pages never print the bit layouts. The element formats are the public
 *  closed forms: E2M1 and E4M3 from the OCP Microscaling (MX) v1.0 and OCP
 *  8-bit Floating Point v1.0 specifications, binary16 from IEEE 754-2008,
 *  bfloat16 as the upper half of an IEEE binary32. The block structure (16 k
 *  per E4M3 scale plus one FP32 tensor scale; 32 k per fp16 scale for Q8_0;
 *  low nibble = lower k) is the workload definition of the method.
 *
 * Every value is decoded from its bits by the closed form, products and sums
 * are taken in fp64 in plain index order, with no blocking or reordering.
 *
 * Parity status: every function below is pinned by the CPU test suite
 * (enumeration against library decoders or the published value tables,
 * hand-computed worked examples, exact-rational brute force, invariants).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* ------------------------------------------------------------ element decoders */

/* E2M1 (OCP MX v1.0, FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 * mantissa. Exponent 0 is subnormal: 0.5 * m. No inf or NaN. */
double oracle_e2m1(uint8_t code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag;
    if (e == 0)
        mag = 0.5 * m;
    else
        mag = ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (OCP 8-bit FP v1.0, "E4M3FN"): bit 7 sign, bits 6..3 exponent (bias 7),
 * bits 2..0 mantissa. Exponent 0 is subnormal: 2^-6 * m/8. The codes with all
 * exponent and mantissa bits set are NaN; there are no infinities. */
double oracle_e4m3(uint8_t b)
{
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp(m / 8.0, -6);
    else
        mag = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_fp16(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double mag;
    if (e == 31)
        mag = f ? NAN : INFINITY;
    else if (e == 0)
        mag = ldexp(f / 1024.0, -14);
    else
        mag = ldexp(1.0 + f / 1024.0, e - 15);
    return s ? -mag : mag;
}

/* bfloat16: the upper 16 bits of an IEEE binary32, i.e. 1 sign, 8 exponent
 * (bias 127), 7 fraction bits. */
double oracle_bf16(uint16_t b)
{
    int s = (b >> 15) & 1;
    int e = (b >> 7) & 255;
    int f = b & 127;
    double mag;
    if (e == 255)
        mag = f ? NAN : INFINITY;
    else if (e == 0)
        mag = ldexp(f / 128.0, -126);
    else
        mag = ldexp(1.0 + f / 128.0, e - 127);
    return s ? -mag : mag;
}

/* ------------------------------------------------------------ weight elements */

/* E2M1 code of element (m, k) of an NVFP4 weight whose codes plane is
 * u8[M][K/2], two codes per byte, the low nibble holding the even k. */
static uint8_t nvfp4_code(const uint8_t *codes, int64_t K, int64_t m, int64_t k)
{
    uint8_t byte = codes[m * (K / 2) + k / 2];
    return (k % 2 == 0) ? (uint8_t)(byte & 0x0F) : (uint8_t)(byte >> 4);
}

/* Real value of NVFP4 element (m, k) without the tensor scale:
 * e2m1(code) * e4m3(scale of block k/16). Exact in fp64. */
static double nvfp4_elem(const uint8_t *codes, const uint8_t *scales, int64_t K,
                         int64_t m, int64_t k)
{
    double v = oracle_e2m1(nvfp4_code(codes, K, m, k));
    double s = oracle_e4m3(scales[m * (K / 16) + k / 16]);
    return v * s;
}

/* Real value of Q8_0 element (m, k): fp16(d of block k/32) * q. */
static double q8_0_elem(const int8_t *q, const uint16_t *d, int64_t K, int64_t m, int64_t k)
{
    return oracle_fp16(d[m * (K / 32) + k / 32]) * (double)q[m * K + k];
}

/* Q4_0 element (m, k): fp16(d of block k/32) * (q - 8), q the 4-bit code
 * of element j = k % 32 of the block: the low nibble of the block's code
 * byte j for j < 16, the high nibble of byte j - 16 otherwise (the order of
 * a GGUF Q4_0 block, whose two fields are the two planes here). */
static int q4_0_code(const uint8_t *codes, int64_t K, int64_t m, int64_t k)
{
    int64_t j = k % 32;
    uint8_t byte = codes[m * (K / 2) + (k / 32) * 16 + (j % 16)];
    return j < 16 ? (byte & 0x0F) : (byte >> 4);
}

static double q4_0_elem(const uint8_t *codes, const uint16_t *d, int64_t K, int64_t m, int64_t k)
{
    return oracle_fp16(d[m * (K / 32) + k / 32]) * (double)(q4_0_code(codes, K, m, k) - 8);
}

/* Q4_1 element (m, k): fp16(d) * q + fp16(m) of the element's 32-block, q
 * its 4-bit code in the Q4_0 block order (low nibbles of the block's 16
 * bytes are elements 0..15, the high nibbles elements 16..31); d and m are
 * the block's two fp16 fields, stored side by side: dm[m][k/32] = (d, m).
 * Exact in fp64 (at most 44 bits between the two terms' extreme bits). */
static double q4_1_elem(const uint8_t *codes, const uint16_t *dm, int64_t K, int64_t m, int64_t k)
{
    const uint16_t *f = dm + (m * (K / 32) + k / 32) * 2;
    return oracle_fp16(f[0]) * (double)q4_0_code(codes, K, m, k) + oracle_fp16(f[1]);
}

/* FP8 block-128 element (m, k): e4m3(code[m][k]) * scale of the 128 x 128
 * tile holding (m, k); scales are fp32 [ceil(M/128)][ceil(K/128)] row-major,
 * so rows 0..127 share scale row 0 and k 0..127 scale column 0. */
static double fp8_b128_elem(const uint8_t *codes, const float *scales, int64_t K, int64_t m, int64_t k)
{
    int64_t kb = (K + 127) / 128;
    return oracle_e4m3(codes[m * K + k]) * (double)scales[(m / 128) * kb + k / 128];
}

/* ------------------------------------------------------------ dequantisation */

/* w[m][k] = e2m1 * e4m3 * ts as a real number (fp64, exact: at most 30
 * significant bits). */
void oracle_nvfp4_dequant_f64(const uint8_t *codes, const uint8_t *scales, float ts,
                              int64_t M, int64_t K, double *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = nvfp4_elem(codes, scales, K, m, k) * (double)ts;
}

/* The dequantised weight as fp32: the exact value rounded once to nearest. */
void oracle_nvfp4_dequant_f32(const uint8_t *codes, const uint8_t *scales, float ts,
                              int64_t M, int64_t K, float *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = (float)(nvfp4_elem(codes, scales, K, m, k) * (double)ts);
}

/* Q8_0 dequantised weight, fp64 (exact) and fp32 (exact too: 11 + 8 bits). */
void oracle_q8_0_dequant_f64(const int8_t *q, const uint16_t *d, int64_t M, int64_t K, double *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = q8_0_elem(q, d, K, m, k);
}

void oracle_q8_0_dequant_f32(const int8_t *q, const uint16_t *d, int64_t M, int64_t K, float *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = (float)q8_0_elem(q, d, K, m, k);
}

/* Q4_0 dequantised weight, fp64 and fp32 (both exact: 11 + 4 bits). */
void oracle_q4_0_dequant_f64(const uint8_t *codes, const uint16_t *d, int64_t M, int64_t K, double *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = q4_0_elem(codes, d, K, m, k);
}

void oracle_q4_0_dequant_f32(const uint8_t *codes, const uint16_t *d, int64_t M, int64_t K, float *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = (float)q4_0_elem(codes, d, K, m, k);
}

/* Q4_1 dequantised weight, fp64 (exact) and fp32 (rounded once). */
void oracle_q4_1_dequant_f64(const uint8_t *codes, const uint16_t *dm, int64_t M, int64_t K, double *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = q4_1_elem(codes, dm, K, m, k);
}

void oracle_q4_1_dequant_f32(const uint8_t *codes, const uint16_t *dm, int64_t M, int64_t K, float *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = (float)q4_1_elem(codes, dm, K, m, k);
}

/* FP8 block-128 dequantised weight: fp64 exact (4 + 24 significant bits);
 * fp32 the exact value rounded once to nearest. */
void oracle_fp8_b128_dequant_f64(const uint8_t *codes, const float *scales, int64_t M, int64_t K, double *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = fp8_b128_elem(codes, scales, K, m, k);
}

void oracle_fp8_b128_dequant_f32(const uint8_t *codes, const float *scales, int64_t M, int64_t K, float *w)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            w[m * K + k] = (float)fp8_b128_elem(codes, scales, K, m, k);
}

/* ------------------------------------------------------------ GEMV */

/*
 * y[n][i] = sum_k W[m][k] * x[n][k] for m = rows[i] (all rows when rows is
 * NULL, then i = m), x given as bf16 bits [N][K]. Accumulated in fp64 in k
 * order. a[n][i] = sum_k |W[m][k] * x[n][k]|, the scale of the tolerance.
 * Output arrays are [N][nrows] with nrows = M when rows is NULL.
 */
void oracle_nvfp4_gemv(const uint8_t *codes, const uint8_t *scales, float ts,
                       const uint16_t *x, int64_t M, int64_t K, int64_t N,
                       const int64_t *rows, int64_t nrows, double *y, double *a)
{
    int64_t R = rows ? nrows : M;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t i = 0; i < R; ++i) {
            int64_t m = rows ? rows[i] : i;
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = nvfp4_elem(codes, scales, K, m, k) * (double)ts;
                double p = w * oracle_bf16(x[n * K + k]);
                sum += p;
                abs_sum += fabs(p);
            }
            y[n * R + i] = sum;
            if (a)
                a[n * R + i] = abs_sum;
        }
    }
}

void oracle_q8_0_gemv(const int8_t *q, const uint16_t *d, const uint16_t *x,
                      int64_t M, int64_t K, int64_t N,
                      const int64_t *rows, int64_t nrows, double *y, double *a)
{
    int64_t R = rows ? nrows : M;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t i = 0; i < R; ++i) {
            int64_t m = rows ? rows[i] : i;
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = q8_0_elem(q, d, K, m, k) * oracle_bf16(x[n * K + k]);
                sum += p;
                abs_sum += fabs(p);
            }
            y[n * R + i] = sum;
            if (a)
                a[n * R + i] = abs_sum;
        }
    }
}

void oracle_q4_0_gemv(const uint8_t *codes, const uint16_t *d, const uint16_t *x,
                      int64_t M, int64_t K, int64_t N,
                      const int64_t *rows, int64_t nrows, double *y, double *a)
{
    int64_t R = rows ? nrows : M;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t i = 0; i < R; ++i) {
            int64_t m = rows ? rows[i] : i;
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = q4_0_elem(codes, d, K, m, k) * oracle_bf16(x[n * K + k]);
                sum += p;
                abs_sum += fabs(p);
            }
            y[n * R + i] = sum;
            if (a)
                a[n * R + i] = abs_sum;
        }
    }
}

void oracle_q4_1_gemv(const uint8_t *codes, const uint16_t *dm, const uint16_t *x,
                      int64_t M, int64_t K, int64_t N,
                      const int64_t *rows, int64_t nrows, double *y, double *a)
{
    int64_t R = rows ? nrows : M;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t i = 0; i < R; ++i) {
            int64_t m = rows ? rows[i] : i;
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = q4_1_elem(codes, dm, K, m, k) * oracle_bf16(x[n * K + k]);
                sum += p;
                abs_sum += fabs(p);
            }
            y[n * R + i] = sum;
            if (a)
                a[n * R + i] = abs_sum;
        }
    }
}

void oracle_fp8_b128_gemv(const uint8_t *codes, const float *scales, const uint16_t *x,
                          int64_t M, int64_t K, int64_t N,
                          const int64_t *rows, int64_t nrows, double *y, double *a)
{
    int64_t R = rows ? nrows : M;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t i = 0; i < R; ++i) {
            int64_t m = rows ? rows[i] : i;
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = fp8_b128_elem(codes, scales, K, m, k) * oracle_bf16(x[n * K + k]);
                sum += p;
                abs_sum += fabs(p);
            }
            y[n * R + i] = sum;
            if (a)
                a[n * R + i] = abs_sum;
        }
    }
}

/* As oracle_nvfp4_gemv, with the activations given as fp64 values [N][K]
 * instead of bf16 bits (used to recompute a down projection from a given h). */
void oracle_nvfp4_gemv_f64x(const uint8_t *codes, const uint8_t *scales, float ts,
                            const double *x, int64_t M, int64_t K, int64_t N,
                            double *y, double *a)
{
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double sum = 0.0, abs_sum = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = nvfp4_elem(codes, scales, K, m, k) * (double)ts * x[n * K + k];
                sum += p;
                abs_sum += fabs(p);
            }
            y[n * M + m] = sum;
            if (a)
                a[n * M + m] = abs_sum;
        }
    }
}

/* ------------------------------------------------------------ MoE */

/*
 * Router of one MoE layer ("robertbfuentes7-cloud/bw24" README, MoE bullet;
 * the routing rule is the workload's: softmax over the E logits, keep the
 * topk largest, renormalise them to sum to one).
 * sel_expert[t][s] is the expert of slot s of token t, slots in decreasing
 * order of probability; equal logits rank the lower expert index first.
 * Selection compares the given fp32 logits themselves (softmax is monotone).
 * sel_weight[t][s] = p_sel / sum of the topk selected p, in fp64.
 * Requires topk <= E.
 */
void oracle_moe_route(const float *logits, int64_t T, int64_t E, int64_t topk,
                      int32_t *sel_expert, double *sel_weight)
{
    char *taken = (char *)malloc((size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        /* softmax over all E experts */
        double lmax = -INFINITY;
        for (int64_t e = 0; e < E; ++e)
            if ((double)l[e] > lmax)
                lmax = (double)l[e];
        double z = 0.0;
        for (int64_t e = 0; e < E; ++e) {
            p[e] = exp((double)l[e] - lmax);
            z += p[e];
        }
        for (int64_t e = 0; e < E; ++e)
            p[e] /= z;
        /* top-k by repeated selection of the largest remaining logit */
        for (int64_t e = 0; e < E; ++e)
            taken[e] = 0;
        double psum = 0.0;
        for (int64_t s = 0; s < topk; ++s) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e; /* strict '>' keeps the lower index on ties */
            }
            taken[best] = 1;
            sel_expert[t * topk + s] = (int32_t)best;
            sel_weight[t * topk + s] = p[best];
            psum += p[best];
        }
        /* renormalise over the selected experts */
        for (int64_t s = 0; s < topk; ++s)
            sel_weight[t * topk + s] /= psum;
    }
    free(p);
    free(taken);
}

/*
 * One routed MoE FFN layer for T tokens, given the routing (sel_expert,
 * sel_weight as from oracle_moe_route or any other source).
 *   gate_up[e] is NVFP4 [2I][H] (rows 0..I-1 gate, I..2I-1 up), scale gu_ts[e];
 *   down[e]    is NVFP4 [H][I], scale dn_ts[e].
 * For token t and slot s with expert e:
 *   g_i = sum_k gate_up[e][i][k] x_t[k],  u_i = sum_k gate_up[e][I+i][k] x_t[k]
 *   h_i = SiLU(g_i) * u_i = g_i / (1 + exp(-g_i)) * u_i
 *   d_j = sum_i down[e][j][i] h_i
 *   y_t[j] = sum_s w_{t,s} d_j   (slots added in order s = 0..topk-1)
 * Optional outputs (any may be NULL), all fp64, indexed [t][s][...]:
 *   g, u, h: [T][topk][I]; ag, au: sum_k |w x| of g and u; d: [T][topk][H];
 *   ad: sum_i |down[e][j][i] h_i|.
 */
void oracle_moe_layer(const uint8_t *gu_codes, const uint8_t *gu_scales, const float *gu_ts,
                      const uint8_t *dn_codes, const uint8_t *dn_scales, const float *dn_ts,
                      const uint16_t *x, const int32_t *sel_expert, const double *sel_weight,
                      int64_t T, int64_t H, int64_t I, int64_t topk,
                      double *y, double *g_out, double *u_out, double *h_out,
                      double *ag_out, double *au_out, double *d_out, double *ad_out)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    const int64_t gu_codes_per_e = 2 * I * (H / 2), gu_scales_per_e = 2 * I * (H / 16);
    const int64_t dn_codes_per_e = H * (I / 2), dn_scales_per_e = H * (I / 16);
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t j = 0; j < H; ++j)
            y[t * H + j] = 0.0;
        for (int64_t s = 0; s < topk; ++s) {
            int64_t e = sel_expert[t * topk + s];
            double wsel = sel_weight[t * topk + s];
            const uint8_t *gc = gu_codes + e * gu_codes_per_e;
            const uint8_t *gs = gu_scales + e * gu_scales_per_e;
            const uint8_t *dc = dn_codes + e * dn_codes_per_e;
            const uint8_t *ds = dn_scales + e * dn_scales_per_e;
            int64_t base = (t * topk + s) * I;
            for (int64_t i = 0; i < I; ++i) {
                double sg = 0.0, su = 0.0, ag = 0.0, au = 0.0;
                for (int64_t k = 0; k < H; ++k) {
                    double xv = oracle_bf16(x[t * H + k]);
                    double pg = nvfp4_elem(gc, gs, H, i, k) * (double)gu_ts[e] * xv;
                    double pu = nvfp4_elem(gc, gs, H, I + i, k) * (double)gu_ts[e] * xv;
                    sg += pg;
                    su += pu;
                    ag += fabs(pg);
                    au += fabs(pu);
                }
                g[i] = sg;
                u[i] = su;
                h[i] = sg / (1.0 + exp(-sg)) * su;
                if (g_out) g_out[base + i] = sg;
                if (u_out) u_out[base + i] = su;
                if (h_out) h_out[base + i] = h[i];
                if (ag_out) ag_out[base + i] = ag;
                if (au_out) au_out[base + i] = au;
            }
            int64_t dbase = (t * topk + s) * H;
            for (int64_t j = 0; j < H; ++j) {
                double sd = 0.0, ad = 0.0;
                for (int64_t i = 0; i < I; ++i) {
                    double p = nvfp4_elem(dc, ds, I, j, i) * (double)dn_ts[e] * h[i];
                    sd += p;
                    ad += fabs(p);
                }
                if (d_out) d_out[dbase + j] = sd;
                if (ad_out) ad_out[dbase + j] = ad;
                y[t * H + j] += wsel * sd;
            }
        }
    }
    free(h);
    free(u);
    free(g);
}
