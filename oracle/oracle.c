/*
 * oracle.c -- fp64 CPU oracle for the dense decoder-layer region
 *             y = x . W^T ; r = r0 + y ; out = RMSNorm(r)
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library.  The
 * product path (libfusedln) never links, loads or calls it, and the two share
 * no code, headers, tables or helpers.
 *
 * What it follows (vLLM "TPSP Design" page, and the torch-spyre "Plugin
 * Architecture" page for the norm semantics):
 *   - row-parallel projection o_proj / down_proj, F.linear semantics
 *     y = x @ W^T with W stored [out, in] = [H, K]
 *       ("Plugin Architecture", "Custom Op Replacement" table, RowParallelLinear
 *        row; "Transposed linear weights");
 *   - residual add then RMSNorm over the complete hidden dimension of each
 *     token ("TPSP Design", section 1 "Motivation": local residual add and norm
 *     keep the full hidden size per token; section 3 "Fusion regions");
 *   - standard RMSNorm without norm bias ("TPSP Design", section 4
 *     "Constraints"), computed in a wider type than the bf16 activations
 *     ("Plugin Architecture", "Transformers backend": the fp16->fp32 upcast of
 *     the native RMSNorm forward);
 *   - Gemma RMSNorm: the same body with a trailing multiply by (1 + gamma),
 *     gamma an fp32 [hidden] weight ("Plugin Architecture", table row
 *     GemmaRMSNorm; "TPSP Design", section 5 "To-do", Gemma family).
 *
 * Readings where the pages print no formula (each listed in the design notes):
 *   - RMSNorm(r)[h] = r[h] / sqrt(mean_h(r^2) + eps) * g[h], eps inside the
 *     square root, mean over the full hidden dimension H;
 *   - the projection output is not rounded before the residual add, and the
 *     norm statistics come from the unrounded sum;
 *   - g[h] = gamma[h] (standard) or 1 + gamma[h] (Gemma).
 *
 * Arithmetic: every bf16 input is widened exactly to double, the dot product
 * is accumulated in double in ascending k, and nothing is blocked, fused or
 * reordered beyond the definition above.  Rows are independent, so rows are
 * spread over OpenMP threads; that changes no result bit.
 *
 * FP8 projection (the "TPSP Design" page, section 5 "To-do": "FP8 dense",
 * quantized projections with scale handling across microchunks).  Reading:
 * x and W hold FP8 E4M3 codes with fp32 dequantisation scales, one per tensor
 * or one per token row of x and one per output row of W, so that
 *   y[t,h] = sx[t] * sw[h] * sum_k e4m3(x[t,k]) * e4m3(W[h,k]);
 * the residual add and the norm are unchanged.  A microchunk uses the scales
 * of its own rows, so chunking changes no value.
 *
 * NVFP4 weights (the same page's "MXFP4 / NVFP4 dense" item, low-bit weight
 * layouts and scaling): W holds E2M1 codes packed two per byte along K with
 * one E4M3 scale per 16 elements and an fp32 tensor scale; x stays bf16.
 * MXFP4 weights: the same codes with one E8M0 (power-of-two) scale per 32
 * elements and no tensor scale.
 *
 * Pins (tests/test_oracle.py, tests/test_oracle_fp8.py, tests/test_oracle_fp4.py,
 * tests/test_oracle_mx.py, tests/test_oracle_moe.py): hand-worked 2x2, 4x4
 * and 1x3x2 cases, the closed form of a constant row, the unit-RMS invariant,
 * Gemma(0)==standard(1) bit for bit, linearity of the residual add, eps=0
 * scale invariance, column permutation of K, the projection against numpy's
 * float64 matmul; for FP8 the decoding of all 256 codes against PyTorch's
 * float8_e4m3fn, a hand-worked scaled case, equality with the bf16 region on
 * the same values at unit scales, and exact power-of-two scale laws.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_NORM_STANDARD 0
#define ORACLE_NORM_GEMMA 1

/* bf16 bit pattern -> double.  bf16 is the top half of an IEEE binary32, so
 * the widening is exact. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> bf16 bit pattern, round to nearest, ties to even, in one rounding
 * step from the exact double value (no intermediate binary32).
 * bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored fraction bits. */
uint16_t oracle_double_to_bf16(double v)
{
    if (isnan(v))
        return (uint16_t)0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);            /* a = m * 2^e, m in [0.5, 1) */
    int exp_unbiased = e - 1;      /* a = 1.f * 2^exp_unbiased */
    int quantum_exp;               /* spacing of representable values near a */
    if (exp_unbiased >= -126)
        quantum_exp = exp_unbiased - 7;  /* 8 significant bits */
    else
        quantum_exp = -126 - 7;          /* subnormal spacing 2^-133 */
    double q = ldexp(a, -quantum_exp);   /* exact: scaling by a power of two */
    double qi = nearbyint(q);            /* default mode: nearest, ties to even */
    double rounded = ldexp(qi, quantum_exp);
    if (rounded >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80); /* overflow to infinity */
    /* rounded has at most 8 significant bits and lies in binary32 range, so
     * the conversion to float is exact and its top 16 bits are the bf16. */
    float f = (float)rounded;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

void oracle_round_to_bf16(const double *v, long n, uint16_t *out)
{
    for (long i = 0; i < n; ++i)
        out[i] = oracle_double_to_bf16(v[i]);
}

static double norm_weight(const float *gamma, long h, int norm_kind)
{
    double g = (double)gamma[h];
    return norm_kind == ORACLE_NORM_GEMMA ? 1.0 + g : g;
}

/* RMSNorm of one row r[0..H) in place into o[0..H); returns mean square. */
static double rmsnorm_row(const double *r, long H, const float *gamma, double eps,
                          int norm_kind, double *o)
{
    double sum_sq = 0.0;
    for (long h = 0; h < H; ++h)
        sum_sq += r[h] * r[h];
    double mean_sq = sum_sq / (double)H;
    double inv_rms = 1.0 / sqrt(mean_sq + eps);
    for (long h = 0; h < H; ++h)
        o[h] = r[h] * inv_rms * norm_weight(gamma, h, norm_kind);
    return mean_sq;
}

static int check_args(long T, long K, long H, int norm_kind, double eps)
{
    if (T < 0 || K < 0 || H <= 0)
        return -1;
    if (norm_kind != ORACLE_NORM_STANDARD && norm_kind != ORACLE_NORM_GEMMA)
        return -1;
    if (!(eps >= 0.0) || isinf(eps))
        return -1;
    return 0;
}

/*
 * Full region for the selected token rows.
 *   x      [T, K] bf16 bits, row-major
 *   W      [H, K] bf16 bits, row-major ([out, in], F.linear layout)
 *   r0     [T, H] bf16 bits, residual before the add
 *   gamma  [H] fp32 norm weight
 *   rows   indices of the token rows to compute, or NULL for all T rows
 *   nrows  number of entries in rows (ignored when rows is NULL)
 *   r_out  [n, H] double: r = r0 + x . W^T        (n = nrows or T)
 *   o_out  [n, H] double: RMSNorm(r)
 *   ms_out [n] double: mean over h of r^2, or NULL
 * Returns 0, or -1 on a bad argument.
 */
int oracle_proj_add_rmsnorm(const uint16_t *x, const uint16_t *W, const uint16_t *r0,
                            const float *gamma, double eps, int norm_kind,
                            long T, long K, long H, const long *rows, long nrows,
                            double *r_out, double *o_out, double *ms_out, int nthreads)
{
    if (check_args(T, K, H, norm_kind, eps))
        return -1;
    long n = rows ? nrows : T;
    for (long i = 0; rows && i < n; ++i)
        if (rows[i] < 0 || rows[i] >= T)
            return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < n; ++i) {
        long t = rows ? rows[i] : i;
        const uint16_t *xt = x + t * K;
        double *r = r_out + i * H;
        for (long h = 0; h < H; ++h) {
            const uint16_t *wh = W + h * K;
            double y = 0.0;
            for (long k = 0; k < K; ++k)
                y += bf16_bits_to_double(xt[k]) * bf16_bits_to_double(wh[k]);
            r[h] = bf16_bits_to_double(r0[t * H + h]) + y;
        }
        double ms = rmsnorm_row(r, H, gamma, eps, norm_kind, o_out + i * H);
        if (ms_out)
            ms_out[i] = ms;
    }
    return 0;
}

/*
 * Add + RMSNorm alone, with a bf16 addend y (the unfused path's second step).
 *   y [T, H] bf16, r0 [T, H] bf16, gamma [H] fp32; outputs as above.
 */
int oracle_add_rmsnorm(const uint16_t *y, const uint16_t *r0, const float *gamma,
                       double eps, int norm_kind, long T, long H,
                       double *r_out, double *o_out, double *ms_out, int nthreads)
{
    if (check_args(T, 0, H, norm_kind, eps))
        return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(static)
    for (long t = 0; t < T; ++t) {
        double *r = r_out + t * H;
        for (long h = 0; h < H; ++h)
            r[h] = bf16_bits_to_double(r0[t * H + h]) + bf16_bits_to_double(y[t * H + h]);
        double ms = rmsnorm_row(r, H, gamma, eps, norm_kind, o_out + t * H);
        if (ms_out)
            ms_out[t] = ms;
    }
    return 0;
}

/*
 * FP8 E4M3 code -> double (the OCP 8-bit floating-point format in its "FN"
 * form): 1 sign bit, 4 exponent bits with bias 7, 3 stored fraction bits.
 * Exponent field 0 holds the subnormals f/8 * 2^-6; exponent field 15 with
 * fraction 7 is the only NaN (no infinities), so the largest finite value is
 * 1.75 * 2^8 = 448.  Every code is exact in double.
 */
double oracle_e4m3_to_double(uint8_t b)
{
    int sign = b >> 7;
    int e = (b >> 3) & 0xF;
    int f = b & 0x7;
    double v;
    if (e == 15 && f == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)f, -9);          /* (f / 8) * 2^-6 */
    else
        v = ldexp(8.0 + (double)f, e - 10); /* (1 + f / 8) * 2^(e - 7) */
    return sign ? -v : v;
}

/*
 * The region with FP8 operands.
 *   x        [T, K] E4M3 codes, row-major
 *   x_scale  [T] fp32 if x_per_row, else [1] (one scale for the tensor)
 *   W        [H, K] E4M3 codes, row-major ([out, in])
 *   w_scale  [H] fp32 if w_per_row, else [1]
 *   the rest as in oracle_proj_add_rmsnorm.
 * y[t,h] = sx * sw * (sum over k ascending of the exact products), in double.
 */
int oracle_proj_add_rmsnorm_fp8(const uint8_t *x, const float *x_scale, int x_per_row,
                                const uint8_t *W, const float *w_scale, int w_per_row,
                                const uint16_t *r0, const float *gamma, double eps, int norm_kind,
                                long T, long K, long H, const long *rows, long nrows,
                                double *r_out, double *o_out, double *ms_out, int nthreads)
{
    if (check_args(T, K, H, norm_kind, eps))
        return -1;
    if (!x_scale || !w_scale)
        return -1;
    long n = rows ? nrows : T;
    for (long i = 0; rows && i < n; ++i)
        if (rows[i] < 0 || rows[i] >= T)
            return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < n; ++i) {
        long t = rows ? rows[i] : i;
        const uint8_t *xt = x + t * K;
        double sx = (double)x_scale[x_per_row ? t : 0];
        double *r = r_out + i * H;
        for (long h = 0; h < H; ++h) {
            const uint8_t *wh = W + h * K;
            double dot = 0.0;
            for (long k = 0; k < K; ++k)
                dot += oracle_e4m3_to_double(xt[k]) * oracle_e4m3_to_double(wh[k]);
            double sw = (double)w_scale[w_per_row ? h : 0];
            r[h] = bf16_bits_to_double(r0[t * H + h]) + sx * sw * dot;
        }
        double ms = rmsnorm_row(r, H, gamma, eps, norm_kind, o_out + i * H);
        if (ms_out)
            ms_out[i] = ms;
    }
    return 0;
}

/*
 * FP4 E2M1 code (low 4 bits of b) -> double (the OCP 4-bit floating-point
 * element): 1 sign bit, 2 exponent bits with bias 1, 1 fraction bit; exponent
 * field 0 holds the subnormal 0.5 * f; no infinities or NaN.  Values
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives.
 */
double oracle_e2m1_to_double(uint8_t b)
{
    int sign = (b >> 3) & 1;
    int e = (b >> 1) & 3;
    int f = b & 1;
    double v = e == 0 ? 0.5 * f : ldexp(1.0 + 0.5 * f, e - 1);
    return (sign != 0) ? -v : v;
}

/*
 * The region with NVFP4 weights ("TPSP Design", section 5 "To-do": MXFP4 /
 * NVFP4 dense, low-bit weight layouts and their scaling).  Reading: W holds
 * E2M1 codes, two per byte along K (element 2j in the low nibble of byte j,
 * element 2j + 1 in the high nibble), each run of 16 elements of a row shares
 * an E4M3 scale, and one fp32 scale applies to the whole tensor:
 *   w[h,k] = gs * e4m3(S[h, k / 16]) * e2m1(W[h,k])
 *   y[t,h] = sum_k x[t,k] * w[h,k]        (x bf16)
 * then the unchanged add and norm.
 *   x      [T, K] bf16 bits
 *   Wq     [H, K / 2] bytes (K even)
 *   S      [H, ceil(K / 16)] E4M3 codes
 *   gs     the tensor's fp32 scale
 */
int oracle_proj_add_rmsnorm_nvfp4(const uint16_t *x, const uint8_t *Wq, const uint8_t *S, float gs,
                                  const uint16_t *r0, const float *gamma, double eps, int norm_kind,
                                  long T, long K, long H, const long *rows, long nrows,
                                  double *r_out, double *o_out, double *ms_out, int nthreads)
{
    if (check_args(T, K, H, norm_kind, eps) || (K & 1))
        return -1;
    long nblk = (K + 15) / 16;
    long n = rows ? nrows : T;
    for (long i = 0; rows && i < n; ++i)
        if (rows[i] < 0 || rows[i] >= T)
            return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < n; ++i) {
        long t = rows ? rows[i] : i;
        const uint16_t *xt = x + t * K;
        double *r = r_out + i * H;
        for (long h = 0; h < H; ++h) {
            const uint8_t *wh = Wq + h * (K / 2);
            const uint8_t *sh = S + h * nblk;
            double acc = 0.0;
            for (long k = 0; k < K; ++k) {
                uint8_t code = (k & 1) ? (uint8_t)(wh[k / 2] >> 4) : (uint8_t)(wh[k / 2] & 0xF);
                double w = (double)gs * oracle_e4m3_to_double(sh[k / 16]) * oracle_e2m1_to_double(code);
                acc += bf16_bits_to_double(xt[k]) * w;
            }
            r[h] = bf16_bits_to_double(r0[t * H + h]) + acc;
        }
        double ms = rmsnorm_row(r, H, gamma, eps, norm_kind, o_out + i * H);
        if (ms_out)
            ms_out[i] = ms;
    }
    return 0;
}

/*
 * OCP microscaling E8M0 scale code -> double: a bare biased exponent, the
 * value 2^(E - 127) for E = 0 .. 254; the code 255 is NaN.
 */
double oracle_e8m0_to_double(uint8_t E)
{
    if (E == 255)
        return NAN;
    return ldexp(1.0, (int)E - 127);
}

/*
 * The region with MXFP4 weights (the same "MXFP4 / NVFP4 dense" item).
 * Reading: the OCP MX layout for FP4 -- E2M1 codes packed two per byte along
 * K exactly as for NVFP4, one E8M0 scale shared by each run of 32 elements
 * of a row, no tensor scale:
 *   w[h,k] = e8m0(S[h, k / 32]) * e2m1(W[h,k])
 *   y[t,h] = sum_k x[t,k] * w[h,k]        (x bf16)
 * then the unchanged add and norm.
 *   S      [H, ceil(K / 32)] E8M0 codes
 */
int oracle_proj_add_rmsnorm_mxfp4(const uint16_t *x, const uint8_t *Wq, const uint8_t *S,
                                  const uint16_t *r0, const float *gamma, double eps, int norm_kind,
                                  long T, long K, long H, const long *rows, long nrows,
                                  double *r_out, double *o_out, double *ms_out, int nthreads)
{
    if (check_args(T, K, H, norm_kind, eps) || (K % 2) != 0)
        return -1;
    long scales_per_row = (K + 31) / 32;
    long nout = rows ? nrows : T;
    for (long i = 0; rows && i < nout; ++i)
        if (rows[i] < 0 || rows[i] >= T)
            return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < nout; ++i) {
        long tok = rows ? rows[i] : i;
        const uint16_t *xrow = x + tok * K;
        double *r = r_out + i * H;
        for (long h = 0; h < H; ++h) {
            const uint8_t *codes = Wq + h * (K / 2);
            const uint8_t *scales = S + h * scales_per_row;
            double sum = 0.0;
            for (long k = 0; k < K; ++k) {
                uint8_t byte = codes[k / 2];
                uint8_t nib = (k % 2 == 0) ? (uint8_t)(byte & 0x0F) : (uint8_t)(byte >> 4);
                double wv = oracle_e8m0_to_double(scales[k / 32]) * oracle_e2m1_to_double(nib);
                sum += bf16_bits_to_double(xrow[k]) * wv;
            }
            r[h] = bf16_bits_to_double(r0[tok * H + h]) + sum;
        }
        double ms = rmsnorm_row(r, H, gamma, eps, norm_kind, o_out + i * H);
        if (ms_out)
            ms_out[i] = ms;
    }
    return 0;
}

/*
 * The MoE region ("TPSP Design", section 3 "Fusion regions": the MoE design
 * extends the dense regions to routing and expert reordering -- routing and
 * permute before the grouped GEMM, grouped GEMM then unpermute and the
 * add / next norm; section 5 "To-do": MoE).  The pages give the order of the
 * steps, not their arithmetic; readings:
 *
 * routing: logits [T, E] fp32 from the router; each token takes the k
 * experts of largest logit (equal logits: the smaller expert index first),
 * listed in that order, with weights softmax over the k chosen logits
 *   w[t,j] = exp(l[t,e_j] - l[t,e_0]) / sum_i exp(l[t,e_i] - l[t,e_0]).
 */
int oracle_moe_route(const float *logits, long T, long E, long k, int32_t *ids, double *w)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E)
        return -1;
    for (long t = 0; t < T; ++t) {
        const float *lt = logits + t * E;
        int32_t *it = ids + t * k;
        for (long j = 0; j < k; ++j) {
            long best = -1;
            for (long e = 0; e < E; ++e) {
                int taken = 0;
                for (long i = 0; i < j; ++i)
                    if (it[i] == e)
                        taken = 1;
                if (taken)
                    continue;
                if (best < 0 || (double)lt[e] > (double)lt[best])
                    best = e;
            }
            it[j] = (int32_t)best;
        }
        double top = (double)lt[it[0]], denom = 0.0;
        for (long j = 0; j < k; ++j)
            denom += exp((double)lt[it[j]] - top);
        for (long j = 0; j < k; ++j)
            w[t * k + j] = exp((double)lt[it[j]] - top) / denom;
    }
    return 0;
}

/*
 * permute: the T * k (token, slot) pairs grouped by expert, experts in
 * ascending order and, within an expert, tokens ascending (a token lists an
 * expert at most once).  offsets [E + 1]: expert e owns rows
 * [offsets[e], offsets[e + 1]); row_token / row_slot [T * k]: the pair of each
 * row; row_of [T * k]: the row of pair (t, j) (the unpermute index).
 */
int oracle_moe_permute(const int32_t *ids, long T, long E, long k, int32_t *offsets, int32_t *row_token,
                       int32_t *row_slot, int32_t *row_of)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E)
        return -1;
    for (long i = 0; i < T * k; ++i)
        if (ids[i] < 0 || ids[i] >= E)
            return -1;
    long next = 0;
    for (long e = 0; e < E; ++e) {
        offsets[e] = (int32_t)next;
        for (long t = 0; t < T; ++t)
            for (long j = 0; j < k; ++j)
                if (ids[t * k + j] == e) {
                    row_token[next] = (int32_t)t;
                    row_slot[next] = (int32_t)j;
                    row_of[t * k + j] = (int32_t)next;
                    ++next;
                }
    }
    offsets[E] = (int32_t)next;
    return 0;
}

/*
 * grouped GEMM, unpermute, add and norm: row r of the grouped activations
 * hg [T * k, K] (bf16, expert e's rows at [offsets[e], offsets[e + 1])) is
 * projected by its expert's down weight We [E, H, K] (bf16),
 *   y[r, h] = sum_c hg[r, c] * We[e(r), h, c];
 * each token gathers its k rows in slot order, weighted by its fp32 gate
 * weights wt [T, k]:  z[t, h] = sum_j wt[t, j] * y[row_of[t, j], h];
 * then r = r0 + z and out = RMSNorm(r) as in the dense region.
 */
int oracle_moe_down_region(const uint16_t *hg, const int32_t *offsets, const int32_t *row_of, const float *wt,
                           const uint16_t *We, const uint16_t *r0, const float *gamma, double eps, int norm_kind,
                           long T, long K, long H, long E, long k, double *r_out, double *o_out, double *ms_out,
                           int nthreads)
{
    if (check_args(T, K, H, norm_kind, eps) || E <= 0 || k <= 0 || k > E)
        return -1;
    long R = T * k;
    if (offsets[0] != 0 || offsets[E] != R)
        return -1;
    for (long e = 0; e < E; ++e)
        if (offsets[e + 1] < offsets[e])
            return -1;
    for (long i = 0; i < R; ++i)
        if (row_of[i] < 0 || row_of[i] >= R)
            return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (long t = 0; t < T; ++t) {
        double *r = r_out + t * H;
        for (long h = 0; h < H; ++h)
            r[h] = 0.0;
        for (long j = 0; j < k; ++j) {
            long row = row_of[t * k + j];
            long e = 0;
            while (!(row >= offsets[e] && row < offsets[e + 1]))
                ++e;
            const uint16_t *a = hg + row * K;
            double gate = (double)wt[t * k + j];
            for (long h = 0; h < H; ++h) {
                const uint16_t *wrow = We + (e * H + h) * K;
                double dot = 0.0;
                for (long c = 0; c < K; ++c)
                    dot += bf16_bits_to_double(a[c]) * bf16_bits_to_double(wrow[c]);
                r[h] += gate * dot;
            }
        }
        for (long h = 0; h < H; ++h)
            r[h] += bf16_bits_to_double(r0[t * H + h]);
        double ms = rmsnorm_row(r, H, gamma, eps, norm_kind, o_out + t * H);
        if (ms_out)
            ms_out[t] = ms;
    }
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
