/*
 * CPU oracle for the FP8_DYNAMIC W8A8 linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline and reference arm use it.  It shares no code, header, table or
 * constant generator with the CUDA library.
 *
 * It is deliberately plain and slow: one value at a time, in the order the
 * pages describe, with fp64 wherever a step has no fixed precision.
 *
 * Sources (page title, section):
 *   [P2] "FP8 Inference Explained, in depth", sections "The numbers in one
 *        byte" (E4M3 layout, the round_e4m3 semantics, the fake_quant worked
 *        row), "Scales and their granularity" (x_fp8 = round(x / s),
 *        s = amax / 448) and "Inside a quantized linear layer" (per-token x
 *        per-channel scales move outside the K sum; FP32 accumulation).
 *   [P3] "FP8 Quantization", sections "FP8 Representation" (bias 7,
 *        96.0 = 0 1101 100) and "How FP8 Matmul Works at the Hardware Level"
 *        (FP8 x FP8 -> FP32 accumulate -> BF16 out).
 *   [P4] "Quantization: FP8 inference and KV-cache quantization", section
 *        "Dynamic scales or static scales" (per-token scale amax/448,
 *        saturating conversion).
 *
 * Readings taken where the pages leave a step open:
 *   - the activation scale is s = fl32(amax / 448) and each value is divided
 *     by s in IEEE fp32 (round to nearest even) before the E4M3 rounding;
 *   - an all-zero row gets s = 1;
 *   - conversion saturates at +-448 (never NaN) and keeps the sign of zero;
 *   - the GEMM result is kept in fp64 (not rounded to BF16).
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fPIC -shared.
 * No -ffast-math: every fp32 division below must be IEEE.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define E4M3_MAX 448.0

/* ------------------------------------------------------------------------ */
/* E4M3 (float8_e4m3fn) codec                                               */
/* ------------------------------------------------------------------------ */

/* Value of one E4M3 code.  [P2 "The numbers in one byte"], [P3 "FP8
 * Representation"]: bit 7 sign, bits 6..3 exponent field E with bias 7,
 * bits 2..0 mantissa m.  E = 0 is subnormal with value m * 2^-9; otherwise
 * (1 + m/8) * 2^(E-7).  The fn variant has no infinities: only E = 15,
 * m = 7 is NaN, so the largest finite value is (1 + 6/8) * 2^8 = 448. */
double orc_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int E = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (E == 15 && m == 7)
        return NAN;
    if (E == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, E - 7);
    return sign ? -v : v;
}

/* Saturating round-to-nearest-even conversion to E4M3, derived from the
 * code table itself rather than from exponent arithmetic.
 * [P2 "The numbers in one byte"] fixes the grid (the decoded codes above),
 * the rounding (to the nearest representable value, halfway cases to the
 * even one, as Python's round does) and the saturation at +-448; [P4
 * "Dynamic scales or static scales"] the saturating (not NaN) overflow.
 * The positive finite codes 0x00..0x7E decode to strictly increasing
 * values, so the two codes that bracket |x| are found by bisection on the
 * code number; the closer one wins, and on an exact tie the one with an even
 * mantissa field, which is the even code number (the mantissa is the low
 * three bits).  Distances are exact: |x| and both bracketing values are
 * dyadic numbers well inside the range of a double.  The sign of x (zero
 * included) becomes bit 7. */
static double g_grid[0x7F];          /* g_grid[c] = orc_e4m3_decode(c), c = 0..0x7E */
static pthread_once_t g_grid_once = PTHREAD_ONCE_INIT;

static void fill_grid(void)
{
    int c;
    for (c = 0; c < 0x7F; ++c)
        g_grid[c] = orc_e4m3_decode((uint8_t)c);
}

uint8_t orc_e4m3_encode(double x)
{
    uint8_t sign;
    double a, d_lo, d_hi;
    int lo, hi;
    pthread_once(&g_grid_once, fill_grid);
    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs(x);
    if (a >= E4M3_MAX)
        return (uint8_t)(sign | 0x7E);
    /* invariant: decode(lo) <= a < decode(hi) */
    lo = 0x00;
    hi = 0x7E;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (g_grid[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    d_lo = a - g_grid[lo];
    d_hi = g_grid[hi] - a;
    if (d_lo < d_hi)
        return (uint8_t)(sign | lo);
    if (d_hi < d_lo)
        return (uint8_t)(sign | hi);
    return (uint8_t)(sign | ((lo % 2 == 0) ? lo : hi));
}

/* The E4M3 value nearest to x (ties to even, saturating at +-448), as a
 * double: the decoded code.  Zero (either sign) and NaN pass through. */
double orc_round_e4m3(double x)
{
    if (x == 0.0 || isnan(x))
        return x;
    return orc_e4m3_decode(orc_e4m3_encode(x));
}

/* Bit pattern of a value that is already on the E4M3 grid (the output of
 * orc_round_e4m3).  Inverse of orc_e4m3_decode by the same field layout. */
uint8_t orc_e4m3_pack(double v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    int ex, e, E, m;
    if (isnan(v))
        return 0x7F;
    if (a == 0.0)
        return sign;
    frexp(a, &ex);
    e = ex - 1;
    if (e < -6) {                         /* subnormal: a = m * 2^-9 */
        m = (int)ldexp(a, 9);
        return (uint8_t)(sign | m);
    }
    E = e + 7;
    m = (int)((ldexp(a, -e) - 1.0) * 8.0);
    return (uint8_t)(sign | (E << 3) | m);
}


/* ------------------------------------------------------------------------ */
/* Dynamic per-token (and per-output-channel) quantization                  */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the top half of an IEEE binary32, so widening is exact. */
static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float orc_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }

/* Quantize one row of fp32 values with its own dynamic scale.
 * [P2 "Scales and their granularity"]: s = amax / 448 and x_fp8 = round(x/s);
 * [P4 "Dynamic scales or static scales"]: one scale per token, computed on
 * every forward pass, so the row maximum lands exactly on 448.
 * Both the scale and every quotient are IEEE fp32 divisions. */
static void quant_row_f32(const float* x, int64_t K, uint8_t* q, float* s_out)
{
    float amax = 0.0f, s;
    int64_t k;
    for (k = 0; k < K; ++k) {
        float a = fabsf(x[k]);
        if (a > amax)
            amax = a;
    }
    s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    for (k = 0; k < K; ++k) {
        volatile float t = x[k] / s;   /* force an fp32 quotient */
        q[k] = orc_e4m3_encode((double)t);
    }
    *s_out = s;
}

/* Rows of bf16 bit patterns (activations [M,K] or weights [N,K]).  The row
 * is widened to fp32 (exact) value by value and read twice: once for amax,
 * once for the quotients. */
void orc_quant_rows_bf16(const uint16_t* x, int64_t R, int64_t K, int64_t ldx,
                         uint8_t* q, int64_t ldq, float* s)
{
    int64_t r;
#pragma omp parallel for schedule(dynamic, 4)
    for (r = 0; r < R; ++r) {
        const uint16_t* xr = x + r * ldx;
        uint8_t* qr = q + r * ldq;
        float amax = 0.0f, sc;
        int64_t k;
        for (k = 0; k < K; ++k) {
            float a = fabsf(bf16_to_f32(xr[k]));
            if (a > amax)
                amax = a;
        }
        sc = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        for (k = 0; k < K; ++k) {
            volatile float t = bf16_to_f32(xr[k]) / sc;   /* fp32 quotient */
            qr[k] = orc_e4m3_encode((double)t);
        }
        s[r] = sc;
    }
}

/* Rows of fp32 values: used to check the pages' fp32 worked examples. */
void orc_quant_rows_f32(const float* x, int64_t R, int64_t K, int64_t ldx,
                        uint8_t* q, int64_t ldq, float* s)
{
    int64_t r;
    for (r = 0; r < R; ++r)
        quant_row_f32(x + r * ldx, K, q + r * ldq, s + r);
}

/* ------------------------------------------------------------------------ */
/* Scaled FP8 GEMM + dequant epilogue                                       */
/* ------------------------------------------------------------------------ */

/* Every finite E4M3 value times 2^9 is an integer of magnitude at most
 * 448 * 512 = 229376 < 2^18, so a product of two scaled codes is an exact
 * integer below 2^36 and a K-term sum stays below 2^51 for K < 2^15: the
 * dot product of the codes is computed exactly in int64. */
static int64_t code_times_512(uint8_t c)
{
    return (int64_t)ldexp(orc_e4m3_decode(c), 9);
}

/* acc[m,n] = sum_k (512 q_x[m,k]) * (512 q_w[n,k])  (exact, int64).
 * q_x is [M,K] row-major, q_w is [N,K] row-major (nn.Linear layout). */
void orc_gemm_exact(const uint8_t* qx, int64_t ldqx, const uint8_t* qw, int64_t ldqw,
                    int64_t M, int64_t N, int64_t K, int64_t* acc)
{
    int64_t tab[256];
    int64_t m;
    int i;
    for (i = 0; i < 256; ++i)
        tab[i] = ((i & 0x7F) == 0x7F) ? 0 : code_times_512((uint8_t)i);
#pragma omp parallel for collapse(2) schedule(static)
    for (m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t sum = 0, k;
            for (k = 0; k < K; ++k)
                sum += tab[qx[m * ldqx + k]] * tab[qw[n * ldqw + k]];
            acc[m * N + n] = sum;
        }
    }
}

/* [P2 "Inside a quantized linear layer"]: both scales are constant along k,
 * so y[m,n] = s_tok[m] * s_w[n] * (q_x[m,:] . q_w[n,:]).  Kept in fp64. */
void orc_epilogue(const int64_t* acc, int64_t M, int64_t N,
                  const float* s_tok, const float* s_w, double* y)
{
    int64_t m, n;
    for (m = 0; m < M; ++m)
        for (n = 0; n < N; ++n)
            y[m * N + n] = ldexp((double)acc[m * N + n], -18)
                           * (double)s_tok[m] * (double)s_w[n];
}

/* The same result at a list of (row, col) points only, for shapes whose full
 * output is too large to compute on the CPU. */
void orc_linear_points(const uint8_t* qx, int64_t ldqx, const float* s_tok,
                       const uint8_t* qw, int64_t ldqw, const float* s_w, int64_t K,
                       int64_t npts, const int64_t* rows, const int64_t* cols, double* y)
{
    int64_t tab[256];
    int64_t p;
    int i;
    for (i = 0; i < 256; ++i)
        tab[i] = ((i & 0x7F) == 0x7F) ? 0 : code_times_512((uint8_t)i);
#pragma omp parallel for schedule(static)
    for (p = 0; p < npts; ++p) {
        int64_t m = rows[p], n = cols[p], k, sum = 0;
        for (k = 0; k < K; ++k)
            sum += tab[qx[m * ldqx + k]] * tab[qw[n * ldqw + k]];
        y[p] = ldexp((double)sum, -18) * (double)s_tok[m] * (double)s_w[n];
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Per-tensor and static scales; KV-cache quantize-on-write                 */
/* ------------------------------------------------------------------------ */

/* Rows quantized with a given scale each: q[r,k] = E4M3(fl32(x[r,k] / s[r])).
 * A static (calibrated) scale is the same s for every row ("Quantization:
 * FP8 inference and KV-cache quantization", "Dynamic scales or static
 * scales": values beyond 448 s clamp to 448 in saturating mode). */
void orc_quant_rows_scaled_bf16(const uint16_t* x, int64_t R, int64_t K, int64_t ldx,
                                const float* s, uint8_t* q, int64_t ldq)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; ++r) {
        int64_t k;
        for (k = 0; k < K; ++k) {
            volatile float t = bf16_to_f32(x[r * ldx + k]) / s[r];
            q[r * ldq + k] = orc_e4m3_encode((double)t);
        }
    }
}

/* Dynamic per-tensor scale ("FP8 Quantization", "Choose Scaling Strategy"
 * and "Granularity": one scale for the whole tensor, from its max |x|,
 * computed at run time): s = fl32(amax / 448) over all R x K values (1 if
 * all are zero), then every value divided by s. */
void orc_quant_tensor_bf16(const uint16_t* x, int64_t R, int64_t K, int64_t ldx,
                           uint8_t* q, int64_t ldq, float* s_out)
{
    float amax = 0.0f, s;
    int64_t r, k;
    for (r = 0; r < R; ++r)
        for (k = 0; k < K; ++k) {
            float a = fabsf(bf16_to_f32(x[r * ldx + k]));
            if (a > amax)
                amax = a;
        }
    s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    for (r = 0; r < R; ++r)
        for (k = 0; k < K; ++k) {
            volatile float t = bf16_to_f32(x[r * ldx + k]) / s;
            q[r * ldq + k] = orc_e4m3_encode((double)t);
        }
    *s_out = s;
}

/* FP8 KV-cache write ("Quantization: FP8 inference and KV-cache
 * quantization", "Turning it on in an engine": one scale per tensor or per
 * attention head, 1.0 when uncalibrated; values beyond 448 are clipped).
 * x is [T, H, D] bf16; scale has H entries (per head) or 1 (per tensor,
 * scale_stride 0); token t goes to cache row slot[t] (or t), skipped when
 * that row is negative or not below n_slots; cache is [n_slots, H, D] E4M3. */
void orc_kv_cache_quant_bf16(const uint16_t* x, int64_t T, int64_t H, int64_t D,
                             const float* scale, int64_t scale_stride,
                             const int64_t* slot, int64_t n_slots, uint8_t* cache)
{
    int64_t t;
    for (t = 0; t < T; ++t) {
        int64_t row = slot ? slot[t] : t, h, d;
        if (row < 0 || row >= n_slots)
            continue;
        for (h = 0; h < H; ++h) {
            const float s = scale[h * scale_stride];
            for (d = 0; d < D; ++d) {
                volatile float v = bf16_to_f32(x[(t * H + h) * D + d]) / s;
                cache[(row * H + h) * D + d] = orc_e4m3_encode((double)v);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Block-wise scales: 1 x G activation groups, Bn x Bk weight blocks         */
/* ------------------------------------------------------------------------ */

/* Each rectangle [r0, r1) x [k0, k1) of x shares one scale:
 * s = fl32(amax / 448) (1 if the rectangle is all zero) and every value in it
 * becomes E4M3(fl32(x / s)) -- the per-token rule applied to a smaller set of
 * values ("FP8 Quantization", "Granularity": per-block, one scale per
 * 128 x 128 tile; "FP8 Inference Explained, in depth", "Scales and their
 * granularity": s = amax / 448 where amax is the largest value the scale
 * covers). */
static float quant_rect_bf16(const uint16_t* x, int64_t ldx, int64_t r0, int64_t r1,
                             int64_t k0, int64_t k1, uint8_t* q, int64_t ldq)
{
    float amax = 0.0f, s;
    int64_t r, k;
    for (r = r0; r < r1; ++r)
        for (k = k0; k < k1; ++k) {
            float a = fabsf(bf16_to_f32(x[r * ldx + k]));
            if (a > amax)
                amax = a;
        }
    s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    for (r = r0; r < r1; ++r)
        for (k = k0; k < k1; ++k) {
            volatile float t = bf16_to_f32(x[r * ldx + k]) / s;
            q[r * ldq + k] = orc_e4m3_encode((double)t);
        }
    return s;
}

/* x [R, K] in blocks of br rows x bk columns (the last block of each
 * dimension may be partial).  s is [ceil(R/br), ceil(K/bk)] row-major.
 * Activations use br = 1, bk = 128 (one scale per token per 128 inputs);
 * weights use br = bk = 128. */
void orc_quant_blocks_bf16(const uint16_t* x, int64_t R, int64_t K, int64_t ldx,
                           int64_t br, int64_t bk, uint8_t* q, int64_t ldq, float* s)
{
    const int64_t RB = (R + br - 1) / br, KB = (K + bk - 1) / bk;
    int64_t b;
#pragma omp parallel for schedule(dynamic, 8)
    for (b = 0; b < RB * KB; ++b) {
        const int64_t rb = b / KB, kb = b % KB;
        const int64_t r0 = rb * br, k0 = kb * bk;
        const int64_t r1 = r0 + br < R ? r0 + br : R, k1 = k0 + bk < K ? k0 + bk : K;
        s[b] = quant_rect_bf16(x, ldx, r0, r1, k0, k1, q, ldq);
    }
}

/* Block-scaled GEMM ("FP8 Inference Explained, in depth", "Inside a quantized
 * linear layer": block-wise scales vary along k, so each block's partial sum
 * is multiplied by that block's scales before the partial sums are added):
 *   y[m,n] = sum_kb  s_x[m, kb] * s_w[n / bn, kb] * P[m, n, kb],
 *   P[m, n, kb] = sum_{k in block kb} e4m3(q_x[m,k]) * e4m3(q_w[n,k]),
 * blocks of bk along K for both operands.  Each P is exact (int64 of codes
 * times 2^9), the sum over kb is in fp64, in increasing kb.  Computed at the
 * npts points (rows[p], cols[p]) only, or everywhere when rows is NULL
 * (then y is [M, N]). */
void orc_gemm_blockwise(const uint8_t* qx, int64_t ldqx, const float* s_x,
                        const uint8_t* qw, int64_t ldqw, const float* s_w,
                        int64_t M, int64_t N, int64_t K, int64_t bn, int64_t bk,
                        int64_t npts, const int64_t* rows, const int64_t* cols, double* y)
{
    const int64_t KB = (K + bk - 1) / bk;
    const int64_t total = rows ? npts : M * N;
    int64_t tab[256];
    int64_t p;
    int i;
    for (i = 0; i < 256; ++i)
        tab[i] = ((i & 0x7F) == 0x7F) ? 0 : code_times_512((uint8_t)i);
#pragma omp parallel for schedule(static)
    for (p = 0; p < total; ++p) {
        const int64_t m = rows ? rows[p] : p / N, n = rows ? cols[p] : p % N;
        double acc = 0.0;
        int64_t kb, k;
        for (kb = 0; kb < KB; ++kb) {
            const int64_t k1 = (kb + 1) * bk < K ? (kb + 1) * bk : K;
            int64_t part = 0;
            for (k = kb * bk; k < k1; ++k)
                part += tab[qx[m * ldqx + k]] * tab[qw[n * ldqw + k]];
            acc += ldexp((double)part, -18) * (double)s_x[m * KB + kb]
                   * (double)s_w[(n / bn) * KB + kb];
        }
        y[p] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm feeding the per-token quantizer (the amax reduction fused into     */
/* the preceding kernel)                                                      */
/* ------------------------------------------------------------------------ */

static uint16_t f32_to_bf16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return (uint16_t)((u >> 16) | 0x40);            /* quiet NaN */
    u += 0x7FFFu + ((u >> 16) & 1u);                     /* round to nearest even */
    return (uint16_t)(u >> 16);
}

/* The normalisation of one row, given its sum of squares ss, as the fp32
 * steps of the reading: mean = fl32(ss / K); r = fl32(sqrt(fl32(mean + eps)));
 * inv = fl32(1 / r); y_k = bf16(fl32(fl32(x_k * inv) * g_k)).  Every step is
 * monotone in ss, so y at two sums brackets y at any sum between them. */
static void rms_row_from_ss(const uint16_t* x, const uint16_t* g, int64_t K, float eps,
                            float ss, uint16_t* y)
{
    volatile float mean = ss / (float)K;
    volatile float t = mean + eps;
    volatile float r = sqrtf(t);
    volatile float inv = 1.0f / r;
    int64_t k;
    for (k = 0; k < K; ++k) {
        volatile float a = bf16_to_f32(x[k]) * inv;
        volatile float b = a * bf16_to_f32(g[k]);
        y[k] = f32_to_bf16_rn(b);
    }
}

/* RMSNorm (y = x / sqrt(mean(x^2) + eps) * g, "FP8 Inference Explained, in
 * depth", "What stays in higher precision": normalisation stays in 16- or
 * 32-bit, and "Scales and their granularity": the amax reduction is fused
 * into the preceding kernel).  The sum of squares is exact here (fp64 sums of
 * bf16 squares, each exact) and the GPU's fp32 sum lies within a relative
 * rel_err of it, so the row is evaluated at ss * (1 - rel_err) and
 * ss * (1 + rel_err) (rounded outwards to fp32): y_lo / y_hi bracket every
 * bf16 value the GPU may produce, element by element.  ss_out is the exact
 * sum. */
void orc_rmsnorm_bracket_bf16(const uint16_t* x, int64_t R, int64_t K, int64_t ldx,
                              const uint16_t* g, float eps, double rel_err,
                              uint16_t* y_lo, uint16_t* y_hi, double* ss_out)
{
    int64_t r;
#pragma omp parallel for schedule(dynamic, 4)
    for (r = 0; r < R; ++r) {
        const uint16_t* xr = x + r * ldx;
        double ss = 0.0, lo, hi;
        float flo, fhi;
        int64_t k;
        for (k = 0; k < K; ++k) {
            double v = (double)bf16_to_f32(xr[k]);
            ss += v * v;
        }
        lo = ss * (1.0 - rel_err);
        hi = ss * (1.0 + rel_err);
        flo = (float)lo;
        if ((double)flo > lo)
            flo = nextafterf(flo, 0.0f);
        fhi = (float)hi;
        if ((double)fhi < hi)
            fhi = nextafterf(fhi, INFINITY);
        /* a larger sum gives a smaller |y| */
        rms_row_from_ss(xr, g, K, eps, fhi, y_lo + r * K);
        rms_row_from_ss(xr, g, K, eps, flo, y_hi + r * K);
        ss_out[r] = ss;
    }
}

/* The same steps in fp64 throughout (no intermediate rounding): the real
 * normalised values, for comparison with an independent library routine. */
void orc_rmsnorm_f64(const uint16_t* x, int64_t R, int64_t K, int64_t ldx, const uint16_t* g,
                     double eps, double* y)
{
    int64_t r, k;
    for (r = 0; r < R; ++r) {
        double ss = 0.0, inv;
        for (k = 0; k < K; ++k) {
            double v = (double)bf16_to_f32(x[r * ldx + k]);
            ss += v * v;
        }
        inv = 1.0 / sqrt(ss / (double)K + eps);
        for (k = 0; k < K; ++k)
            y[r * K + k] = (double)bf16_to_f32(x[r * ldx + k]) * inv * (double)bf16_to_f32(g[k]);
    }
}
