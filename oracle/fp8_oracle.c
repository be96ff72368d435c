/*
 * CPU oracle for the FP8 E4M3 quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this file's library.  The
 * GPU library shares no source, header, table or helper with it.
 *
 * Everything here is the plain definition of what the layer computes, written
 * for a reader to check by eye: linear loops, double-precision accumulation,
 * no blocking, no fusion, no reordering.  Build with -O2 -fno-fast-math
 * -ffp-contract=off so that the single-precision division of the quantizer is
 * one IEEE operation and no multiply-add is contracted.
 *
 * Sources (page title, then the part of the page):
 *  - "RFC: FP8 Quantization Schema in vLLM", Scope: the number format is
 *    FP8_E4M3 as defined by OCP; per-tensor scaling; static input and output
 *    scaling factors.
 *  - "[Kernel][FP8] Initial support with dynamic per-tensor scaling",
 *    Algorithm: the weight scale is computed once after loading and the
 *    activation scale in every forward pass; the forward pass is a cast to
 *    torch.float8_e4m3fn followed by torch._scaled_mm.
 *  - "Marlin fp8", kernel argument checks: the FP8 weight scale of the
 *    weight-only kernel is one value per output channel (shape [1, N]).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* OCP E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * No infinities; S.1111.111 is NaN; the largest finite magnitude is
 * S.1111.110 = 448.  Exponent field 0 encodes subnormals m/8 * 2^-6.        */

double fp8o_e4m3_decode(unsigned code)
{
    unsigned s = (code >> 7) & 1u;
    unsigned e = (code >> 3) & 15u;
    unsigned m = code & 7u;
    double mag;
    if (e == 15u && m == 7u)
        return NAN;
    if (e == 0u)
        mag = ((double)m / 8.0) * ldexp(1.0, -6);
    else
        mag = (1.0 + (double)m / 8.0) * ldexp(1.0, (int)e - 7);
    return s ? -mag : mag;
}

void fp8o_e4m3_decode_table(double out[256])
{
    for (unsigned c = 0; c < 256u; ++c)
        out[c] = fp8o_e4m3_decode(c);
}

/* The same 256 values, computed once by fp8o_e4m3_decode and kept for the
 * loops below (a cache, not a second definition). */
static double g_value[256];
static int g_value_ready = 0;

static const double *value_table(void)
{
    if (!g_value_ready) {
        fp8o_e4m3_decode_table(g_value);
        g_value_ready = 1;
    }
    return g_value;
}

/* Saturating round-to-nearest-even encode of a real value.
 *
 * The 127 non-negative finite codes 0x00..0x7E have strictly increasing
 * values, so the nearest code to |v| is found by bisection on that list;
 * the exact midpoint between two neighbours is representable in double, so
 * the nearer/tie decision is exact.  On a tie the code with the even
 * mantissa (even code, since the mantissa is the low 3 bits) wins.
 * Magnitudes at or above 448 saturate to 448.  The sign of v is kept, so a
 * negative value that rounds to zero gives 0x80.  NaN gives 0x7F (NaN input
 * is outside the layer's contract).                                        */
unsigned fp8o_e4m3_encode(double v)
{
    const double *val = value_table();
    unsigned sign, lo, hi;
    double a, mid;
    if (v != v)
        return 0x7Fu;
    sign = signbit(v) ? 0x80u : 0x00u;
    a = fabs(v);
    if (a >= 448.0)
        return sign | 0x7Eu;
    /* invariant: value(lo) <= a < value(hi) */
    lo = 0u;
    hi = 0x7Eu;
    while (hi - lo > 1u) {
        unsigned m = (lo + hi) / 2u;
        if (val[m] <= a)
            lo = m;
        else
            hi = m;
    }
    mid = 0.5 * (val[lo] + val[hi]);
    if (a < mid)
        return sign | lo;
    if (a > mid)
        return sign | hi;
    return sign | ((lo % 2u == 0u) ? lo : hi);
}

void fp8o_e4m3_encode_f64_array(const double *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)fp8o_e4m3_encode(v[i]);
}

void fp8o_e4m3_encode_f32_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)fp8o_e4m3_encode((double)v[i]);
}

/* ------------------------------------------------------------------------ */
/* Per-tensor quantization ("[Kernel][FP8] Initial support ...", Algorithm).
 * amax = max |x_i| (exact); scale = amax / 448 as one fp32 division; a zero
 * scale (all-zero tensor, or a quotient that underflows) is replaced by 1 so
 * that every code is zero; q_i = E4M3(fp32(x_i / scale)).                  */

float fp8o_amax(const float *x, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > m)
            m = a;
    }
    return m;
}

float fp8o_scale_from_amax(float amax)
{
    float s = amax / 448.0f;
    if (s == 0.0f)
        s = 1.0f;
    return s;
}

void fp8o_quant_with_scale(const float *x, int64_t n, float scale, uint8_t *q)
{
    for (int64_t i = 0; i < n; ++i) {
        float t = x[i] / scale;
        q[i] = (uint8_t)fp8o_e4m3_encode((double)t);
    }
}

/* Dynamic per-tensor quantization; writes the scale it used. */
void fp8o_quant_per_tensor(const float *x, int64_t n, uint8_t *q, float *scale)
{
    float s = fp8o_scale_from_amax(fp8o_amax(x, n));
    fp8o_quant_with_scale(x, n, s, q);
    *scale = s;
}

/* One scale per row of a [rows, cols] matrix (per-output-channel weight
 * scale, the [1, N] scale shape of "Marlin fp8").                          */
void fp8o_quant_per_row(const float *x, int64_t rows, int64_t cols,
                        uint8_t *q, float *row_scale)
{
    for (int64_t r = 0; r < rows; ++r)
        fp8o_quant_per_tensor(x + r * cols, cols, q + r * cols, &row_scale[r]);
}

/* ------------------------------------------------------------------------ */
/* W8A8 scaled matrix product, brute force in double precision.
 *   y[m,n] = (sa * sw[n]) * sum_k dec(qa[m,k]) * dec(qw[n,k])
 * qa is [M,K] and qw is [N,K], both row-major (K contiguous, nn.Linear
 * layout); sw has one entry (per-tensor) or N entries (per-channel).       */
void fp8o_scaled_mm_f64(const uint8_t *qa, const uint8_t *qw,
                        int64_t M, int64_t N, int64_t K,
                        float sa, const float *sw, int per_channel,
                        double *y)
{
    const double *val = value_table();
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += val[qa[m * K + k]] * val[qw[n * K + k]];
            double wscale = per_channel ? (double)sw[n] : (double)sw[0];
            y[m * N + n] = ((double)sa * wscale) * acc;
        }
    }
}

/* The same product with one activation scale per row of qa (per token):
 *   y[m,n] = (sa[m] * sw[n]) * sum_k dec(qa[m,k]) * dec(qw[n,k])
 * The RFC (Scope) supports per-tensor scales and leaves per-channel and
 * finer granularities for later; one scale per activation row is such a
 * finer granularity on the activation side, the weight side unchanged.     */
void fp8o_scaled_mm_rows_f64(const uint8_t *qa, const uint8_t *qw,
                             int64_t M, int64_t N, int64_t K,
                             const float *sa, const float *sw, int per_channel,
                             double *y)
{
    const double *val = value_table();
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += val[qa[m * K + k]] * val[qw[n * K + k]];
            double wscale = per_channel ? (double)sw[n] : (double)sw[0];
            y[m * N + n] = ((double)sa[m] * wscale) * acc;
        }
    }
}

/* W8A16 weight-only product ("Marlin fp8"): 16-bit activations (passed here
 * already widened to fp32, which is exact) times FP8 weights with one scale
 * per output channel.
 *   y[m,n] = sw[n] * sum_k x[m,k] * dec(qw[n,k])                           */
void fp8o_w8a16_mm_f64(const float *x, const uint8_t *qw, const float *sw,
                       int64_t M, int64_t N, int64_t K, double *y)
{
    const double *val = value_table();
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)x[m * K + k] * val[qw[n * K + k]];
            y[m * N + n] = (double)sw[n] * acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* RMS normalization feeding the quantizer.  "Condition to achieve linear
 * speedup?" (the QQQ issue) names fusing the activation quantization into
 * an element-wise kernel such as RMSNorm; the pages do not define RMSNorm,
 * so this is its plain reading (the Llama layer norm):
 *   h[m,k] = x[m,k] * gamma[k] / sqrt( (1/K) sum_j x[m,j]^2 + eps )
 * in double precision.  The layer stores h in the activation's 16-bit
 * format before quantizing it: fp8o_round_binary rounds a double to the
 * nearest value of a binary format with `p` significand bits (including the
 * implicit one) and minimum normal exponent `emin`, ties to even, with
 * gradual underflow (bfloat16: p = 8, emin = -126; fp16: p = 11,
 * emin = -14).  Values beyond the format's range are not produced by the
 * inputs used here.                                                        */

void fp8o_rmsnorm_f64(const float *x, const float *gamma, int64_t M, int64_t K,
                      double eps, double *h)
{
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k)
            ss += (double)x[m * K + k] * (double)x[m * K + k];
        double rms = sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k)
            h[m * K + k] = (double)x[m * K + k] * (double)gamma[k] / rms;
    }
}

double fp8o_round_binary(double v, int p, int emin)
{
    if (v == 0.0 || v != v)
        return v;
    int e = ilogb(v);
    if (e < emin)
        e = emin;
    double ulp = ldexp(1.0, e - (p - 1));
    return rint(v / ulp) * ulp; /* v / ulp is exact; rint rounds ties to even */
}

void fp8o_round_binary_array(const double *v, int64_t n, int p, int emin, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = fp8o_round_binary(v[i], p, emin);
}

/* ------------------------------------------------------------------------ */
/* Grouped W8A8 product for mixture-of-experts layers.  "RFC: FP8
 * Quantization Schema in vLLM", the gate_proj question: FP8 GEMMs need
 * shapes divisible by 16, which is why an 8-expert gate stays in 16-bit;
 * the expert products themselves are FP8.  Tokens routed to expert e are
 * the rows offs[e] .. offs[e+1]-1 of qa; expert e has its own weights
 * qw[e] ([N, K]) and scales (one per expert, or N per expert):
 *   y[m,n] = (sa(m) * sw_e(n)) * sum_k dec(qa[m,k]) * dec(qw[e][n,k])
 * for offs[e] <= m < offs[e+1].  sa has 1 or M entries.                    */
void fp8o_grouped_mm_f64(const uint8_t *qa, const uint8_t *qw, const int32_t *offs,
                         int64_t E, int64_t M, int64_t N, int64_t K,
                         const float *sa, int sa_per_row, const float *sw, int per_channel,
                         double *y)
{
    const double *val = value_table();
    for (int64_t e = 0; e < E; ++e) {
        const uint8_t *we = qw + e * N * K;
        for (int64_t m = offs[e]; m < offs[e + 1] && m < M; ++m) {
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += val[qa[m * K + k]] * val[we[n * K + k]];
                double ws = per_channel ? (double)sw[e * N + n] : (double)sw[e];
                double as = sa_per_row ? (double)sa[m] : (double)sa[0];
                y[m * N + n] = (as * ws) * acc;
            }
        }
    }
}
