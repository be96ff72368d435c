/*
 * Host replay of how the quantizer kernels form the quotient x / s without a
 * division, checked against the IEEE single-precision division x / s.
 *
 * With y = RN(1/s) (a correctly rounded reciprocal):
 *   q0 = RN(x * y)
 *   q1 = RN(q0 + r0 * y),  r0 = RN(x - s * q0)   (two fused multiply-adds)
 *   q2 = RN(q1 + r1 * y),  r1 = RN(x - s * q1)
 * The kernels use q1 for 16-bit inputs and q2 for fp32 inputs.  Scaling x or
 * s by a power of two scales y, q0, r0, q1, ... exactly (as long as nothing
 * under- or overflows, which the kernels' range check on s guarantees), so
 * the claim q1 == RN(x / s) for 16-bit x reduces to the pairs (significand
 * of x, significand of s) with x and s in [1, 2).
 *
 * Built with -O2 -fno-fast-math -ffp-contract=off: every product, sum and
 * quotient below is one IEEE single-precision operation, and fmaf() is the
 * correctly rounded fused multiply-add of the C library.  Test code only.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static float f_of(uint32_t b)
{
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

static uint32_t b_of(float f)
{
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    return b;
}

static float corrected(float x, float s, float y, int corrections)
{
    float q = x * y;
    for (int i = 0; i < corrections; ++i) {
        float r = fmaf(-s, q, x);
        q = fmaf(r, y, q);
    }
    return q;
}

/* Every x in [1, 2) with `x_bits` stored significand bits (7: bfloat16,
 * 10: fp16) against every s in [1, 2) whose 23 stored significand bits are
 * s_lo, s_lo + s_step, ... below s_hi.  Counts the pairs whose quotient
 * after `corrections` corrections differs (in bits) from x / s, and
 * records the first one. */
int64_t qs_sweep16(int x_bits, uint32_t s_lo, uint32_t s_hi, uint32_t s_step, int corrections,
                   uint32_t *bad_x, uint32_t *bad_s)
{
    const uint32_t nx = 1u << x_bits;
    int64_t bad = 0;
    uint32_t fx = 0, fs = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad)
    for (int64_t ms = s_lo; ms < (int64_t)s_hi; ms += s_step) {
        const float s = f_of(0x3F800000u | (uint32_t)ms);
        const float y = 1.0f / s;
        for (uint32_t mx = 0; mx < nx; ++mx) {
            const float x = f_of(0x3F800000u | (mx << (23 - x_bits)));
            if (b_of(corrected(x, s, y, corrections)) != b_of(x / s)) {
                ++bad;
#pragma omp critical
                if (fx == 0 && fs == 0) {
                    fx = b_of(x);
                    fs = b_of(s);
                }
            }
        }
    }
    *bad_x = fx;
    *bad_s = fs;
    return bad;
}

/* Given pairs of fp32 bit patterns (x[i], s[i]), the number of pairs whose
 * quotient after `corrections` corrections differs from x / s. */
int64_t qs_pairs(const uint32_t *x, const uint32_t *s, int64_t n, int corrections)
{
    int64_t bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : bad)
    for (int64_t i = 0; i < n; ++i) {
        const float xs = f_of(x[i]), ss = f_of(s[i]);
        if (b_of(corrected(xs, ss, 1.0f / ss, corrections)) != b_of(xs / ss))
            ++bad;
    }
    return bad;
}
