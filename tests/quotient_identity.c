/* Host check of the division-free quotient the page-quantise kernel uses
 * (round-to-nearest fp32, the C float arithmetic of the host):
 *
 *   rcp = RN(1 / s);  xc = clamp(x, -1024 s, +1024 s), NaN kept
 *   q0 = RN(xc * rcp);  r = RN(s * q0 - xc) (one fma);  q = RN(q0 - r * rcp) (one fma)
 *
 * Part 1, every bf16 significand of x against every fp32 significand of s
 * (x in [1, 2), s in [1, 2): within the normal range the outcome depends on
 * the significands only): q must equal RN(x / s) bit for bit.
 * Part 2, every bf16 bit pattern of x against scales spread over
 * [2^-90, 2^100] (edges included): q must match RN(x / s) wherever that
 * decides an e4m3 code -- equal for 2^-12 <= |x/s| < 464, beyond the
 * saturation point for |x/s| >= 464, below 2^-10 with the same sign under
 * 2^-12, NaN for NaN.
 * Prints "cases N mismatches M" and exits 1 on any mismatch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float min_nan(float a, float b) { return (isnan(a) || isnan(b)) ? NAN : (a < b ? a : b); }
static float max_nan(float a, float b) { return (isnan(a) || isnan(b)) ? NAN : (a > b ? a : b); }

static float corrected_quotient(float x, float s, float rcp)
{
    const float lim = 1024.0f * s;
    const float xc = max_nan(min_nan(x, lim), -lim);
    const float q0 = xc * rcp;
#ifdef QI_DROP_CORRECTION   /* a planted mistake: the check must then fail */
    return q0;
#else
    const float r = fmaf(s, q0, -xc);
    return fmaf(r, -rcp, q0);
#endif
}

#ifndef QI_SCALE_SIGNIFICANDS
#define QI_SCALE_SIGNIFICANDS (1u << 23)
#endif

int main(void)
{
    long n = 0, bad = 0;
    for (uint32_t xm = 0; xm < 128; ++xm) {
        const float x = from_bits(0x3F800000u | (xm << 16));
        for (uint32_t sm = 0; sm < QI_SCALE_SIGNIFICANDS; ++sm) {
            const float s = from_bits(0x3F800000u | sm);
            const float q = corrected_quotient(x, s, 1.0f / s);
            ++n;
            if (bits_of(q) != bits_of(x / s)) {
                if (bad < 5) printf("x=%a s=%a q=%a x/s=%a\n", x, s, q, x / s);
                ++bad;
            }
        }
    }
    uint64_t st = 88172645463325252ull;   /* xorshift64 */
    const float edges[] = {0x1p-90f, 0x1.000002p-90f, 0x1p100f, 0x1.fffffep99f,
                           1.0f, 1.0f / 448.0f, 448.0f, 0x1.fffffep-1f};
    for (int k = 0; k < 600; ++k) {
        float s;
        if (k < 8) {
            s = edges[k];
        } else {
            st ^= st << 13; st ^= st >> 7; st ^= st << 17;
            const int e = -90 + (int)(st % 190);
            s = ldexpf(from_bits(0x3F800000u | ((uint32_t)(st >> 20) & 0x7FFFFFu)), e);
            if (s > 0x1p100f) s = 0x1p100f;
        }
        const float rcp = 1.0f / s;
        for (uint32_t b = 0; b < 65536; ++b) {
            const float x = from_bits(b << 16);
            const float q = corrected_quotient(x, s, rcp), t = x / s;
            int ok;
            if (isnan(x))
                ok = isnan(q);
            else if (fabsf(t) >= 464.0f)
                ok = fabsf(q) >= 464.0f && signbit(q) == signbit(t);
            else if (fabsf(t) >= 0x1p-12f)
                ok = bits_of(q) == bits_of(t);
            else
                ok = fabsf(q) < 0x1p-10f && signbit(q) == signbit(t);
            ++n;
            if (!ok) {
                if (bad < 5) printf("x=%a s=%a q=%a x/s=%a\n", x, s, q, t);
                ++bad;
            }
        }
    }
    printf("cases %ld mismatches %ld\n", n, bad);
    return bad != 0;
}
