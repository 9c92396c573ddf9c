/*
 * Exhaustive check of the oracle's E2M1 and E4M3 encoders over every binary32
 * bit pattern, against a brute-force definition written independently here:
 * the encoded value is the representable value nearest to v (ties: the code
 * with the even significand), magnitudes beyond the largest finite value
 * saturate to it, and the sign of zero is kept.
 *
 * Includes the oracle source so that the functions under test are the
 * oracle's own.  Prints "<e2m1 mismatches> <e4m3 mismatches> <checked>".
 */
#include "../../oracle/h3fp4_oracle.c"

#include <stdio.h>

/* positive magnitudes of the codes, built from the bit fields */
static double e2m1_mag_bf(int c)
{
    int e = (c >> 1) & 3, m = c & 1;
    return e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
}

static double e4m3_mag_bf(int c)
{
    int e = (c >> 3) & 15, m = c & 7;
    return e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
}

static int nearest(double a, const double *mags, int n)
{
    /* mags ascending: bisect for the last code with magnitude <= a, then take
     * the closer of it and its successor; on a tie, the even code */
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (mags[mid] <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    if (lo == n - 1)
        return lo;
    double d0 = a - mags[lo], d1 = mags[lo + 1] - a;
    if (d0 < d1)
        return lo;
    if (d1 < d0)
        return lo + 1;
    return (lo & 1) == 0 ? lo : lo + 1;
}

int main(void)
{
    double e2[8], e4[127];
    for (int c = 0; c < 8; ++c)
        e2[c] = e2m1_mag_bf(c);
    for (int c = 0; c < 127; ++c)
        e4[c] = e4m3_mag_bf(c);
    long long bad2 = 0, bad4 = 0, checked = 0;
#pragma omp parallel for reduction(+ : bad2, bad4, checked) schedule(static)
    for (long long hi = 0; hi < 65536; ++hi) {
        for (long long lo = 0; lo < 65536; ++lo) {
            uint32_t u = (uint32_t)((hi << 16) | lo);
            float f;
            memcpy(&f, &u, 4);
            if (f != f)
                continue;
            double v = (double)f;
            double a = fabs(v);
            int neg = signbit(v) != 0;
            int c2 = (a >= 6.0) ? 7 : nearest(a, e2, 8);
            int c4 = (a >= 448.0) ? 126 : nearest(a, e4, 127);
            uint8_t want2 = (uint8_t)((neg ? 8 : 0) | c2);
            uint8_t want4 = (uint8_t)((neg ? 0x80 : 0) | c4);
            bad2 += orc_e2m1_encode(v) != want2;
            bad4 += orc_e4m3_encode(v) != want4;
            checked += 1;
        }
    }
    printf("%lld %lld %lld\n", bad2, bad4, checked);
    return 0;
}
