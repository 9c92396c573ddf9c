/* Host check of the division-free quotient the pack kernels use:
 *   r = RN(1/b), q = RN(a r), e = RN(q b - a) (fused), q' = RN(q - e r) (fused)
 * must equal the IEEE quotient RN(a / b).  Runs over every bf16 significand
 * of a (128), every STRIDE-th f32 significand of b in [1, 2) and a-exponents
 * giving quotients in [2^-5, 2^5), both signs, plus signed zeros; by
 * power-of-two scaling the significands decide the result at every exponent
 * where the residual keeps its bits.  Prints "checks N mismatches K".
 *
 *   rcp_quotient_check [STRIDE]
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u)
{
    float x;
    memcpy(&x, &u, 4);
    return x;
}

static uint32_t bits(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    return u;
}

static float quotient(float a, float b, float r)
{
    const float q = a * r;
    const float e = fmaf(q, b, -a);
    return fmaf(-e, r, q);
}

int main(int argc, char **argv)
{
    const long stride = argc > 1 ? atol(argv[1]) : 1;
    long checks = 0, bad = 0;
#pragma omp parallel for reduction(+ : checks, bad) schedule(dynamic, 256)
    for (long ms = 0; ms < (1L << 23); ms += stride) {
        const float b = from_bits(0x3F800000u | (uint32_t)ms);
        const float r = 1.0f / b;
        for (int k = -4; k <= 4; ++k) {
            for (uint32_t my = 0; my < 128; ++my) {
                const float a = from_bits(((uint32_t)(127 + k) << 23) | (my << 16));
                checks += 2;
                bad += bits(quotient(a, b, r)) != bits(a / b);
                bad += bits(quotient(-a, b, r)) != bits(-a / b);
            }
        }
    }
    const float zeros[2] = {0.0f, -0.0f};
    for (int i = 0; i < 2; ++i) {
        checks += 1;
        bad += bits(quotient(zeros[i], 1.2345f, 1.0f / 1.2345f)) != bits(zeros[i]);
    }
    printf("checks %ld mismatches %ld\n", checks, bad);
    return bad != 0;
}
