/* Exhaustive check of the quantizer's division by 127 (host arithmetic).
 *
 * The kernels compute d = RN(a / 127) without a divide: q0 = RN(a y) with
 * y = RN(1/127), the exact remainder r = a - 127 q0 (one fma), then
 * q = RN(q0 + r y) (one fma).  This program checks q == a / 127.0f (IEEE
 * division) for every non-negative finite a in the binades where rounding can
 * depend on the exponent, and in one binade that stands for all the others:
 *  - biased exponent 0..32: subnormal a and quotients, and every a whose
 *    remainder r can be subnormal (r is a multiple of ulp(q0) ~ 2^(e - 30));
 *  - 250..254: the top of the range;
 *  - 127: [1, 2).  For exponents 33..249 every intermediate is normal, so the
 *    whole computation scales exactly by powers of two from this binade.
 * Arguments: none.  Exit status 0 when every input agrees. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int main(void)
{
    volatile float divisor = 127.0f;
    const float y = 0x1.020408p-7f;
    if (y != 1.0f / divisor) {
        printf("constant is not RN(1/127)\n");
        return 2;
    }
    static const int ranges[][2] = {{0, 32}, {127, 127}, {250, 254}};
    long checked = 0, bad = 0;
    for (int k = 0; k < 3; k++) {
        for (uint32_t e = (uint32_t)ranges[k][0]; e <= (uint32_t)ranges[k][1]; e++) {
            for (uint32_t m = 0; m < (1u << 23); m++) {
                const float a = from_bits((e << 23) | m);
                const float q0 = a * y;
                const float r = fmaf(-q0, 127.0f, a);
                const float q = fmaf(r, y, q0);
                const float ref = a / divisor;
                checked++;
                if (memcmp(&q, &ref, sizeof q) != 0) {
                    if (bad < 5) printf("mismatch a=%a q=%a ref=%a\n", a, q, ref);
                    bad++;
                }
            }
        }
    }
    printf("checked %ld inputs, %ld mismatches\n", checked, bad);
    return bad != 0;
}
