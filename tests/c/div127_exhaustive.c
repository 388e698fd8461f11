/* Exhaustive check of the division-free row scale of the mixed decode kernel:
 * for every finite FP32 a >= 1e-8, q0 = RN(a * RN(1/127)) followed by one
 * exact-remainder correction q = RN(q0 + RN(a - 127 q0) * RN(1/127)) equals
 * the IEEE quotient RN(a / 127).  Prints the number of values checked and of
 * mismatches; exits 1 on any mismatch.  Built with -ffp-contract=off so that
 * every operation rounds once, as on the GPU. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

int main(void) {
    const float y = 1.0f / 127.0f;
    const float lo = 1e-8f;
    uint32_t b;
    memcpy(&b, &lo, 4);
    unsigned long long n = 0, bad = 0;
    for (;; ++b) {
        float a;
        memcpy(&a, &b, 4);
        if (!isfinite(a)) break;
        const float ref = a / 127.0f;
        const float q0 = a * y;
        const float q = fmaf(fmaf(-q0, 127.0f, a), y, q0);
        if (memcmp(&q, &ref, 4) != 0) ++bad;
        ++n;
    }
    printf("%llu %llu\n", n, bad);
    return bad != 0;
}
