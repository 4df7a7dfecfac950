/*
 * gen.c -- counter-based generator of seeded synthetic bf16 tensors.
 *
 * Holds none of the Float8 method's arithmetic: it only draws the inputs
 * (activations X, weights W, output gradients dY) that both the CUDA library
 * and the CPU oracle are fed.  The steps are stated in workloads/__init__.py.
 *
 * splitmix64: Steele, Lea, Flood, "Fast splittable pseudorandom number
 * generators" (OOPSLA 2014).  Box-Muller for normals, inverse CDF for Laplace.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static double uniform01(uint64_t key, uint64_t i, uint64_t j) {
    uint64_t z = splitmix64(key + 2ull * i + j);
    return ((double)(z >> 11) + 0.5) * 0x1.0p-53;
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    b = b + 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

/* dist: 0 = normal(0, param) (param = standard deviation),
 *       1 = Laplace(0, param) (param = scale b). */
void gen_bf16(uint16_t *out, int64_t n, uint64_t key, int dist, double param) {
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double u0 = uniform01(key, (uint64_t)i, 0);
        double u1 = uniform01(key, (uint64_t)i, 1);
        double x;
        if (dist == 0) {
            x = sqrt(-2.0 * log(u0)) * cos(two_pi * u1) * param;
        } else {
            double t = u0 - 0.5;
            double sg = (t > 0) ? 1.0 : ((t < 0) ? -1.0 : 0.0);
            x = -param * sg * log1p(-2.0 * fabs(t));
        }
        out[i] = f32_to_bf16_rne((float)x);
    }
}
