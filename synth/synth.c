/*
 * synth.c -- seeded, counter-based synthetic inputs shared by the tests, the
 * bench and the oracle's CPU baseline.  It holds none of the products'
 * arithmetic: it only draws numbers.
 *
 * Element i of tensor t under seed s uses two 64-bit draws,
 *     u = splitmix64(s ^ splitmix64(t) ^ (2i)),  v = splitmix64(s ^ splitmix64(t) ^ (2i+1)),
 * where splitmix64 is the published finaliser of Steele, Lea and Flood
 * ("Fast splittable pseudorandom number generators", OOPSLA 2014).  The two
 * draws become a standard normal by the Box-Muller transform in double,
 *     z = sqrt(-2 ln u1) cos(2 pi u2),  u1 = ((u >> 11) + 1) 2^-53,  u2 = (v >> 11) 2^-53,
 * scaled by sigma.  f32 outputs are (float)(sigma z); f16 outputs are the C
 * compiler's own IEEE conversion (_Float16)(sigma z) -- the weights are inputs
 * handed to the method, not something the method computes.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t z)
{
    z += 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

static inline double normal_at(uint64_t key, uint64_t i)
{
    uint64_t u = splitmix64(key ^ (2 * i));
    uint64_t v = splitmix64(key ^ (2 * i + 1));
    double u1 = (double)((u >> 11) + 1) * 0x1p-53;
    double u2 = (double)(v >> 11) * 0x1p-53;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

/* out[j] = element (offset + j) of tensor `tensor`, for j < n. */
void synth_normal_f32(uint64_t seed, uint64_t tensor, double sigma, int64_t offset, int64_t n,
                      float *out)
{
    uint64_t key = seed ^ splitmix64(tensor);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; j++) out[j] = (float)(sigma * normal_at(key, (uint64_t)(offset + j)));
}

void synth_normal_f16(uint64_t seed, uint64_t tensor, double sigma, int64_t offset, int64_t n,
                      uint16_t *out)
{
    uint64_t key = seed ^ splitmix64(tensor);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; j++) {
        _Float16 h = (_Float16)(sigma * normal_at(key, (uint64_t)(offset + j)));
        memcpy(&out[j], &h, 2);
    }
}

/* Raw draws, for tests of the generator itself. */
uint64_t synth_splitmix64(uint64_t z) { return splitmix64(z); }
