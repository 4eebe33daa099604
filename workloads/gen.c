/*
 * Seeded synthetic input generator shared by the tests, the bench and the
 * CPU oracle's callers.  It holds none of the attention arithmetic: it only
 * turns (seed, stream, element index) into a bf16 bit pattern.
 *
 * Each element is drawn independently of every other one, so any slice of a
 * large tensor can be generated on its own and in parallel, and the result
 * does not depend on the thread count or on the platform:
 *
 *   1. Three 64-bit words come from the splitmix64 finaliser (Steele, Lea and
 *      Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014)
 *      applied to a per-(seed, stream) key plus a Weyl sequence in the
 *      element index.
 *   2. The twelve 16-bit fields of those words are summed.  The sum of twelve
 *      independent uniforms on {0..65535} has mean 12*32767.5 and variance
 *      65536^2-1 (Irwin-Hall); subtracting the mean and dividing by the
 *      standard deviation gives an approximately N(0,1) value (support +-6).
 *   3. That double is rounded to float32 and then to bf16 (the top 16 bits of
 *      a float32) with round-to-nearest-even.
 *
 * Every operation is an exact integer operation or a single correctly rounded
 * IEEE operation, so the bits are identical on x86-64 and AArch64.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static const uint64_t WL_GAMMA = 0x9E3779B97F4A7C15ULL;

static inline uint64_t wl_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t wl_key(uint64_t seed, uint64_t stream) {
    return wl_mix64(wl_mix64(seed * WL_GAMMA + 0x632BE59BD9B4E019ULL) ^ (stream * 0xD1B54A32D192ED03ULL));
}

/* float32 -> bf16 bits, round to nearest, ties to even (inputs are finite). */
static inline uint16_t wl_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline uint16_t wl_one(uint64_t key, uint64_t index, double inv_sd) {
    int64_t sum = 0;
    for (int r = 0; r < 3; ++r) {
        uint64_t w = wl_mix64(key + (3 * index + (uint64_t)r + 1) * WL_GAMMA);
        sum += (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) +
               (int64_t)((w >> 32) & 0xFFFF) + (int64_t)(w >> 48);
    }
    /* 12 * 32767.5 = 393210 exactly; (sum - 393210) is an exact integer. */
    double z = (double)(sum - 393210) * inv_sd;
    return wl_f32_to_bf16((float)z);
}

/* out[j] = bf16 draw for element (offset + j) of stream `stream` under `seed`. */
void wl_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset,
                    int num_threads) {
    const uint64_t key = wl_key(seed, stream);
    const double inv_sd = 1.0 / sqrt(65536.0 * 65536.0 - 1.0);
#ifdef _OPENMP
    if (num_threads < 1) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(num_threads)
#endif
    for (int64_t j = 0; j < n; ++j) out[j] = wl_one(key, (uint64_t)(offset + j), inv_sd);
    (void)num_threads;
}

/* Raw 64-bit draws of the same family (used for cheap seeded integer choices). */
void wl_u64(uint64_t* out, int64_t n, uint64_t seed, uint64_t stream, int64_t offset) {
    const uint64_t key = wl_key(seed, stream);
    for (int64_t j = 0; j < n; ++j) out[j] = wl_mix64(key + ((uint64_t)(offset + j) + 1) * WL_GAMMA);
}

/* Fill n uint16 with a constant (poisoning large caches without numpy temporaries). */
void wl_fill_u16(uint16_t* out, int64_t n, uint16_t value, int num_threads) {
#ifdef _OPENMP
    if (num_threads < 1) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(num_threads)
#endif
    for (int64_t j = 0; j < n; ++j) out[j] = value;
    (void)num_threads;
}

int wl_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
