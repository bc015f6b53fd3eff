/* CPU version of synth.normal_tensor (seeded input generation only; no arithmetic of the
 * verify method): for element i of a tensor with 64-bit key k,
 *   h_j = splitmix64(k + (3 i + j) * 0x9E3779B97F4A7C15), j = 1, 2, 3 (wrapping 64-bit),
 *   n   = 2 * (sum of the twelve 16-bit fields of h_1..h_3) - 12 * 65535,
 *   v   = float(n) * scale (one IEEE single multiply), rounded to bfloat16 (nearest, ties
 *         to even) when bf16 != 0,
 * written as doubles.  Bit-identical to the torch implementation (tested). */
#include <stdint.h>
#include <string.h>

static inline uint64_t splitmix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void synth_normal_f64(uint64_t key, int64_t start, int64_t n, float scale, int bf16, double* out) {
    for (int64_t i = 0; i < n; ++i) {
        const uint64_t idx = (uint64_t)(start + i);
        int64_t total = 0;
        for (uint64_t j = 1; j <= 3; ++j) {
            const uint64_t h = splitmix64((idx * 3u + j) * 0x9E3779B97F4A7C15ull + key);
            total += (int64_t)(h & 0xFFFFu) + (int64_t)((h >> 16) & 0xFFFFu) + (int64_t)((h >> 32) & 0xFFFFu) +
                     (int64_t)((h >> 48) & 0xFFFFu);
        }
        const float num = (float)(total * 2 - 12 * 65535);
        float v = num * scale;
        if (bf16) {
            uint32_t b;
            memcpy(&b, &v, 4);
            b += 0x7FFFu + ((b >> 16) & 1u);
            b &= 0xFFFF0000u;
            memcpy(&v, &b, 4);
        }
        out[i] = (double)v;
    }
}
