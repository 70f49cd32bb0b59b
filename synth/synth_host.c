/*
 * Seeded synthetic inputs for the MXFP4 MoE layer: host-side byte generator.
 *
 * This file holds none of the method's arithmetic. It only fills expert
 * records with reproducible pseudo-random bytes, so that the CPU oracle and
 * the CUDA path can be fed identical inputs. The device-side twin lives in
 * synth_dev.cu and must produce bit-identical bytes (a CPU/GPU test checks it).
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), used counter-based: output i
 * of a stream whose state starts at `key` is mix64(key + (i + 1) * GAMMA).
 *
 * Record layout (per expert, contiguous; d = d_model, f = d_ff):
 *   [gate codes f*d/2][gate scales f*d/32][up codes f*d/2][up scales f*d/32]
 *   [down codes d*f/2][down scales d*f/32][zero padding up to `stride`]
 * Code bytes are uniform in 0..255 (two uniform 4-bit E2M1 codes, low nibble
 * first). Scale bytes are E8M0 exponents 127 + e with e uniform in {-6..-2}.
 */
#include <stdint.h>
#include <string.h>

#define K3S_GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t k3s_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Stream key for (seed, kind, layer, expert, matrix). */
uint64_t k3s_key(uint64_t seed, uint32_t kind, uint32_t layer, uint32_t expert, uint32_t matrix) {
    uint64_t tag = ((uint64_t)(kind & 0xFFu) << 56) | ((uint64_t)(layer & 0xFFFFu) << 40) |
                   ((uint64_t)(expert & 0xFFFFFFFFu) << 8) | (uint64_t)(matrix & 0xFFu);
    return k3s_mix64(seed * K3S_GAMMA ^ k3s_mix64(tag));
}

uint64_t k3s_value(uint64_t key, uint64_t i) { return k3s_mix64(key + (i + 1) * K3S_GAMMA); }

/* Bytes of one expert record: 3 * d * f * 17 / 32. */
int64_t k3s_record_bytes(int64_t d, int64_t f) { return 3 * (d * f / 2 + d * f / 32); }

enum { K3S_KIND_CODES = 1, K3S_KIND_SCALES = 2 };

static void fill_codes(uint8_t* dst, int64_t n, uint64_t key) {
    int64_t i = 0;
    for (; i + 8 <= n; i += 8) {
        uint64_t w = k3s_value(key, (uint64_t)(i / 8));
        uint8_t le[8];
        for (int b = 0; b < 8; ++b) le[b] = (uint8_t)(w >> (8 * b)); /* byte b = bits 8b..8b+7 */
        memcpy(dst + i, le, 8);
    }
    if (i < n) {
        uint64_t w = k3s_value(key, (uint64_t)(i / 8));
        for (int b = 0; i + b < n; ++b) dst[i + b] = (uint8_t)(w >> (8 * b));
    }
}

static void fill_scales(uint8_t* dst, int64_t n, uint64_t key) {
    for (int64_t i = 0; i < n; ++i) {
        uint64_t v = k3s_value(key, (uint64_t)i);
        uint32_t e5 = (uint32_t)(((v >> 32) * 5ull) >> 32); /* uniform in 0..4 */
        dst[i] = (uint8_t)(121u + e5);                      /* 127 + (-6 .. -2) */
    }
}

/*
 * Fill `n` consecutive expert records (expert ids e0 .. e0+n-1 of `layer`)
 * into dst, `stride` bytes apart. Shared experts use ids n_routed + s.
 * Returns 0, or -1 on a bad argument.
 */
int k3s_fill_records(uint8_t* dst, int64_t d, int64_t f, uint64_t seed, uint32_t layer,
                     uint32_t e0, int64_t n, int64_t stride) {
    int64_t rec = k3s_record_bytes(d, f);
    if (!dst || d <= 0 || f <= 0 || (d % 32) || (f % 32) || stride < rec || n < 0) return -1;
    int64_t nc = d * f / 2, ns = d * f / 32;
    for (int64_t r = 0; r < n; ++r) {
        uint8_t* p = dst + r * stride;
        uint32_t e = e0 + (uint32_t)r;
        for (uint32_t m = 0; m < 3; ++m) {
            uint8_t* pm = p + (int64_t)m * (nc + ns);
            fill_codes(pm, nc, k3s_key(seed, K3S_KIND_CODES, layer, e, m));
            fill_scales(pm + nc, ns, k3s_key(seed, K3S_KIND_SCALES, layer, e, m));
        }
        if (stride > rec) memset(p + rec, 0, (size_t)(stride - rec));
    }
    return 0;
}
