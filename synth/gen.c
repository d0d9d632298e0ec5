/*
 * Seeded synthetic inputs for the routed-MoE workloads.
 *
 * This file holds no MoE arithmetic: it only turns (seed, tensor tag, slab,
 * element index) into numbers.  Both the CPU oracle (through the Python
 * wrapper in synth/__init__.py) and the GPU path (through the bit-identical
 * torch restatement in the same module) consume what it defines.
 *
 * Generator, stated once so that any implementation can be checked:
 *   fmix32(h)      : the MurmurHash3 32-bit finaliser
 *                    (h ^= h>>16; h *= 0x85ebca6b; h ^= h>>13;
 *                     h *= 0xc2b2ae35; h ^= h>>16), arithmetic mod 2^32.
 *   key(seed,tag,slab) = fmix32(fmix32(fmix32(seed ^ 0x9e3779b9)
 *                         ^ (tag*0x85ebca77 + 0x27d4eb2f))
 *                         ^ (slab*0xc2b2ae3d + 0x165667b1))
 *   draw(key, i)   = fmix32(key ^ fmix32(i + 0x61c88647))
 *   normal(idx)    : a = draw(key, 2 idx), b = draw(key, 2 idx + 1);
 *                    s = sum of the four 16-bit halves of a and b
 *                    (Irwin-Hall sum of four discrete uniforms);
 *                    c = 2 s - 262140 (an even integer, exact in fp32);
 *                    value = fp32(c) * scale, one IEEE round-to-nearest
 *                    multiply, scale = fp32(sigma / 75674.44...) so that
 *                    the value has mean 0 and standard deviation sigma.
 *   bf16           : round-to-nearest-even of the fp32 value.
 *   uniform(i, n)  = (draw(key, i) * n) >> 32  (64-bit product).
 */
#include <stdint.h>
#include <string.h>

static inline uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85ebca6bu;
    h ^= h >> 13;
    h *= 0xc2b2ae35u;
    h ^= h >> 16;
    return h;
}

uint32_t synth_key(uint32_t seed, uint32_t tag, uint32_t slab) {
    uint32_t k = fmix32(seed ^ 0x9e3779b9u);
    k = fmix32(k ^ (tag * 0x85ebca77u + 0x27d4eb2fu));
    k = fmix32(k ^ (slab * 0xc2b2ae3du + 0x165667b1u));
    return k;
}

static inline uint32_t draw(uint32_t key, uint32_t i) {
    return fmix32(key ^ fmix32(i + 0x61c88647u));
}

uint32_t synth_draw(uint32_t key, uint32_t i) { return draw(key, i); }

static inline float normal_at(uint32_t key, uint32_t idx, float scale) {
    uint32_t a = draw(key, 2u * idx), b = draw(key, 2u * idx + 1u);
    int32_t s = (int32_t)((a & 0xffffu) + (a >> 16) + (b & 0xffffu) + (b >> 16));
    int32_t c = 2 * s - 262140;
    return (float)c * scale;
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* values idx in [start, start+count) of one slab, as fp32 */
void synth_normal_f32(uint32_t key, uint32_t start, uint32_t count, float scale,
                      float* out) {
    for (uint32_t i = 0; i < count; ++i) out[i] = normal_at(key, start + i, scale);
}

/* values idx in [start, start+count) of one slab, rounded to bf16 (raw bits) */
void synth_normal_bf16(uint32_t key, uint32_t start, uint32_t count, float scale,
                       uint16_t* out) {
    for (uint32_t i = 0; i < count; ++i)
        out[i] = f32_to_bf16_rne(normal_at(key, start + i, scale));
}

/* uniform integers in [0, n) */
void synth_uniform_i32(uint32_t key, uint32_t start, uint32_t count, uint32_t n,
                       int32_t* out) {
    for (uint32_t i = 0; i < count; ++i)
        out[i] = (int32_t)(((uint64_t)draw(key, start + i) * (uint64_t)n) >> 32);
}

/* Durstenfeld shuffle of 0..n-1; the j-th swap partner is uniform(i, i+1). */
void synth_permutation(uint32_t key, int32_t n, int32_t* out) {
    for (int32_t i = 0; i < n; ++i) out[i] = i;
    for (int32_t i = n - 1; i > 0; --i) {
        int32_t j = (int32_t)(((uint64_t)draw(key, (uint32_t)i) * (uint64_t)(i + 1)) >> 32);
        int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}

/*
 * Rows of a token-id -> expert-id table: row v holds k distinct experts of E,
 * the first k picks of a partial Fisher-Yates shuffle of 0..E-1 keyed by
 * synth_key(seed, tag, v).  scratch must hold E ints.
 */
void synth_distinct_rows(uint32_t seed, uint32_t tag, int64_t v0, int64_t nrows,
                         int32_t E, int32_t k, int32_t* scratch, int32_t* out) {
    for (int32_t e = 0; e < E; ++e) scratch[e] = e;
    for (int64_t r = 0; r < nrows; ++r) {
        uint32_t key = synth_key(seed, tag, (uint32_t)(v0 + r));
        int32_t pick[64];
        for (int32_t j = 0; j < k; ++j) {
            int32_t span = E - j;
            int32_t q = j + (int32_t)(((uint64_t)draw(key, (uint32_t)j) * (uint64_t)span) >> 32);
            pick[j] = q;
            int32_t t = scratch[j];
            scratch[j] = scratch[q];
            scratch[q] = t;
            out[r * k + j] = scratch[j];
        }
        for (int32_t j = k - 1; j >= 0; --j) { /* undo, so scratch is identity again */
            int32_t q = pick[j];
            int32_t t = scratch[j];
            scratch[j] = scratch[q];
            scratch[q] = t;
        }
    }
}
