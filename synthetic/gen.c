/*
 * Seeded synthetic inputs for the attention workloads (shared by the tests, the bench and the
 * oracle's callers). This file holds no attention arithmetic: only a counter-based random number
 * generator, the Box-Muller transform and the rounding of fp32 values to fp16 / bf16 bit patterns.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014). The n-th output (n >= 0) of the sequence whose state starts at s is
 * mix(s + (n + 1) * GAMMA); being a pure function of (s, n), any element of any tensor can be
 * regenerated on its own, independent of thread count.
 *
 * Element stream of one tensor: state s_t = sm64_at(seed, tensor_id). Logical element index e of a
 * [B,H,N,d] tensor (SDPA order, e = ((b*H + h)*N + n)*d + c) belongs to pair p = e / 2; the pair
 * draws w1 = sm64_at(s_t, 2p), w2 = sm64_at(s_t, 2p + 1) and forms u1 = ((w1 >> 11) + 1) * 2^-53 in
 * (0, 1], u2 = (w2 >> 11) * 2^-53 in [0, 1). Box-Muller (G. Box, M. Muller, Ann. Math. Stat. 1958)
 * gives r = sqrt(-2 ln u1), theta = 2 pi u2, z_{2p} = r cos theta, z_{2p+1} = r sin theta in double,
 * then z is rounded to fp32, multiplied in fp32 by `mul` (1 for N(0,1); 3 for the peaked-K workload)
 * and rounded once, to nearest even, to the storage type.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_sm64_at(uint64_t state, uint64_t n) { return sm64_mix(state + (n + 1) * SM64_GAMMA); }

/* fp32 -> fp16 bits, round to nearest even (IEEE 754 binary16, subnormals kept, overflow -> inf). */
static uint16_t f32_to_f16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7fffffffu;
    if (ax > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);            /* NaN */
    if (ax >= 0x47800000u) return (uint16_t)(sign | 0x7c00u);           /* >= 65536: inf */
    if (ax < 0x33000000u) return (uint16_t)sign;                        /* < 2^-25: rounds to 0 */
    int32_t e = (int32_t)(ax >> 23) - 127;                              /* unbiased exponent */
    uint32_t m = (ax & 0x7fffffu) | 0x800000u;                          /* 24-bit significand */
    /* target: integer multiple of 2^(max(e,-14) - 10) */
    int32_t shift = (e < -14 ? (-14 - e) : 0) + 13;                     /* bits dropped from m */
    uint32_t kept = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (kept & 1u))) kept++;
    uint32_t bits;
    if (e < -14) {
        bits = kept;                                                    /* subnormal (may carry to normal) */
    } else {
        /* kept in [2^10, 2^11]; carry into the exponent is handled by the addition */
        bits = ((uint32_t)(e + 15) << 10) + (kept - 0x400u);
    }
    if (bits >= 0x7c00u) bits = 0x7c00u;                                /* rounded up to inf */
    return (uint16_t)(sign | bits);
}

/* fp32 -> bf16 bits, round to nearest even. */
static uint16_t f32_to_bf16_bits(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((x >> 16) | 0x40u); /* quiet NaN */
    uint32_t lsb = (x >> 16) & 1u;
    x += 0x7fffu + lsb;
    return (uint16_t)(x >> 16);
}

uint16_t synth_f32_to_f16(float f) { return f32_to_f16_bits(f); }
uint16_t synth_f32_to_bf16(float f) { return f32_to_bf16_bits(f); }

/* The fp32 value of logical element e of tensor stream `state` (before the storage rounding). */
static inline float synth_value(uint64_t state, int64_t e, float mul) {
    uint64_t p = (uint64_t)e >> 1;
    uint64_t w1 = sm64_mix(state + (2 * p + 1) * SM64_GAMMA);
    uint64_t w2 = sm64_mix(state + (2 * p + 2) * SM64_GAMMA);
    double u1 = (double)((w1 >> 11) + 1) * 0x1p-53;
    double u2 = (double)(w2 >> 11) * 0x1p-53;
    double r = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586476925286766559 * u2;
    double z = (e & 1) ? r * sin(th) : r * cos(th);
    float zf = (float)z;
    return zf * mul;
}

/*
 * Fill `out` with the B*H*N*d elements of tensor `tensor_id` under `seed`, stored in `layout`
 * (0: [B,H,N,d]; 1: token-major [B,N,H,d]) as `dtype` (0: fp16, 1: bf16, 2: fp32 bits in pairs of
 * uint16). Only tokens [n0, n0 + n_cnt) are written, packed as a [B,H,n_cnt,d] or [B,n_cnt,H,d]
 * array; the values are those of the full tensor, so a chunk equals the slice of the whole.
 */
void synth_normal(void* out, int64_t B, int64_t H, int64_t N, int64_t d, int64_t n0, int64_t n_cnt,
                  int layout, int dtype, uint64_t seed, uint64_t tensor_id, float mul) {
    uint64_t state = synth_sm64_at(seed, tensor_id);
    int64_t rows = B * H * n_cnt;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t b, h, n;
        if (layout == 0) {
            b = r / (H * n_cnt);
            h = (r / n_cnt) % H;
            n = r % n_cnt;
        } else {
            b = r / (n_cnt * H);
            n = (r / H) % n_cnt;
            h = r % H;
        }
        int64_t e0 = ((b * H + h) * N + (n0 + n)) * d;
        for (int64_t c = 0; c < d; ++c) {
            float f = synth_value(state, e0 + c, mul);
            if (dtype == 0) {
                ((uint16_t*)out)[r * d + c] = f32_to_f16_bits(f);
            } else if (dtype == 1) {
                ((uint16_t*)out)[r * d + c] = f32_to_bf16_bits(f);
            } else {
                ((float*)out)[r * d + c] = f;
            }
        }
    }
}

/* Raw 64-bit draws: out[i] = sm64_at(sm64_at(seed, stream_id), first + i). */
void synth_words(uint64_t* out, int64_t n, uint64_t seed, uint64_t stream_id, uint64_t first) {
    uint64_t state = synth_sm64_at(seed, stream_id);
    for (int64_t i = 0; i < n; ++i) out[i] = synth_sm64_at(state, first + (uint64_t)i);
}
