/*
 * Seeded synthetic inputs for the MXFP4 MoE layer: one counter-based generator,
 * written once, compiled for the host (synth_host.c) and for the GPU
 * (synth_cuda.cu).  It holds no arithmetic of the method itself: no MX
 * quantisation, no routing, no GEMM.  Everything here is integer hashing plus
 * IEEE operations that round identically on any conforming host or device, so
 * both builds produce bit-identical tensors.
 *
 * Generator
 *   mix64:  the SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable
 *           pseudorandom number generators", OOPSLA 2014).
 *   key    = mix64(seed * G + stream * C + D)      one key per (seed, tensor)
 *   bits_i = mix64(key + i * G)                    counter mode
 *   normal_i: Irwin-Hall approximation of N(0, 1): the sum of twelve uniform
 *           variates (k + 1/2) / 2^16, k a 16-bit lane of bits_{3i..3i+2},
 *           minus 6.  Mean 0, variance 1 - 2^-32, support [-6, 6].  The sum
 *           is an integer divided by 2^16, so it is exact in fp32 and fp64.
 *
 * Derived values (all rounded once, round-to-nearest-even):
 *   normal_f32(sigma) = fp32( fp64(sigma) * normal_i )
 *   bf16 values       = bf16_rne( fp32(normal_i) )   (fp32(normal_i) is exact)
 */
#ifndef MOE_SYNTH_H
#define MOE_SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_FN __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ull
#define SYNTH_STREAM 0xD1B54A32D192ED03ull
#define SYNTH_OFFSET 0x632BE59BD9B4E019ull

/* Tensor streams.  A tensor's stream id keeps every tensor of one seed on its
 * own sequence. */
enum {
    SYNTH_STREAM_X = 1,        /* activations x [T, H], bf16, N(0,1)        */
    SYNTH_STREAM_LOGITS = 2,   /* router logits [T, Eg], fp32, N(0,1)+bias  */
    SYNTH_STREAM_ROUTER = 3,   /* router matrix Wr [H, Eg], fp32            */
    SYNTH_STREAM_W1 = 4,       /* W1 [expert, 2I, H], fp32                  */
    SYNTH_STREAM_W2 = 5,       /* W2 [expert, H, I], fp32                   */
    SYNTH_STREAM_SHARED = 6    /* shared-expert gate logit [T], bf16        */
};

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

SYNTH_FN uint64_t synth_key(uint64_t seed, uint64_t stream) {
    return synth_mix64(seed * SYNTH_GOLDEN + stream * SYNTH_STREAM + SYNTH_OFFSET);
}

SYNTH_FN uint64_t synth_bits(uint64_t key, uint64_t ctr) {
    return synth_mix64(key + ctr * SYNTH_GOLDEN);
}

/* Irwin-Hall(12) - 6, exact: returns an integer n with value n / 65536. */
SYNTH_FN int32_t synth_normal_q16(uint64_t key, uint64_t i) {
    int64_t s = 0;
    for (int c = 0; c < 3; ++c) {
        uint64_t b = synth_bits(key, 3ull * i + (uint64_t)c);
        s += (int64_t)(b & 0xFFFFull) + (int64_t)((b >> 16) & 0xFFFFull) +
             (int64_t)((b >> 32) & 0xFFFFull) + (int64_t)(b >> 48);
    }
    /* sum_{12} (k + 1/2)/2^16 - 6 = (s + 6 - 6 * 2^16) / 2^16 */
    return (int32_t)(s + 6 - 393216);
}

SYNTH_FN double synth_normal(uint64_t key, uint64_t i) {
    return (double)synth_normal_q16(key, i) * (1.0 / 65536.0);
}

SYNTH_FN uint32_t synth_f32_bits(float f) {
    union { float f; uint32_t u; } v;
    v.f = f;
    return v.u;
}

/* fp32 -> bf16, round to nearest even (inputs here are finite). */
SYNTH_FN uint16_t synth_bf16_rne(float f) {
    uint32_t u = synth_f32_bits(f);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* fp64 -> fp32 with one IEEE rounding, identical on host and device. */
SYNTH_FN float synth_to_f32(double d) {
#if defined(__CUDA_ARCH__)
    return __double2float_rn(d);
#else
    return (float)d;
#endif
}

SYNTH_FN double synth_mul(double a, double b) {
#if defined(__CUDA_ARCH__)
    return __dmul_rn(a, b);
#else
    return a * b;
#endif
}

SYNTH_FN double synth_add(double a, double b) {
#if defined(__CUDA_ARCH__)
    return __dadd_rn(a, b);
#else
    return a + b;
#endif
}

/* fp32( sigma * N_i ) */
SYNTH_FN float synth_normal_f32(uint64_t key, uint64_t i, double sigma) {
    return synth_to_f32(synth_mul(sigma, synth_normal(key, i)));
}

/* fp32( N_i + bias ) */
SYNTH_FN float synth_normal_plus_f32(uint64_t key, uint64_t i, double bias) {
    return synth_to_f32(synth_add(synth_normal(key, i), bias));
}

/* bf16( N_i ) */
SYNTH_FN uint16_t synth_normal_bf16(uint64_t key, uint64_t i) {
    return synth_bf16_rne((float)synth_normal(key, i));
}

#endif /* MOE_SYNTH_H */
