/*
 * Host build of the seeded input generator (see synth.h).  Plain C, one thread.
 * Fills caller-owned host arrays; no method arithmetic.
 */
#include "synth.h"

/* x [T, H] bf16 bits, rows t0 .. t0 + T - 1 of the seed's token stream. */
void synth_x(uint64_t seed, int64_t t0, int64_t T, int64_t H, uint16_t* out) {
    uint64_t key = synth_key(seed, SYNTH_STREAM_X);
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h)
            out[t * H + h] = synth_normal_bf16(key, (uint64_t)((t0 + t) * H + h));
}

/* logits [T, Eg] fp32 = fp32(N(0,1) + bias[e]); bias may be NULL (zero). */
void synth_logits(uint64_t seed, int64_t t0, int64_t T, int64_t Eg, const double* bias, float* out) {
    uint64_t key = synth_key(seed, SYNTH_STREAM_LOGITS);
    for (int64_t t = 0; t < T; ++t)
        for (int64_t e = 0; e < Eg; ++e)
            out[t * Eg + e] = synth_normal_plus_f32(key, (uint64_t)((t0 + t) * Eg + e), bias ? bias[e] : 0.0);
}

/* router matrix Wr [H, Eg] fp32 = fp32(sigma * N(0,1)). */
void synth_router(uint64_t seed, int64_t H, int64_t Eg, double sigma, float* out) {
    uint64_t key = synth_key(seed, SYNTH_STREAM_ROUTER);
    for (int64_t i = 0; i < H * Eg; ++i) out[i] = synth_normal_f32(key, (uint64_t)i, sigma);
}

/* shared-expert gate logit [T] bf16 bits. */
void synth_shared_logit(uint64_t seed, int64_t t0, int64_t T, uint16_t* out) {
    uint64_t key = synth_key(seed, SYNTH_STREAM_SHARED);
    for (int64_t t = 0; t < T; ++t) out[t] = synth_normal_bf16(key, (uint64_t)(t0 + t));
}

/* W1 [n, 2I, H] fp32 for the listed global expert ids (the shared expert has
 * id E_global). */
void synth_w1(uint64_t seed, int64_t H, int64_t I, const int64_t* experts, int64_t n, double sigma, float* out) {
    uint64_t key = synth_key(seed, SYNTH_STREAM_W1);
    int64_t per = 2 * I * H;
    for (int64_t k = 0; k < n; ++k) {
        uint64_t base = (uint64_t)(experts[k] * per);
        float* o = out + k * per;
        for (int64_t i = 0; i < per; ++i) o[i] = synth_normal_f32(key, base + (uint64_t)i, sigma);
    }
}

/* W2 [n, H, I] fp32 for the listed global expert ids. */
void synth_w2(uint64_t seed, int64_t H, int64_t I, const int64_t* experts, int64_t n, double sigma, float* out) {
    uint64_t key = synth_key(seed, SYNTH_STREAM_W2);
    int64_t per = H * I;
    for (int64_t k = 0; k < n; ++k) {
        uint64_t base = (uint64_t)(experts[k] * per);
        float* o = out + k * per;
        for (int64_t i = 0; i < per; ++i) o[i] = synth_normal_f32(key, base + (uint64_t)i, sigma);
    }
}

/* Raw generator outputs, for cross-build checks. */
void synth_normal_q16_range(uint64_t seed, uint64_t stream, uint64_t i0, int64_t n, int32_t* out) {
    uint64_t key = synth_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = synth_normal_q16(key, i0 + (uint64_t)i);
}
