/*
 * GPU build of the seeded input generator (see synth.h): the same counter
 * hash, writing device arrays.  Used to materialise full-size synthetic
 * inputs (the fp32 weights of a 896-expert layer are ~15 GB) directly in HBM.
 * Every function returns a cudaError_t value cast to int (0 = success).
 */
#include <cuda_runtime.h>
#include "synth.h"

namespace {

constexpr int kThreads = 256;

inline unsigned grid_for(int64_t n) {
    int64_t g = (n + kThreads - 1) / kThreads;
    if (g > 65535LL * 64) g = 65535LL * 64;
    return (unsigned)(g < 1 ? 1 : g);
}

__global__ void k_x(uint64_t key, int64_t t0, int64_t n, int64_t H, uint16_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = synth_normal_bf16(key, (uint64_t)(t0 * H + i));
}

__global__ void k_logits(uint64_t key, int64_t t0, int64_t n, int64_t Eg, const double* bias, float* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        double b = bias ? bias[i % Eg] : 0.0;
        out[i] = synth_normal_plus_f32(key, (uint64_t)(t0 * Eg + i), b);
    }
}

__global__ void k_shared(uint64_t key, int64_t t0, int64_t n, uint16_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = synth_normal_bf16(key, (uint64_t)(t0 + i));
}

/* out [n, per] for expert ids experts[0..n) (device array). */
__global__ void k_expert(uint64_t key, int64_t per, const int64_t* experts, int64_t n, double sigma, float* out) {
    int64_t total = per * n;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t k = i / per, j = i - k * per;
        out[i] = synth_normal_f32(key, (uint64_t)(experts[k] * per + j), sigma);
    }
}

__global__ void k_q16(uint64_t key, uint64_t i0, int64_t n, int32_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = synth_normal_q16(key, i0 + (uint64_t)i);
}

}  // namespace

extern "C" {

int synth_x_cuda(uint64_t seed, int64_t t0, int64_t T, int64_t H, uint16_t* out, cudaStream_t s) {
    int64_t n = T * H;
    k_x<<<grid_for(n), kThreads, 0, s>>>(synth_key(seed, SYNTH_STREAM_X), t0, n, H, out);
    return (int)cudaGetLastError();
}

int synth_logits_cuda(uint64_t seed, int64_t t0, int64_t T, int64_t Eg, const double* bias_dev, float* out, cudaStream_t s) {
    int64_t n = T * Eg;
    k_logits<<<grid_for(n), kThreads, 0, s>>>(synth_key(seed, SYNTH_STREAM_LOGITS), t0, n, Eg, bias_dev, out);
    return (int)cudaGetLastError();
}

int synth_shared_logit_cuda(uint64_t seed, int64_t t0, int64_t T, uint16_t* out, cudaStream_t s) {
    k_shared<<<grid_for(T), kThreads, 0, s>>>(synth_key(seed, SYNTH_STREAM_SHARED), t0, T, out);
    return (int)cudaGetLastError();
}

int synth_w1_cuda(uint64_t seed, int64_t H, int64_t I, const int64_t* experts_dev, int64_t n, double sigma, float* out,
                  cudaStream_t s) {
    int64_t per = 2 * I * H;
    k_expert<<<grid_for(per * n), kThreads, 0, s>>>(synth_key(seed, SYNTH_STREAM_W1), per, experts_dev, n, sigma, out);
    return (int)cudaGetLastError();
}

int synth_w2_cuda(uint64_t seed, int64_t H, int64_t I, const int64_t* experts_dev, int64_t n, double sigma, float* out,
                  cudaStream_t s) {
    int64_t per = H * I;
    k_expert<<<grid_for(per * n), kThreads, 0, s>>>(synth_key(seed, SYNTH_STREAM_W2), per, experts_dev, n, sigma, out);
    return (int)cudaGetLastError();
}

int synth_normal_q16_range_cuda(uint64_t seed, uint64_t stream, uint64_t i0, int64_t n, int32_t* out, cudaStream_t s) {
    k_q16<<<grid_for(n), kThreads, 0, s>>>(synth_key(seed, stream), i0, n, out);
    return (int)cudaGetLastError();
}

}  // extern "C"
