// Top-k routing with renormalised softmax weights and the optional appended
// shared expert.
//
// One warp per token.  Lane l holds the logits of experts l, l+32, ... in
// registers (coalesced loads of the token's row) and keeps its best untaken
// entry.  Each of the k rounds is two warp reductions: the maximum of an
// order-preserving integer key of the logit, then the smallest expert id
// among the lanes holding that maximum (ties go to the lower id); only the
// winning lane rescans its entries.  Weights: exp(l_j - l_0) / sum over the
// picks (softmax renormalised over the selected experts).  The shared expert
// gets id E_global + s and weight sigmoid(fp32(bf16 logit)) * scale, computed
// in fp32 in the same kernel ("[sglang] SGLang MoE shared expert: fuse 3
// kernels into 1": the sigmoid and the bf16->fp32 cast fused into the append).
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kRouteWarps = 8;
constexpr int kMaxPerLane = 32;  // E_global <= 1024

// Monotone map of a finite fp32 to uint32 (a < b  <=>  key(a) < key(b));
// -0 is folded onto +0 so that equal values tie; every finite value and
// -inf map above 0.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Best (largest key, lowest index on ties) of a lane's entries by a
// pairwise tree; taken / absent entries hold key 0, which no finite logit
// maps to.
__device__ __forceinline__ void lane_best(const uint32_t (&key)[kMaxPerLane], uint32_t& bk, int& bi) {
    uint32_t k[kMaxPerLane];
    int ix[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        k[i] = key[i];
        ix[i] = i;
    }
#pragma unroll
    for (int w = kMaxPerLane / 2; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i)
            if (k[i + w] > k[i]) {  // the upper half holds higher indices: ties keep the lower one
                k[i] = k[i + w];
                ix[i] = ix[i + w];
            }
    bk = k[0];
    bi = ix[0];
}

__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(RouteParams p) {
    ptx::pdl_wait();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t < p.T) {
        const float* row = p.logits + static_cast<size_t>(t) * p.Eg;
        uint32_t key[kMaxPerLane];
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int e = lane + 32 * i;
            key[i] = (e < p.Eg) ? order_key(row[e]) : 0u;
        }
        uint32_t bk;
        int bi;
        lane_best(key, bk, bi);
        uint32_t my_key = 0, my_id = 0;
        for (int j = 0; j < p.k; ++j) {
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t cand = (bk == kmax && bk != 0) ? static_cast<uint32_t>(lane + 32 * bi) : 0xFFFFFFFFu;
            const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
            if (lane == static_cast<int>(win & 31)) {
#pragma unroll
                for (int i = 0; i < kMaxPerLane; ++i)
                    if (i == static_cast<int>(win >> 5)) key[i] = 0;
                lane_best(key, bk, bi);
            }
            if (lane == j) {
                my_key = kmax;
                my_id = win;
            }
        }
        const float my_val = key_value(my_key);
        const float m = __shfl_sync(0xffffffffu, my_val, 0);
        const float ex = (lane < p.k) ? expf(my_val - m) : 0.f;
        float sum = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const size_t base = static_cast<size_t>(t) * p.kp;
        if (lane < p.k) {
            p.ids[base + lane] = static_cast<int32_t>(my_id);
            p.w[base + lane] = ex / sum;
        }
        if (lane < p.S) {
            const float x = bf16_bits_to_float(p.shared_logit[static_cast<size_t>(t) * p.S + lane]);
            p.ids[base + p.k + lane] = p.Eg + lane;
            p.w[base + p.k + lane] = p.shared_scale / (1.0f + expf(-x));
        }
    }
    ptx::pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_route(const RouteParams& p, cudaStream_t stream, bool pdl) {
    if (p.T == 0) return cudaSuccess;
    const int blocks = (p.T + kRouteWarps - 1) / kRouteWarps;
    return launch_kernel(route_kernel, dim3(blocks), dim3(kRouteWarps * 32), 0, stream, pdl, p);
}

}  // namespace moe
