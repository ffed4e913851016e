// Top-k routing with renormalised softmax weights and the optional appended
// shared expert.
//
// One warp per token.  Lane l holds the logits of experts l, l+32, ... in
// registers (coalesced loads of the token's row).  Each of the k rounds takes
// a warp-wide argmax of (logit, -id) with butterfly shuffles, so ties go to
// the lower expert id, and removes the winner.  Weights: exp(l_j - l_0) / sum
// over the picks (softmax renormalised over the selected experts).  The
// shared expert gets id E_global + s and weight sigmoid(fp32(bf16 logit)) *
// scale, computed in fp32 in the same kernel ("[sglang] SGLang MoE shared
// expert: fuse 3 kernels into 1": the sigmoid and the bf16->fp32 cast fused
// into the append).
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kRouteWarps = 8;
constexpr int kMaxPerLane = 32;  // E_global <= 1024

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(RouteParams p) {
    ptx::pdl_wait();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t < p.T) {
        const float* row = p.logits + static_cast<size_t>(t) * p.Eg;
        const int nper = (p.Eg + 31) / 32;
        float v[kMaxPerLane];
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int e = lane + 32 * i;
            v[i] = (i < nper && e < p.Eg) ? row[e] : -INFINITY;
        }
        uint32_t taken = 0;
        for (int i = 0; i < kMaxPerLane; ++i)
            if (i >= nper || lane + 32 * i >= p.Eg) taken |= 1u << i;

        float my_val = 0.f;
        int my_id = 0;
        for (int j = 0; j < p.k; ++j) {
            // lane-local best among untaken entries (lower index = lower id)
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF;
#pragma unroll
            for (int i = 0; i < kMaxPerLane; ++i) {
                const int e = lane + 32 * i;
                if (!((taken >> i) & 1u) && better(v[i], e, bv, bi)) {
                    bv = v[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (better(ov, oi, bv, bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == j) {
                my_val = bv;
                my_id = bi;
            }
        }
        const float m = __shfl_sync(0xffffffffu, my_val, 0);
        const float ex = (lane < p.k) ? expf(my_val - m) : 0.f;
        float sum = ex;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const size_t base = static_cast<size_t>(t) * p.kp;
        if (lane < p.k) {
            p.ids[base + lane] = my_id;
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
