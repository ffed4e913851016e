// Top-k routing with renormalised softmax weights and the optional appended
// shared expert: one warp per token (rs::route_token; the selection is
// described at rs::warp_topk).  Weights: exp(l_j - l_0) / sum over the picks
// (softmax renormalised over the selected experts).
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "route_sort.cuh"

namespace moe {

namespace {

constexpr int kRouteWarps = 8;

__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(RouteParams p) {
    __shared__ uint2 s_cand[kRouteWarps][rs::kMaxCand];
    ptx::pdl_wait();
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * kRouteWarps + warp;
    if (t < p.T) rs::route_token(p, t, s_cand[warp], nullptr);
    ptx::pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_route(const RouteParams& p, cudaStream_t stream, bool pdl) {
    if (p.T == 0) return cudaSuccess;
    const int blocks = (p.T + kRouteWarps - 1) / kRouteWarps;
    return launch_kernel(route_kernel, dim3(blocks), dim3(kRouteWarps * 32), 0, stream, pdl, p);
}

}  // namespace moe
