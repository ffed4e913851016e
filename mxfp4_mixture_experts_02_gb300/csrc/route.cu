// Top-k routing with renormalised softmax weights and the optional appended
// shared expert: one warp per token (rs::route_token; the selection is
// described at rs::warp_topk).  Weights: exp(l_j - l_0) / sum over the picks
// (softmax renormalised over the selected experts).
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "route_sort.cuh"

namespace moe {

namespace {

constexpr int kRouteWarps = 8;
constexpr int kRouteCtasPerSm = 3;  // resident CTAs per SM: long batches loop several tokens per warp

// Each warp routes tokens t, t + stride, ...; while it routes one, its lanes
// prefetch the next token's logits row (one 128-byte line per lane) into L2,
// so the next token's loads do not wait for DRAM.  fuse_x (decode tilings,
// x kept in token order): the whole grid then also quantises x to MXFP8, one
// 32-element block per thread and step (the sort that follows writes each
// row's routing weight), so the quantiser needs no launch of its own.
__global__ void __launch_bounds__(kRouteWarps * 32, kRouteCtasPerSm)
    route_kernel(RouteParams p, GatherParams gp, int fuse_x) {
    __shared__ uint2 s_cand[kRouteWarps][rs::kMaxCand];
    ptx::pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stride = gridDim.x * kRouteWarps;
    const int lines = (p.Eg * 4 + 127) / 128;  // <= 32 for E_global <= 1024
    for (int t = blockIdx.x * kRouteWarps + warp; t < p.T; t += stride) {
        const int tn = t + stride;
        if (tn < p.T && lane < lines)
            ptx::prefetch_l2(reinterpret_cast<const char*>(p.logits + static_cast<size_t>(tn) * p.Eg) + 128 * lane);
        rs::route_token(p, t, s_cand[warp], nullptr);
    }
    if (fuse_x) {
        const int64_t nq = static_cast<int64_t>(p.T) * (gp.H / 32);
        for (int64_t blk = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; blk < nq;
             blk += static_cast<int64_t>(gridDim.x) * blockDim.x)
            quant_x_block(gp.x, gp.xq, gp.xsf, static_cast<size_t>(blk));
    }
    ptx::pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_route(const RouteParams& p, cudaStream_t stream, bool pdl, const GatherParams* gp) {
    if (p.T == 0) return cudaSuccess;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
        return cudaErrorUnknown;
    int64_t blocks = (p.T + kRouteWarps - 1) / kRouteWarps;
    if (gp) {  // enough CTAs for one x block per thread, up to one CTA per SM
        const int64_t xb = (static_cast<int64_t>(p.T) * (gp->H / 32) + kRouteWarps * 32 - 1) / (kRouteWarps * 32);
        blocks = std::max(blocks, std::min<int64_t>(xb, nsm));
    }
    blocks = std::min<int64_t>(blocks, static_cast<int64_t>(nsm) * kRouteCtasPerSm);
    const GatherParams g = gp ? *gp : GatherParams{};
    return launch_kernel(route_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kRouteWarps * 32), 0, stream, pdl, p,
                         g, gp ? 1 : 0);
}

}  // namespace moe
