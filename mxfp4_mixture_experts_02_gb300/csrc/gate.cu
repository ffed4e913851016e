// The GEMM2 gate ("[FlashInfer] Device-side gating for the MoE GEMM2 path",
// sections 1 and 2): one warp, launched after the sort, reads the sorted
// table and chooses the GEMM2 strategy on the device, so one fixed launch
// chain (one CUDA graph) serves every routing:
//   split: FC2 writes each routed row (w * Y); the combine sums a token's rows
//          in slot order (bit-reproducible);
//   dense: FC2's epilogue reduces w * Y straight into an fp32 [T, H]
//          accumulator at the L2 (the finalize fused into GEMM2); the combine
//          only converts it to bf16.  The order of the reductions varies
//          from run to run, so the last bits of the sums may too.
// The rule: dense when the rows' reductions are few, rows * H <=
// dense_max_elems (the accumulator then stays in L2 and the reductions cost
// less than writing and re-reading the rows); split otherwise.  A caller may
// force either path.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(32) gemm2_gate_kernel(GateParams p) {
    ptx::pdl_wait();  // the sort's table is complete and visible
    if (threadIdx.x == 0) {
        const int R = p.header[kHdrRows];  // routed rows of this call
        int path;
        if (p.force == 1)
            path = kPathSplit;
        else if (p.force == 2)
            path = kPathDense;
        else
            path = static_cast<int64_t>(R) * p.H <= p.dense_max_elems ? kPathDense : kPathSplit;
        p.header[kHdrGemm2Path] = path;
    }
    ptx::pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_gate(const GateParams& p, cudaStream_t stream, bool pdl) {
    return launch_kernel(gemm2_gate_kernel, dim3(1), dim3(32), 0, stream, pdl, p);
}

}  // namespace moe
