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
// dense_max_elems, and the accumulator is small, T * H * 4 bytes <= 32 MiB
// (well inside the 126 MiB L2, so the reductions run at the L2 and cost less
// than writing the rows and reading them back); split otherwise.  Measured on
// GB300: dense is faster at every decode workload (the 4352-row skewed batch
// by 10 %), and 2x slower at the 32768-token prefill, whose 470 MB
// accumulator lives in DRAM.  A caller may force either path.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(32) gemm2_gate_kernel(GateParams p) {
    // The next launch may start its prologue now: it waits for this grid
    // (griddepcontrol.wait) before it reads the path or the sort's table.
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();  // the sort's table is complete and visible
    if (threadIdx.x == 0) {
        const int R = p.header[kHdrRows];  // routed rows of this call
        int path;
        if (p.force == 1)
            path = kPathSplit;
        else if (p.force == 2)
            path = kPathDense;
        else
            path = (static_cast<int64_t>(R) * p.H <= p.dense_max_elems &&
                    static_cast<int64_t>(p.T) * p.H * 4 <= (int64_t(32) << 20))
                       ? kPathDense
                       : kPathSplit;
        p.header[kHdrGemm2Path] = path;
    }
}

}  // namespace

cudaError_t launch_gate(const GateParams& p, cudaStream_t stream, bool pdl) {
    return launch_kernel(gemm2_gate_kernel, dim3(1), dim3(32), 0, stream, pdl, p);
}

}  // namespace moe
