// Weighted un-permute combine ("[SGLang] CUTLASS MoE", section 5
// apply_shuffle_mul_sum): out[t] = bf16( sum_j Y[c_map[t, j]] ) over the
// token's slots j in ascending order, skipping slots with no local row
// (c_map = -1, "[sglang] ... MXFP4 decode MoE ... shape templates", section
// 5).  Y rows already carry the routing weight (FC2 epilogue), so this is a
// gather-sum: no atomics, bitwise deterministic.
//
// When the GEMM2 gate chose the dense path ("[FlashInfer] Device-side gating
// for the MoE GEMM2 path"), FC2 has already summed every token's rows into
// the fp32 accumulator, and this launch is the finalize's last step: out[t] =
// bf16(acc[t]).
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kCombineThreads = 128;   // one float4 of the hidden dim per thread
constexpr int kMaxSlots = 64;

// Block (chunk of 512 hidden columns, token).  The token's rows are read
// once into shared memory; each thread sums its float4 over the slots in
// ascending order, issuing the loads of up to kBatch slots before adding
// them (one memory round trip for a decode token's 16 slots).
constexpr int kBatch = 16;

// Dense GEMM2 path: columns 8 * c8 .. 8 * c8 + 7 of token t's fp32 sums to bf16.
__device__ __forceinline__ void convert_acc_row8(const CombineParams& p, int t, int c8) {
    const float4* a = reinterpret_cast<const float4*>(p.acc + static_cast<int64_t>(t) * p.H) + 2 * c8;
    const float4 u = a[0], v = a[1];
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(u.x, u.y), b1 = __floats2bfloat162_rn(u.z, u.w);
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(v.x, v.y), b3 = __floats2bfloat162_rn(v.z, v.w);
    reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(t) * p.H)[c8] =
        make_uint4(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1),
                   *reinterpret_cast<const uint32_t*>(&b2), *reinterpret_cast<const uint32_t*>(&b3));
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
    __shared__ int rows[kMaxSlots];
    ptx::pdl_wait();
    const int t = p.t0 + static_cast<int>(blockIdx.y);
    if (p.header[kHdrGemm2Path] == kPathDense) {
        // this block's 512 columns: 64 groups of 8 on the first 64 threads
        const int c8 = blockIdx.x * (kCombineThreads / 2) + threadIdx.x;
        if (threadIdx.x < kCombineThreads / 2 && c8 < p.H / 8) convert_acc_row8(p, t, c8);
        ptx::pdl_launch_dependents();
        return;
    }
    if (threadIdx.x < p.kp) rows[threadIdx.x] = p.c_map[static_cast<size_t>(t) * p.kp + threadIdx.x];
    __syncthreads();
    const int c = blockIdx.x * kCombineThreads + threadIdx.x;  // float4 column
    if (c < p.H / 4) {
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 acc = zero;
        for (int j0 = 0; j0 < p.kp; j0 += kBatch) {
            float4 v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int r = (j0 + u < p.kp) ? rows[j0 + u] : -1;
                v[u] = r >= 0 ? reinterpret_cast<const float4*>(p.y + static_cast<size_t>(r) * p.H)[c] : zero;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (j0 + u >= p.kp || rows[j0 + u] < 0) continue;  // skipped slots add nothing
                acc.x += v[u].x;
                acc.y += v[u].y;
                acc.z += v[u].z;
                acc.w += v[u].w;
            }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t*>(&lo);
        packed.y = *reinterpret_cast<const uint32_t*>(&hi);
        reinterpret_cast<uint2*>(p.out + static_cast<size_t>(t) * p.H)[c] = packed;
    }
    ptx::pdl_launch_dependents();
}

// bf16 Y rows (prefill tiling): one uint4 (8 columns) per thread.
__global__ void __launch_bounds__(kCombineThreads) combine_bf16_kernel(CombineParams p) {
    __shared__ int rows[kMaxSlots];
    ptx::pdl_wait();
    const int t = p.t0 + static_cast<int>(blockIdx.y);
    if (p.header[kHdrGemm2Path] == kPathDense) {
        const int c8 = blockIdx.x * kCombineThreads + threadIdx.x;  // this block's 1024 columns
        if (c8 < p.H / 8) convert_acc_row8(p, t, c8);
        ptx::pdl_launch_dependents();
        return;
    }
    if (threadIdx.x < p.kp) rows[threadIdx.x] = p.c_map[static_cast<size_t>(t) * p.kp + threadIdx.x];
    __syncthreads();
    const int c = blockIdx.x * kCombineThreads + threadIdx.x;  // uint4 column (8 bf16)
    if (c < p.H / 8) {
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = 0.f;
        int j = 0;
        for (; j + 4 <= p.kp; j += 4) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = rows[j + u];
                v[u] = r >= 0 ? reinterpret_cast<const uint4*>(p.y_bf16 + static_cast<size_t>(r) * p.H)[c]
                              : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    acc[2 * m] += __uint_as_float(w4[m] << 16);
                    acc[2 * m + 1] += __uint_as_float(w4[m] & 0xFFFF0000u);
                }
            }
        }
        for (; j < p.kp; ++j) {
            const int r = rows[j];
            if (r < 0) continue;
            const uint4 v = reinterpret_cast<const uint4*>(p.y_bf16 + static_cast<size_t>(r) * p.H)[c];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                acc[2 * m] += __uint_as_float(w4[m] << 16);
                acc[2 * m + 1] += __uint_as_float(w4[m] & 0xFFFF0000u);
            }
        }
        uint32_t pk[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * m], acc[2 * m + 1]);
            pk[m] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * p.H)[c] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    ptx::pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl) {
    if (p.T <= p.t0) return cudaSuccess;
    if (p.y_bf16) {
        const dim3 grid((p.H / 8 + kCombineThreads - 1) / kCombineThreads, p.T - p.t0);
        return launch_kernel(combine_bf16_kernel, grid, dim3(kCombineThreads), 0, stream, pdl, p);
    }
    const dim3 grid((p.H / 4 + kCombineThreads - 1) / kCombineThreads, p.T - p.t0);
    return launch_kernel(combine_kernel, grid, dim3(kCombineThreads), 0, stream, pdl, p);
}

}  // namespace moe
