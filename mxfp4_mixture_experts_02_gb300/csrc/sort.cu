// Token-to-expert sort ("[SGLang] CUTLASS MoE", section 1 prepare_moe_input:
// expert_offsets, a_map, c_map; "[sglang] ... MXFP4 decode MoE ... shape
// templates", sections 1 and 5: virtual experts of kBlockN rows, ids outside
// the local slice get -1, ranks in ascending token order).
//
// One CTA of 32 warps; warp w owns a contiguous run of slots.  Two passes
// over the slots in rounds of 32, each round grouping equal experts with
// __match_any_sync:
//   count: the group leader adds the group size to the warp's histogram row;
//   rank : row = offsets[e] + (slots of e in earlier warps) + (slots of e
//          earlier in this warp) + (lower lanes of the group this round).
// Ranks therefore follow ascending slot index t*k' + j whatever the timing,
// with no atomics on the data path.  Between the passes a block-wide scan of
// (count, tiles, groups) over experts places every expert's rows, virtual
// experts (chunks of B rows) and GEMM work groups (G virtual experts).
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;

__device__ __forceinline__ int local_expert(int32_t id, const SortParams& p) {
    if (id >= p.Eg && id < p.Eg + p.S) return p.E + (id - p.Eg);
    if (id >= p.off && id < p.off + p.E) return id - p.off;
    return -1;
}

// Exclusive scan of three ints across the block (one expert per thread).
__device__ __forceinline__ void block_scan3(int a, int b, int c, int& ea, int& eb, int& ec, int& ta, int& tb, int& tc,
                                            int (*s_tot)[kSortWarps]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ia = a, ib = b, ic = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xa = __shfl_up_sync(0xffffffffu, ia, o);
        const int xb = __shfl_up_sync(0xffffffffu, ib, o);
        const int xc = __shfl_up_sync(0xffffffffu, ic, o);
        if (lane >= o) {
            ia += xa;
            ib += xb;
            ic += xc;
        }
    }
    if (lane == 31) {
        s_tot[0][warp] = ia;
        s_tot[1][warp] = ib;
        s_tot[2][warp] = ic;
    }
    __syncthreads();
    if (warp == 0) {
        int va = s_tot[0][lane], vb = s_tot[1][lane], vc = s_tot[2][lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int xa = __shfl_up_sync(0xffffffffu, va, o);
            const int xb = __shfl_up_sync(0xffffffffu, vb, o);
            const int xc = __shfl_up_sync(0xffffffffu, vc, o);
            if (lane >= o) {
                va += xa;
                vb += xb;
                vc += xc;
            }
        }
        s_tot[0][lane] = va;  // inclusive prefix of warp totals
        s_tot[1][lane] = vb;
        s_tot[2][lane] = vc;
    }
    __syncthreads();
    const int pa = warp ? s_tot[0][warp - 1] : 0;
    const int pb = warp ? s_tot[1][warp - 1] : 0;
    const int pc = warp ? s_tot[2][warp - 1] : 0;
    ea = pa + ia - a;
    eb = pb + ib - b;
    ec = pc + ic - c;
    ta = s_tot[0][kSortWarps - 1];
    tb = s_tot[1][kSortWarps - 1];
    tc = s_tot[2][kSortWarps - 1];
}

__global__ void __launch_bounds__(kSortThreads, 1) sort_kernel(SortParams p) {
    extern __shared__ int s_dyn[];
    int* hist = s_dyn;                     // [32][Et]: per-warp counts, then per-warp bases
    int* s_off = s_dyn + kSortWarps * p.Et;  // [Et]
    __shared__ int s_tot[3][kSortWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kSortWarps * p.Et; i += kSortThreads) hist[i] = 0;
    ptx::pdl_wait();
    __syncthreads();

    const int n = p.T * p.kp;
    const int per = (((n + kSortWarps - 1) / kSortWarps) + 31) & ~31;
    const int s0 = warp * per;
    const int s1 = min(n, s0 + per);
    int* my_hist = hist + warp * p.Et;

    // pass 1: per-warp histogram
    for (int base = s0; base < s1; base += 32) {
        const int s = base + lane;
        const int e = (s < s1) ? local_expert(p.ids[s], p) : -1;
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my_hist[e] += __popc(peers);
    }
    __syncthreads();

    // per expert: prefix over warps (in place) and totals
    int cnt = 0;
    if (tid < p.Et) {
        for (int w = 0; w < kSortWarps; ++w) {
            const int c = hist[w * p.Et + tid];
            hist[w * p.Et + tid] = cnt;
            cnt += c;
        }
    }
    const int tiles = (cnt + p.B - 1) / p.B;
    const int grps = (tiles + p.G - 1) / p.G;
    int off, vb, gb, R, V, NG;
    block_scan3(cnt, tiles, grps, off, vb, gb, R, V, NG, s_tot);

    if (tid < p.Et) {
        s_off[tid] = off;
        p.counts[tid] = cnt;
        p.offsets[tid] = off;
        for (int c = 0; c < tiles; ++c)
            p.vinfo[vb + c] = make_int4(tid, off + c * p.B, min(p.B, cnt - c * p.B), c);
        for (int g = 0; g < grps; ++g) p.groups[gb + g] = make_int4(tid, vb + g * p.G, min(p.G, tiles - g * p.G), 0);
    }
    if (tid == 0) {
        p.offsets[p.Et] = R;
        p.header[kHdrRows] = R;
        p.header[kHdrNumV] = V;
        p.header[kHdrNumGroups] = NG;
        p.header[kHdrStatus] = 0;
        p.header[kHdrDetail] = 0;
    }
    __syncthreads();

    // pass 2: ranks -> c_map / a_map
    for (int base = s0; base < s1; base += 32) {
        const int s = base + lane;
        const int e = (s < s1) ? local_expert(p.ids[s], p) : -1;
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (s < s1) {
            if (e >= 0) {
                const int row = s_off[e] + my_hist[e] + __popc(peers & ptx::lanemask_lt());
                p.c_map[s] = row;
                p.a_map[row] = s;
            } else {
                p.c_map[s] = -1;
            }
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) my_hist[e] += __popc(peers);
        __syncwarp();
    }
    ptx::pdl_launch_dependents();
}

}  // namespace

size_t sort_smem_bytes(int Et) { return static_cast<size_t>(kSortWarps + 1) * Et * sizeof(int); }

cudaError_t launch_sort(const SortParams& p, cudaStream_t stream, bool pdl) {
    const size_t smem = sort_smem_bytes(p.Et);
    cudaError_t err = cudaFuncSetAttribute(sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_kernel(sort_kernel, dim3(1), dim3(kSortThreads), smem, stream, pdl, p);
}

}  // namespace moe
