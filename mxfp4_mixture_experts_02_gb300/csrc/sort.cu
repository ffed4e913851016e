// Token-to-expert sort ("[SGLang] CUTLASS MoE", section 1 prepare_moe_input:
// expert_offsets, a_map, c_map; "[sglang] ... MXFP4 decode MoE ... shape
// templates", sections 1 and 5: virtual experts of kBlockN rows, ids outside
// the local slice get -1, ranks in ascending token order).
//
// Small slot counts: one CTA of 32 warps; warp w owns a contiguous run of
// slots.  Large slot counts: the same per-warp passes spread over CTAs of 8
// warps (4096 slots each) with a one-CTA scan in between.  Two passes
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

// Expert-level part shared by both paths (one CTA of kSortThreads, thread
// tid = expert): given each expert's row count, scan (count, tiles, groups),
// write counts / offsets / virtual experts / work groups and the header, and
// leave each expert's first row in s_off.
__device__ __forceinline__ void place_experts(const SortParams& p, int cnt, int* s_off, int (*s_tot)[kSortWarps]) {
    const int tid = threadIdx.x;
    const int tiles = (cnt + p.B - 1) / p.B;
    const int grps = (tiles + p.G - 1) / p.G;
    int off, vb, gb, R, V, NG;
    block_scan3(cnt, tiles, grps, off, vb, gb, R, V, NG, s_tot);
    if (tid < p.Et) {
        if (s_off) s_off[tid] = off;
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
}

// Per-warp histogram of the slots [s0, s1) into my_hist (rounds of 32).
__device__ __forceinline__ void warp_count(const SortParams& p, int s0, int s1, int* my_hist) {
    const int lane = threadIdx.x & 31;
    for (int base = s0; base < s1; base += 32) {
        const int s = base + lane;
        const int e = (s < s1) ? local_expert(p.ids[s], p) : -1;
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my_hist[e] += __popc(peers);
    }
}

// Ranks of the slots [s0, s1): row = my_base[e] + earlier slots of e in this
// warp + lower lanes of e in this round.  my_base advances in place.
__device__ __forceinline__ void warp_rank(const SortParams& p, int s0, int s1, int* my_base) {
    const int lane = threadIdx.x & 31;
    for (int base = s0; base < s1; base += 32) {
        const int s = base + lane;
        const int e = (s < s1) ? local_expert(p.ids[s], p) : -1;
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        if (s < s1) {
            if (e >= 0) {
                const int row = my_base[e] + __popc(peers & ptx::lanemask_lt());
                p.c_map[s] = row;
                p.a_map[row] = s;
            } else {
                p.c_map[s] = -1;
            }
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) my_base[e] += __popc(peers);
        __syncwarp();
    }
}

// Small slot counts: the whole sort in one CTA of 32 warps.
__global__ void __launch_bounds__(kSortThreads, 1) sort_kernel(SortParams p) {
    extern __shared__ int s_dyn[];
    int* hist = s_dyn;                       // [32][Et]: per-warp counts, then per-warp bases
    int* s_off = s_dyn + kSortWarps * p.Et;  // [Et]
    __shared__ int s_tot[3][kSortWarps];

    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < kSortWarps * p.Et; i += kSortThreads) hist[i] = 0;
    ptx::pdl_wait();
    __syncthreads();

    const int n = p.T * p.kp;
    const int per = (((n + kSortWarps - 1) / kSortWarps) + 31) & ~31;
    const int s0 = warp * per;
    const int s1 = min(n, s0 + per);
    int* my_hist = hist + warp * p.Et;

    warp_count(p, s0, s1, my_hist);
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
    place_experts(p, cnt, s_off, s_tot);
    __syncthreads();
    // per-warp bases: expert offset + earlier warps
    for (int i = tid; i < kSortWarps * p.Et; i += kSortThreads) hist[i] += s_off[i % p.Et];
    __syncthreads();
    warp_rank(p, s0, s1, my_hist);
    ptx::pdl_launch_dependents();
}

// Large slot counts: CTA c owns slots [c * kBigChunk, (c + 1) * kBigChunk),
// warp w of it the w-th sub-run of kBigWarpSlots.
constexpr int kBigWarps = 8;
constexpr int kBigWarpSlots = 512;
constexpr int kBigChunk = kBigWarps * kBigWarpSlots;

// Pass 1: per-CTA expert counts -> cta_hist[c][e].
__global__ void __launch_bounds__(kBigWarps * 32) sort_count_kernel(SortParams p) {
    extern __shared__ int s_dyn[];
    int* hist = s_dyn;  // [kBigWarps][Et]
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < kBigWarps * p.Et; i += kBigWarps * 32) hist[i] = 0;
    ptx::pdl_wait();
    __syncthreads();
    const int n = p.T * p.kp;
    const int s0 = blockIdx.x * kBigChunk + warp * kBigWarpSlots;
    warp_count(p, s0, min(n, s0 + kBigWarpSlots), hist + warp * p.Et);
    __syncthreads();
    for (int e = tid; e < p.Et; e += kBigWarps * 32) {
        int c = 0;
        for (int w = 0; w < kBigWarps; ++w) c += hist[w * p.Et + e];
        p.cta_hist[static_cast<size_t>(blockIdx.x) * p.Et + e] = c;
    }
    ptx::pdl_launch_dependents();
}

// Pass 2 (one CTA): per expert, exclusive prefix over CTAs in place and the
// total; then the expert-level placement.
__global__ void __launch_bounds__(kSortThreads, 1) sort_scan_kernel(SortParams p, int nctas) {
    __shared__ int s_tot[3][kSortWarps];
    ptx::pdl_wait();
    const int tid = threadIdx.x;
    int cnt = 0;
    if (tid < p.Et) {
        for (int c = 0; c < nctas; ++c) {
            int* h = p.cta_hist + static_cast<size_t>(c) * p.Et + tid;
            const int v = *h;
            *h = cnt;
            cnt += v;
        }
    }
    place_experts(p, cnt, nullptr, s_tot);
    ptx::pdl_launch_dependents();
}

// Pass 3: ranks.  Per-warp bases = expert offset + earlier CTAs + earlier
// warps of this CTA (recounted).
__global__ void __launch_bounds__(kBigWarps * 32) sort_rank_kernel(SortParams p) {
    extern __shared__ int s_dyn[];
    int* hist = s_dyn;  // [kBigWarps][Et]
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < kBigWarps * p.Et; i += kBigWarps * 32) hist[i] = 0;
    ptx::pdl_wait();
    __syncthreads();
    const int n = p.T * p.kp;
    const int s0 = blockIdx.x * kBigChunk + warp * kBigWarpSlots;
    const int s1 = min(n, s0 + kBigWarpSlots);
    warp_count(p, s0, s1, hist + warp * p.Et);
    __syncthreads();
    for (int e = tid; e < p.Et; e += kBigWarps * 32) {
        int run = p.offsets[e] + p.cta_hist[static_cast<size_t>(blockIdx.x) * p.Et + e];
        for (int w = 0; w < kBigWarps; ++w) {
            const int c = hist[w * p.Et + e];
            hist[w * p.Et + e] = run;
            run += c;
        }
    }
    __syncthreads();
    warp_rank(p, s0, s1, hist + warp * p.Et);
    ptx::pdl_launch_dependents();
}

}  // namespace

size_t sort_smem_bytes(int Et) { return static_cast<size_t>(kSortWarps + 1) * Et * sizeof(int); }

int sort_big_ctas(int n) { return (n + kBigChunk - 1) / kBigChunk; }

cudaError_t launch_sort(const SortParams& p, cudaStream_t stream, bool pdl) {
    const int n = p.T * p.kp;
    if (n <= kSortWarps * kBigWarpSlots) {
        const size_t smem = sort_smem_bytes(p.Et);
        cudaError_t err = cudaFuncSetAttribute(sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        return launch_kernel(sort_kernel, dim3(1), dim3(kSortThreads), smem, stream, pdl, p);
    }
    const int nctas = sort_big_ctas(n);
    const size_t smem = static_cast<size_t>(kBigWarps) * p.Et * sizeof(int);
    cudaError_t err = launch_kernel(sort_count_kernel, dim3(nctas), dim3(kBigWarps * 32), smem, stream, pdl, p);
    if (err != cudaSuccess) return err;
    err = launch_kernel(sort_scan_kernel, dim3(1), dim3(kSortThreads), 0, stream, true, p, nctas);
    if (err != cudaSuccess) return err;
    return launch_kernel(sort_rank_kernel, dim3(nctas), dim3(kBigWarps * 32), smem, stream, true, p);
}

}  // namespace moe
