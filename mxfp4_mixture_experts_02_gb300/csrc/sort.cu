// Token-to-expert sort ("[SGLang] CUTLASS MoE", section 1 prepare_moe_input:
// expert_offsets, a_map, c_map; "[sglang] ... MXFP4 decode MoE ... shape
// templates", sections 1 and 5: virtual experts of kBlockN rows, ids outside
// the local slice get -1, ranks in ascending token order).
//
// Small slot counts: one CTA of 32 warps; warp w owns a contiguous run of
// slots (the slots' local experts are staged in shared memory first).  Large
// slot counts: the same per-warp passes spread over CTAs of 8 warps (4096
// slots each, a warp's 512 ids held in registers) with a one-CTA scan in
// between.  Two passes over the slots in rounds of 32, each round grouping
// equal experts (same_expert_lanes, the lanes holding the same expert):
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
#include "route_sort.cuh"

#include <cooperative_groups.h>

namespace moe {

namespace {

constexpr int kSortThreads = 1024;
constexpr int kSortWarps = kSortThreads / 32;
using rs::local_expert;
using rs::place_experts;

constexpr int kBigWarps = 8;
constexpr int kBigWarpSlots = 512;
constexpr int kBigRounds = kBigWarpSlots / 32;

// The lanes of the warp holding the same local expert as this lane (the
// mask match.any returns), from one ballot per bit: e in [-1, 1023] is taken
// as 11 bits (-1 -> 2047) and a lane matches where every bit agrees.  Eleven
// ballots cost far less than match.any over 32 distinct experts (on GB300
// a count round went from ~1400 to ~100 cycles).
__device__ __forceinline__ uint32_t same_expert_lanes(int e) {
    const uint32_t v = static_cast<uint32_t>(e) & 2047u;
    uint32_t m = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < 11; ++b) {
        const bool bit = (v >> b) & 1u;
        const uint32_t x = __ballot_sync(0xffffffffu, bit);
        m &= bit ? x : ~x;
    }
    return m;
}

// The local experts of a warp's kBigWarpSlots slots [s0, s1), round r in
// e[r] (lane = slot within the round; -1 past s1 or without a local row).
// All loads are issued before any is used.
__device__ __forceinline__ void load_experts(const SortParams& p, int s0, int s1, int (&e)[kBigRounds]) {
    const int lane = threadIdx.x & 31;
    int id[kBigRounds];
#pragma unroll
    for (int r = 0; r < kBigRounds; ++r) {
        const int s = s0 + 32 * r + lane;
        id[r] = s < s1 ? p.ids[s] : -1;
    }
#pragma unroll
    for (int r = 0; r < kBigRounds; ++r) e[r] = (s0 + 32 * r + lane < s1) ? local_expert(id[r], p) : -1;
}

// Per-warp histogram of a warp's slots into my_hist, in rounds of 32: equal
// experts are grouped (same_expert_lanes) and the group's leader adds the
// group size.  Here on experts already in registers.
__device__ __forceinline__ void warp_count_regs(const int (&e)[kBigRounds], int* my_hist) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kBigRounds; ++r) {
        const uint32_t peers = same_expert_lanes(e[r]);
        if (e[r] >= 0 && lane == __ffs(peers) - 1) my_hist[e[r]] += __popc(peers);
    }
}

// Ranks of a warp's slots [s0, s1): row = my_base[e] + earlier slots of e in
// this warp + lower lanes of e in this round; my_base advances in place.
// Here on experts held in registers (round r in e[r]).
__device__ __forceinline__ void warp_rank_regs(const SortParams& p, int s0, int s1, const int (&e)[kBigRounds],
                                               int* my_base) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < kBigRounds; ++r) {
        const int s = s0 + 32 * r + lane;
        const uint32_t peers = same_expert_lanes(e[r]);
        if (s < s1) {
            if (e[r] >= 0) {
                const int row = my_base[e[r]] + __popc(peers & ptx::lanemask_lt());
                p.c_map[s] = row;
                p.a_map[row] = s;
            } else {
                p.c_map[s] = -1;
            }
        }
        __syncwarp();
        if (e[r] >= 0 && lane == __ffs(peers) - 1) my_base[e[r]] += __popc(peers);
        __syncwarp();
    }
}

// The same two passes on the slots' local experts staged in shared memory.
__device__ __forceinline__ void warp_count_smem(const int* s_e, int s0, int s1, int* my_hist) {
    const int lane = threadIdx.x & 31;
    for (int base = s0; base < s1; base += 32) {
        const int s = base + lane;
        const int e = s < s1 ? s_e[s] : -1;
        const uint32_t peers = same_expert_lanes(e);
        if (e >= 0 && lane == __ffs(peers) - 1) my_hist[e] += __popc(peers);
    }
}

// my_base[e]: this warp's first rank inside expert e; e_off[e]: the expert's
// first row.
__device__ __forceinline__ void warp_rank_smem(const SortParams& p, const int* s_e, int s0, int s1, int* my_base,
                                               const int* e_off) {
    const int lane = threadIdx.x & 31;
    for (int base = s0; base < s1; base += 32) {
        const int s = base + lane;
        const int e = s < s1 ? s_e[s] : -1;
        const uint32_t peers = same_expert_lanes(e);
        if (s < s1) {
            if (e >= 0) {
                const int row = e_off[e] + my_base[e] + __popc(peers & ptx::lanemask_lt());
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
    __shared__ int s_tot[3][rs::kScanWarps];

    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < kSortWarps * p.Et; i += kSortThreads) hist[i] = 0;
    ptx::pdl_wait();
    __syncthreads();

    const int n = p.T * p.kp;
    // every slot's local expert, loaded once (eight loads in flight per
    // thread) into shared memory; both passes read it from there
    int* s_e = s_off + p.Et;  // [n]
    for (int i0 = 0; i0 < n; i0 += 8 * kSortThreads) {
        int id[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * kSortThreads + tid;
            id[u] = i < n ? p.ids[i] : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * kSortThreads + tid;
            if (i < n) s_e[i] = local_expert(id[u], p);
        }
    }
    __syncthreads();
    const int per = (((n + kSortWarps - 1) / kSortWarps) + 31) & ~31;
    const int s0 = min(n, warp * per);
    const int s1 = min(n, s0 + per);
    int* my_hist = hist + warp * p.Et;
    warp_count_smem(s_e, s0, s1, my_hist);
    __syncthreads();

    // per expert: exclusive prefix over the warps (in place), in batches of 8
    // loads so that they overlap, and the total
    int cnt = 0;
    if (tid < p.Et) {
#pragma unroll
        for (int w0 = 0; w0 < kSortWarps; w0 += 8) {
            int c[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) c[u] = hist[(w0 + u) * p.Et + tid];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                hist[(w0 + u) * p.Et + tid] = cnt;
                cnt += c[u];
            }
        }
    }
    place_experts(p, cnt, s_off, s_tot);
    __syncthreads();
    // ranks: the expert's first row (s_off) + earlier warps + this warp's
    warp_rank_smem(p, s_e, s0, s1, my_hist, s_off);
    ptx::pdl_launch_dependents();
}

// Ranks the T * k' slots whose picked ids sit in s_ids, in one CTA of
// kSortThreads threads, with per-expert bitmasks over the tokens (s_mask:
// [nw][Et] words, word w of every expert side by side so that the counting
// pass -- thread = expert -- reads consecutive words; zeroed by the caller).
// Valid when a token picks an expert at most once, as the routing's picks do
// (the top-k are distinct experts and the shared experts are distinct from
// them): token t sets bit t of each picked expert's mask; the expert's row
// count is the popcount of its mask and slot (t, j)'s row is the expert's
// first row plus the number of its bits below t -- ascending token inside
// each expert, the rows of the ballot-grouped passes (the popcount rank of
// "[sglang] ... MXFP4 decode MoE ... shape templates", section 5, over the
// whole batch).  row_w (optional) receives each row's routing weight w[slot].
// s_ids is overwritten with each slot's local expert (-1: not local).
// s_pref (optional, [nw][Et] 16-bit): the popcount of each expert's mask
// words below word w, so a slot's rank takes one masked popcount instead of
// one per earlier word.  s_rows (optional, R ints of shared memory): the
// rank pass records each row's slot there, and a second pass writes a_map
// and row_w in row order (coalesced) instead of one scattered store per
// slot.  One CTA of kSortThreads threads: the passes are bound by its
// instruction issue, so a thread steps its slots' token index by addition
// rather than dividing by k'.
__device__ __forceinline__ void rank_by_token_masks(const SortParams& p, int* s_ids, uint32_t* s_mask,
                                                    uint16_t* s_pref, int* s_off, int (*s_tot)[rs::kScanWarps],
                                                    const float* w, float* row_w, int* s_rows) {
    const int tid = threadIdx.x;
    const int n = p.T * p.kp;
    const int nw = (p.T + 31) >> 5;
    const int t0 = tid / p.kp;                             // token of this thread's first slot
    const int dt = kSortThreads / p.kp, dj = kSortThreads - dt * p.kp;
    const int j0 = tid - t0 * p.kp;
    for (int sl = tid, t = t0, j = j0; sl < n; sl += kSortThreads) {
        const int e = local_expert(s_ids[sl], p);
        s_ids[sl] = e;
        if (e >= 0) atomicOr(&s_mask[(t >> 5) * p.Et + e], 1u << (t & 31));
        t += dt;
        j += dj;
        if (j >= p.kp) {
            j -= p.kp;
            ++t;
        }
    }
    __syncthreads();
    int cnt = 0;
    if (tid < p.Et) {
#pragma unroll 8
        for (int wd = 0; wd < nw; ++wd) {
            if (s_pref) s_pref[wd * p.Et + tid] = static_cast<uint16_t>(cnt);
            cnt += __popc(s_mask[wd * p.Et + tid]);
        }
    }
    place_experts(p, cnt, s_off, s_tot);
    __syncthreads();
    for (int sl = tid, t = t0, j = j0; sl < n; sl += kSortThreads) {
        const int e = s_ids[sl];
        if (e >= 0) {
            const int wt = t >> 5;
            const uint32_t* m = s_mask + e;  // word w at m[w * Et]
            int r = __popc(m[wt * p.Et] & ((1u << (t & 31)) - 1u));
            if (s_pref) {
                r += s_pref[wt * p.Et + e];
            } else {
                for (int wd = 0; wd < wt; ++wd) r += __popc(m[wd * p.Et]);
            }
            const int row = s_off[e] + r;
            p.c_map[sl] = row;
            if (s_rows) {
                s_rows[row] = sl;
            } else {
                p.a_map[row] = sl;
                if (row_w) row_w[row] = w[sl];
            }
        } else {
            p.c_map[sl] = -1;
        }
        t += dt;
        j += dj;
        if (j >= p.kp) {
            j -= p.kp;
            ++t;
        }
    }
    if (s_rows) {
        __syncthreads();
        const int R = p.offsets[p.Et];  // written by place_experts before the barrier above
        for (int row = tid; row < R; row += kSortThreads) {
            const int sl = s_rows[row];
            p.a_map[row] = sl;
            if (row_w) row_w[row] = w[sl];
        }
    }
}

// The layer's own routing past the fused range: the ids are the routing's,
// so one CTA ranks them with token bitmasks (rank_by_token_masks) instead of
// the ballot-grouped passes that arbitrary ids (duplicates, masked -1) need.
// Shared memory holds the masks and prefixes (Et * T/32 words and
// half-words), then the slots' experts, their routing weights (row_w given)
// and the row -> slot table (T * k' each): up to kSortTokensMaxT tokens when
// that fits (T 512 at k' 17 and 896 experts does).
constexpr int kSortTokensMaxT = 512;
constexpr size_t kSortTokensMaxSmem = 220 * 1024;

size_t sort_tokens_smem(int T, int kp, int Et, bool with_w) {
    const size_t n = static_cast<size_t>(T) * kp;
    const size_t nw = (static_cast<size_t>(T) + 31) / 32;
    const size_t pref = ((static_cast<size_t>(Et) * nw * 2 + 3) / 4) * 4;
    return static_cast<size_t>(Et) * nw * 4 + pref + n * 4 * (with_w ? 3 : 2);
}

__device__ __forceinline__ size_t sort_tokens_pref_bytes(int Et, int T) {
    return ((static_cast<size_t>(Et) * ((T + 31) / 32) * 2 + 3) / 4) * 4;
}

__global__ void __launch_bounds__(kSortThreads, 1) sort_tokens_kernel(SortParams p, const float* w, float* row_w) {
    __shared__ int s_off[1024];
    __shared__ int s_tot[3][rs::kScanWarps];
    extern __shared__ uint32_t s_mask[];
    const int tid = threadIdx.x;
    const int nw = (p.T + 31) >> 5;
    const int n = p.T * p.kp;
    uint16_t* s_pref = reinterpret_cast<uint16_t*>(s_mask + p.Et * nw);
    int* s_ids = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(s_pref) + sort_tokens_pref_bytes(p.Et, p.T));
    float* s_w = reinterpret_cast<float*>(s_ids + n);
    int* s_rows = reinterpret_cast<int*>(s_w + (row_w ? n : 0));
    for (int wd = tid; wd < p.Et * nw; wd += kSortThreads) s_mask[wd] = 0;
    ptx::pdl_wait();
#pragma unroll 4
    for (int sl = tid; sl < n; sl += kSortThreads) {
        s_ids[sl] = p.ids[sl];
        if (row_w) s_w[sl] = w[sl];
    }
    __syncthreads();
    rank_by_token_masks(p, s_ids, s_mask, s_pref, s_off, s_tot, s_w, row_w, s_rows);
    ptx::pdl_launch_dependents();
}

// Route and sort in one launch when the batch has at most kFusedMaxT tokens
// (decode).  A cluster of kRouteCtas CTAs routes the tokens (token t on CTA
// t % kRouteCtas, so the routing spreads over that many SMs) and stores the
// picked ids straight into CTA 0's shared memory; after the cluster barrier
// CTA 0 ranks the slots with per-expert token bitmasks (rank_by_token_masks).
//
// fuse_x (decode tilings, x kept in token order): the warps that route no
// token quantise the CTA's tokens' x rows to MXFP8 meanwhile, and CTA 0
// writes each row's routing weight while ranking -- the launch then also
// does the gather's work, and no launch of its own is spent on it.  Past 64
// tokens every warp routes, and x on 8 SMs would run after the routing at
// those SMs' bandwidth: the route kernel over the whole GPU (quantising x on
// its grid) followed by sort_tokens_kernel is faster there (measured on
// GB300 at T 72 to 256).
constexpr int kFusedMaxT = 64;
constexpr int kFuseXMaxT = 64;
constexpr int kRouteCtas = 8;

__global__ void __cluster_dims__(kRouteCtas, 1, 1) __launch_bounds__(kSortThreads, 1)
    route_sort_small_kernel(RouteParams rp, SortParams p, GatherParams gp, int fuse_x) {
    __shared__ uint2 s_cand[kSortWarps][rs::kMaxCand];
    __shared__ int s_off[1024];
    __shared__ int s_tot[3][rs::kScanWarps];
    // dynamic: [nw][Et] token bitmasks (word w of every expert side by side,
    // so the per-expert counting pass -- thread = expert -- reads consecutive
    // words), then the slots' picked ids [T * k']
    extern __shared__ uint32_t s_mask[];
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int nw = (p.T + 31) >> 5;  // mask words per expert
    int* s_ids = reinterpret_cast<int*>(s_mask + p.Et * nw);
    int* ids0 = cluster.map_shared_rank(s_ids, 0);  // CTA 0's id table
    ptx::pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5;
    if (rank == 0)
        for (int w = tid; w < p.Et * nw; w += kSortThreads) s_mask[w] = 0;
    for (int t = rank + kRouteCtas * warp; t < rp.T; t += kRouteCtas * kSortWarps)
        rs::route_token(rp, t, s_cand[warp], ids0);
    if (fuse_x) {
        // x -> MXFP8 of this CTA's tokens (rank, rank + 8, ...), one
        // 32-element block per job, on the warps that route no token while
        // the others route (on every warp, after routing, when all route);
        // token order, row-major scales
        const int nt = (p.T - rank + kRouteCtas - 1) / kRouteCtas;
        const int nb = gp.H / 32;
        const int nr = 32 * min(nt, kSortWarps);  // routing threads
        const bool all_route = nr == kSortThreads;
        const int first = all_route ? tid : tid - nr;
        const int stride = all_route ? kSortThreads : kSortThreads - nr;
        for (int job = first; first >= 0 && job < nt * nb; job += stride) {
            const int j = job / nb, b = job - j * nb;
            const size_t blk = static_cast<size_t>(rank + kRouteCtas * j) * nb + b;
            quant_x_block(gp.x, gp.xq, gp.xsf, blk);
        }
    }
    cluster.sync();
    if (rank != 0) {
        ptx::pdl_launch_dependents();
        return;  // nothing reads the other CTAs' shared memory
    }

    rank_by_token_masks(p, s_ids, s_mask, nullptr, s_off, s_tot, rp.w, fuse_x ? gp.row_w : nullptr, nullptr);
    // The launch that follows (FC1 at the decode tilings, the gather at
    // 128-row tiles) reads the work list only after its griddepcontrol.wait.
    ptx::pdl_launch_dependents();
}

// Large slot counts: CTA c owns slots [c * kBigChunk, (c + 1) * kBigChunk),
// warp w of it the w-th sub-run of kBigWarpSlots.
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
    int e[kBigRounds];
    load_experts(p, s0, min(n, s0 + kBigWarpSlots), e);
    warp_count_regs(e, hist + warp * p.Et);
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
    __shared__ int s_tot[3][rs::kScanWarps];
    ptx::pdl_wait();
    const int tid = threadIdx.x;
    int cnt = 0;
    if (tid < p.Et) {
        // 16 CTAs' counts are loaded together (independent loads), then
        // replaced by their exclusive prefix
        int* h = p.cta_hist + tid;
        for (int c0 = 0; c0 < nctas; c0 += 16) {
            int v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = (c0 + j < nctas) ? h[static_cast<size_t>(c0 + j) * p.Et] : 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (c0 + j < nctas) h[static_cast<size_t>(c0 + j) * p.Et] = cnt;
                cnt += v[j];
            }
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
    int e[kBigRounds];
    load_experts(p, s0, s1, e);
    warp_count_regs(e, hist + warp * p.Et);
    __syncthreads();
    for (int x = tid; x < p.Et; x += kBigWarps * 32) {
        int run = p.offsets[x] + p.cta_hist[static_cast<size_t>(blockIdx.x) * p.Et + x];
        for (int w = 0; w < kBigWarps; ++w) {
            const int c = hist[w * p.Et + x];
            hist[w * p.Et + x] = run;
            run += c;
        }
    }
    __syncthreads();
    warp_rank_regs(p, s0, s1, e, hist + warp * p.Et);
    ptx::pdl_launch_dependents();
}

}  // namespace

// per-warp histograms [32][Et], expert offsets [Et] and the slots' experts [n]
size_t sort_smem_bytes(int Et, int n) { return (static_cast<size_t>(kSortWarps + 1) * Et + n) * sizeof(int); }

int sort_big_ctas(int n) { return (n + kBigChunk - 1) / kBigChunk; }

cudaError_t launch_sort(const SortParams& p, cudaStream_t stream, bool pdl) {
    const int n = p.T * p.kp;
    if (n <= kSortWarps * kBigWarpSlots) {
        const size_t smem = sort_smem_bytes(p.Et, n);
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

int sort_launch_count(int64_t slots) { return slots <= kSortWarps * kBigWarpSlots ? 1 : 3; }

bool route_sort_fusable(int T, int kp) { return T <= kFusedMaxT && kp <= 33; }

bool route_sort_fuses_x(int T) { return T > 0 && T <= kFuseXMaxT; }

bool sort_tokens_ok(int T, int kp, int Et) {
    return T <= kSortTokensMaxT && sort_tokens_smem(T, kp, Et, true) <= kSortTokensMaxSmem;
}

cudaError_t launch_sort_tokens(const SortParams& p, cudaStream_t stream, bool pdl, const float* w, float* row_w) {
    const size_t smem = sort_tokens_smem(p.T, p.kp, p.Et, row_w != nullptr);
    cudaError_t err = cudaFuncSetAttribute(sort_tokens_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_kernel(sort_tokens_kernel, dim3(1), dim3(kSortThreads), smem, stream, pdl, p, w, row_w);
}

cudaError_t launch_route_sort_small(const RouteParams& rp, const SortParams& p, const GatherParams* gp,
                                    cudaStream_t stream, bool pdl) {
    const size_t smem = (static_cast<size_t>(p.Et) * ((p.T + 31) / 32) + static_cast<size_t>(p.T) * p.kp) * 4;
    cudaError_t err = cudaFuncSetAttribute(route_sort_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const GatherParams g = gp ? *gp : GatherParams{};
    return launch_kernel(route_sort_small_kernel, dim3(kRouteCtas), dim3(kSortThreads), smem, stream, pdl, rp, p, g,
                         gp ? 1 : 0);
}

}  // namespace moe
