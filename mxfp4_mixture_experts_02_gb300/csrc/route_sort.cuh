// Device pieces shared by the routing and sort kernels: the per-token top-k
// of one warp and the expert-level placement of rows into virtual experts.
#pragma once

#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace rs {

constexpr int kMaxPerLane = 32;  // E_global <= 1024: expert lane + 32 i in lane `lane`
constexpr int kMaxCand = 64;     // candidate list of the fast top-k path
constexpr uint32_t kNoId = 0xFFFFFFFFu;

// Monotone map of a finite fp32 to uint32 (a < b  <=>  key(a) < key(b));
// -0 is folded onto +0 so that equal values tie; every finite value and
// -inf map above 0, so key 0 marks an absent or taken entry.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Best (largest key, lowest index on ties) of a lane's entries by a
// pairwise tree; a tie compares the indices (after the first level an upper
// entry may carry a lower index than the entry it meets).
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
            if (k[i + w] > k[i] || (k[i + w] == k[i] && ix[i + w] < ix[i])) {
                k[i] = k[i + w];
                ix[i] = ix[i + w];
            }
    bk = k[0];
    bi = ix[0];
}

// (key, id) a ranks before b: larger key, or equal key and smaller id.
__device__ __forceinline__ bool ranks_before(uint2 a, uint2 b) { return a.x > b.x || (a.x == b.x && a.y < b.y); }

// Top-k (k <= 32) of one token's logits row[0, Eg) by one warp: lane j < k
// receives the key and expert id of the j-th pick (descending logit, ties to
// the lower id).  `cand` is this warp's shared-memory scratch of kMaxCand
// entries.
//
// Fast path: let thr be the k-th largest of the 32 lane maxima.  At least k
// lane maxima are >= thr, so an entry below thr has k entries above it and
// cannot be picked: the top-k of the whole row is the top-k of the entries
// >= thr (typically a few dozen).  Those are compacted into `cand` and picked
// in k rounds of two warp reductions (maximum key, then minimum id among the
// lanes holding it) over two entries per lane.  With more than kMaxCand
// candidates (heavy ties) the same rounds run over all entries, the winning
// lane rescanning its own 32 with a pairwise tree.
__device__ __forceinline__ void warp_topk(const float* row, int Eg, int k, uint2* cand, uint32_t& my_key,
                                          uint32_t& my_id) {
    const int lane = threadIdx.x & 31;
    uint32_t key[kMaxPerLane];
    uint32_t lmax = 0;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        key[i] = (e < Eg) ? order_key(row[e]) : 0u;
        lmax = max(lmax, key[i]);
    }
    // bitonic sort of the lane maxima, descending across lanes
    uint32_t v = lmax;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool desc = (lane & size) == 0;
            const bool lower = (lane & stride) == 0;
            v = (desc == lower) ? max(v, o) : min(v, o);
        }
    const uint32_t thr = __shfl_sync(0xffffffffu, v, k - 1);
    int c = 0;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) c += (key[i] != 0 && key[i] >= thr) ? 1 : 0;
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    const int total = __shfl_sync(0xffffffffu, inc, 31);
    my_key = 0;
    my_id = 0;
    if (thr != 0 && total <= kMaxCand) {
        int pos = inc - c;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i)
            if (key[i] != 0 && key[i] >= thr) cand[pos++] = make_uint2(key[i], static_cast<uint32_t>(lane + 32 * i));
        __syncwarp();
        uint2 a = lane < total ? cand[lane] : make_uint2(0u, kNoId);
        uint2 b = lane + 32 < total ? cand[lane + 32] : make_uint2(0u, kNoId);
        __syncwarp();  // the scratch may be reused by the next token
        if (ranks_before(b, a)) {
            const uint2 t = a;
            a = b;
            b = t;
        }
        for (int j = 0; j < k; ++j) {
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, a.x);
            const uint32_t win = __reduce_min_sync(0xffffffffu, (a.x == kmax && a.x != 0) ? a.y : kNoId);
            if (a.x != 0 && a.y == win) {
                a = b;
                b = make_uint2(0u, kNoId);
            }
            if (lane == j) {
                my_key = kmax;
                my_id = win;
            }
        }
    } else {
        uint32_t bk;
        int bi;
        lane_best(key, bk, bi);
        for (int j = 0; j < k; ++j) {
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t cid = (bk == kmax && bk != 0) ? static_cast<uint32_t>(lane + 32 * bi) : kNoId;
            const uint32_t win = __reduce_min_sync(0xffffffffu, cid);
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
    }
}

// Routes token t with one warp: top-k picks and their renormalised softmax
// weights, then the shared experts (id E_global + s, weight
// sigmoid(fp32(bf16 logit)) * scale, in fp32: "[sglang] SGLang MoE shared
// expert: fuse 3 kernels into 1").  Writes ids / weights of the token's k'
// slots to global memory and, when s_ids is given, the ids to s_ids too.
__device__ __forceinline__ void route_token(const RouteParams& p, int t, uint2* cand, int* s_ids) {
    const int lane = threadIdx.x & 31;
    uint32_t my_key, my_id;
    warp_topk(p.logits + static_cast<size_t>(t) * p.Eg, p.Eg, p.k, cand, my_key, my_id);
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
        if (s_ids) s_ids[base + lane] = static_cast<int32_t>(my_id);
    }
    if (lane < p.S) {
        const float x = bf16_bits_to_float(p.shared_logit[static_cast<size_t>(t) * p.S + lane]);
        p.ids[base + p.k + lane] = p.Eg + lane;
        p.w[base + p.k + lane] = p.shared_scale / (1.0f + expf(-x));
        if (s_ids) s_ids[base + p.k + lane] = p.Eg + lane;
    }
}

// Local row owner of a global id: the slice [off, off + E) maps to 0..E-1,
// shared experts E_global + s to E + s, anything else (masked -1, other
// slices) to -1.
__device__ __forceinline__ int local_expert(int32_t id, const SortParams& p) {
    if (id >= p.Eg && id < p.Eg + p.S) return p.E + (id - p.Eg);
    if (id >= p.off && id < p.off + p.E) return id - p.off;
    return -1;
}

constexpr int kScanWarps = 32;  // block_scan3 / place_experts run on 1024 threads

// Exclusive scan of three ints across a block of 1024 threads.
__device__ __forceinline__ void block_scan3(int a, int b, int c, int& ea, int& eb, int& ec, int& ta, int& tb, int& tc,
                                            int (*s_tot)[kScanWarps]) {
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
    ta = s_tot[0][kScanWarps - 1];
    tb = s_tot[1][kScanWarps - 1];
    tc = s_tot[2][kScanWarps - 1];
}

// The GEMM2 gate ("[FlashInfer] Device-side gating for the MoE GEMM2 path",
// sections 1 and 2): chosen on the device once the sorted table's row count
// R is known, so one fixed launch chain (one CUDA graph) serves every
// routing:
//   split: FC2 writes each routed row (w * Y); the combine sums a token's rows
//          in slot order (bit-reproducible);
//   dense: FC2's epilogue reduces w * Y straight into an fp32 [T, H]
//          accumulator at the L2 (the finalize fused into GEMM2); the combine
//          only converts it to bf16.  The order of the reductions varies from
//          run to run, so the last bits of the sums may too.
// The rule: dense needs the accumulator to stay in L2, T * H * 4 bytes <=
// 32 MiB (well inside the 126 MiB L2: the reductions then run at the L2).
// Within that, the split rows' format decides.  The decode tilings' split
// rows are fp32 (8 bytes per element written and read back), which costs
// more than the reductions at every such batch: dense.  The 128-row tiling's
// rows are bf16 (4 bytes per element), cheaper than the reductions once
// there are many: dense only while R * H <= dense_max_128.  Measured on
// GB300 (H 3584, top-16): decode tilings dense faster at every T up to 2340
// (742 against 848 us per layer there); 128-row tiles dense faster up to
// T 1024 (R * H = 56 Mi; 470 against 475 us), split from T 1280 (484 against
// 491 us) and 2x faster at the 32768-token prefill, whose 470 MB accumulator
// lives in DRAM.  A caller may force either path.  The pages give the gate
// a one-warp launch after the sort; here the thread that writes the sort's
// header decides, and the chain has no launch for it.
__device__ __forceinline__ int gemm2_path(int R, int T, int H, int B, int force, int64_t dense_max_128) {
    if (force == 1) return kPathSplit;
    if (force == 2) return kPathDense;
    const bool acc_in_l2 = static_cast<int64_t>(T) * H * 4 <= (int64_t(32) << 20);
    const bool rows_ok = B < 128 || static_cast<int64_t>(R) * H <= dense_max_128;
    return acc_in_l2 && rows_ok ? kPathDense : kPathSplit;
}

// Expert-level placement (one CTA of 1024 threads, thread tid = expert):
// given each expert's row count, scan (count, tiles, groups), write counts /
// offsets / virtual experts / work groups and the header (with the GEMM2
// gate's path), and leave each expert's first row in s_off (when given).
__device__ __forceinline__ void place_experts(const SortParams& p, int cnt, int* s_off, int (*s_tot)[kScanWarps]) {
    const int tid = threadIdx.x;
    const int tiles = (cnt + p.B - 1) / p.B;
    const int grps = (tiles + p.G - 1) / p.G;
    int off, vb, gb, R, V, NG;
    block_scan3(cnt, tiles, grps, off, vb, gb, R, V, NG, s_tot);
    if (tid < p.Et) {
        if (s_off) s_off[tid] = off;
        p.counts[tid] = cnt;
        p.offsets[tid] = off;
        p.vbase[tid] = vb;
        for (int c = 0; c < tiles; ++c)
            p.vinfo[vb + c] = make_int4(tid, off + c * p.B, min(p.B, cnt - c * p.B), c);
        for (int g = 0; g < grps; ++g) p.groups[gb + g] = make_int4(tid, vb + g * p.G, min(p.G, tiles - g * p.G), 0);
    }
    if (tid == 0) {
        p.offsets[p.Et] = R;
        p.header[kHdrRows] = R;
        p.header[kHdrNumV] = V;
        p.header[kHdrNumGroups] = NG;
        p.header[kHdrGemm2Path] = gemm2_path(R, p.T, p.H, p.B, p.gemm2_force, p.dense_max_elems);
        if (!p.keep_status) {
            p.header[kHdrStatus] = 0;
            p.header[kHdrDetail] = 0;
        }
    }
}

}  // namespace rs
}  // namespace moe
