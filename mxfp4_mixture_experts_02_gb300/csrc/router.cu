// Router GEMM: logits[t][e] = sum_h x[t][h] * wr[e][h] with bf16 x [T, H] and
// bf16 router rows wr [E_global, H], fp32 accumulation -- the step in front of
// the routing of "... MXFP4 decode MoE ... shape templates" (section 5 starts
// from the top-k ids of these logits), run on the tensor cores in the same
// launch chain.
//
// Tile = 128 tokens x N router rows (experts).  One tcgen05.mma kind::f16
// (bf16 x bf16 -> fp32) per 16-wide K step: A = the token tile, B = the router
// rows, both K-major in 128-byte-swizzled tiles of 64 K; accumulator 128 lanes
// x N columns in TMEM.  Tokens past T and rows past E_global are zero-filled
// by TMA and masked on output.
//
// Short batches (the decode tiling) split K over the KS CTAs of a cluster:
// N = 64, KS = 8, so a 32-token batch at E_global 896 runs 112 CTAs that each
// stream 1/112 of the router matrix.  Each CTA stages its fp32 partial tile in
// its own shared memory; after a cluster barrier every CTA sums a slice of
// the tile over the KS partials in rank order (distributed shared memory
// loads, a fixed order: the logits are bit-reproducible), then a second
// barrier keeps the partials alive until all reads are done.  Long batches
// use N = 224 (E_global 896 = 4 tiles), no split, and a persistent grid with
// two TMEM accumulators (below).
//
// Warps: 0..3 epilogue (TMEM lane quadrant = warp), 4 TMA producer, 5 TMEM
// allocator and single-thread MMA issuer.  Every mbarrier wait is bounded; on
// expiry the CTA records MOE_ERR_TIMEOUT in the status word, skips the rest of
// its work, still reaches both cluster barriers, lets its MMAs and copies
// drain, frees TMEM and exits.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

namespace cg = cooperative_groups;

constexpr int kRtWarps = 6;
constexpr int kRtThreads = kRtWarps * 32;
constexpr int kRtProducerWarp = 4;
constexpr int kRtMmaWarp = 5;
constexpr int kRtStages = 5;
constexpr int kRtKChunk = 64;  // bf16 elements per 128-byte row of a stage

enum { kRtSiteProducer = 11, kRtSiteMma = 12, kRtSiteEpi = 13 };

template <int N>
struct RtCfg {
    static constexpr int kATile = 128 * 128;  // 128 token rows x 64 bf16
    static constexpr int kBTile = N * 128;    // N router rows x 64 bf16
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kRtStages * kATile;
    static constexpr int kPipeBytes = kOffB + kRtStages * kBTile;
    static constexpr int kPartStride = N + 4;  // floats per staged partial row (16-byte rows, odd in 16-byte units)
    static constexpr int kOffBar = kPipeBytes;
    static constexpr int kSmemBytes = kOffBar + (2 * kRtStages + 2) * 8 + 16 + 1024;
    static constexpr uint32_t kTmemCols = N <= 64 ? 64 : 256;
    static constexpr uint32_t kStageTx = kATile + kBTile;
    static_assert(N % 32 == 0, "N: whole 32-column TMEM loads");
    static_assert(N % 16 == 0 && N >= 16 && N <= 256, "kind::f16 with M = 128 needs N % 16 == 0, 16..256");
    static_assert(128 * kPartStride * 4 <= kPipeBytes, "the partial tile fits in the drained pipeline buffers");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ void rt_record_timeout(const RouterParams& p, volatile int* abort_flag, int site) {
    *abort_flag = 1;
    if (p.status && atomicCAS(p.status, 0, MOE_ERR_TIMEOUT) == 0) p.status[1] = site * 65536 + static_cast<int>(blockIdx.x);
}

__device__ __forceinline__ bool rt_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, volatile int* abort_flag) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > limit_ns) return false;
    }
}

// Writes 32 consecutive fp32 logits of one token row (columns e0..e0+31),
// masked at E_global.
__device__ __forceinline__ void store_logits_32(float* row, int e0, int Eg, const uint32_t (&r)[32]) {
    if (e0 + 32 <= Eg && (Eg & 3) == 0) {
        float4* dst = reinterpret_cast<float4*>(row + e0);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                                 __uint_as_float(r[4 * j + 3]));
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (e0 + j < Eg) row[e0 + j] = __uint_as_float(r[j]);
    }
}

template <int N>
__global__ void __launch_bounds__(kRtThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                       const RouterParams p) {
    using C = RtCfg<N>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* empty = full + kRtStages;
    uint64_t* accfull = empty + kRtStages;
    uint64_t* done = accfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ks = p.ks;
    const int rank = static_cast<int>(blockIdx.x) % ks;  // == the cluster rank along x
    const int tile = static_cast<int>(blockIdx.x) / ks;
    const int m0 = (tile / p.n_tiles) * 128;
    const int n0 = (tile % p.n_tiles) * N;
    const int kc_per_rank = p.H / kRtKChunk / ks;
    const int kc0 = rank * kc_per_rank;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(accfull, 1);
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == kRtProducerWarp && lane == 0) {
        ptx::tma_prefetch_desc(&tmX);
        ptx::tma_prefetch_desc(&tmW);
    }
    if (warp == kRtMmaWarp) {
        ptx::tmem_alloc(tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // x and the logits buffer may belong to the preceding kernel of the chain
    ptx::pdl_wait();

    if (warp == kRtProducerWarp) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            for (int kc = 0; kc < kc_per_rank; ++kc) {
                if (!rt_wait(&empty[stage], phase ^ 1, p.wait_ns, abort_flag)) {
                    if (!*abort_flag) rt_record_timeout(p, abort_flag, kRtSiteProducer);
                    break;
                }
                ptx::mbar_arrive_expect_tx(&full[stage], C::kStageTx);
                const int k = (kc0 + kc) * kRtKChunk;
                ptx::tma_load_2d(smem + C::kOffA + stage * C::kATile, &tmX, &full[stage], k, m0);
                ptx::tma_load_2d(smem + C::kOffB + stage * C::kBTile, &tmW, &full[stage], k, n0);
                ++issued;
                if (++stage == kRtStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            // every issued stage lands before the buffers are reused or the CTA exits (bounded)
            for (int i = issued > kRtStages ? issued - kRtStages : 0; i < issued; ++i)
                ptx::mbar_wait(&full[i % kRtStages], static_cast<uint32_t>(i / kRtStages) & 1, 10ull * 1000 * 1000);
        }
    } else if (warp == kRtMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t kIdesc = ptx::idesc_f16_bf16(128, N);
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int kc = 0; kc < kc_per_rank; ++kc) {
                if (!rt_wait(&full[stage], phase, p.wait_ns, abort_flag)) {
                    if (!*abort_flag) rt_record_timeout(p, abort_flag, kRtSiteMma);
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t xa = ptx::smem_u32(smem + C::kOffA + stage * C::kATile);
                const uint32_t wa = ptx::smem_u32(smem + C::kOffB + stage * C::kBTile);
#pragma unroll
                for (int kk = 0; kk < kRtKChunk / 16; ++kk)
                    ptx::mma_f16(tmem, ptx::sdesc_sw128(xa + kk * 32), ptx::sdesc_sw128(wa + kk * 32), kIdesc,
                                 (kc | kk) != 0);
                ptx::tc_commit(&empty[stage]);
                if (++stage == kRtStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (ok) ptx::tc_commit(accfull);
            ptx::tc_commit(done);
            ptx::mbar_wait(done, 0, 10ull * 1000 * 1000);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int row = warp * 32 + lane;  // token row within the tile = TMEM lane
        bool ok = rt_wait(accfull, 0, p.wait_ns, abort_flag);
        if (!ok && lane == 0 && !*abort_flag) rt_record_timeout(p, abort_flag, kRtSiteEpi);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            ptx::tc_fence_after();
            const uint32_t tq = tmem + (static_cast<uint32_t>(warp * 32) << 16);
            if (ks == 1) {
                const bool valid = m0 + row < p.T;
                float* out = p.logits + static_cast<int64_t>(m0 + row) * p.Eg;
#pragma unroll 1
                for (int c = 0; c < N / 32; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld32(tq + 32 * c, r);
                    ptx::tmem_wait_ld();
                    if (valid) store_logits_32(out, n0 + 32 * c, p.Eg, r);
                }
            } else {
                // the pipeline buffers are drained (accfull: every MMA, and so
                // every stage it read, has completed): stage the partial there
                float* part = reinterpret_cast<float*>(smem) + row * C::kPartStride;
#pragma unroll 1
                for (int c = 0; c < N / 32; ++c) {
                    uint32_t r[32];
                    ptx::tmem_ld32(tq + 32 * c, r);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        reinterpret_cast<float4*>(part + 32 * c)[j] =
                            make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                        __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                }
            }
        }
    }

    if (ks > 1) {
        // Every CTA of the cluster reaches both barriers, aborted or not; each
        // CTA converges first (the producer and MMA lanes left their loops at
        // different times).
        cg::cluster_group cluster = cg::this_cluster();
        __syncthreads();
        cluster.sync();
        const int rows = min(128, p.T - m0);
        const int total = rows * N;
        for (int idx = rank * kRtThreads + static_cast<int>(threadIdx.x); idx < total; idx += ks * kRtThreads) {
            const int r = idx / N, c = idx - r * N;
            if (n0 + c >= p.Eg) continue;
            float acc = 0.f;
            for (int q = 0; q < ks; ++q) {
                const float* src = cluster.map_shared_rank(reinterpret_cast<float*>(smem), q);
                acc += src[r * C::kPartStride + c];
            }
            if (!*abort_flag) p.logits[static_cast<int64_t>(m0 + r) * p.Eg + n0 + c] = acc;
        }
        __syncthreads();
        cluster.sync();
    }

    ptx::pdl_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kRtMmaWarp) {
        __syncwarp();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Long batches: a persistent grid (one CTA per SM) takes the 128 x 224 tiles
// round-robin.  Two accumulators of 224 columns in TMEM (kind::f16 needs no
// scale columns, so 2 x 224 fit in 512): the MMA issuer fills one while the
// four epilogue warps drain the other to global memory, so a tile's epilogue
// overlaps the next tile's MMAs.
constexpr int kRpWarps = 6;  // 0..3 epilogue, 4 producer, 5 MMA
constexpr int kRpThreads = kRpWarps * 32;
constexpr int kRpN = 224;
constexpr int kRpAccStride = 256;  // TMEM columns between the two accumulators
// pipeline buffers, 13 mbarriers + TMEM slot + abort flag, 1 KiB alignment slack
constexpr int kRpSmemBytes = RtCfg<kRpN>::kOffBar + 16 * 8 + 1024;
static_assert(kRpSmemBytes <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kRpThreads, 1)
    router_gemm_persistent_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                                  const RouterParams p) {
    using C = RtCfg<kRpN>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* empty = full + kRtStages;
    uint64_t* accfull = empty + kRtStages;  // [2]
    uint64_t* accempty = accfull + 2;       // [2]
    uint64_t* done = accempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = ((p.T + 127) / 128) * p.n_tiles;
    const int KC = p.H / kRtKChunk;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRtStages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&accfull[a], 1);
            ptx::mbar_init(&accempty[a], 4);  // the four epilogue warps
        }
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == kRtProducerWarp && lane == 0) {
        ptx::tma_prefetch_desc(&tmX);
        ptx::tma_prefetch_desc(&tmW);
    }
    if (warp == kRtMmaWarp) {
        ptx::tmem_alloc(tmem_slot, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    ptx::pdl_wait();

    if (warp == kRtProducerWarp) {
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
                const int m0 = (tile / p.n_tiles) * 128, n0 = (tile % p.n_tiles) * kRpN;
                for (int kc = 0; kc < KC; ++kc) {
                    if (!rt_wait(&empty[stage], phase ^ 1, p.wait_ns, abort_flag)) {
                        if (!*abort_flag) rt_record_timeout(p, abort_flag, kRtSiteProducer);
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[stage], C::kStageTx);
                    ptx::tma_load_2d(smem + C::kOffA + stage * C::kATile, &tmX, &full[stage], kc * kRtKChunk, m0);
                    ptx::tma_load_2d(smem + C::kOffB + stage * C::kBTile, &tmW, &full[stage], kc * kRtKChunk, n0);
                    ++issued;
                    if (++stage == kRtStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            for (int i = issued > kRtStages ? issued - kRtStages : 0; i < issued; ++i)
                ptx::mbar_wait(&full[i % kRtStages], static_cast<uint32_t>(i / kRtStages) & 1, 10ull * 1000 * 1000);
        }
    } else if (warp == kRtMmaWarp) {
        if (lane == 0) {
            constexpr uint32_t kIdesc = ptx::idesc_f16_bf16(128, kRpN);
            uint32_t stage = 0, phase = 0;
            uint32_t aphase[2] = {0, 0};
            bool ok = true;
            int j = 0;  // this CTA's tile count
            for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++j) {
                const int a = j & 1;
                if (!rt_wait(&accempty[a], aphase[a] ^ 1, p.wait_ns, abort_flag)) {
                    if (!*abort_flag) rt_record_timeout(p, abort_flag, kRtSiteMma);
                    break;
                }
                aphase[a] ^= 1;
                ptx::tc_fence_after();
                const uint32_t acc = tmem + a * kRpAccStride;
                for (int kc = 0; kc < KC; ++kc) {
                    if (!rt_wait(&full[stage], phase, p.wait_ns, abort_flag)) {
                        if (!*abort_flag) rt_record_timeout(p, abort_flag, kRtSiteMma);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t xa = ptx::smem_u32(smem + C::kOffA + stage * C::kATile);
                    const uint32_t wa = ptx::smem_u32(smem + C::kOffB + stage * C::kBTile);
#pragma unroll
                    for (int kk = 0; kk < kRtKChunk / 16; ++kk)
                        ptx::mma_f16(acc, ptx::sdesc_sw128(xa + kk * 32), ptx::sdesc_sw128(wa + kk * 32), kIdesc,
                                     (kc | kk) != 0);
                    ptx::tc_commit(&empty[stage]);
                    if (++stage == kRtStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok) ptx::tc_commit(&accfull[a]);
            }
            ptx::tc_commit(done);
            ptx::mbar_wait(done, 0, 10ull * 1000 * 1000);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int row = warp * 32 + lane;
        uint32_t aphase[2] = {0, 0};
        int j = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++j) {
            const int a = j & 1;
            bool ok = rt_wait(&accfull[a], aphase[a], p.wait_ns, abort_flag);
            if (!ok && lane == 0 && !*abort_flag) rt_record_timeout(p, abort_flag, kRtSiteEpi);
            if (!__all_sync(0xffffffffu, ok)) break;
            aphase[a] ^= 1;
            ptx::tc_fence_after();
            const int m0 = (tile / p.n_tiles) * 128, n0 = (tile % p.n_tiles) * kRpN;
            const bool valid = m0 + row < p.T;
            float* out = p.logits + static_cast<int64_t>(m0 + row) * p.Eg;
            const uint32_t tq = tmem + a * kRpAccStride + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < kRpN / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld32(tq + 32 * c, r);
                ptx::tmem_wait_ld();
                if (c == kRpN / 32 - 1) {
                    // the accumulator is free once its last columns are in registers
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&accempty[a]);
                }
                if (valid) store_logits_32(out, n0 + 32 * c, p.Eg, r);
            }
        }
    }

    ptx::pdl_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kRtMmaWarp) {
        __syncwarp();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int N>
cudaError_t launch_router_impl(const CUtensorMap& tmX, const CUtensorMap& tmW, const RouterParams& p, int grid,
                               cudaStream_t stream, bool pdl) {
    using C = RtCfg<N>;
    auto kern = router_gemm_kernel<N>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kRtThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = p.ks;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, p);
}

}  // namespace

RouterTiling router_tiling(int T, int Eg, int num_sms) {
    RouterTiling t{};
    if (T <= 256) {
        t.N = 64;
        t.ks = 8;
    } else {
        t.N = kRpN;
        t.ks = 1;
    }
    t.n_tiles = (Eg + t.N - 1) / t.N;
    t.grid = ((T + 127) / 128) * t.n_tiles * t.ks;
    if (t.ks == 1 && t.grid > num_sms) t.grid = num_sms;  // persistent: tiles round-robin over one CTA per SM
    return t;
}

cudaError_t launch_router(const CUtensorMap& tmX, const CUtensorMap& tmW, const RouterParams& p, int grid,
                          cudaStream_t stream, bool pdl) {
    if (p.N == 64) return launch_router_impl<64>(tmX, tmW, p, grid, stream, pdl);
    cudaError_t err = cudaFuncSetAttribute(router_gemm_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kRpSmemBytes);
    if (err != cudaSuccess) return err;
    return launch_kernel(router_gemm_persistent_kernel, dim3(grid), dim3(kRpThreads), kRpSmemBytes, stream, pdl, tmX,
                         tmW, p);
}

}  // namespace moe
