// Grouped block-scaled GEMMs of the MoE layer, decode tiling (block_n 16/32).
//
// Orientation ("swap AB"): the expert weights are the M = 128 operand and a
// virtual expert's B token rows are N, so a handful of tokens per expert
// still runs a full-height tensor-core tile while the kernel streams weights
// ("[sglang] ... MXFP4 decode MoE ... shape templates", section 1: FC1 items
// of 128 weight rows x kBlockN tokens).
//   FC1: per (group of <= G virtual experts of expert e, 128 intermediate
//        features f0..f0+127): gate rows f0.. and up rows I+f0.. of W1[e]
//        against the group's x tiles, K = H.  Epilogue: h = silu(gate) * up
//        in fp32, per token and 32-feature block MXFP8 (E4M3, E8M0 scale)
//        into act / act_sf ("[SGLang] CUTLASS MoE", section 4 silu_and_mul,
//        fused).
//   FC2: per (group, 128 hidden rows): W2[e] rows against the group's act
//        tiles, K = I.  Epilogue: multiply by the routing weight of the row's
//        slot and store fp32 Y rows (section 5's multiply, fused).
//
// Pipeline (one CTA per SM, persistent over a static round-robin of items):
//   warp 0      TMA producer: W tiles (E2M1, packed 16x4-bit -> 16-byte
//               smem chunks by the tensor map type), activation tiles (E4M3),
//               and the 512-byte scale blocks by bulk copy; STAGES-deep ring.
//   warp 1      TMEM allocator and single-thread MMA issuer: tcgen05.cp of the
//               scale blocks into TMEM, tcgen05.mma kind::mxf8f6f4 block_scale
//               (E2M1 x E4M3, scale_vec 1X = one E8M0 per 32 K), commits to
//               free smem stages and to publish accumulators.
//   warps 2..5  epilogue: tcgen05.ld of the fp32 accumulators (double
//               buffered in TMEM), fused math, global stores.
// Every wait is bounded; on expiry the CTA records MOE_ERR_TIMEOUT in the
// workspace status word, stops issuing work, lets its MMAs drain, frees TMEM
// and exits.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kGemmThreads = 192;

template <int B, int G, int NA, int STAGES>
struct Cfg {
    static constexpr int kATile = 128 * 128;  // smem bytes of a 128 x 128 W tile (E2M1 in 16-byte chunks)
    static constexpr int kBTile = B * 128;    // smem bytes of a B x 128 E4M3 tile
    static constexpr int kOffB = NA * kATile;
    static constexpr int kOffSFA = kOffB + G * kBTile;
    static constexpr int kOffSFB = kOffSFA + NA * 512;
    static constexpr int kStageBytes = ((kOffSFB + G * 512) + 1023) & ~1023;
    static constexpr int kAccCols = NA * G * B;       // fp32 columns of one accumulator buffer
    static constexpr int kSfCols = ((4 * NA + 4 * G) + 15) & ~15;  // TMEM columns of one stage's scale blocks
    static constexpr int kSfBase = 2 * kAccCols;
    static constexpr int kTmemCols = 512;
    static constexpr int kBarBytes = (2 * STAGES + 5) * 8 + 16;
    static constexpr int kSmemBytes = STAGES * kStageBytes + kBarBytes + 1024;
    static_assert(kSfBase + STAGES * kSfCols <= kTmemCols, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(B == 16 || B == 32, "decode tile rows");
};

struct Shared {
    uint64_t* full;
    uint64_t* empty;
    uint64_t* accfull;
    uint64_t* accempty;
    uint64_t* done;
    uint32_t* tmem_slot;
    volatile int* abort_flag;
};

__device__ __forceinline__ void record_timeout(const GemmParams& p, volatile int* abort_flag, int site) {
    *abort_flag = 1;
    if (atomicCAS(p.status, 0, MOE_ERR_TIMEOUT) == 0) p.status[1] = site * 65536 + static_cast<int>(blockIdx.x);
}

// Bounded wait that also gives up as soon as another role of the CTA aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              volatile int* abort_flag) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

template <int B, int G, bool FC1, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_decode_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const GemmParams p) {
    constexpr int NA = FC1 ? 2 : 1;
    using C = Cfg<B, G, NA, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared sh;
    sh.full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
    sh.empty = sh.full + STAGES;
    sh.accfull = sh.empty + STAGES;
    sh.accempty = sh.accfull + 2;
    sh.done = sh.accempty + 2;
    sh.tmem_slot = reinterpret_cast<uint32_t*>(sh.done + 1);
    sh.abort_flag = reinterpret_cast<volatile int*>(sh.tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&sh.full[s], 1);
            ptx::mbar_init(&sh.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&sh.accfull[b], 1);
            ptx::mbar_init(&sh.accempty[b], 4);
        }
        ptx::mbar_init(sh.done, 1);
        *sh.abort_flag = 0;
        ptx::fence_mbarrier_init();
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(sh.tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *sh.tmem_slot;

    ptx::pdl_wait();
    const int ngroups = p.header[kHdrNumGroups];
    const int MT = FC1 ? p.I / 128 : p.H / 128;   // 128-row weight tiles per item row
    const int KC = FC1 ? p.H / 128 : p.I / 128;   // 128-wide K chunks
    const int nitems = ngroups * MT;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x) {
                const int g = it / MT, mt = it - g * MT;
                const int4 grp = p.groups[g];
                const int e = grp.x, v0 = grp.y, nt = grp.z;
                int fr[G];
#pragma unroll
                for (int j = 0; j < G; ++j) fr[j] = (j < nt) ? p.vinfo[v0 + j].y : 0;
                // tile-major packed weights: (expert, row block, K chunk) tiles
                const int64_t tile0 = (static_cast<int64_t>(e) * MT + mt) * KC;
                const uint32_t tx = p.a_tx_bytes + nt * (C::kBTile + 512) + NA * 512;
                for (int kc = 0; kc < KC; ++kc) {
                    if (!wait_or_abort(&sh.empty[stage], phase ^ 1, p.wait_ns, sh.abort_flag)) {
                        if (!*sh.abort_flag) record_timeout(p, sh.abort_flag, kSiteProducerEmpty);
                        ok = false;
                        break;
                    }
                    uint8_t* st = smem + stage * C::kStageBytes;
                    ptx::mbar_arrive_expect_tx(&sh.full[stage], tx);
                    ptx::tma_load_2d(st, &tmA, &sh.full[stage], 0, static_cast<int32_t>((tile0 + kc) * (NA * 128)));
#pragma unroll
                    for (int j = 0; j < G; ++j)
                        if (j < nt) ptx::tma_load_2d(st + C::kOffB + j * C::kBTile, &tmB, &sh.full[stage], kc * 128, fr[j]);
                    ptx::bulk_load(st + C::kOffSFA, p.a_sf + static_cast<size_t>(tile0 + kc) * (NA * 512), NA * 512,
                                   &sh.full[stage]);
#pragma unroll
                    for (int j = 0; j < G; ++j)
                        if (j < nt)
                            ptx::bulk_load(st + C::kOffSFB + j * 512,
                                           p.b_sf + static_cast<size_t>(v0 + j) * p.b_sf_tile_bytes + kc * 512,
                                           512, &sh.full[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // Drain: every issued stage must have landed before the CTA may
            // exit (bounded; a stage consumed by the MMA already has).
            for (int s = 0; s < STAGES; ++s) {
                // Stages filled in the current lap have parity `phase`; earlier
                // laps' fills of the later stages have parity phase ^ 1.
                const uint32_t par = (static_cast<uint32_t>(s) < stage) ? phase : (phase ^ 1);
                ptx::mbar_wait(&sh.full[s], par, 10ull * 1000 * 1000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t kIdesc = ptx::idesc_mx(ptx::kFmtE2M1, ptx::kFmtE4M3, 128, B);
            uint32_t stage = 0, phase = 0, abuf = 0, aphase = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < nitems; it += gridDim.x) {
                const int g = it / MT;
                const int nt = p.groups[g].z;
                if (!wait_or_abort(&sh.accempty[abuf], aphase ^ 1, p.wait_ns, sh.abort_flag)) {
                    if (!*sh.abort_flag) record_timeout(p, sh.abort_flag, kSiteMmaAccEmpty);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t acc = tmem + abuf * C::kAccCols;
                for (int kc = 0; kc < KC; ++kc) {
                    if (!wait_or_abort(&sh.full[stage], phase, p.wait_ns, sh.abort_flag)) {
                        if (!*sh.abort_flag) record_timeout(p, sh.abort_flag, kSiteMmaFull);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint8_t* st = smem + stage * C::kStageBytes;
                    const uint32_t sf = tmem + C::kSfBase + stage * C::kSfCols;
#pragma unroll
                    for (int a = 0; a < NA; ++a)
                        ptx::tc_cp_32x128b_warpx4(sf + 4 * a, ptx::sdesc_sf(ptx::smem_u32(st + C::kOffSFA + a * 512)));
#pragma unroll
                    for (int j = 0; j < G; ++j)
                        if (j < nt)
                            ptx::tc_cp_32x128b_warpx4(sf + 4 * NA + 4 * j,
                                                      ptx::sdesc_sf(ptx::smem_u32(st + C::kOffSFB + j * 512)));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t idesc = ptx::idesc_with_sf_id(kIdesc, kk, kk);
#pragma unroll
                        for (int j = 0; j < G; ++j) {
                            if (j >= nt) continue;
                            const uint64_t bdesc = ptx::sdesc_sw128(ptx::smem_u32(st + C::kOffB + j * C::kBTile) + kk * 32);
                            const uint32_t sfb = sf + 4 * NA + 4 * j;
#pragma unroll
                            for (int a = 0; a < NA; ++a) {
                                const uint64_t adesc = ptx::sdesc_sw128(ptx::smem_u32(st + a * C::kATile) + kk * 32);
                                ptx::mma_mxf8f6f4(acc + (j * NA + a) * B, adesc, bdesc, idesc, sf + 4 * a, sfb,
                                                  (kc | kk) != 0);
                            }
                        }
                    }
                    ptx::tc_commit(&sh.empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                ptx::tc_commit(&sh.accfull[abuf]);
                abuf ^= 1;
                if (abuf == 0) aphase ^= 1;
            }
            // all MMAs issued by this thread complete before TMEM is released
            ptx::tc_commit(sh.done);
            ptx::mbar_wait(sh.done, 0, 10ull * 1000 * 1000);
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        uint32_t abuf = 0, aphase = 0;
        for (int it = blockIdx.x; it < nitems; it += gridDim.x) {
            const int g = it / MT, mt = it - g * MT;
            const int4 grp = p.groups[g];
            const int v0 = grp.y, nt = grp.z;
            // FC2: lane i holds the routing weight of tile row i, loaded before
            // the accumulator wait so the dependent loads overlap the MMAs.
            float wrow[G];
            if constexpr (!FC1) {
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    wrow[j] = 0.f;
                    if (j < nt) {
                        const int4 vi = p.vinfo[v0 + j];
                        if (lane < vi.z) wrow[j] = p.topk_w[p.a_map[vi.y + lane]];
                    }
                }
            }
            if (!wait_or_abort(&sh.accfull[abuf], aphase, p.wait_ns, sh.abort_flag)) {
                if (lane == 0 && !*sh.abort_flag) record_timeout(p, sh.abort_flag, kSiteEpiAccFull);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t acc = tmem + abuf * C::kAccCols + (static_cast<uint32_t>(32 * q) << 16);
            const int f = mt * 128 + 32 * q + lane;  // feature (FC1) / hidden row (FC2) of this lane
            for (int j = 0; j < nt; ++j) {
                const int4 vi = p.vinfo[v0 + j];
                const int first = vi.y, rows = vi.z;
                if constexpr (FC1) {
                    uint32_t gr[B], ur[B];
                    if constexpr (B == 32) {
                        ptx::tmem_ld32(acc + (2 * j) * B, gr);
                        ptx::tmem_ld32(acc + (2 * j + 1) * B, ur);
                    } else {
                        ptx::tmem_ld16(acc + (2 * j) * B, gr);
                        ptx::tmem_ld16(acc + (2 * j + 1) * B, ur);
                    }
                    ptx::tmem_wait_ld();
                    uint8_t* sf_tile = p.act_sf + static_cast<size_t>(v0 + j) * p.out_sf_tile_bytes;
                    const int sf_off = ((mt * 128 + 32 * q) >> 7) * 512 + (((mt * 128 + 32 * q) >> 5) & 3);
#pragma unroll
                    for (int n = 0; n < B; ++n) {
                        if (n < rows) {
                            const float h = silu(__uint_as_float(gr[n])) * __uint_as_float(ur[n]);
                            const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h)));
                            const int ex = mx_shared_exponent(__uint_as_float(amax_bits), 8);
                            const uint8_t code = static_cast<uint8_t>(e4m3x2(h * exp2_int(-ex), 0.f) & 0xFF);
                            p.act[static_cast<size_t>(first + n) * p.I + f] = code;
                            if (lane == 0) sf_tile[sf_off + n * 16] = static_cast<uint8_t>(ex + 127);
                        }
                    }
                } else {
                    uint32_t yr[B];
                    if constexpr (B == 32)
                        ptx::tmem_ld32(acc + j * B, yr);
                    else
                        ptx::tmem_ld16(acc + j * B, yr);
                    ptx::tmem_wait_ld();
                    float wj = 0.f;
#pragma unroll
                    for (int jj = 0; jj < G; ++jj)
                        if (jj == j) wj = wrow[jj];
#pragma unroll
                    for (int n = 0; n < B; ++n) {
                        const float w = __shfl_sync(0xffffffffu, wj, n);
                        if (n < rows) p.y[static_cast<size_t>(first + n) * p.H + f] = __uint_as_float(yr[n]) * w;
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sh.accempty[abuf]);
            abuf ^= 1;
            if (abuf == 0) aphase ^= 1;
        }
    }

    ptx::pdl_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int B, int G, bool FC1, int STAGES>
cudaError_t launch_impl(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int grid,
                        cudaStream_t stream, bool pdl) {
    using C = Cfg<B, G, FC1 ? 2 : 1, STAGES>;
    auto kern = gemm_decode_kernel<B, G, FC1, STAGES>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, dim3(grid), dim3(kGemmThreads), C::kSmemBytes, stream, pdl, tmA, tmB, p);
}

}  // namespace

cudaError_t launch_fc1_decode(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int B, int grid,
                              cudaStream_t stream, bool pdl) {
    if (B == 32) return launch_impl<32, 2, true, 5>(tmA, tmB, p, grid, stream, pdl);
    return launch_impl<16, 4, true, 5>(tmA, tmB, p, grid, stream, pdl);
}

cudaError_t launch_fc2_decode(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int B, int grid,
                              cudaStream_t stream, bool pdl) {
    if (B == 32) return launch_impl<32, 2, false, 8>(tmA, tmB, p, grid, stream, pdl);
    return launch_impl<16, 4, false, 8>(tmA, tmB, p, grid, stream, pdl);
}

}  // namespace moe
