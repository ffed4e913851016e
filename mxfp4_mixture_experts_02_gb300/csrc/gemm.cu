// Grouped block-scaled GEMMs of the MoE layer (FC1 and FC2), one kernel
// template for the decode tilings (token tiles of 16 / 32 rows) and the
// prefill tiling (128-row token tiles).
//
// Work item = (virtual expert v: a tile of TM token rows of expert e,
// weight block nb of 256 rows).  One tcgen05.mma kind::mxf8f6f4 block_scale
// per 32-wide K step: A = the token tile (M = 128, E4M3, K-major), B = the
// 256 weight rows (N = 256, E2M1, K-major), fp32 accumulator of 128 lanes x
// 256 columns in TMEM, E8M0 scales (one per 32 K) copied into TMEM with
// tcgen05.cp.  The weights are the N operand because an MMA instruction costs
// the same for any N <= 256: 256 weight rows per instruction halves the
// instruction count of a weight-streaming (decode) GEMM against 128 rows.
//
//   FC1: B = W1[e] gate rows f0..f0+127 and up rows I+f0.. (packed adjacent),
//        K = H.  Epilogue: the activation h(gate, up) in fp32 and MXFP8 per
//        token and 32 features -> act / act_sf ("[SGLang] CUTLASS MoE",
//        section 4 silu_and_mul, fused into the GEMM; the clamped SwiGLU and
//        SiTU variants of "... MXFP4 decode MoE ... shape templates",
//        section 4).
//   FC2: B = W2[e] rows nb*256.., K = I.  Epilogue: times the routing weight
//        of the row's slot -> Y rows (the multiply of section 5's
//        apply_shuffle_mul_sum, fused).
//
// With TM < 128 only the tile's TM rows are loaded; the MMA still reads 128
// rows, the rest alias the next stages' token tiles (their accumulator lanes
// are never read).
//
// Warp roles (11 warps): 0..7 epilogue (warp w reads TMEM lane quadrant w % 4
// and column half w / 4; with TM <= 32 only quadrant 0 holds tokens, so only
// warps 0 and 4 work), 8 weight producer (one thread, TMA) and 10 token
// producer filling the same STAGES-deep ring (a single issuing thread could
// not keep up with the MMAs): one thread issuing TMA boxes of expert-ordered
// rows, except in the decode FC1, where all 32 lanes gather the tile's rows
// from the token-order MXFP8 x with cp.async; 9 TMEM allocator and
// single-thread MMA issuer.  The epilogue releases the accumulator as soon as
// its TMEM loads complete, so the next item's MMAs overlap the activation /
// quantise / store math.  Every wait is bounded; on expiry the CTA records
// MOE_ERR_TIMEOUT in the workspace status word, stops, lets its MMAs drain,
// frees TMEM and exits.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

// Ring depths (stages of 256 weight rows x 128 K).  The decode GEMMs stream
// weights at close to the MMA issue rate, so their rings are as deep as the
// shared memory of a 32-row token tile allows; the prefill rings share shared
// memory with 128-row token tiles (and FC2's output staging).
#ifndef MOE_STAGES_DEC_FC1
#define MOE_STAGES_DEC_FC1 6
#endif
#ifndef MOE_STAGES_DEC_FC2
#define MOE_STAGES_DEC_FC2 6
#endif
#ifndef MOE_STAGES_PRE_FC1
#define MOE_STAGES_PRE_FC1 4
#endif
#ifndef MOE_STAGES_PRE_FC2
#define MOE_STAGES_PRE_FC2 3
#endif
constexpr int kStagesDecFc1 = MOE_STAGES_DEC_FC1;
constexpr int kStagesDecFc2 = MOE_STAGES_DEC_FC2;

constexpr int kStagesPreFc1 = MOE_STAGES_PRE_FC1;
constexpr int kStagesPreFc2 = MOE_STAGES_PRE_FC2;
// NVFP4 (128-row tiles): a 128-K stage is 8 KB of tokens, 16 KB of packed
// weights and 3 KB of scales, so the rings are deeper in the same memory.
constexpr int kStagesNvFc1 = 7;
constexpr int kStagesNvFc2 = 5;

constexpr int kWarps = 11;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = 8;  // weight tiles and weight scales
constexpr int kMmaWarp = 9;
constexpr int kTokenWarp = 10;    // token tiles and token scales

// Shared memory: token tiles first (TM rows x 128 B per stage; the MMA
// reads 128 rows, so a short tile's reads run on into the following slots
// and the weight tiles -- bytes whose accumulator lanes are never read),
// then the weight tiles (32 KiB per stage: 256 rows x 128 E2M1 codes in
// 16-byte chunks), then each stage's scales (1 KiB weight + 512 B token).
// NV: the NVFP4 variant -- packed E2M1 rows of 64 bytes (128 K) in both
// operands, 64-byte swizzle, scales per 16 K (3 KB per stage: 2 KB weights,
// 1 KB tokens; 24 TMEM columns: 4 + 4 token, 8 + 8 weight, one set per 64-K
// MMA).
template <int TM, int STAGES, bool STAGE_Y, bool NV = false>
struct Cfg {
    static constexpr int kRow = NV ? 64 : 128;         // shared-memory bytes of one 128-K row
    static constexpr int kXTile = TM * kRow;           // bytes of the loaded token rows
    static constexpr int kWTile = 256 * kRow;          // 256 weight rows x 128 K
    static constexpr int kSfStage = NV ? 3072 : 1536;
    static constexpr int kSfW = NV ? 2048 : 1024;      // weight scales per stage
    static constexpr int kSfX = NV ? 1024 : 512;       // token scales per stage
    static constexpr int kOffX = 0;
    static constexpr int kOffW = STAGES * kXTile;      // 1024-byte aligned: TM * 128 is
    static constexpr int kOffSF = kOffW + STAGES * kWTile;
    // bf16 FC2 rows of 128-row tiles are staged per epilogue warp (two
    // 1024-byte-aligned 32-row x 64-column boxes) and leave by TMA stores
    static constexpr int kOffEpi = (kOffSF + STAGES * kSfStage + 1023) & ~1023;
    static constexpr int kEpiBytes = STAGE_Y ? 8 * 32 * 256 : 0;
    static constexpr int kOffBar = kOffEpi + kEpiBytes;
    static constexpr int kSmemBytes = kOffBar + (2 * STAGES + 6) * 8 + 16 + 1024;
    static constexpr int kAccCols = 256;
    static constexpr int kSfCols = NV ? 24 : 16;        // per stage: token-scale + weight-scale columns
    static constexpr int kTmemCols = 512;
    static constexpr int kEpiWarps = TM <= 32 ? 2 : 8;  // warps holding token lanes
    static_assert(!NV || TM == 128, "the NVFP4 variant has 128-row tiles");
    static_assert(kOffX + STAGES * kXTile + 128 * kRow <= kOffSF, "a 128-row read of the last token slot stays inside");
    static_assert(kAccCols + STAGES * kSfCols <= kTmemCols, "TMEM budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(TM == 16 || TM == 32 || TM == 128, "token tile rows");
    static __device__ __forceinline__ int x_off(int s) { return kOffX + s * kXTile; }
    static __device__ __forceinline__ int w_off(int s) { return kOffW + s * kWTile; }
    static __device__ __forceinline__ int sfw_off(int s) { return kOffSF + s * kSfStage; }
    static __device__ __forceinline__ int sfx_off(int s) { return kOffSF + s * kSfStage + kSfW; }
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

// silu(g) = g / (1 + e^-g) with the fast exponential and divide (relative
// error about 1e-6, far below the E4M3 step the result is quantised to).
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Descriptor of work item `it` (NB weight blocks per virtual expert), or
// `none` past the item count.  The load does not wait for the count: the
// index is clamped into the array and the value dropped when the item does
// not exist, so a CTA's first descriptor loads overlap its header load.
__device__ __forceinline__ int4 item_desc(const GemmParams& p, int it, int NB, int iend, int4 none) {
    const int4 d = p.vinfo[min(it / NB, p.max_v - 1)];
    return it < iend ? d : none;
}

// FC1 activations h(gate, up) ("... MXFP4 decode MoE ... shape templates",
// section 4).  c0 / c1 are the constants, i0 / i1 their reciprocals.
//   SwiGLU         silu(g) * u
//   clamped SwiGLU silu(min(g, L)) * clamp(u, -L, L), L = c0
//   SiTU           beta tanh(g / beta) sigmoid(g) * lb tanh(u / lb), beta = c0,
//                  lb = c1, evaluated as (beta / 2) tanh(g / beta)
//                  (1 + tanh(g / 2)) * lb tanh(u / lb) with the hardware
//                  tanh approximation, as the section's kernel does (beta 4,
//                  lb 25 give its fixed form 2 tanh(g/4) (1 + tanh(g/2)) *
//                  25 tanh(u/25))
template <int ACT>
__device__ __forceinline__ float activation(float g, float u, float c0, float c1, float i0, float i1) {
    if constexpr (ACT == MOE_ACT_SWIGLU_CLAMP) {
        return silu(fminf(g, c0)) * fminf(fmaxf(u, -c0), c0);
    } else if constexpr (ACT == MOE_ACT_SITU) {
        return (0.5f * c0) * ptx::tanh_approx(g * i0) * (1.0f + ptx::tanh_approx(0.5f * g)) *
               (c1 * ptx::tanh_approx(u * i1));
    } else {
        return silu(g) * u;
    }
}

template <int ACT>
__device__ __forceinline__ void activation_block(const uint32_t (&g)[32], const uint32_t (&u)[32], float (&h)[32],
                                                 float c0, float c1, float i0, float i1) {
#pragma unroll
    for (int c = 0; c < 32; ++c) h[c] = activation<ACT>(__uint_as_float(g[c]), __uint_as_float(u[c]), c0, c1, i0, i1);
}

// NVFP4: the product's scale 1 / (gs_in * gs_w[e]) of the item's expert (the
// E2M1 x E2M1 MMA sums e2m1 * e4m3 products; each operand's value is that
// over its global scale).  0 past the last item.
__device__ __forceinline__ float nv_alpha(const GemmParams& p, const int4& vi) {
    return vi.z > 0 ? __frcp_rn(p.nv_in_gs * p.nv_w_gs[vi.x]) : 0.f;
}

// 32 fp32 -> MXFP8 (E4M3 codes in 8 words, E8M0 code returned).
__device__ __forceinline__ uint32_t mxfp8_block(const float* v, uint32_t (&w)[8]) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int ex = mx_shared_exponent(amax, 8);
    const float inv = exp2_int(-ex);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv);
        const uint32_t hi = e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv);
        w[i] = lo | (hi << 16);
    }
    return static_cast<uint32_t>(ex + 127);
}

// ACT: the FC1 activation (MOE_ACT_*), a template parameter so that each
// epilogue carries only its own arithmetic.  Tensor maps: tmW the packed
// weights, tmX the token rows, tmAux the bf16 FC2 rows (TMA stores, 128-row
// tiling) or, for the MXFP8 FC1 at 128-row tiles, the x scale blocks (one 4-D
// box per stage, see the token producer).
template <int TM, bool FC1, bool YBF16, int STAGES, int ACT, bool NV>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmAux, const GemmParams p) {
    constexpr bool kStageY = !FC1 && YBF16 && TM == 128;
    // decode FC1: the token producer gathers x rows from the token-order MXFP8
    // rows with cp.async (128-row tiles read expert-ordered rows by TMA)
    constexpr bool kGatherX = FC1 && TM <= 32;
    // FC1 at 128-row tiles: the x scales come by TMA from the lane-major tile
    // layout the token-major gathers write
    constexpr bool kXScaleMap = FC1 && TM == 128;
    using C = Cfg<TM, STAGES, kStageY, NV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* empty = full + STAGES;
    uint64_t* accfull = empty + STAGES;
    uint64_t* accempty = accfull + 1;
    uint64_t* done = accempty + 1;
    uint64_t* stall = done + 1;  // test hook: nothing ever arrives on it
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stall + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // gathered x rows: the weight producer's arrive (with the weight
            // bytes) and one arrive per token-producer lane when its row copies
            // have landed
            ptx::mbar_init(&full[s], kGatherX ? 1 + 32 : 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(accfull, 1);
        ptx::mbar_init(accempty, C::kEpiWarps);
        ptx::mbar_init(done, 1);
        ptx::mbar_init(stall, 1);
        *abort_flag = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == kProducerWarp && lane == 0) ptx::tma_prefetch_desc(&tmW);
    if (warp == kTokenWarp && lane == 0) {
        ptx::tma_prefetch_desc(&tmX);
        if constexpr (kXScaleMap) ptx::tma_prefetch_desc(&tmAux);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // The work list (header, virtual experts) comes from the sort.  In the
    // decode FC1 the sort may be the launch just before this one (the fused
    // route + sort), so every thread waits for that grid's completion, which
    // makes its writes visible, before reading the list.  Everywhere else a
    // kernel in between already waited for the sort's grid to complete before
    // it triggered this launch, so the list is read at once, and only the
    // token operands -- written by the immediately preceding kernel -- need
    // griddepcontrol.wait, which the token producer issues while the weight
    // producer streams the first weight stages.
    if constexpr (kGatherX) ptx::pdl_wait();
    const int num_v = p.header[kHdrNumV];
    const int NB = FC1 ? p.I / 128 : p.H / 256;  // 256-row weight blocks per expert
    const int KC = FC1 ? p.H / 128 : p.I / 128;  // 128-wide K chunks
    const int nitems = num_v * NB;
    // This CTA's items: it0, it0 + istep, ... below iend (round-robin over the
    // grid: the token tiles of one expert run side by side and share its
    // weights in L2).
    const int it0 = blockIdx.x, istep = gridDim.x, iend = nitems;

    // Descriptors of the next three items stay in flight in each producer (an
    // FC2 item streams only I/128 stages, less than an L2 round trip under
    // load).
    const int4 kNone = make_int4(0, 0, 0, 0);
    const int g = istep;
    if (warp == kProducerWarp) {
        if (lane == 0) {
            // ------------------------------------------------- weight producer
            // Weight tiles and weight scales need nothing the immediately
            // preceding kernel writes: once the work list is read (above)
            // they stream without griddepcontrol.wait.  This thread sets each
            // stage's expected bytes (weights and tokens); the token
            // producer's copies may land before or after.
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            // global bytes: 256 rows x 64 B of weights (E2M1 either way) plus
            // the weight scales, and the token tile and its scales where they
            // come by TMA (the decode FC1's gathered rows arrive by cp.async)
            const uint32_t tx = kGatherX ? 256 * 64 + C::kSfW : 256 * 64 + C::kXTile + C::kSfStage;
            int4 vq0 = item_desc(p, it0, NB, iend, kNone);
            int4 vq1 = item_desc(p, it0 + g, NB, iend, kNone);
            int4 vq2 = item_desc(p, it0 + 2 * g, NB, iend, kNone);
            for (int it = it0; ok && it < iend; it += g) {
                const int v = it / NB, nb = it - v * NB;
                const int4 vi = vq0;
                vq0 = vq1;
                vq1 = vq2;
                vq2 = item_desc(p, it + 3 * g, NB, iend, kNone);
                const int64_t tile0 = (static_cast<int64_t>(vi.x) * NB + nb) * KC;
                for (int kc = 0; kc < KC; ++kc) {
                    if (!wait_or_abort(&empty[stage], phase ^ 1, p.wait_ns, abort_flag)) {
                        if (!*abort_flag) record_timeout(p, abort_flag, kSiteProducerEmpty);
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&full[stage], tx);
                    ptx::tma_load_2d(smem + C::w_off(stage), &tmW, &full[stage], 0,
                                     static_cast<int32_t>((tile0 + kc) * 256));
                    ptx::bulk_load(smem + C::sfw_off(stage), p.a_sf + static_cast<size_t>(tile0 + kc) * C::kSfW,
                                   C::kSfW, &full[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // every issued stage lands before the CTA may exit (bounded)
            for (int s = 0; s < STAGES; ++s) {
                const uint32_t par = (static_cast<uint32_t>(s) < stage) ? phase : (phase ^ 1);
                ptx::mbar_wait(&full[s], par, 10ull * 1000 * 1000);
            }
        }
    } else if (warp == kTokenWarp && kGatherX) {
        // ------------------------------------- decode FC1 token producer
        // The x rows of each tile are gathered from the token-order MXFP8 rows
        // (written by the preceding kernel) with cp.async.  Each copy
        // instruction moves 4 whole 128-byte row segments (lanes 8r..8r+7 take
        // the 16-byte chunks of one row: full cache lines per request); chunk c
        // of tile row i lands at chunk c ^ (i % 8), the 128-byte swizzle the
        // MMA descriptors expect.  Lane l also copies the 4 block scales of
        // the 128-K chunk of rows l, l + 32, ... to the tile scale layout, then
        // arrives on the stage's full barrier once its copies have landed.
        constexpr int kRowsPerLane = TM >= 32 ? TM / 32 : 1;
        ptx::pdl_wait();
        uint32_t stage = 0, phase = 0;
        bool ok = true;
        const int sf_row = p.H / 32;
        const int chunk = lane & 7, rsub = lane >> 3;
        int4 vq0 = item_desc(p, it0, NB, iend, kNone);
        int4 vq1 = item_desc(p, it0 + g, NB, iend, kNone);
        int4 vq2 = item_desc(p, it0 + 2 * g, NB, iend, kNone);
        for (int it = it0; ok && it < iend; it += g) {
            const int4 vi = vq0;
            vq0 = vq1;
            vq1 = vq2;
            vq2 = item_desc(p, it + 3 * g, NB, iend, kNone);
            int tok[kRowsPerLane];  // token of tile row lane + 32 q, or -1
#pragma unroll
            for (int q = 0; q < kRowsPerLane; ++q) {
                const int i = lane + 32 * q;
                tok[q] = (i < TM && i < vi.z) ? p.a_map[vi.y + i] / p.kp : -1;
            }
            for (int kc = 0; kc < KC; ++kc) {
                const bool waited = wait_or_abort(&empty[stage], phase ^ 1, p.wait_ns, abort_flag);
                if (!__all_sync(0xffffffffu, waited)) {
                    if (lane == 0 && !*abort_flag) record_timeout(p, abort_flag, kSiteProducerEmpty);
                    ok = false;
                    break;
                }
                uint8_t* xs = smem + C::x_off(stage);
                uint8_t* ss = smem + C::sfx_off(stage);
#pragma unroll
                for (int k = 0; k < TM / 4; ++k) {
                    const int i = 4 * k + rsub;  // tile row of this lane's chunk
                    const int t = __shfl_sync(0xffffffffu, tok[k >> 3], i & 31);
                    if (t >= 0)
                        ptx::cp_async_16(xs + i * 128 + ((chunk ^ (i & 7)) << 4),
                                         p.xq + static_cast<size_t>(t) * p.H + kc * 128 + chunk * 16);
                }
#pragma unroll
                for (int q = 0; q < kRowsPerLane; ++q) {
                    const int i = lane + 32 * q;
                    if (tok[q] >= 0)
                        ptx::cp_async_4(ss + (i & 31) * 16 + (i >> 5) * 4,
                                        p.xsf + static_cast<size_t>(tok[q]) * sf_row + kc * 4);
                }
                ptx::cp_async_mbar_arrive_noinc(&full[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        ptx::cp_async_wait_all();  // no copy lands after the CTA has moved on
    } else if (warp == kTokenWarp) {
        if (lane == 0) {
            // -------------------------------------------------- token producer
            // The token operands are written by the immediately preceding
            // kernel: wait for it once, then follow the same stage sequence.
            ptx::pdl_wait();
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            int4 vq0 = item_desc(p, it0, NB, iend, kNone);
            int4 vq1 = item_desc(p, it0 + g, NB, iend, kNone);
            int4 vq2 = item_desc(p, it0 + 2 * g, NB, iend, kNone);
            for (int it = it0; ok && it < iend; it += g) {
                const int v = it / NB;
                const int4 vi = vq0;
                vq0 = vq1;
                vq1 = vq2;
                vq2 = item_desc(p, it + 3 * g, NB, iend, kNone);
                const uint8_t* sfx = p.b_sf + static_cast<size_t>(v) * p.b_sf_tile_bytes;
                for (int kc = 0; kc < KC; ++kc) {
                    if (!wait_or_abort(&empty[stage], phase ^ 1, p.wait_ns, abort_flag)) {
                        if (!*abort_flag) record_timeout(p, abort_flag, kSiteProducerEmpty);
                        ok = false;
                        break;
                    }
                    ptx::tma_load_2d(smem + C::x_off(stage), &tmX, &full[stage], kc * C::kRow, vi.y);
                    if constexpr (kXScaleMap) {
                        // tile v's x scales are stored lane-major (16-byte cell
                        // of lane l and chunk kc at (l * chunks + kc) * 16; the
                        // NVFP4 halves as 32 further lanes), so the gather
                        // writes each row's words close together; the box
                        // {16 B, chunk kc, 32 (NVFP4: 64) lanes, tile v} lands
                        // as the block(s) the scale copies read
                        ptx::tma_load_4d(smem + C::sfx_off(stage), &tmAux, &full[stage], 0, kc, 0, v);
                    } else {
                        ptx::bulk_load(smem + C::sfx_off(stage), sfx + kc * C::kSfX, C::kSfX, &full[stage]);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            constexpr uint32_t kIdesc = ptx::idesc_mx(ptx::kFmtE4M3, ptx::kFmtE2M1, 128, 256);
            uint32_t stage = 0, phase = 0, aphase = 0;
            bool ok = true;
            // test hook: a wait that cannot complete, so that the timeout path
            // (status word, abort of the other roles, drain) runs on demand
            if (p.test_stall_ns && !wait_or_abort(stall, 0, p.test_stall_ns, abort_flag)) {
                if (!*abort_flag) record_timeout(p, abort_flag, kSiteTestStall);
                ok = false;
            }
            for (int it = it0; ok && it < iend; it += istep) {
                // FC2 at the decode tilings and in NVFP4 (items of I / 128 = 3
                // stages): an item's first stage copies its scales (scale
                // columns, not the accumulator) before the wait for the
                // epilogue to free the accumulator, overlapping that hand-off.
                // Elsewhere the wait comes first: FC1's items are H / 128
                // stages long and rarely wait, and the extra fence between
                // the copies and the MMAs measured slower there and in the
                // MXFP8 FC2 at 128-row tiles.
                constexpr bool kCopyFirst = !FC1 && (TM <= 32 || NV);
                auto acc_free = [&]() -> bool {
                    if (!wait_or_abort(accempty, aphase ^ 1, p.wait_ns, abort_flag)) {
                        if (!*abort_flag) record_timeout(p, abort_flag, kSiteMmaAccEmpty);
                        return false;
                    }
                    ptx::tc_fence_after();
                    return true;
                };
                if constexpr (!kCopyFirst) {
                    if (!acc_free()) break;
                }
                for (int kc = 0; kc < KC; ++kc) {
                    if (!wait_or_abort(&full[stage], phase, p.wait_ns, abort_flag)) {
                        if (!*abort_flag) record_timeout(p, abort_flag, kSiteMmaFull);
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    // gathered token rows arrive through cp.async (the
                    // generic proxy): make them visible to the tensor core
                    if constexpr (kGatherX) ptx::fence_proxy_async_smem();
                    const uint32_t sf = tmem + C::kAccCols + stage * C::kSfCols;
                    const uint32_t xa = ptx::smem_u32(smem + C::x_off(stage));
                    const uint32_t wa = ptx::smem_u32(smem + C::w_off(stage));
                    if constexpr (NV) {
                        // two 64-K MMAs; each reads a 32-bit cell of four 16-K
                        // block scales per row: tokens at sf + 4 kk, weights
                        // (rows 0-127, 128-255) at sf + 8 + 8 kk
                        constexpr uint32_t kIdescNv = ptx::idesc_nvf4(128, 256);
                        const uint32_t sx = ptx::smem_u32(smem + C::sfx_off(stage));
                        const uint32_t sw = ptx::smem_u32(smem + C::sfw_off(stage));
                        ptx::tc_cp_32x128b_warpx4(sf, ptx::sdesc_sf(sx));
                        ptx::tc_cp_32x128b_warpx4(sf + 4, ptx::sdesc_sf(sx + 512));
#pragma unroll
                        for (int q = 0; q < 4; ++q) ptx::tc_cp_32x128b_warpx4(sf + 8 + 4 * q, ptx::sdesc_sf(sw + 512 * q));
                        if (kCopyFirst && kc == 0 && !acc_free()) {
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk)
                            ptx::mma_mxf4nvf4(tmem, ptx::sdesc_sw64(xa + kk * 32), ptx::sdesc_sw64(wa + kk * 32),
                                              kIdescNv, sf + 4 * kk, sf + 8 + 8 * kk, (kc | kk) != 0);
                    } else {
                        ptx::tc_cp_32x128b_warpx4(sf, ptx::sdesc_sf(ptx::smem_u32(smem + C::sfx_off(stage))));
                        ptx::tc_cp_32x128b_warpx4(sf + 4, ptx::sdesc_sf(ptx::smem_u32(smem + C::sfw_off(stage))));
                        ptx::tc_cp_32x128b_warpx4(sf + 8,
                                                  ptx::sdesc_sf(ptx::smem_u32(smem + C::sfw_off(stage) + 512)));
                        if (kCopyFirst && kc == 0 && !acc_free()) {
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            ptx::mma_mxf8f6f4(tmem, ptx::sdesc_sw128(xa + kk * 32), ptx::sdesc_sw128(wa + kk * 32),
                                              ptx::idesc_with_sf_id(kIdesc, kk, kk), sf, sf + 4, (kc | kk) != 0);
                    }
                    ptx::tc_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                ptx::tc_commit(accfull);
                aphase ^= 1;
            }
            ptx::tc_commit(done);
            ptx::mbar_wait(done, 0, 10ull * 1000 * 1000);
        }
    } else if (warp < 8) {
        // -------------------------------------------------------- epilogue
        const int q = warp & 3, half = warp >> 2;
        const bool active = (TM > 32) || q == 0;
        uint32_t aphase = 0;
        const int i = q * 32 + lane;  // token row of this lane within a tile
        // reciprocals of the SiTU constants (unused by the other activations)
        const float act_i0 = ACT == MOE_ACT_SITU ? 1.0f / p.act_c0 : 0.f;
        const float act_i1 = ACT == MOE_ACT_SITU ? 1.0f / p.act_c1 : 0.f;
        // FC2: the GEMM2 path the gate chose (dense: reduce w * Y into the
        // token's accumulator row instead of writing the routed row).  The
        // sort decided it before FC1, which waited for the sort's grid (itself
        // or through the gather), and this grid launched after FC1 finished its
        // work, so the word is final.
        const bool dense = !FC1 && p.header[kHdrGemm2Path] == kPathDense;
        // Descriptors two items ahead and row weights (dense: and tokens) one
        // item ahead are loaded early, so no dependent load chain sits between
        // two items.
        const int4 kNoTile = kNone;
        int4 vi_cur = active ? item_desc(p, it0, NB, iend, kNoTile) : kNoTile;
        int4 vi_nxt = active ? item_desc(p, it0 + g, NB, iend, kNoTile) : kNoTile;
        float w_cur = (!FC1 && i < vi_cur.z) ? p.row_w[vi_cur.y + i] : 0.f;
        int t_cur = (dense && i < vi_cur.z) ? p.a_map[vi_cur.y + i] / p.kp : 0;
        float a_cur = NV ? nv_alpha(p, vi_cur) : 1.f;
        for (int it = it0; active && it < iend; it += g) {
            const int v = it / NB, nb = it - v * NB;
            const int4 vi = vi_cur;
            // FC2: the row's routing weight, times the NVFP4 product scale
            const float w_row = NV ? w_cur * a_cur : w_cur;
            const float alpha = a_cur;
            const int t_row = t_cur;
            const int4 vi_n2 = item_desc(p, it + 2 * g, NB, iend, kNoTile);
            w_cur = (!FC1 && i < vi_nxt.z) ? p.row_w[vi_nxt.y + i] : 0.f;
            t_cur = (dense && i < vi_nxt.z) ? p.a_map[vi_nxt.y + i] / p.kp : 0;
            if constexpr (NV) a_cur = nv_alpha(p, vi_nxt);
            vi_cur = vi_nxt;
            vi_nxt = vi_n2;
            const int first = vi.y, rows = vi.z;
            const bool valid = i < rows;
            if (!wait_or_abort(accfull, aphase, p.wait_ns, abort_flag)) {
                if (lane == 0 && !*abort_flag) record_timeout(p, abort_flag, kSiteEpiAccFull);
                break;
            }
            aphase ^= 1;
            ptx::tc_fence_after();
            const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
            uint32_t r[4][32];
            if constexpr (FC1) {
                // gate features half*64 .. +64 and the matching up features
                ptx::tmem_ld32(tq + half * 64, r[0]);
                ptx::tmem_ld32(tq + half * 64 + 32, r[1]);
                ptx::tmem_ld32(tq + 128 + half * 64, r[2]);
                ptx::tmem_ld32(tq + 128 + half * 64 + 32, r[3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tq + half * 128 + 32 * c, r[c]);
            }
            ptx::tmem_wait_ld();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(accempty);  // accumulator free for the next item
            if (dense) {
                // finalize fused into GEMM2: out_acc[token] += w * Y, four
                // columns per reduction, performed at the L2
                if (valid) {
                    float* dst = p.acc + static_cast<int64_t>(t_row) * p.H + nb * 256 + half * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            ptx::red_add_v4(dst + c * 32 + q4 * 4, __uint_as_float(r[c][4 * q4]) * w_row,
                                            __uint_as_float(r[c][4 * q4 + 1]) * w_row,
                                            __uint_as_float(r[c][4 * q4 + 2]) * w_row,
                                            __uint_as_float(r[c][4 * q4 + 3]) * w_row);
                }
            } else if constexpr (kStageY) {
                // lane = tile row q*32+lane.  Its 128 weighted bf16 values are
                // staged as two 32-row x 64-column boxes in the 128-byte TMA
                // swizzle (16-byte chunk j of row r at chunk j ^ (r % 8)); a
                // slab of 32 valid rows leaves with two tensor stores, a slab
                // cut by the tile's last row with row stores of its valid rows
                // (a tensor store would overwrite the next tile's rows).
                uint8_t* stg = smem + C::kOffEpi + warp * (32 * 256);
                const int slab_rows = rows - q * 32;
                if (slab_rows > 0) {
                    if (lane == 0) ptx::bulk_wait_read_all();  // previous item's stores left the buffer
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        uint32_t pk[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __nv_bfloat162 b2 =
                                __floats2bfloat162_rn(__uint_as_float(r[c >> 2][8 * (c & 3) + 2 * u]) * w_row,
                                                      __uint_as_float(r[c >> 2][8 * (c & 3) + 2 * u + 1]) * w_row);
                            pk[u] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        *reinterpret_cast<uint4*>(stg + (c >> 3) * 4096 + lane * 128 + (((c & 7) ^ (lane & 7)) << 4)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                    const int n0 = nb * 256 + half * 128;
                    if (slab_rows >= 32) {
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&tmAux, stg, n0, first + q * 32);
                            ptx::tma_store_2d(&tmAux, stg + 4096, n0 + 64, first + q * 32);
                            ptx::bulk_commit_group();
                        }
                    } else {
                        __syncwarp();
                        // lane owns columns n0 + 4*lane .. +3: chunk lane/2, half lane%2
                        const int cb = lane >> 1;
                        for (int rr = 0; rr < slab_rows; ++rr) {
                            const uint2 v2 = *reinterpret_cast<const uint2*>(
                                stg + (cb >> 3) * 4096 + rr * 128 + (((cb & 7) ^ (rr & 7)) << 4) + (lane & 1) * 8);
                            *reinterpret_cast<uint2*>(p.y_bf16 + static_cast<int64_t>(first + q * 32 + rr) * p.H +
                                                      n0 + lane * 4) = v2;
                        }
                    }
                    __syncwarp();
                }
            } else if (valid) {
                const int64_t row = first + i;
                if constexpr (FC1 && NV) {
                    // NVFP4 intermediate: features f0 .. f0 + 63 are the 64-K half
                    // `half` of 128-feature chunk nb: four blocks of 16, their four
                    // E4M3 scales one 32-bit cell of the chunk's tile block
                    const int f0 = nb * 128 + half * 64;
                    uint32_t cell = 0;
                    uint32_t wq[8];
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        float h[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            h[c] = activation<ACT>(__uint_as_float(r[b][c]) * alpha, __uint_as_float(r[2 + b][c]) * alpha,
                                                   p.act_c0, p.act_c1, act_i0, act_i1);
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb)
                            cell |= nvfp4_block(h + 16 * hb, p.nv_out_gs, wq[4 * b + 2 * hb], wq[4 * b + 2 * hb + 1])
                                    << (8 * (2 * b + hb));
                    }
                    uint4* dst = reinterpret_cast<uint4*>(p.act + row * (p.I / 2) + f0 / 2);
                    dst[0] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                    dst[1] = make_uint4(wq[4], wq[5], wq[6], wq[7]);
                    *reinterpret_cast<uint32_t*>(p.act_sf + static_cast<size_t>(v) * p.out_sf_tile_bytes +
                                                 nb * 1024 + half * 512 + (i & 31) * 16 + (i >> 5) * 4) = cell;
                } else if constexpr (FC1) {
                    const int f0 = nb * 128 + half * 64;  // first intermediate feature of this lane
                    uint8_t* sf_tile = p.act_sf + static_cast<size_t>(v) * p.out_sf_tile_bytes + nb * 512 +
                                       (i & 31) * 16 + (i >> 5) * 4 + half * 2;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        float h[32];
                        activation_block<ACT>(r[b], r[2 + b], h, p.act_c0, p.act_c1, act_i0, act_i1);
                        uint32_t wq[8];
                        const uint32_t sc = mxfp8_block(h, wq);
                        uint4* dst = reinterpret_cast<uint4*>(p.act + row * p.I + f0 + 32 * b);
                        dst[0] = make_uint4(wq[0], wq[1], wq[2], wq[3]);
                        dst[1] = make_uint4(wq[4], wq[5], wq[6], wq[7]);
                        sf_tile[b] = static_cast<uint8_t>(sc);
                    }
                } else {
                    const int n0 = nb * 256 + half * 128;  // first hidden column of this lane
                    if constexpr (YBF16) {
                        uint4* dst = reinterpret_cast<uint4*>(p.y_bf16 + row * p.H + n0);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int g = 0; g < 4; ++g) {
                                uint32_t pk[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const __nv_bfloat162 b2 =
                                        __floats2bfloat162_rn(__uint_as_float(r[c][8 * g + 2 * u]) * w_row,
                                                              __uint_as_float(r[c][8 * g + 2 * u + 1]) * w_row);
                                    pk[u] = *reinterpret_cast<const uint32_t*>(&b2);
                                }
                                dst[c * 4 + g] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            }
                    } else {
                        float4* dst = reinterpret_cast<float4*>(p.y + row * p.H + n0);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int g = 0; g < 8; ++g)
                                dst[c * 8 + g] = make_float4(__uint_as_float(r[c][4 * g]) * w_row,
                                                             __uint_as_float(r[c][4 * g + 1]) * w_row,
                                                             __uint_as_float(r[c][4 * g + 2]) * w_row,
                                                             __uint_as_float(r[c][4 * g + 3]) * w_row);
                    }
                }
            }
        }
        if constexpr (kStageY) {
            if (lane == 0) ptx::bulk_wait_all();  // tensor stores complete before the CTA exits
            __syncwarp();
        }
        if constexpr (kGatherX) {
            // Decode FC1: the six epilogue warps that hold no token lane zero
            // the dense GEMM2 accumulator when the gate chose that path (every
            // thread of this grid waited for the sort's grid, which decided
            // it, above), so FC2's reductions start from zero.
            if (!active && p.header[kHdrGemm2Path] == kPathDense) {
                const int wi = (q - 1) + 3 * half;  // 0..5
                const int64_t n4 = static_cast<int64_t>(p.T) * p.H / 4;
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int64_t k = (static_cast<int64_t>(blockIdx.x) * 6 + wi) * 32 + lane; k < n4;
                     k += static_cast<int64_t>(gridDim.x) * 6 * 32)
                    reinterpret_cast<float4*>(p.acc)[k] = z;
            }
        }
    }

    ptx::pdl_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int TM, bool FC1, bool YBF16, int STAGES, int ACT = MOE_ACT_SWIGLU, bool NV = false>
cudaError_t launch_impl(const CUtensorMap& tmW, const CUtensorMap& tmX, const CUtensorMap& tmAux, const GemmParams& p,
                        int grid, cudaStream_t stream, bool pdl) {
    using C = Cfg<TM, STAGES, !FC1 && YBF16 && TM == 128, NV>;
    auto kern = moe_gemm_kernel<TM, FC1, YBF16, STAGES, ACT, NV>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, pdl, tmW, tmX, tmAux, p);
}

template <int ACT>
cudaError_t launch_fc1(const CUtensorMap& tmW, const CUtensorMap& tmX, const CUtensorMap& tmAux, const GemmParams& p,
                       int TM, int grid, cudaStream_t stream, bool pdl) {
    if (p.nv) return launch_impl<128, true, true, kStagesNvFc1, ACT, true>(tmW, tmX, tmAux, p, grid, stream, pdl);
    if (TM == 16) return launch_impl<16, true, false, kStagesDecFc1, ACT>(tmW, tmX, tmAux, p, grid, stream, pdl);
    if (TM == 32) return launch_impl<32, true, false, kStagesDecFc1, ACT>(tmW, tmX, tmAux, p, grid, stream, pdl);
    return launch_impl<128, true, true, kStagesPreFc1, ACT>(tmW, tmX, tmAux, p, grid, stream, pdl);
}

}  // namespace

cudaError_t launch_gemm(bool fc1, const CUtensorMap& tmW, const CUtensorMap& tmX, const CUtensorMap& tmAux,
                        const GemmParams& p, int TM, int grid, cudaStream_t stream, bool pdl) {
    if (fc1) {
        if (p.act_kind == MOE_ACT_SWIGLU_CLAMP) return launch_fc1<MOE_ACT_SWIGLU_CLAMP>(tmW, tmX, tmAux, p, TM, grid, stream, pdl);
        if (p.act_kind == MOE_ACT_SITU) return launch_fc1<MOE_ACT_SITU>(tmW, tmX, tmAux, p, TM, grid, stream, pdl);
        return launch_fc1<MOE_ACT_SWIGLU>(tmW, tmX, tmAux, p, TM, grid, stream, pdl);
    }
    if (p.nv) return launch_impl<128, false, true, kStagesNvFc2, MOE_ACT_SWIGLU, true>(tmW, tmX, tmAux, p, grid, stream, pdl);
    if (TM == 16) return launch_impl<16, false, false, kStagesDecFc2>(tmW, tmX, tmAux, p, grid, stream, pdl);
    if (TM == 32) return launch_impl<32, false, false, kStagesDecFc2>(tmW, tmX, tmAux, p, grid, stream, pdl);
    return launch_impl<128, false, true, kStagesPreFc2>(tmW, tmX, tmAux, p, grid, stream, pdl);
}

}  // namespace moe
