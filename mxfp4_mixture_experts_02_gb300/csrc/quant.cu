// MX quantisers (OCP MX v1.0 conversion: shared exponent floor(log2 amax) -
// emax, elements rounded to nearest even and saturated by the cvt.satfinite
// instructions):
//   quant_x_kernel       : decode tilings (16 / 32-row tiles): x bf16 ->
//                          MXFP8 (E4M3, emax 8) in token order, row-major
//                          E8M0 scales, and each expert row's routing weight
//                          (the "[SGLang] CUTLASS MoE" section 2 shuffle_rows
//                          is done by the FC1 token producer, which gathers
//                          each tile's rows);
//   gather_token_kernel  : 128-row tiles: x quantised once per token and
//                          written to each of its expert rows (shuffle_rows
//                          folded into the quantiser), with the tile scale
//                          layout the FC1 kernel copies into tensor memory;
//   quantize_mxfp4_kernel: fp32 weights -> MXFP4 (E2M1, emax 2), offline;
//   pack_codes_kernel,
//   pack_scales_kernel   : row-major MXFP4 -> tile-major codes (one contiguous
//                          run per TMA box) and 512-byte tensor-memory scale
//                          blocks, offline.
#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kGatherThreads = 256;

// x -> MXFP8 in natural token order plus the per-row routing weight.  Job j <
// T * H/32: token j / (H/32), 32-element block j % (H/32) (consecutive
// threads take consecutive blocks of a row: 64-byte reads, 32-byte code
// writes and 1-byte scale writes, all contiguous across the warp); the
// remaining R jobs copy topk_w[a_map[row]] to row_w[row].  The GEMM's token
// producer gathers the rows of each tile from here.
__global__ void __launch_bounds__(kGatherThreads) quant_x_kernel(GatherParams p) {
    ptx::pdl_wait();
    const int nb = p.H / 32;
    const int64_t nq = static_cast<int64_t>(p.T) * nb;
    const int64_t total = nq + p.header[kHdrRows];
    for (int64_t job = static_cast<int64_t>(blockIdx.x) * kGatherThreads + threadIdx.x; job < total;
         job += static_cast<int64_t>(gridDim.x) * kGatherThreads) {
        if (job >= nq) {
            const int row = static_cast<int>(job - nq);
            p.row_w[row] = p.topk_w[p.a_map[row]];
            continue;
        }
        quant_x_block(p.x, p.xq, p.xsf, static_cast<size_t>(job));
    }
    ptx::pdl_launch_dependents();
}

// Token-major pass (128-row tiles, long batches): one warp per token
// quantises the token's row once and writes it to every row the token's
// slots occupy (c_map), with the row's routing weight and its scale words.
// Lane l holds the 16-element half-blocks l, l + 32, ... of each 4096-column
// slab (lanes 2k, 2k+1 share MX block k: one shuffle gives the block amax),
// so each store instruction writes 512 contiguous bytes; the four K-block
// scales of 128-K chunk kc form one word, stored by lane kc.  The tile scales
// are lane-major: tile row i's word of chunk kc sits at word
// ((i % 32) * chunks + kc) * 4 + i / 32 of tile v's block, so one store
// instruction puts a row's words into 448 bytes (4 lines at H 3584) instead
// of one line per chunk; the FC1 token producer picks a chunk's 512-byte
// block out of it with a 4-D TMA box.  Each x row is read once, so the pass
// costs the x read plus the expert-ordered write.  A row's expert is the last one whose first row is
// <= it (binary search over the offsets, cached in shared memory); its tile
// is vbase[e] + (row - off) / B.
constexpr int kTokWarps = 8;
constexpr int kTokMaxExperts = 1024;

__device__ __forceinline__ int last_le(const int* a, int n, int x) {  // largest i < n with a[i] <= x (a[0] <= x)
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= x)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kTokWarps * 32) gather_token_kernel(GatherParams p) {
    __shared__ int s_off[kTokMaxExperts + 1];
    __shared__ int s_vb[kTokMaxExperts];
    __shared__ uint32_t s_exp[kTokWarps][32];  // a slab's 128 block scales (bytes) per warp
    ptx::pdl_wait();
    for (int e = threadIdx.x; e <= p.Et; e += kTokWarps * 32) {
        s_off[e] = p.offsets[e];
        if (e < p.Et) s_vb[e] = p.vbase[e];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* exp_bytes = reinterpret_cast<uint8_t*>(s_exp[warp]);
    const int nh = p.H / 16;  // half-blocks per row
    // the sort, which decided the GEMM2 path, ran before this launch: with the
    // dense path, each token's fp32 accumulator row is zeroed here, before FC2
    // reduces into it
    const bool zero_acc = p.header[kHdrGemm2Path] == kPathDense;
    for (int t = p.t0 + blockIdx.x * kTokWarps + warp; t < p.T; t += gridDim.x * kTokWarps) {
        if (zero_acc) {
            float4* a = reinterpret_cast<float4*>(p.acc + static_cast<int64_t>(t) * p.H);
            for (int c = lane; c < p.H / 4; c += 32) a[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int j0 = 0; j0 < p.kp; j0 += 32) {
            // slot j0 + lane: its row, tile and tile row
            const int j = j0 + lane;
            int row = -1, v = 0, i = 0;
            if (j < p.kp) {
                row = p.c_map[static_cast<size_t>(t) * p.kp + j];
                if (row >= 0) {
                    const int e = last_le(s_off, p.Et, row);
                    const int rel = row - s_off[e];
                    v = s_vb[e] + rel / p.B;
                    i = rel % p.B;
                    p.row_w[row] = p.topk_w[static_cast<size_t>(t) * p.kp + j];
                }
            }
            const int nj = min(32, p.kp - j0);
            for (int h0 = 0; h0 < nh; h0 += 256) {  // 4096-column slabs
                uint4 q[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int h = h0 + lane + 32 * m;
                    float f[16];
                    float amax = 0.f;
                    if (h < nh) {
                        const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * p.H + h * 16);
                        uint4 raw[2];
                        raw[0] = __ldg(src);
                        raw[1] = __ldg(src + 1);
                        const uint16_t* hv = reinterpret_cast<const uint16_t*>(raw);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            f[e] = bf16_bits_to_float(hv[e]);
                            amax = fmaxf(amax, fabsf(f[e]));
                        }
                    }
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                    if (h < nh) {
                        const int ex = mx_shared_exponent(amax, 8);
                        const float inv = exp2_int(-ex);
                        uint32_t packed[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t lo = e4m3x2(f[4 * e] * inv, f[4 * e + 1] * inv);
                            const uint32_t hi = e4m3x2(f[4 * e + 2] * inv, f[4 * e + 3] * inv);
                            packed[e] = lo | (hi << 16);
                        }
                        q[m] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        if ((lane & 1) == 0) exp_bytes[(h - h0) >> 1] = static_cast<uint8_t>(ex + 127);
                    }
                }
                __syncwarp();
                const int kc = h0 / 8 + lane;  // this lane's 128-K chunk
                const bool has_sf = 8 * kc < nh;
                const int chunks = nh / 8;
                const uint32_t sfw = has_sf ? s_exp[warp][lane] : 0u;
                __syncwarp();  // s_exp is rewritten by the next slab
                for (int jj = 0; jj < nj; ++jj) {
                    const int r = __shfl_sync(0xffffffffu, row, jj);
                    const int rv = __shfl_sync(0xffffffffu, v, jj);
                    const int ri = __shfl_sync(0xffffffffu, i, jj);
                    if (r < 0) continue;  // warp-uniform
                    uint4* dst = reinterpret_cast<uint4*>(p.xq + static_cast<size_t>(r) * p.H);
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const int h = h0 + lane + 32 * m;
                        if (h < nh) dst[h] = q[m];
                    }
                    if (has_sf) {
                        uint32_t* sf_tile =
                            reinterpret_cast<uint32_t*>(p.xsf + static_cast<size_t>(rv) * p.xsf_tile_bytes);
                        sf_tile[((ri & 31) * chunks + kc) * 4 + (ri >> 5)] = sfw;
                    }
                }
            }
        }
    }
    ptx::pdl_launch_dependents();
}

// NVFP4 x for 128-row tiles, token-major like gather_token_kernel: one warp
// per token quantises its row once (lane l takes the 16-element blocks l, l +
// 32, ... of each 4096-column slab: one NVFP4 block each, global scale
// x_gscale) and writes it to every row its slots occupy: packed E2M1 codes
// [rows, H / 2] (each store instruction writes 256 contiguous bytes) and the
// block scales of each virtual expert lane-major: 16-byte cells (64-K half,
// tile lane l, 128-K chunk kc) at ((half * 32 + l) * chunks + kc) * 16, tile
// row i's word at (i / 32) * 4 of cell (half, i % 32, kc), byte b = the
// half's 16-element block b.  A chunk's cells of both halves are the two
// 512-byte blocks the scale_vec::4X MMA reads, fetched by FC1 as one 4-D
// TMA box.
__global__ void __launch_bounds__(kTokWarps * 32) gather_token_nvfp4_kernel(GatherParams p) {
    __shared__ int s_off[kTokMaxExperts + 1];
    __shared__ int s_vb[kTokMaxExperts];
    __shared__ uint32_t s_sf[kTokWarps][64];  // a slab's 256 block scales (bytes) per warp
    ptx::pdl_wait();
    for (int e = threadIdx.x; e <= p.Et; e += kTokWarps * 32) {
        s_off[e] = p.offsets[e];
        if (e < p.Et) s_vb[e] = p.vbase[e];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* sf_bytes = reinterpret_cast<uint8_t*>(s_sf[warp]);
    const int nh = p.H / 16;  // NVFP4 blocks per row
    const bool zero_acc = p.header[kHdrGemm2Path] == kPathDense;
    for (int t = p.t0 + blockIdx.x * kTokWarps + warp; t < p.T; t += gridDim.x * kTokWarps) {
        if (zero_acc) {
            float4* a = reinterpret_cast<float4*>(p.acc + static_cast<int64_t>(t) * p.H);
            for (int c = lane; c < p.H / 4; c += 32) a[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int j0 = 0; j0 < p.kp; j0 += 32) {
            const int j = j0 + lane;
            int row = -1, v = 0, i = 0;
            if (j < p.kp) {
                row = p.c_map[static_cast<size_t>(t) * p.kp + j];
                if (row >= 0) {
                    const int e = last_le(s_off, p.Et, row);
                    const int rel = row - s_off[e];
                    v = s_vb[e] + rel / p.B;
                    i = rel % p.B;
                    p.row_w[row] = p.topk_w[static_cast<size_t>(t) * p.kp + j];
                }
            }
            const int nj = min(32, p.kp - j0);
            for (int h0 = 0; h0 < nh; h0 += 256) {  // 4096-column slabs
                uint2 q[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int h = h0 + lane + 32 * m;
                    if (h < nh) {
                        const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * p.H + h * 16);
                        uint4 raw[2];
                        raw[0] = __ldg(src);
                        raw[1] = __ldg(src + 1);
                        const uint16_t* hv = reinterpret_cast<const uint16_t*>(raw);
                        float f[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) f[e] = bf16_bits_to_float(hv[e]);
                        uint32_t w0, w1;
                        sf_bytes[h - h0] = static_cast<uint8_t>(nvfp4_block(f, p.x_gscale, w0, w1));
                        q[m] = make_uint2(w0, w1);
                    }
                }
                __syncwarp();
                const int kc = h0 / 8 + lane;  // this lane's 128-K chunk (8 blocks)
                const bool has_sf = 8 * kc < nh;
                const int chunks = nh / 8;
                const uint32_t sf_lo = has_sf ? s_sf[warp][2 * lane] : 0u;      // blocks 0-3 of the chunk
                const uint32_t sf_hi = has_sf ? s_sf[warp][2 * lane + 1] : 0u;  // blocks 4-7
                __syncwarp();  // s_sf is rewritten by the next slab
                for (int jj = 0; jj < nj; ++jj) {
                    const int r = __shfl_sync(0xffffffffu, row, jj);
                    const int rv = __shfl_sync(0xffffffffu, v, jj);
                    const int ri = __shfl_sync(0xffffffffu, i, jj);
                    if (r < 0) continue;  // warp-uniform
                    uint2* dst = reinterpret_cast<uint2*>(p.xq + static_cast<size_t>(r) * (p.H / 2));
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const int h = h0 + lane + 32 * m;
                        if (h < nh) dst[h] = q[m];
                    }
                    if (has_sf) {
                        // lane-major cells (half, tile lane, chunk): half 0 at
                        // ((i % 32) * chunks + kc) * 16, half 1 32 * chunks
                        // cells further
                        uint32_t* tile = reinterpret_cast<uint32_t*>(p.xsf + static_cast<size_t>(rv) * p.xsf_tile_bytes);
                        const int w = ((ri & 31) * chunks + kc) * 4 + (ri >> 5);
                        tile[w] = sf_lo;
                        tile[w + 32 * chunks * 4] = sf_hi;
                    }
                }
            }
        }
    }
    ptx::pdl_launch_dependents();
}

// One thread per 32-element block of a row.
__global__ void quantize_mxfp4_kernel(QuantParams p) {
    const int64_t nb = p.K / 32;
    const int64_t total = p.rows * nb;
    for (int64_t job = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; job < total;
         job += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = job / nb, b = job - r * nb;
        const float4* src = reinterpret_cast<const float4*>(p.w + r * p.K + b * 32);
        float f[32];
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float4 q = src[c];
            f[4 * c] = q.x;
            f[4 * c + 1] = q.y;
            f[4 * c + 2] = q.z;
            f[4 * c + 3] = q.w;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(f[e]));
        const int ex = mx_shared_exponent(amax, 2);
        const float inv = exp2_int(-ex);
        uint32_t words[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t acc = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                acc |= static_cast<uint32_t>(e2m1x2(f[8 * w + 2 * q] * inv, f[8 * w + 2 * q + 1] * inv)) << (8 * q);
            words[w] = acc;
        }
        *reinterpret_cast<uint4*>(p.codes + r * (p.K / 2) + b * 16) = make_uint4(words[0], words[1], words[2], words[3]);
        p.scales[r * nb + b] = static_cast<uint8_t>(ex + 127);
    }
}

// Source row of row rr of 256-row block b (see moe_pack_weights).
__device__ __forceinline__ int64_t packed_src_row(int64_t b, int rr, int64_t N, int pair) {
    if (!pair) return b * 256 + rr;
    return rr < 128 ? b * 128 + rr : N / 2 + b * 128 + (rr - 128);
}

// Codes: one thread per 16-byte piece of the output.
__global__ void pack_codes_kernel(PackParams p) {
    const int RB = 256;
    const int64_t NB = p.N / RB, KC = p.K / 128;
    const int64_t total = p.experts * p.N * (p.K / 2) / 16;
    for (int64_t o = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; o < total;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = o / (RB * 4);
        const int within = static_cast<int>(o - tile * RB * 4);
        const int rr = within >> 2, piece = within & 3;
        const int64_t e = tile / (NB * KC), rem = tile - e * NB * KC;
        const int64_t b = rem / KC, c = rem - b * KC;
        const int64_t row = e * p.N + packed_src_row(b, rr, p.N, p.pair);
        reinterpret_cast<uint4*>(p.packed_codes)[o] =
            *reinterpret_cast<const uint4*>(p.codes + row * (p.K / 2) + c * 64 + piece * 16);
    }
}

// Scales: one thread per output byte.
__global__ void pack_scales_kernel(PackParams p) {
    const int RB = 256;
    const int64_t NB = p.N / RB, KC = p.K / 128;
    const int64_t total = p.experts * p.N * (p.K / 32);
    for (int64_t o = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; o < total;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = o / (RB * 4);
        const int within = static_cast<int>(o - tile * RB * 4);
        const int grp = within >> 9, pos = within & 511;
        const int line = pos >> 4, quarter = (pos >> 2) & 3, kb = pos & 3;
        const int rr = grp * 128 + quarter * 32 + line;
        const int64_t e = tile / (NB * KC), rem = tile - e * NB * KC;
        const int64_t b = rem / KC, c = rem - b * KC;
        const int64_t row = e * p.N + packed_src_row(b, rr, p.N, p.pair);
        p.packed_scales[o] = p.scales[row * (p.K / 32) + c * 4 + kb];
    }
}

// NVFP4 weight quantiser, pass 1: each expert matrix's global scale
// fp32(2688 / amax) (2688 = 448 * 6: the largest E4M3 block scale times the
// largest E2M1 element; 1 for an all-zero matrix).  One CTA per expert.
constexpr int kGsThreads = 512;
__global__ void __launch_bounds__(kGsThreads) nvfp4_gscale_kernel(NvQuantParams p) {
    __shared__ float s_max[kGsThreads / 32];
    const int64_t n = p.rows_per_expert * p.K;
    const float4* w = reinterpret_cast<const float4*>(p.w + static_cast<int64_t>(blockIdx.x) * n);
    float amax = 0.f;
    for (int64_t i = threadIdx.x; i < n / 4; i += kGsThreads) {
        const float4 q = w[i];
        amax = fmaxf(fmaxf(amax, fmaxf(fabsf(q.x), fabsf(q.y))), fmaxf(fabsf(q.z), fabsf(q.w)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int i = 0; i < kGsThreads / 32; ++i) m = fmaxf(m, s_max[i]);
        p.gscale[blockIdx.x] = m > 0.f ? __fdiv_rn(2688.0f, m) : 1.0f;
    }
}

// NVFP4 weight quantiser, pass 2: one thread per block of 16 elements.
__global__ void quantize_nvfp4_kernel(NvQuantParams p) {
    const int64_t nb = p.K / 16;
    const int64_t rows = p.experts * p.rows_per_expert;
    for (int64_t job = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; job < rows * nb;
         job += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = job / nb, b = job - r * nb;
        const float4* src = reinterpret_cast<const float4*>(p.w + r * p.K + b * 16);
        float v[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const float4 q = src[c];
            v[4 * c] = q.x;
            v[4 * c + 1] = q.y;
            v[4 * c + 2] = q.z;
            v[4 * c + 3] = q.w;
        }
        uint32_t w0, w1;
        const uint32_t sf = nvfp4_block(v, p.gscale[r / p.rows_per_expert], w0, w1);
        *reinterpret_cast<uint2*>(p.codes + r * (p.K / 2) + b * 8) = make_uint2(w0, w1);
        p.scales[r * nb + b] = static_cast<uint8_t>(sf);
    }
}

// NVFP4 scales in the layout tcgen05.mma .scale_vec::4X reads from tensor
// memory, one thread per output byte.  Per (expert, 256-row block, 128-K
// chunk) tile 2 KB: for each 64-K half kk (one MMA) two 512-byte blocks (block
// rows 0-127, 128-255); row r's 4-byte cell at (r % 32) * 16 + (r / 32) * 4,
// byte b = the half's 16-element block b.
__global__ void pack_scales_nvfp4_kernel(PackParams p) {
    const int RB = 256;
    const int64_t NB = p.N / RB, KC = p.K / 128;
    const int64_t total = p.experts * p.N * (p.K / 16);
    for (int64_t o = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; o < total;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t tile = o / 2048;
        const int within = static_cast<int>(o - tile * 2048);
        const int kk = within >> 10, grp = (within >> 9) & 1, pos = within & 511;
        const int line = pos >> 4, quarter = (pos >> 2) & 3, b = pos & 3;
        const int rr = grp * 128 + quarter * 32 + line;
        const int64_t e = tile / (NB * KC), rem = tile - e * NB * KC;
        const int64_t blk = rem / KC, c = rem - blk * KC;
        const int64_t row = e * p.N + packed_src_row(blk, rr, p.N, p.pair);
        p.packed_scales[o] = p.scales[row * (p.K / 16) + c * 8 + kk * 4 + b];
    }
}

unsigned grid_for(int64_t n, int threads) {
    int64_t g = (n + threads - 1) / threads;
    if (g > 1 << 20) g = 1 << 20;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream, bool pdl) {
    if (p.token_order) {
        const int64_t jobs = static_cast<int64_t>(p.T) * (p.H / 32) + p.R_max;
        int64_t blocks = (jobs + kGatherThreads - 1) / kGatherThreads;
        if (blocks > p.max_blocks) blocks = p.max_blocks;
        if (blocks < 1) blocks = 1;
        return launch_kernel(quant_x_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kGatherThreads), 0, stream, pdl,
                             p);
    }
    int64_t blocks = (static_cast<int64_t>(p.T - p.t0) + kTokWarps - 1) / kTokWarps;
    if (blocks > p.max_blocks) blocks = p.max_blocks;
    if (blocks < 1) blocks = 1;
    return launch_kernel(gather_token_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kTokWarps * 32), 0, stream, pdl,
                         p);
}

cudaError_t launch_gather_nvfp4(const GatherParams& p, cudaStream_t stream, bool pdl) {
    int64_t blocks = (static_cast<int64_t>(p.T - p.t0) + kTokWarps - 1) / kTokWarps;
    if (blocks > p.max_blocks) blocks = p.max_blocks;
    if (blocks < 1) blocks = 1;
    return launch_kernel(gather_token_nvfp4_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kTokWarps * 32), 0,
                         stream, pdl, p);
}

cudaError_t launch_quantize_mxfp4(const QuantParams& p, cudaStream_t stream) {
    quantize_mxfp4_kernel<<<grid_for(p.rows * (p.K / 32), 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_quantize_nvfp4(const NvQuantParams& p, cudaStream_t stream) {
    nvfp4_gscale_kernel<<<static_cast<unsigned>(p.experts), kGsThreads, 0, stream>>>(p);
    quantize_nvfp4_kernel<<<grid_for(p.experts * p.rows_per_expert * (p.K / 16), 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_pack_weights_nvfp4(const PackParams& p, cudaStream_t stream) {
    pack_codes_kernel<<<grid_for(p.experts * p.N * (p.K / 2) / 16, 256), 256, 0, stream>>>(p);
    pack_scales_nvfp4_kernel<<<grid_for(p.experts * p.N * (p.K / 16), 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_pack_weights(const PackParams& p, cudaStream_t stream) {
    pack_codes_kernel<<<grid_for(p.experts * p.N * (p.K / 2) / 16, 256), 256, 0, stream>>>(p);
    pack_scales_kernel<<<grid_for(p.experts * p.N * (p.K / 32), 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace moe
