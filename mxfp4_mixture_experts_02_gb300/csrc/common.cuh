// Shared definitions of the GPU library: derived dimensions, the workspace
// carve, status codes and the MX (OCP MX v1.0) element quantiser used by the
// activation paths.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/moe_api.h"

namespace moe {

constexpr int kHeaderWords = 64;
enum HeaderWord { kHdrRows = 0, kHdrNumV = 1, kHdrNumGroups = 2, kHdrStatus = 3, kHdrDetail = 4, kHdrGemm2Path = 5 };

// GEMM2 strategies the gate chooses between ("[FlashInfer] Device-side gating
// for the MoE GEMM2 path"): split = FC2 writes each routed row, the combine
// sums a token's rows; dense = FC2's epilogue reduces w * Y straight into an
// fp32 [T, H] accumulator (the finalize fused), the combine converts it.
enum Gemm2Path { kPathSplit = 0, kPathDense = 1 };

// Where a bounded wait expired (status detail = site * 65536 + block index).
enum WaitSite { kSiteProducerEmpty = 1, kSiteMmaFull = 2, kSiteMmaAccEmpty = 3, kSiteEpiAccFull = 4, kSiteTestStall = 5 };

constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 200 ms per wait

enum Mode { kModeDecode = 0, kModePrefill = 1 };

// Dimensions derived from a moe_shape.
struct Dims {
    int T, max_T, Eg, E, off, k, S, kp, Et, H, I, B;
    int G;           // virtual experts per sort work group (1: a GEMM item is one tile)
    int R_max;       // routed rows bound: max_T * k'
    int V_max;       // virtual-expert bound: Et + R_max / B
    int rows_alloc;  // activation rows incl. the last tile's TMA tail box
    int mode;
    float shared_scale;
};

// Byte offsets of the workspace regions (256-byte aligned).
struct Layout {
    size_t header, counts, offsets, vinfo, groups, a_map, c_map, sort_hist, row_w;
    size_t xq, xsf, act, asf, y, vbase, acc;
    size_t st_logits, st_shared, st_x, st_ids, st_w, st_out;
    size_t total;
    int xsf_tile_bytes, asf_tile_bytes, y_bf16, x_token_order;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline Dims make_dims(const moe_shape& s) {
    Dims d{};
    d.T = s.T;
    d.max_T = s.max_T;
    d.Eg = s.E_global;
    d.E = s.E_local;
    d.off = s.expert_offset;
    d.k = s.top_k;
    d.S = s.num_shared;
    d.kp = s.top_k + s.num_shared;
    d.Et = s.E_local + s.num_shared;
    d.H = s.hidden;
    d.I = s.inter;
    d.B = s.block_n;
    d.mode = (s.block_n == 128) ? kModePrefill : kModeDecode;
    d.G = 1;
    d.R_max = s.max_T * d.kp;
    d.V_max = d.Et + d.R_max / d.B;
    d.rows_alloc = d.R_max + d.B;
    d.shared_scale = s.shared_scale;
    return d;
}

inline Layout make_layout(const Dims& d) {
    Layout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align256(o + bytes);
        return at;
    };
    L.header = take(kHeaderWords * 4);
    L.counts = take(size_t(d.Et) * 4);
    L.offsets = take(size_t(d.Et + 1) * 4);
    L.vinfo = take(size_t(d.V_max) * 16);
    L.groups = take(size_t(d.V_max) * 16);
    L.a_map = take(size_t(d.R_max) * 4);
    L.c_map = take(size_t(d.R_max) * 4);
    L.sort_hist = take(size_t((d.R_max + 4095) / 4096) * d.Et * 4);
    L.row_w = take(size_t(d.R_max) * 4);
    // Tile scale layout (the FC1 output's scales; the FC1 token producer
    // builds the same layout in shared memory for x): per virtual expert and
    // 128-K chunk one 512-byte block, tile row r / K-block b at (r % 32) * 16 +
    // (r / 32) * 4 + b: one tcgen05.cp .32x128b.warpx4 puts it in 4 TMEM
    // columns, row r at lane r % 32, column r / 32, byte b.
    L.xsf_tile_bytes = (d.H / 128) * 512;
    L.asf_tile_bytes = (d.I / 128) * 512;
    L.y_bf16 = (d.mode == kModeDecode) ? 0 : 1;
    // x in MXFP8.  Decode tilings: token order, codes [max_T, H] and scales
    // [max_T, H / 32] (the FC1 token producer gathers each tile's rows).
    // 128-row tiles: expert-row order [rows_alloc, H] (TMA boxes), scales per
    // tile in the 16-byte cells of the tile scale layout ordered lane-major,
    // cell (lane l, chunk kc) at (l * H / 128 + kc) * 16, so the token-major
    // gather writes a row's words close together and a 4-D TMA box fetches a
    // chunk's 512-byte block.
    L.x_token_order = (d.mode == kModeDecode) ? 1 : 0;
    // (The NVFP4 variant of the 128-row tiling stores half the code bytes and
    // twice the scale bytes -- one E4M3 per 16 -- in the same regions.)
    L.xq = take(size_t(L.x_token_order ? d.max_T : d.rows_alloc) * d.H);
    L.xsf = take(L.x_token_order ? size_t(d.max_T) * (d.H / 32) : size_t(d.V_max) * L.xsf_tile_bytes * 2);
    L.act = take(size_t(d.rows_alloc) * d.I);
    L.asf = take(size_t(d.V_max) * L.asf_tile_bytes * (d.mode == kModePrefill ? 2 : 1));
    // bf16 rows carry the TMA tail too: the store map's row extent is
    // rows_alloc (>= 128), so a 32-row box never exceeds it
    L.y = take(size_t(L.y_bf16 ? d.rows_alloc : d.R_max) * d.H * (L.y_bf16 ? 2 : 4));
    L.vbase = take(size_t(d.Et) * 4);
    // fp32 [max_T, H]: the dense GEMM2 path's accumulator (zeroed in the call
    // that uses it, before FC2)
    L.acc = take(size_t(d.max_T) * d.H * 4);
    L.st_logits = take(size_t(d.max_T) * d.Eg * 4);
    L.st_shared = take(size_t(d.max_T) * (d.S > 0 ? d.S : 1) * 2);
    L.st_x = take(size_t(d.max_T) * d.H * 2);
    L.st_ids = take(size_t(d.R_max) * 4);
    L.st_w = take(size_t(d.R_max) * 4);
    L.st_out = take(size_t(d.max_T) * d.H * 2);
    L.total = o;
    return L;
}

// ---------------------------------------------------------------- device MX
// floor(log2 |amax|) - emax for a finite non-negative fp32, clamped to
// [-127, 127]; amax == 0 gives -127 (E8M0 code 0).
__device__ __forceinline__ int mx_shared_exponent(float amax, int emax) {
    const uint32_t b = __float_as_uint(amax);
    const int ex = static_cast<int>((b >> 23) & 0xFF);
    int fl;
    if (ex == 0) {
        const uint32_t m = b & 0x7FFFFF;
        if (m == 0) return -127;
        fl = (31 - __clz(m)) - 149;  // subnormal: m * 2^-149
    } else {
        fl = ex - 127;
    }
    const int e = fl - emax;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^n as fp32 for n in [-127, 127] (exact).
__device__ __forceinline__ float exp2_int(int n) {
    return n >= -126 ? __uint_as_float(static_cast<uint32_t>(n + 127) << 23) : __uint_as_float(0x00400000u);
}

// Two fp32 -> two E4M3 codes (RNE, saturating); v0 in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float v0, float v1) {
    return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3));
}

// Two fp32 -> two E2M1 codes (RNE, saturating); v0 in the low nibble.
__device__ __forceinline__ uint8_t e2m1x2(float v0, float v1) {
    return static_cast<uint8_t>(__nv_cvt_float2_to_fp4x2(make_float2(v0, v1), __NV_E2M1, cudaRoundNearest));
}

// A non-negative finite E4M3 code to fp32, exactly: subnormals m * 2^-9,
// normals (1 + m / 8) * 2^(e - 7).
__device__ __forceinline__ float e4m3_pos_to_float(uint32_t c) {
    const uint32_t e = (c >> 3) & 15, m = c & 7;
    return e == 0 ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120) << 23) | (m << 20));
}

// NVFP4 ("[SGLang] CUTLASS MoE", section 6): one block of 16 fp32 values with
// global scale gs -> the E4M3 block scale code (returned) and the 16 E2M1
// codes, element 2i in the low nibble of byte i (w0: elements 0-7, w1: 8-15).
// Every decision in fp32: s = (amax * gs) / 6 rounded to E4M3 (nearest even,
// saturating), r = gs / dec(s), codes = E2M1(v_i * r) (nearest even,
// saturating; r = 0 when the scale underflows, giving signed zeros).
__device__ __forceinline__ uint32_t nvfp4_block(const float* v, float gs, uint32_t& w0, uint32_t& w1) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float s = __fdiv_rn(__fmul_rn(amax, gs), 6.0f);
    const uint32_t sf = __nv_cvt_float2_to_fp8x2(make_float2(s, 0.f), __NV_SATFINITE, __NV_E4M3) & 0xFFu;
    const float d = e4m3_pos_to_float(sf);
    const float r = d > 0.f ? __fdiv_rn(gs, d) : 0.f;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t b = static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(
            make_float2(__fmul_rn(v[2 * i], r), __fmul_rn(v[2 * i + 1], r)), __NV_E2M1, cudaRoundNearest));
        w[i >> 2] |= b << (8 * (i & 3));
    }
    w0 = w[0];
    w1 = w[1];
    return sf;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// x -> MXFP8 in token order, one 32-element block: blk = t * (H / 32) + b of
// the bf16 rows x [T, H] gives the E8M0 code xsf[blk] (emax 8) and the 32
// E4M3 codes xq[32 blk ..] (nearest even, saturating).
__device__ __forceinline__ void quant_x_block(const uint16_t* x, uint8_t* xq, uint8_t* xsf, size_t blk) {
    const uint4* src = reinterpret_cast<const uint4*>(x) + blk * 4;
    uint4 raw[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) raw[c] = __ldg(src + c);
    // word k holds elements 2k (low half) and 2k + 1 (high half)
    const uint32_t* wd = reinterpret_cast<const uint32_t*>(raw);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wd[k] << 16)), fabsf(__uint_as_float(wd[k] & 0xFFFF0000u))));
    const int ex = mx_shared_exponent(amax, 8);
    const float inv = exp2_int(-ex);
    uint32_t packed[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t w0 = wd[2 * e], w1 = wd[2 * e + 1];
        const uint32_t lo = e4m3x2(__uint_as_float(w0 << 16) * inv, __uint_as_float(w0 & 0xFFFF0000u) * inv);
        const uint32_t hi = e4m3x2(__uint_as_float(w1 << 16) * inv, __uint_as_float(w1 & 0xFFFF0000u) * inv);
        packed[e] = lo | (hi << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(xq) + blk * 2;
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    xsf[blk] = static_cast<uint8_t>(ex + 127);
}

}  // namespace moe
