// Kernel parameter blocks and launchers of the GPU library.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

// cudaLaunchKernelEx with programmatic dependent launch (the kernel may start
// while its predecessor in the stream drains; it calls griddepcontrol.wait
// before touching the predecessor's outputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                          Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct RouteParams {
    const float* logits;
    const uint16_t* shared_logit;
    int32_t* ids;
    float* w;
    int T, Eg, k, S, kp;
    float shared_scale;
};

struct SortParams {
    const int32_t* ids;
    int32_t* header;
    int32_t* counts;
    int32_t* offsets;
    int4* vinfo;
    int4* groups;
    int32_t* a_map;
    int32_t* c_map;
    int32_t* vbase;     // [Et]: index of each expert's first virtual expert
    int32_t* cta_hist;  // [ceil(T*k' / 4096)][Et]: large-sort scratch
    int T, kp, Eg, E, off, S, Et, B, G;
    int keep_status;    // 1: leave the status word as the router GEMM left it (it was reset before the router)
    // the GEMM2 gate, decided where the expert placement writes the header
    int H;
    int gemm2_force;    // 0 the rule (rs::gemm2_path), 1 split, 2 dense
    int64_t dense_max_elems;  // 128-row tiles: dense when rows * H <= this (and the accumulator fits)
};

// Router GEMM (x bf16 [T, H] times router rows bf16 [Eg, H] -> fp32 logits).
struct RouterParams {
    float* logits;    // [T, Eg]
    int32_t* status;  // status word pair, or nullptr
    int T, Eg, H;
    int N;            // router rows per tile (64 or 224)
    int n_tiles;      // tiles over Eg
    int ks;           // K splits = cluster size
    uint64_t wait_ns;
};

struct RouterTiling {
    int N, ks, n_tiles, grid;
};

struct GatherParams {  // x -> MXFP8 + the routing weight of each expert row
    const uint16_t* x;      // [T, H] bf16
    const int32_t* header;  // rows R
    const int32_t* a_map;
    uint8_t* xq;            // token order [T, H], or expert-row order [rows_alloc, H]
    uint8_t* xsf;           // token order [T, H / 32], or per 128-row tile the lane-major scale cells
    const float* topk_w;
    float* row_w;           // routing weight of each row: topk_w[a_map[row]]
    // expert-row order (128-row tiles): slot -> row map and expert placement
    const int32_t* c_map;
    const int32_t* offsets;
    const int32_t* vbase;
    float* acc;             // dense GEMM2 accumulator [T, H] (zeroed here when the gate chose dense)
    float x_gscale;         // NVFP4: global scale of x
    int token_order;        // 1: decode tilings (the FC1 kernel gathers the rows)
    int H, T, R_max, max_blocks, kp, B, Et, xsf_tile_bytes;
    int t0;                 // token-major gathers: first token (tokens t0 .. T - 1)
};

struct GemmParams {
    const int32_t* header;
    int32_t* status;  // header + kHdrStatus (status, detail)
    const int4* groups;
    const int4* vinfo;
    const int32_t* a_map;
    const float* topk_w;
    const float* row_w;    // routing weight per row (written by the gather)
    const uint8_t* a_sf;   // packed weight scales
    const uint8_t* b_sf;   // tile scales of the activation operand
    uint8_t* act;          // FC1 output codes [rows_alloc, I]
    uint8_t* act_sf;       // FC1 output tile scales
    float* y;              // FC2 output [R, H], fp32 (decode tilings)
    uint16_t* y_bf16;      // FC2 output [R, H], bf16 (prefill tiling)
    int H, I;
    int b_sf_tile_bytes, out_sf_tile_bytes;
    int a_tx_bytes;        // transaction bytes of a stage's weight box (packed E2M1 bytes)
    uint64_t wait_ns;
    int act_kind;          // FC1 epilogue activation (MOE_ACT_*)
    int max_v;             // entries of vinfo (virtual-expert bound)
    // FC1 token rows: gathered per tile from the token-order MXFP8 x
    const uint8_t* xq;     // [T, H] E4M3
    const uint8_t* xsf;    // [T, H / 32] E8M0
    int kp;                // slots per token (a_map / kp = token)
    float act_c0, act_c1;  // its constants: clamp limit, or SiTU beta and linear beta
    uint64_t test_stall_ns;  // test hook: the MMA thread first waits this long on a barrier nothing arrives on (0: off)
    float* acc;              // dense GEMM2 accumulator [T, H] fp32
    int T;
    // NVFP4 variant (128-row tiles): operands packed E2M1 with E4M3 scales per 16
    int nv;
    const float* nv_w_gs;    // per local expert: global scale of this GEMM's weights
    float nv_in_gs;          // global scale of this GEMM's token operand (x, or the intermediate)
    float nv_out_gs;         // FC1: global scale the intermediate is quantised with
};

struct CombineParams {
    const int32_t* header;  // the gate's GEMM2 path
    const float* acc;       // dense path: fp32 [T, H] sums
    const int32_t* c_map;
    const float* y;         // fp32 rows, or NULL when y_bf16 is used
    const uint16_t* y_bf16; // bf16 rows (prefill tiling)
    uint16_t* out;
    int T, kp, H;
    int t0;  // first token (tokens t0 .. T - 1; 0 for the whole batch)
};

struct QuantParams {
    const float* w;
    uint8_t* codes;
    uint8_t* scales;
    int64_t rows, K;
};

// NVFP4 weights: rows of experts x rows_per_expert, each expert with its own
// global scale.
struct NvQuantParams {
    const float* w;
    float* gscale;   // [experts]
    uint8_t* codes;  // [rows, K / 2]
    uint8_t* scales; // [rows, K / 16]
    int64_t experts, rows_per_expert, K;
};

struct PackParams {
    const uint8_t* codes;
    const uint8_t* scales;
    uint8_t* packed_codes;
    uint8_t* packed_scales;
    int64_t experts, N, K;
    int pair;
};

// gp (optional, token-order x only): the launch also quantises x.
cudaError_t launch_route(const RouteParams& p, cudaStream_t stream, bool pdl, const GatherParams* gp = nullptr);
cudaError_t launch_sort(const SortParams& p, cudaStream_t stream, bool pdl);
// Route + sort fused in one cluster launch, for batches of at most 128 tokens.
bool route_sort_fusable(int T, int kp);
// Whether that launch also quantises token-order x (batches of at most 64 tokens).
bool route_sort_fuses_x(int T);
// One-CTA sort of the layer's own routing (ids distinct per token) by token
// bitmasks, for batches of at most 512 tokens whose tables fit in shared memory.
bool sort_tokens_ok(int T, int kp, int Et);
// row_w (optional): each row's routing weight w[slot] is written too.
cudaError_t launch_sort_tokens(const SortParams& p, cudaStream_t stream, bool pdl, const float* w = nullptr,
                               float* row_w = nullptr);
// Kernels launch_sort issues for T*k' slots (1, or 3 above one CTA's share).
int sort_launch_count(int64_t slots);
// gp (optional, token-order x only): the launch also quantises x and writes
// each row's routing weight -- the work of launch_gather.
cudaError_t launch_route_sort_small(const RouteParams& rp, const SortParams& p, const GatherParams* gp,
                                    cudaStream_t stream, bool pdl);
cudaError_t launch_gather(const GatherParams& p, cudaStream_t stream, bool pdl);
// NVFP4 x for 128-row tiles (xsf_tile_bytes: 1024 per 128-K chunk).
cudaError_t launch_gather_nvfp4(const GatherParams& p, cudaStream_t stream, bool pdl);
// tmAux: for FC2 at 128-row tiles the bf16 rows as boxes of 64 columns x 32
// rows; for FC1 at 128-row tiles the x scale blocks as 4-D boxes {16 bytes,
// 1 chunk, 32 lanes (NVFP4: 64), 1 tile} over the lane-major tile layout; any
// valid map otherwise (not read).
cudaError_t launch_gemm(bool fc1, const CUtensorMap& tmW, const CUtensorMap& tmX, const CUtensorMap& tmAux,
                        const GemmParams& p, int TM, int grid, cudaStream_t stream, bool pdl);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream, bool pdl);
RouterTiling router_tiling(int T, int Eg, int num_sms);
cudaError_t launch_router(const CUtensorMap& tmX, const CUtensorMap& tmW, const RouterParams& p, int grid,
                          cudaStream_t stream, bool pdl);
cudaError_t launch_quantize_mxfp4(const QuantParams& p, cudaStream_t stream);
cudaError_t launch_pack_weights(const PackParams& p, cudaStream_t stream);
cudaError_t launch_quantize_nvfp4(const NvQuantParams& p, cudaStream_t stream);
cudaError_t launch_pack_weights_nvfp4(const PackParams& p, cudaStream_t stream);

}  // namespace moe
