/*
 * moe_api.h -- C ABI of the GB300 (sm_103a) fused MXFP4 Mixture-of-Experts
 * layer forward.
 *
 * The layer (reference pages: "[SGLang] CUTLASS MoE", structure diagram;
 * "[sglang] Kimi-K3.1 MXFP4 decode MoE kernel generalised to shape templates",
 * sections 1-5; "[sglang] SGLang MoE shared expert: fuse 3 kernels into 1"):
 *
 *   route  : top-k of the router logits, weights renormalised over the picks,
 *            optional appended shared expert with weight sigmoid(logit)*scale
 *   sort   : token -> expert rows (expert_offsets, a_map, c_map) and virtual
 *            experts of block_n rows
 *   forward: x -> MXFP8, FC1 = [gate | up] on E2M1 weights, activation
 *            h(gate, up) -> MXFP8, FC2, weighted un-permute combine -> bf16 out
 *
 * Ownership: the caller allocates every buffer (device memory unless stated).
 * The library never allocates device memory, never frees and never
 * synchronises the stream; every call is asynchronous on `stream` and, except
 * moe_layer_host, capturable in a CUDA graph.
 *
 * Errors: calls return MOE_OK (0) or a negative MOE_ERR_* code.  Argument
 * errors are detected on the host and launch nothing.  Errors found on the
 * device (a bounded wait that expired) are recorded in the workspace status
 * word, read with moe_get_status after the stream has been synchronised.
 *
 * Data formats:
 *   bf16       : uint16_t bit patterns.
 *   E2M1       : 4-bit codes, two per byte, element 2i in the low nibble.
 *   E4M3 / E8M0: one byte per element / per 32-element block.
 *   MX blocks  : one E8M0 scale per 32 consecutive elements along K (the
 *                contiguous dimension), OCP MX v1.0 conversion rule.
 */
#ifndef MOE_API_H
#define MOE_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
    MOE_OK = 0,
    MOE_ERR_NULL = -1,      /* a required pointer is NULL */
    MOE_ERR_SHAPE = -2,     /* shape outside moe_is_supported */
    MOE_ERR_ALIGN = -3,     /* a pointer misses its documented alignment */
    MOE_ERR_WORKSPACE = -4, /* workspace smaller than moe_workspace_bytes */
    MOE_ERR_CUDA = -5,      /* a CUDA runtime/driver call failed */
    MOE_ERR_TIMEOUT = -6    /* device status: a bounded wait expired */
};

/* FC1 epilogue activation h(g, u) of gate g = W1 rows [0, I) and up u =
 * rows [I, 2I), evaluated in fp32 before the MXFP8 requantisation
 * ("... MXFP4 decode MoE ... shape templates", section 4: the epilogue's
 * activation is a parameter, SiTU<beta, linear_beta> or SwiGLU<limit>).
 *   MOE_ACT_SWIGLU        silu(g) * u,  silu(g) = g / (1 + exp(-g))
 *   MOE_ACT_SWIGLU_CLAMP  silu(min(g, L)) * clamp(u, -L, L),
 *                         L = act_params[0] > 0 (the clamped SwiGLU)
 *   MOE_ACT_SITU          (beta tanh(g / beta)) sigmoid(g) * lb tanh(u / lb),
 *                         beta = act_params[0] > 0, lb = act_params[1] > 0
 *                         (beta 4, lb 25 give the section's fixed form
 *                         2 tanh(g/4) (1 + tanh(g/2)) * 25 tanh(u/25)) */
enum { MOE_ACT_SWIGLU = 0, MOE_ACT_SWIGLU_CLAMP = 1, MOE_ACT_SITU = 2 };

/* Shape of one layer call.
 *   T            tokens in this call (0 <= T <= max_T)
 *   max_T        tokens the workspace is sized for
 *   E_global     routed experts in the logit space (columns of the logits)
 *   E_local      routed experts whose weights live here
 *   expert_offset global id of local expert 0; ids outside
 *                [expert_offset, expert_offset + E_local) get no row
 *                ("... MXFP4 decode MoE ... shape templates", section 5)
 *   top_k        routed experts per token
 *   num_shared   0 or 1 shared experts appended to every token, global id
 *                E_global + s, local weight slot E_local + s
 *   hidden, inter H and I
 *   block_n      rows per virtual expert = token rows of a GEMM tile: 16 or
 *                32 (decode tiling, fp32 FC2 rows) or 128 (prefill tiling,
 *                bf16 FC2 rows); the layer's value does not depend on it
 *   activation   MOE_ACT_SWIGLU, MOE_ACT_SWIGLU_CLAMP or MOE_ACT_SITU
 *   shared_scale multiplies the shared expert's sigmoid weight (e.g.
 *                1/ep_size, "... shared expert: fuse 3 kernels into 1")
 *   act_params   the activation's constants (finite, > 0 where used; unused
 *                entries are ignored) */
typedef struct moe_shape {
    int32_t T, max_T, E_global, E_local, expert_offset, top_k, num_shared;
    int32_t hidden, inter, block_n, activation;
    float shared_scale;
    float act_params[2];
} moe_shape;

/* Packed expert weights (device, read only), E_tot = E_local + num_shared,
 * produced by moe_pack_weights from row-major MXFP4 (moe_quantize_mxfp4):
 *   w1, w1_sf  W1 [E_tot, 2I, H] packed with pair_halves = 1 (gate/up tiles
 *              of the same features adjacent)
 *   w2, w2_sf  W2 [E_tot, H, I] packed with pair_halves = 0
 * Codes 32-byte aligned, scales 16-byte aligned. */
typedef struct moe_weights {
    const uint8_t *w1, *w1_sf, *w2, *w2_sf;
} moe_weights;

/* NVFP4 variant ("[SGLang] CUTLASS MoE", section 6, cutlass_moe_fp4: FP4 in
 * blocks of 16, with a per-tensor scale for the narrow E2M1 range).  A tensor
 * holds E2M1 codes (two per byte, element 2i in the low nibble), one E4M3
 * block scale (sign bit clear) per 16 consecutive K elements and one fp32
 * global scale gs: value = e2m1 * e4m3 / gs.  A block of 16 is quantised with
 * every decision in fp32: s = (amax * gs) / 6 rounded to E4M3 (nearest even,
 * saturating at 448); r = gs / dec(s); each element = E2M1(v * r) (nearest
 * even, saturating at 6; signed zeros when s underflows).  The FC1 / FC2
 * products are E2M1 x E2M1 on tcgen05 kind::mxf4nvf4 tensor cores, scaled by
 * 1 / (gs_in * gs_w[e]) in the epilogue; the activation's output is
 * requantised to NVFP4 with h_gscale.
 *   x_gscale, h_gscale  global scales of x and of the FC1 activation output
 *                       (calibrated by the caller: 2688 / (the largest |value|
 *                       expected) keeps every block scale in range)
 *   w1_gscale, w2_gscale device fp32 [E_tot]: each expert matrix's global
 *                       scale, written by moe_quantize_nvfp4 */
typedef struct moe_nvfp4 {
    float x_gscale, h_gscale;
    const float *w1_gscale, *w2_gscale;
} moe_nvfp4;

/* fp32 weights of `experts` matrices [experts, rows, K] (device, 16-byte
 * aligned, K % 16 == 0) -> NVFP4: gscale [experts] (fp32(2688 / amax) of each
 * matrix, 1 for all zeros), codes [experts * rows, K / 2] and E4M3 scales
 * [experts * rows, K / 16], row-major. */
int moe_quantize_nvfp4(const float* w, int64_t experts, int64_t rows, int64_t K, float* gscale, uint8_t* codes,
                       uint8_t* scales, moe_stream_t stream);

/* moe_pack_weights for NVFP4: the codes are packed exactly as for MXFP4
 * (per expert, 256-row block and 128-K chunk one contiguous 16 KiB run); the
 * scales (row-major [experts, N, K / 16]) become one 2 KiB block per tile in
 * the layout the scale_vec::4X MMA reads from tensor memory: for each 64-K
 * half kk two 512-byte blocks (block rows 0-127, 128-255), row r's 4-byte
 * cell at (r % 32) * 16 + (r / 32) * 4, byte b = the half's 16-element block
 * b.  Sizes: codes experts * N * K / 2, scales experts * N * K / 16 bytes.
 * N % 256 == 0, K % 128 == 0. */
int moe_pack_weights_nvfp4(const uint8_t* codes, const uint8_t* scales, int64_t experts, int64_t N, int64_t K,
                           int32_t pair_halves, uint8_t* packed_codes, uint8_t* packed_scales, moe_stream_t stream);

/* moe_layer in the NVFP4 variant, for 128-row tiles (block_n == 128; other
 * tilings return MOE_ERR_SHAPE): weights packed by moe_pack_weights_nvfp4,
 * global scales in `nv`.  Same launch chain, GEMM2 gate and outputs as
 * moe_layer; in the workspace, x and the intermediate hold NVFP4 codes [rows,
 * H / 2] / [rows, I / 2] with 1 KiB scale blocks per 128-K chunk of a virtual
 * expert (the layout above, tile rows for matrix rows). */
int moe_layer_nvfp4(const moe_shape* shape, const moe_nvfp4* nv, const float* logits, const uint16_t* shared_logit,
                    const uint16_t* x, const moe_weights* weights, int32_t* topk_ids, float* topk_w, void* workspace,
                    size_t workspace_bytes, uint16_t* out, moe_stream_t stream);

/* moe_layer_nvfp4 with the timing events of moe_layer_events. */
int moe_layer_nvfp4_events(const moe_shape* shape, const moe_nvfp4* nv, const float* logits,
                           const uint16_t* shared_logit, const uint16_t* x, const moe_weights* weights,
                           int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes, uint16_t* out,
                           void* const* events, moe_stream_t stream);

/* Device pointers into a workspace, for inspection and parity checks.
 *   header       int32[64]: [0] rows R, [1] virtual experts, [2] groups,
 *                [3] status, [4] status detail, [5] GEMM2 path (0 split,
 *                1 dense)
 *   expert_counts int32[E_tot], expert_offsets int32[E_tot + 1]
 *   vinfo        int32[max_v][4] {local expert, first row, rows, chunk}
 *   a_map        int32[R] row -> slot t*k' + j;  c_map int32[T*k'] slot -> row or -1
 *   xq, xq_sf    x in MXFP8.  x_token_order = 1 (block_n 16 / 32): E4M3
 *                [max_T, H], row t = MXFP8(x[t]), and E8M0 [max_T, H / 32]
 *                row-major (the decode FC1 gathers each tile's rows from
 *                here).  x_token_order = 0 (block_n 128): E4M3 [rows_alloc,
 *                H] in expert-row order, row r = MXFP8(x[a_map[r] / k']),
 *                and E8M0 per virtual expert v in sf_tile_bytes_x bytes at
 *                v * sf_tile_bytes_x, lane-major: tile row i / K-block b at
 *                ((i % 32) * (H / 128) + b / 4) * 16 + (i / 32) * 4 + b % 4
 *                (the 16-byte cells of act_sf's layout, chunk-minor)
 *   act          E4M3 [rows_alloc, I]: the FC1 output (the activation
 *                h(gate, up), MXFP8) in expert-row order
 *   act_sf       E8M0 of act in the tile layout: per virtual expert v and
 *                128-K chunk kc a 512-byte block (v * sf_tile_bytes_act +
 *                kc * 512), tile row i / K-block b at (i % 32) * 16 +
 *                (i / 32) * 4 + b
 *   y            the FC2 output rows [R, H], already multiplied by the routing
 *                weight: fp32 for block_n 16/32, bf16 for block_n 128 */
typedef struct moe_views {
    int32_t *header, *expert_counts, *expert_offsets, *vinfo, *a_map, *c_map;
    uint8_t *xq, *xq_sf, *act, *act_sf;
    void* y;
    int32_t max_v, rows_alloc, y_is_bf16, sf_tile_bytes_x, sf_tile_bytes_act, x_token_order;
} moe_views;

/* 1 if the shape is supported, else 0.  Limits: hidden % 512 == 0,
 * inter % 128 == 0, block_n in {16, 32, 128}, 1 <= top_k <= 32,
 * top_k <= E_global <= 1024, 1 <= E_local + num_shared <= 1024,
 * num_shared in {0, 1}, 0 <= expert_offset, expert_offset + E_local <=
 * E_global, 0 <= T <= max_T, max_T * (top_k + num_shared) < 2^24.
 * (The compile-time limits of "... MXFP4 decode MoE ... shape templates",
 * section 2, restated as runtime checks.) */
int moe_is_supported(const moe_shape* shape);

/* Bytes of the single workspace buffer that every other call carves, at
 * 256-byte alignment, into the routing header, expert counts / offsets,
 * virtual-expert descriptors, a_map / c_map, the MXFP8 x, the intermediate
 * (codes + tile scales, with block_n rows of padding for the last tile's TMA
 * box) and the FC2 rows.  ("... MXFP4 decode MoE ... shape templates",
 * section 3: one byte tensor carved once at 256-byte alignment, so the host
 * allocates a single buffer; the padded intermediate rows are the same
 * section's last-virtual-expert box.)  Returns MOE_ERR_SHAPE for an
 * unsupported shape. */
int moe_workspace_bytes(const moe_shape* shape, size_t* bytes);

/* fp32 [rows, K] -> MXFP4: codes [rows, K/2] and E8M0 scales [rows, K/32]
 * (row-major), shared exponent floor(log2 amax) - 2, elements rounded to
 * nearest even and saturated to +-6 (OCP MX v1.0).  K % 32 == 0.  codes must
 * be 16-byte aligned. */
int moe_quantize_mxfp4(const float* w, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                       moe_stream_t stream);

/* Tile-major packing of one weight matrix per expert for the tensor-core
 * path.  Input: row-major E2M1 codes [experts, N, K/2] and E8M0 scales
 * [experts, N, K/32] (moe_quantize_mxfp4).  A row block holds 256 rows: rows
 * b*256.. (pair_halves = 0, W2), or the 128 rows b*128.. of the first half
 * [0, N/2) followed by the 128 rows N/2 + b*128.. of the second half
 * (pair_halves = 1, W1: the gate and up rows of the same 128 features).
 * Output, for each expert e, row block b and 128-K chunk c in that order:
 *   packed_codes : the block's 256 rows x 64 bytes (the chunk's 128 codes of
 *                  each row), one contiguous 16 KiB run;
 *   packed_scales: two 512-byte blocks (block rows 0-127, 128-255), row r /
 *                  K-block j of the chunk at byte (r % 32) * 16 + (r / 32) * 4
 *                  + j (the tensor-memory scale layout, one tcgen05.cp each).
 * N % 256 == 0, K % 128 == 0.  Sizes: moe_packed_weight_bytes. */
/* Rows per block (256) and the byte sizes of moe_pack_weights' outputs for
 * one weight matrix per expert [experts, N, K] (equal to the inputs').
 *
 * moe_pack_weights: the operand shapes are those of "[SGLang] CUTLASS MoE",
 * structure diagram (GEMM1 (m*topk, k) x (E, k, 2n), GEMM2 (m*topk, n) x
 * (E, n, k), E2M1 weights with one E8M0 scale per 32 K as in "... MXFP4
 * decode MoE ... shape templates", section 1); the tile-major order is this
 * library's own layout for its TMA stages.  Asynchronous on `stream`; the
 * outputs must not alias the inputs. */
int moe_packed_weight_bytes(int64_t experts, int64_t N, int64_t K, int32_t pair_halves, int32_t* block_rows,
                            size_t* code_bytes, size_t* scale_bytes);

int moe_pack_weights(const uint8_t* codes, const uint8_t* scales, int64_t experts, int64_t N, int64_t K,
                     int32_t pair_halves, uint8_t* packed_codes, uint8_t* packed_scales, moe_stream_t stream);

/* Routing.  logits fp32 [T, E_global]; shared_logit bf16 [T, num_shared] or
 * NULL when num_shared == 0.  Writes topk_ids int32 [T, k'] and topk_w fp32
 * [T, k'], k' = top_k + num_shared: the top_k largest logits in descending
 * order (ties to the lower expert id), weights exp(l_j - m) / sum_sel exp(l_i
 * - m) (softmax renormalised over the picks), then the shared expert (id
 * E_global + s, weight sigmoid(fp32(logit)) * shared_scale).  NaN logits are
 * not supported. */
int moe_route(const moe_shape* shape, const float* logits, const uint16_t* shared_logit, int32_t* topk_ids,
              float* topk_w, moe_stream_t stream);

/* Token-to-expert sort of topk_ids int32 [T, k'] into the workspace:
 * expert counts/offsets, a_map/c_map (rows of an expert in ascending slot
 * order t*k' + j), virtual experts (chunks of block_n rows per expert) and the
 * GEMM work list; resets the status word.  ("[SGLang] CUTLASS MoE", section 1
 * prepare_moe_input; "... MXFP4 decode MoE ... shape templates", sections 1,
 * 5.)  The workspace must be 256-byte aligned. */
int moe_sort(const moe_shape* shape, const int32_t* topk_ids, void* workspace, size_t workspace_bytes,
             moe_stream_t stream);

/* Forward after moe_sort ("[SGLang] CUTLASS MoE", structure diagram:
 * quantise + shuffle_rows (section 2), GEMM1, silu_and_mul (section 4),
 * GEMM2 and apply_shuffle_mul_sum (section 5)): x bf16 [T, H] -> out bf16
 * [T, H].
 *   out[t] = bf16( sum_{j: c_map[t,j] >= 0, ascending j} topk_w[t,j] *
 *                  Y_j(t) ),  Y_j = FC2(MXFP8(h(G, U))), [G | U] =
 *                  FC1(MXFP8(x[t])) with expert topk_ids[t,j]'s weights and h
 *                  the shape's activation.
 * FC1/FC2 run on tcgen05 block-scaled tensor cores (E4M3 x E2M1, fp32
 * accumulation), the activation + MXFP8 requantisation is fused into the FC1
 * epilogue and the routing-weight multiply into the FC2 epilogue.
 * x, out 16-byte aligned. */
int moe_forward(const moe_shape* shape, const uint16_t* x, const moe_weights* weights, const float* topk_w,
                void* workspace, size_t workspace_bytes, uint16_t* out, moe_stream_t stream);

/* Router GEMM: logits[t][e] = fp32 sum_h x[t][h] * wr[e][h] for x bf16
 * [T, H] and the router matrix wr bf16 [E_global, H] (row e = expert e),
 * written to logits fp32 [T, E_global].  The step in front of routing: the
 * pages' kernel ("... MXFP4 decode MoE ... shape templates", section 5)
 * starts from the top-k of these logits.  tcgen05 kind::f16 tensor cores
 * (bf16 products, fp32 accumulation); for T <= 256 the H reduction is split
 * over the 8 CTAs of a cluster and summed in a fixed order, so the logits are
 * bit-reproducible.  The fp32 sums differ from an exactly rounded dot
 * product by the accumulation order only.  Resets the workspace status word,
 * then records MOE_ERR_TIMEOUT there if a bounded wait expires.  x, wr,
 * logits 16-byte aligned. */
int moe_router(const moe_shape* shape, const uint16_t* x, const uint16_t* wr, float* logits, void* workspace,
               size_t workspace_bytes, moe_stream_t stream);

/* moe_router + route + sort + forward as one fixed launch chain: the layer
 * from x and the router matrix (logits written to `logits`, ids and weights
 * to topk_ids / topk_w).  Graph capturable; the status word covers the
 * router and the GEMMs. */
int moe_layer_router(const moe_shape* shape, const uint16_t* wr, const uint16_t* shared_logit, const uint16_t* x,
                     const moe_weights* weights, float* logits, int32_t* topk_ids, float* topk_w, void* workspace,
                     size_t workspace_bytes, uint16_t* out, moe_stream_t stream);

/* route + sort + forward as one fixed launch chain: programmatic dependent
 * launch between kernels, no host synchronisation, and kernels that find no
 * work exit at once, so one captured CUDA graph serves every routing of the
 * shape ("[FlashInfer] Device-side gating for the MoE GEMM2 path", section 2
 * "fixed launch chain for CUDA Graph"; "... MXFP4 decode MoE ... shape
 * templates", introduction: routing and the MoE launched from one host
 * entry with PDL).  Same arguments and layouts as moe_route + moe_sort +
 * moe_forward; topk_ids / topk_w receive the routing. */
int moe_layer(const moe_shape* shape, const float* logits, const uint16_t* shared_logit, const uint16_t* x,
              const moe_weights* weights, int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
              uint16_t* out, moe_stream_t stream);

/* moe_layer from HOST buffers: copies logits, shared_logit and x (host,
 * preferably pinned) into the workspace's staging area, runs the chain and
 * copies out (host) back; the call is asynchronous on `stream`, and the
 * caller synchronises `stream` before reading out.  Weights stay on the
 * device.  The layer is the one of "[SGLang] CUTLASS MoE", structure diagram
 * (input a (m, k) -> output (m, k)); the host copies around it are this
 * library's end-to-end entry point.  Decode tilings: every copy on `stream`.
 * 128-row tilings (long batches): the copies run on two streams the library
 * creates once per device, one per direction -- logits first, then x in 8
 * token chunks host-to-device; out in 8 token chunks device-to-host -- so
 * routing starts when the logits have landed, each chunk's x gather when its
 * rows have landed, and each chunk's output leaves once combined,
 * overlapping the copies with the gather and the combine.  The input copies
 * wait for `stream` at the call and `stream` waits for the last output copy,
 * so the call is ordered on `stream` like any other.  Calls issued on two
 * streams, each with its own workspace and output buffer, overlap: one
 * call's output copies share the full-duplex host link with the other's
 * input copies while the GPU computes.  Calls on one device enqueue one at a
 * time (a mutex).  Not capturable (host memory). */
int moe_layer_host(const moe_shape* shape, const float* logits_host, const uint16_t* shared_logit_host,
                   const uint16_t* x_host, const moe_weights* weights, void* workspace, size_t workspace_bytes,
                   uint16_t* out_host, moe_stream_t stream);

/* moe_layer with timing events: events[0..6] (cudaEvent_t, created by the
 * caller) are recorded on `stream` before route and after route, sort, the x
 * quantise/gather, FC1, FC2 and combine, so each kernel's device time is
 * cudaEventElapsedTime(events[i], events[i+1]).  The records sit between the
 * launches (no programmatic overlap across them); use moe_layer for the
 * production chain. */
int moe_layer_events(const moe_shape* shape, const float* logits, const uint16_t* shared_logit, const uint16_t* x,
                     const moe_weights* weights, int32_t* topk_ids, float* topk_w, void* workspace,
                     size_t workspace_bytes, uint16_t* out, void* const* events, moe_stream_t stream);

/* moe_layer for callers that cannot allocate device memory (for example code
 * running under another framework's allocator with allocation disabled, or a
 * runtime that must not call cudaMalloc after start-up).  The reference pages
 * have no counterpart to this call.  The layer's scratch is one 32 MiB
 * file-scope device array that every GPU loading this library holds until
 * the process exits; shapes whose moe_workspace_bytes exceeds 32 MiB are
 * rejected with MOE_ERR_WORKSPACE (decode with T <= 32 at E 896, k 16,
 * H 3584, I 384 fits).  The caller passes inputs and outputs as for
 * moe_layer; the call allocates nothing.  Each call looks up the array's
 * device address (cudaGetSymbolAddress, with the call's device current), so
 * a device reset that reloads the library's module is picked up.  Every call
 * on a device shares the one array and leaves its contents behind: calls
 * whose executions overlap on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.  Device-side errors are recorded
 * in that array's status word: read it with moe_noalloc_get_status. */
int moe_layer_noalloc(const moe_shape* shape, const float* logits, const uint16_t* shared_logit, const uint16_t* x,
                      const moe_weights* weights, int32_t* topk_ids, float* topk_w, uint16_t* out,
                      moe_stream_t stream);

/* moe_get_status for moe_layer_noalloc: reads the status word of the
 * current device's fixed scratch array (synchronous copy; call after the
 * stream has finished).  The array starts zeroed, so before the first
 * moe_layer_noalloc call on a device this reads (MOE_OK, 0). */
int moe_noalloc_get_status(int32_t* status, int32_t* detail);

/* Workspace views (device pointers) for inspection. */
int moe_get_views(const moe_shape* shape, void* workspace, moe_views* views);

/* Reads the status word (and its detail) from the workspace header with a
 * synchronous device-to-host copy: call after the stream has finished.
 * *status is MOE_OK or MOE_ERR_TIMEOUT; *detail = site * 65536 + block of the
 * first expired wait (site 1 producer ring slot, 2 MMA data, 3 MMA
 * accumulator, 4 epilogue accumulator, 5 the test stall below).  The word
 * lives in the counters region of the single workspace ("... MXFP4 decode MoE
 * ... shape templates", section 3); the bounded waits that write it are this
 * library's guard against a kernel that would otherwise spin forever.  The
 * sort resets it on every call. */
int moe_get_status(const void* workspace, int32_t* status, int32_t* detail);

/* GEMM2 strategy ("[FlashInfer] Device-side gating for the MoE GEMM2
 * path", sections 1-2).  Every sort decides it on the device: the thread
 * that places the experts and writes the sorted table's header (rows R)
 * also picks:
 *   MOE_GEMM2_SPLIT  FC2 writes each routed row w * Y; the combine sums a
 *                    token's rows in ascending slot order (bit-reproducible);
 *   MOE_GEMM2_DENSE  FC2's epilogue reduces w * Y into an fp32 [T, H]
 *                    accumulator in the workspace (the finalize fused into
 *                    GEMM2, reductions performed at the L2); the combine
 *                    converts it to bf16.  The reductions' order varies, so
 *                    the result is within the layer's tolerance but not
 *                    bit-reproducible.
 * The gate's own rule (MOE_GEMM2_AUTO, the default) takes dense when the
 * accumulator stays in L2, T * H * 4 bytes <= 32 MiB, and, at block_n 128
 * (whose split rows are bf16, cheaper to write and re-read than the decode
 * tilings' fp32 rows), rows * H <= 56 Mi; split otherwise (the long
 * prefill); the chain of launches is the same either way.  moe_set_gemm2_path forces one path for every later sort
 * (moe_sort, moe_layer*) issued from this process (a captured graph keeps
 * the value of its capture); MOE_ERR_SHAPE for another value.  The path a
 * call took is header word 5 of its workspace (0 split, 1 dense). */
enum { MOE_GEMM2_AUTO = 0, MOE_GEMM2_SPLIT = 1, MOE_GEMM2_DENSE = 2 };
int moe_set_gemm2_path(int32_t path);

/* Test hook for the device-error path, off (0) by default.  While stall_ns is
 * nonzero, every later launch of the FC1 GEMM (on any device) makes its MMA
 * thread first wait stall_ns on a barrier that nothing arrives on; the wait
 * expires, the CTA records MOE_ERR_TIMEOUT (site 5) in the status word,
 * stops its producers and epilogue, lets their copies land, frees tensor
 * memory and exits.  FC2 and the combine still run, on stale data: the
 * output of such a call is garbage, its status says so.  The value is read
 * when a call is issued (a captured graph keeps the value of its capture).
 * Not thread safe against concurrent calls; for tests only.  No counterpart
 * on the reference pages. */
int moe_test_set_stall(uint64_t stall_ns);

/* Number of SMs the launches are sized for on the current device. */
int moe_num_sms(int32_t* num_sms);

/* Number of kernel launches moe_layer (and moe_layer_host, besides its
 * copies) issues for the shape: route + sort (one fused launch up to 64
 * tokens, else route and a one- or three-kernel sort), then for T > 0 the x
 * gather (not in the decode tilings up to 512 tokens, where the route launch
 * quantises x), FC1, FC2 and the combine. */
int moe_layer_launch_count(const moe_shape* shape, int32_t* count);

#ifdef __cplusplus
}
#endif
#endif /* MOE_API_H */
