// C ABI of the library (declared in include/moe_api.h): argument checks, the
// workspace carve, TMA tensor maps and the fixed launch chain
//   route -> sort -> gather/quantise x -> FC1 -> FC2 -> combine
// with programmatic dependent launch between kernels and no host
// synchronisation (graph capturable).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

// A 16U4_ALIGN16B box completes its packed global byte count (8 bytes per 16
// E2M1 elements), not its 16-byte-per-16-element shared-memory footprint.
constexpr int kFp4BytesPer128Row = 64;

// moe_test_set_stall: read by every FC1 launch that is issued
std::atomic<uint64_t> g_test_stall_ns{0};
// moe_set_gemm2_path: read by every sort launch that is issued (the sort's
// placement thread decides the GEMM2 path)
std::atomic<int> g_gemm2_path{MOE_GEMM2_AUTO};

// The gate's rule at 128-row tiles: the dense GEMM2 path when rows * H <=
// this many fp32 reductions and the accumulator fits well inside L2; the
// decode tilings take dense whenever the accumulator fits (rs::gemm2_path).
constexpr int64_t kDenseMaxElems = int64_t(56) << 20;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// 2-D K-major tensor map: dim0 = K elements (contiguous), dim1 = rows.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t K, uint64_t rows,
              uint64_t row_bytes, uint32_t box_k, uint32_t box_rows,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    if (!get_encode()) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_k, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Byte tensor [d3][d2][d1][d0], densely packed (strides d0, d0 * d1,
// d0 * d1 * d2 bytes), no swizzle; boxes of {d0, b1, b2, b3} elements.
bool make_map_4d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3, uint32_t b1,
                 uint32_t b2, uint32_t b3) {
    if (!get_encode() || d0 > 256) return false;
    cuuint64_t dims[4] = {d0, d1, d2, d3};
    cuuint64_t strides[3] = {d0, d0 * d1, d0 * d1 * d2};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(d0), b1, b2, b3};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int num_sms_cached() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static int cache[64] = {0};
    if (dev < 64 && cache[dev]) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev] = n;
    return n;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_NULL;
    return moe_is_supported(s) ? MOE_OK : MOE_ERR_SHAPE;
}

int check_ws(const moe_shape* s, const void* ws, size_t ws_bytes) {
    if (!ws) return MOE_ERR_NULL;
    if (!aligned(ws, 256)) return MOE_ERR_ALIGN;
    size_t need = 0;
    moe_workspace_bytes(s, &need);
    return ws_bytes >= need ? MOE_OK : MOE_ERR_WORKSPACE;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// gp (optional): the launch also quantises token-order x.
int run_route(const moe_shape* s, const float* logits, const uint16_t* shared_logit, int32_t* ids, float* w,
              cudaStream_t st, bool pdl, const GatherParams* gp = nullptr) {
    const Dims d = make_dims(*s);
    RouteParams p{logits, shared_logit, ids, w, d.T, d.Eg, d.k, d.S, d.kp, d.shared_scale};
    return cuda_rc(launch_route(p, st, pdl, gp));
}

// routed: the ids are the layer's own routing (each token's picks distinct),
// so batches of up to 512 tokens take the one-CTA token-bitmask sort, which
// also writes each row's routing weight w[slot] to row_w when given.
int run_sort(const moe_shape* s, const int32_t* ids, void* ws, cudaStream_t st, bool pdl, bool keep_status = false,
             bool routed = false, const float* w = nullptr, float* row_w = nullptr) {
    const Dims d = make_dims(*s);
    const Layout L = make_layout(d);
    SortParams p{ids, at<int32_t>(ws, L.header), at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
                 at<int4>(ws, L.vinfo), at<int4>(ws, L.groups), at<int32_t>(ws, L.a_map), at<int32_t>(ws, L.c_map),
                 at<int32_t>(ws, L.vbase), at<int32_t>(ws, L.sort_hist), d.T, d.kp, d.Eg, d.E, d.off, d.S, d.Et, d.B,
                 d.G, keep_status ? 1 : 0, d.H, g_gemm2_path.load(), kDenseMaxElems};
    if (routed && sort_tokens_ok(d.T, d.kp, d.Et)) return cuda_rc(launch_sort_tokens(p, st, pdl, w, row_w));
    return cuda_rc(launch_sort(p, st, pdl));
}

// Route then sort, fused into one launch when the batch has at most 64
// tokens.  `ev` (optional) gets events 1 (routed) and 2 (sorted); fused, both
// are recorded after the one kernel.  after_router: the logits come from the
// router GEMM launched just before (PDL launch; the status word it may have
// set survives the sort).  x (optional): in the decode tilings the fused
// launch also quantises x (the gather's work) up to 64 tokens; *gathered
// says whether it did.
int run_route_sort(const moe_shape* s, const float* logits, const uint16_t* shared_logit, int32_t* ids, float* w,
                   void* ws, cudaStream_t st, void* const* ev, bool after_router = false,
                   const uint16_t* x = nullptr, bool* gathered = nullptr);

// Records events[i] on the stream when an events array is given.
inline bool rec(void* const* ev, int i, cudaStream_t st) {
    return !ev || cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st) == cudaSuccess;
}

int run_route_sort(const moe_shape* s, const float* logits, const uint16_t* shared_logit, int32_t* ids, float* w,
                   void* ws, cudaStream_t st, void* const* ev, bool after_router, const uint16_t* x, bool* gathered) {
    const Dims d = make_dims(*s);
    if (gathered) *gathered = false;
    if (route_sort_fusable(d.T, d.kp)) {
        const Layout L = make_layout(d);
        RouteParams rp{logits, shared_logit, ids, w, d.T, d.Eg, d.k, d.S, d.kp, d.shared_scale};
        SortParams sp{ids, at<int32_t>(ws, L.header), at<int32_t>(ws, L.counts), at<int32_t>(ws, L.offsets),
                      at<int4>(ws, L.vinfo), at<int4>(ws, L.groups), at<int32_t>(ws, L.a_map), at<int32_t>(ws, L.c_map),
                      at<int32_t>(ws, L.vbase), at<int32_t>(ws, L.sort_hist), d.T, d.kp, d.Eg, d.E, d.off, d.S, d.Et,
                      d.B, d.G, after_router ? 1 : 0, d.H, g_gemm2_path.load(), kDenseMaxElems};
        GatherParams gp{};
        const bool fuse_x = x != nullptr && L.x_token_order && route_sort_fuses_x(d.T);
        if (fuse_x) {
            gp.x = x;
            gp.xq = at<uint8_t>(ws, L.xq);
            gp.xsf = at<uint8_t>(ws, L.xsf);
            gp.row_w = at<float>(ws, L.row_w);
            gp.H = d.H;
        }
        if (launch_route_sort_small(rp, sp, fuse_x ? &gp : nullptr, st, after_router && ev == nullptr) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (gathered) *gathered = fuse_x;
        return (rec(ev, 1, st) && rec(ev, 2, st)) ? MOE_OK : MOE_ERR_CUDA;
    }
    // Past the fused range the decode tilings quantise x in the route launch
    // (over the whole grid) and the token-bitmask sort writes each row's
    // routing weight: the gather's work, with no launch of its own.
    const Layout L = make_layout(d);
    const bool x_in_route = x != nullptr && L.x_token_order && d.T > 0 && sort_tokens_ok(d.T, d.kp, d.Et);
    GatherParams gp{};
    if (x_in_route) {
        gp.x = x;
        gp.xq = at<uint8_t>(ws, L.xq);
        gp.xsf = at<uint8_t>(ws, L.xsf);
        gp.H = d.H;
    }
    int rc = run_route(s, logits, shared_logit, ids, w, st, after_router && ev == nullptr, x_in_route ? &gp : nullptr);
    if (rc) return rc;
    if (!rec(ev, 1, st)) return MOE_ERR_CUDA;
    if ((rc = run_sort(s, ids, ws, st, ev == nullptr, after_router, true, w,
                       x_in_route ? at<float>(ws, L.row_w) : nullptr)))
        return rc;
    if (gathered) *gathered = x_in_route;
    return rec(ev, 2, st) ? MOE_OK : MOE_ERR_CUDA;
}

// gathered: the route + sort launch already quantised x (decode tilings).
// nv: the NVFP4 variant (128-row tiles only; null for MXFP8 x MXFP4).
// moe_layer_host at 128-row tiles: the host copies run on two more streams
// (one per direction: the host link is full duplex) in token chunks, so the
// x gather of each chunk starts as soon as its rows land and the output of
// each chunk leaves as soon as it is combined.
constexpr int kHostChunks = 8;

struct HostPipe {
    cudaStream_t cs;                      // host-to-device copies
    cudaStream_t ds;                      // device-to-host copies
    cudaEvent_t x_in[kHostChunks];        // chunk c of x has landed (recorded on cs)
    cudaEvent_t out_ready[kHostChunks];   // chunk c of the output is combined (recorded on the compute stream)
    uint16_t* out_host;
};

inline int chunk_begin(int T, int c) { return static_cast<int>(static_cast<int64_t>(T) * c / kHostChunks); }

int run_forward(const moe_shape* s, const uint16_t* x, const moe_weights* wt, const float* topk_w, void* ws,
                uint16_t* out, cudaStream_t st, bool pdl, void* const* ev = nullptr, bool gathered = false,
                const moe_nvfp4* nv = nullptr, const HostPipe* hp = nullptr) {
    const Dims d = make_dims(*s);
    const Layout L = make_layout(d);
    if (d.T == 0) {
        for (int i = 3; ev && i < 7; ++i)
            if (!rec(ev, i, st)) return MOE_ERR_CUDA;
        return MOE_OK;
    }
    const int nsm = num_sms_cached();
    if (nsm <= 0) return MOE_ERR_CUDA;

    GatherParams gp{};
    gp.x = x;
    gp.acc = at<float>(ws, L.acc);
    gp.header = at<int32_t>(ws, L.header);
    gp.a_map = at<int32_t>(ws, L.a_map);
    gp.xq = at<uint8_t>(ws, L.xq);
    gp.xsf = at<uint8_t>(ws, L.xsf);
    gp.topk_w = topk_w;
    gp.row_w = at<float>(ws, L.row_w);
    gp.c_map = at<int32_t>(ws, L.c_map);
    gp.offsets = at<int32_t>(ws, L.offsets);
    gp.vbase = at<int32_t>(ws, L.vbase);
    gp.token_order = L.x_token_order;
    gp.H = d.H;
    gp.T = d.T;
    gp.R_max = d.R_max;
    gp.max_blocks = L.x_token_order ? 16 * nsm : 8 * nsm * 8;
    gp.kp = d.kp;
    gp.B = d.B;
    gp.Et = d.Et;
    gp.xsf_tile_bytes = L.xsf_tile_bytes;
    // NVFP4: scale tiles of 1 KB per 128-K chunk (two 64-K halves)
    const int xsf_tile = nv ? 2 * L.xsf_tile_bytes : L.xsf_tile_bytes;
    const int asf_tile = nv ? 2 * L.asf_tile_bytes : L.asf_tile_bytes;
    cudaError_t e;
    if (nv) {
        gp.xsf_tile_bytes = xsf_tile;
        gp.x_gscale = nv->x_gscale;
        e = launch_gather_nvfp4(gp, st, pdl);
    } else {
        if (gathered) {
            e = cudaSuccess;
        } else if (hp && !L.x_token_order) {
            // token chunk c after its rows have landed
            e = cudaSuccess;
            for (int c = 0; c < kHostChunks && e == cudaSuccess; ++c) {
                gp.t0 = chunk_begin(d.T, c);
                gp.T = chunk_begin(d.T, c + 1);
                if (gp.T == gp.t0) continue;
                e = cudaStreamWaitEvent(st, hp->x_in[c], 0);
                if (e == cudaSuccess) e = launch_gather(gp, st, pdl);
            }
            gp.t0 = 0;
            gp.T = d.T;
        } else {
            e = launch_gather(gp, st, pdl);
        }
    }
    if (e != cudaSuccess || !rec(ev, 3, st)) return MOE_ERR_CUDA;

    // Tile-major packed weights viewed as rows of 128 E2M1 codes (64 bytes):
    // a GEMM stage is one 256-row box, one contiguous 16 KiB run of global
    // memory.  Token operands: boxes of B rows x 128 K of expert-ordered MXFP8
    // rows (the intermediate; x in the 128-row tiling -- the decode FC1
    // gathers its x rows itself).
    CUtensorMap mw1, mw2, mx, mact, my;
    const uint64_t Et = static_cast<uint64_t>(d.Et);
    if (nv) {
        // NVFP4: packed E2M1 rows of 64 bytes (128 K) with 64-byte swizzle, in
        // the weights (tile-major as for MXFP4), x and the intermediate
        constexpr CUtensorMapSwizzle kSw64 = CU_TENSOR_MAP_SWIZZLE_64B;
        if (!make_map(&mw1, CU_TENSOR_MAP_DATA_TYPE_UINT8, wt->w1, 64, Et * 2 * d.I * (d.H / 128), 64, 64, 256,
                      kSw64) ||
            !make_map(&mw2, CU_TENSOR_MAP_DATA_TYPE_UINT8, wt->w2, 64, Et * d.H * (d.I / 128), 64, 64, 256, kSw64) ||
            !make_map(&mact, CU_TENSOR_MAP_DATA_TYPE_UINT8, at<uint8_t>(ws, L.act), d.I / 2, d.rows_alloc, d.I / 2,
                      64, d.B, kSw64) ||
            !make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, at<uint8_t>(ws, L.xq), d.H / 2, d.rows_alloc, d.H / 2, 64,
                      d.B, kSw64))
            return MOE_ERR_CUDA;
    } else if (!make_map(&mw1, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, wt->w1, 128, Et * 2 * d.I * (d.H / 128),
                         kFp4BytesPer128Row, 128, 256) ||
               !make_map(&mw2, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, wt->w2, 128, Et * d.H * (d.I / 128),
                         kFp4BytesPer128Row, 128, 256) ||
               !make_map(&mact, CU_TENSOR_MAP_DATA_TYPE_UINT8, at<uint8_t>(ws, L.act), d.I, d.rows_alloc, d.I, 128,
                         d.B)) {
        return MOE_ERR_CUDA;
    }
    if (nv) {
        // x map made above
    } else if (L.x_token_order) {
        mx = mact;  // decode FC1 gathers its token rows with cp.async; the map is not read
    } else if (!make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, at<uint8_t>(ws, L.xq), d.H, d.rows_alloc, d.H, 128, d.B)) {
        return MOE_ERR_CUDA;
    }
    // bf16 FC2 rows (128-row tiling): each epilogue warp stores 32 rows x 64
    // columns per box
    if (L.y_bf16) {
        if (!make_map(&my, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, at<uint16_t>(ws, L.y), d.H, d.rows_alloc, d.H * 2, 64, 32))
            return MOE_ERR_CUDA;
    } else {
        my = mact;
    }

    GemmParams g{};
    g.header = at<int32_t>(ws, L.header);
    g.status = at<int32_t>(ws, L.header) + kHdrStatus;
    g.groups = at<int4>(ws, L.groups);
    g.vinfo = at<int4>(ws, L.vinfo);
    g.a_map = at<int32_t>(ws, L.a_map);
    g.topk_w = topk_w;
    g.row_w = at<float>(ws, L.row_w);
    g.act = at<uint8_t>(ws, L.act);
    g.act_sf = at<uint8_t>(ws, L.asf);
    g.y = L.y_bf16 ? nullptr : at<float>(ws, L.y);
    g.y_bf16 = L.y_bf16 ? at<uint16_t>(ws, L.y) : nullptr;
    g.H = d.H;
    g.I = d.I;
    g.out_sf_tile_bytes = asf_tile;
    g.a_tx_bytes = 256 * kFp4BytesPer128Row;
    g.wait_ns = kWaitLimitNs;
    g.act_kind = s->activation;
    g.max_v = d.V_max;
    g.xq = at<uint8_t>(ws, L.xq);
    g.xsf = at<uint8_t>(ws, L.xsf);
    g.kp = d.kp;
    g.act_c0 = s->act_params[0];
    g.act_c1 = s->act_params[1];
    g.test_stall_ns = g_test_stall_ns.load();
    g.acc = at<float>(ws, L.acc);
    g.T = d.T;
    if (nv) {
        g.nv = 1;
        g.nv_w_gs = nv->w1_gscale;
        g.nv_in_gs = nv->x_gscale;
        g.nv_out_gs = nv->h_gscale;
    }

    g.a_sf = wt->w1_sf;
    g.b_sf = L.x_token_order ? nullptr : at<uint8_t>(ws, L.xsf);
    g.b_sf_tile_bytes = L.x_token_order ? 0 : xsf_tile;
    // x scales at 128-row tiles, lane-major per tile: 16-byte cells (lane l,
    // chunk kc) at (l * chunks + kc) * 16 (NVFP4: the second 64-K half as
    // lanes 32..63), viewed as 4-D [tiles][32 or 64 lanes][chunks][16 bytes];
    // a stage reads the box of one chunk
    CUtensorMap mxs = my;
    const uint32_t sf_lanes = nv ? 64 : 32;
    if (!L.x_token_order && !make_map_4d(&mxs, at<uint8_t>(ws, L.xsf), 16, d.H / 128, sf_lanes,
                                         static_cast<uint64_t>(d.V_max), 1, sf_lanes, 1))
        return MOE_ERR_CUDA;
    e = launch_gemm(true, mw1, mx, mxs, g, d.B, nsm, st, pdl);
    if (e != cudaSuccess || !rec(ev, 4, st)) return MOE_ERR_CUDA;

    g.test_stall_ns = 0;  // the hook stalls FC1 only
    if (nv) {
        g.nv_w_gs = nv->w2_gscale;
        g.nv_in_gs = nv->h_gscale;
    }
    g.a_sf = wt->w2_sf;
    g.b_sf = at<uint8_t>(ws, L.asf);
    g.b_sf_tile_bytes = asf_tile;
    e = launch_gemm(false, mw2, mact, my, g, d.B, nsm, st, pdl);
    if (e != cudaSuccess || !rec(ev, 5, st)) return MOE_ERR_CUDA;

    CombineParams cp{at<int32_t>(ws, L.header), at<float>(ws, L.acc), at<int32_t>(ws, L.c_map),
                     L.y_bf16 ? nullptr : at<float>(ws, L.y),
                     L.y_bf16 ? at<uint16_t>(ws, L.y) : nullptr, out, d.T, d.kp, d.H};
    if (hp) {
        // token chunk c, then its output rows back to the host on the
        // device-to-host stream
        e = cudaSuccess;
        for (int c = 0; c < kHostChunks && e == cudaSuccess; ++c) {
            cp.t0 = chunk_begin(d.T, c);
            cp.T = chunk_begin(d.T, c + 1);
            if (cp.T == cp.t0) continue;
            e = launch_combine(cp, st, pdl);
            if (e == cudaSuccess) e = cudaEventRecord(hp->out_ready[c], st);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->ds, hp->out_ready[c], 0);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(hp->out_host + static_cast<size_t>(cp.t0) * d.H, out + static_cast<size_t>(cp.t0) * d.H,
                                    static_cast<size_t>(cp.T - cp.t0) * d.H * 2, cudaMemcpyDeviceToHost, hp->ds);
        }
    } else {
        e = launch_combine(cp, st, pdl);
    }
    if (e != cudaSuccess || !rec(ev, 6, st)) return MOE_ERR_CUDA;
    return MOE_OK;
}

// Router GEMM x [T, H] bf16 x wr [Eg, H] bf16 -> logits [T, Eg] fp32.  The
// status words are reset first (a copy node on the stream), so a timeout the
// router records survives until the sort that follows (keep_status).
int run_router(const moe_shape* s, const uint16_t* x, const uint16_t* wr, float* logits, void* ws, cudaStream_t st) {
    const Dims d = make_dims(*s);
    int32_t* status = at<int32_t>(ws, make_layout(d).header) + kHdrStatus;
    if (cudaMemsetAsync(status, 0, 2 * sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (d.T == 0) return MOE_OK;
    const int nsm = num_sms_cached();
    if (nsm <= 0) return MOE_ERR_CUDA;
    const RouterTiling t = router_tiling(d.T, d.Eg, nsm);
    CUtensorMap mx, mw;
    if (!make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, d.H, d.T, size_t(d.H) * 2, 64, 128) ||
        !make_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, wr, d.H, d.Eg, size_t(d.H) * 2, 64, t.N))
        return MOE_ERR_CUDA;
    RouterParams p{logits, status, d.T, d.Eg, d.H, t.N, t.n_tiles, t.ks, kWaitLimitNs};
    return cuda_rc(launch_router(mx, mw, p, t.grid, st, false));
}

int check_weights(const moe_weights* w) {
    if (!w || !w->w1 || !w->w1_sf || !w->w2 || !w->w2_sf) return MOE_ERR_NULL;
    if (!aligned(w->w1, 32) || !aligned(w->w2, 32) || !aligned(w->w1_sf, 16) || !aligned(w->w2_sf, 16))
        return MOE_ERR_ALIGN;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_is_supported(const moe_shape* s) {
    if (!s) return 0;
    const int64_t kp = static_cast<int64_t>(s->top_k) + s->num_shared;
    if (s->hidden <= 0 || s->hidden % 512 != 0) return 0;
    if (s->inter <= 0 || s->inter % 128 != 0) return 0;
    if (!(s->block_n == 16 || s->block_n == 32 || s->block_n == 128)) return 0;
    if (s->top_k < 1 || s->top_k > 32 || s->top_k > s->E_global || s->E_global > 1024) return 0;
    if (s->num_shared < 0 || s->num_shared > 1) return 0;
    if (s->E_local < 1 || s->E_local + s->num_shared > 1024) return 0;
    if (s->expert_offset < 0 || s->expert_offset + s->E_local > s->E_global) return 0;
    if (s->T < 0 || s->T > s->max_T || s->max_T < 1) return 0;
    if (static_cast<int64_t>(s->max_T) * kp >= (1 << 24)) return 0;
    const auto positive = [](float c) { return c > 0.f && c <= 3.0e38f; };  // finite and > 0
    if (s->activation == MOE_ACT_SWIGLU_CLAMP) {
        if (!positive(s->act_params[0])) return 0;
    } else if (s->activation == MOE_ACT_SITU) {
        if (!positive(s->act_params[0]) || !positive(s->act_params[1])) return 0;
    } else if (s->activation != MOE_ACT_SWIGLU) {
        return 0;
    }
    return 1;
}

int moe_workspace_bytes(const moe_shape* s, size_t* bytes) {
    if (!s || !bytes) return MOE_ERR_NULL;
    if (!moe_is_supported(s)) return MOE_ERR_SHAPE;
    *bytes = make_layout(make_dims(*s)).total;
    return MOE_OK;
}

int moe_quantize_mxfp4(const float* w, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales,
                       moe_stream_t stream) {
    if (!w || !codes || !scales) return MOE_ERR_NULL;
    if (rows <= 0 || K <= 0 || K % 32) return MOE_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(codes, 16)) return MOE_ERR_ALIGN;
    QuantParams p{w, codes, scales, rows, K};
    return cuda_rc(launch_quantize_mxfp4(p, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_packed_weight_bytes(int64_t experts, int64_t N, int64_t K, int32_t pair_halves, int32_t* block_rows,
                            size_t* code_bytes, size_t* scale_bytes) {
    (void)pair_halves;
    if (experts <= 0 || N <= 0 || K <= 0 || K % 128 || N % 256) return MOE_ERR_SHAPE;
    if (block_rows) *block_rows = 256;
    if (code_bytes) *code_bytes = static_cast<size_t>(experts) * N * (K / 2);
    if (scale_bytes) *scale_bytes = static_cast<size_t>(experts) * N * (K / 32);
    return MOE_OK;
}

int moe_pack_weights(const uint8_t* codes, const uint8_t* scales, int64_t experts, int64_t N, int64_t K,
                     int32_t pair_halves, uint8_t* packed_codes, uint8_t* packed_scales, moe_stream_t stream) {
    if (!codes || !scales || !packed_codes || !packed_scales) return MOE_ERR_NULL;
    int rc = moe_packed_weight_bytes(experts, N, K, pair_halves, nullptr, nullptr, nullptr);
    if (rc) return rc;
    if (!aligned(codes, 16) || !aligned(packed_codes, 16)) return MOE_ERR_ALIGN;
    PackParams p{codes, scales, packed_codes, packed_scales, experts, N, K, pair_halves ? 1 : 0};
    return cuda_rc(launch_pack_weights(p, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_route(const moe_shape* s, const float* logits, const uint16_t* shared_logit, int32_t* topk_ids,
              float* topk_w, moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (s->T > 0 && (!logits || !topk_ids || !topk_w || (s->num_shared > 0 && !shared_logit))) return MOE_ERR_NULL;
    return run_route(s, logits, shared_logit, topk_ids, topk_w, reinterpret_cast<cudaStream_t>(stream), false);
}

int moe_sort(const moe_shape* s, const int32_t* topk_ids, void* ws, size_t ws_bytes, moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (s->T > 0 && !topk_ids) return MOE_ERR_NULL;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    return run_sort(s, topk_ids, ws, reinterpret_cast<cudaStream_t>(stream), false);
}

int moe_forward(const moe_shape* s, const uint16_t* x, const moe_weights* w, const float* topk_w, void* ws,
                size_t ws_bytes, uint16_t* out, moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (s->T > 0 && (!x || !topk_w || !out)) return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
    if ((rc = check_weights(w))) return rc;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    return run_forward(s, x, w, topk_w, ws, out, reinterpret_cast<cudaStream_t>(stream), false);
}

int moe_layer(const moe_shape* s, const float* logits, const uint16_t* shared_logit, const uint16_t* x,
              const moe_weights* w, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, uint16_t* out,
              moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (s->T > 0 && (!logits || !x || !topk_ids || !topk_w || !out || (s->num_shared > 0 && !shared_logit)))
        return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
    if ((rc = check_weights(w))) return rc;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    bool gathered = false;
    if ((rc = run_route_sort(s, logits, shared_logit, topk_ids, topk_w, ws, st, nullptr, false, x, &gathered))) return rc;
    return run_forward(s, x, w, topk_w, ws, out, st, true, nullptr, gathered);
}

int moe_quantize_nvfp4(const float* w, int64_t experts, int64_t rows, int64_t K, float* gscale, uint8_t* codes,
                       uint8_t* scales, moe_stream_t stream) {
    if (!w || !gscale || !codes || !scales) return MOE_ERR_NULL;
    if (experts <= 0 || rows <= 0 || K <= 0 || K % 16) return MOE_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(codes, 8)) return MOE_ERR_ALIGN;
    NvQuantParams p{w, gscale, codes, scales, experts, rows, K};
    return cuda_rc(launch_quantize_nvfp4(p, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_pack_weights_nvfp4(const uint8_t* codes, const uint8_t* scales, int64_t experts, int64_t N, int64_t K,
                           int32_t pair_halves, uint8_t* packed_codes, uint8_t* packed_scales, moe_stream_t stream) {
    if (!codes || !scales || !packed_codes || !packed_scales) return MOE_ERR_NULL;
    if (experts <= 0 || N <= 0 || K <= 0 || K % 128 || N % 256) return MOE_ERR_SHAPE;
    if (!aligned(codes, 16) || !aligned(packed_codes, 16)) return MOE_ERR_ALIGN;
    PackParams p{codes, scales, packed_codes, packed_scales, experts, N, K, pair_halves ? 1 : 0};
    return cuda_rc(launch_pack_weights_nvfp4(p, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
int check_nvfp4(const moe_shape* s, const moe_nvfp4* nv) {
    if (!nv || !nv->w1_gscale || !nv->w2_gscale) return MOE_ERR_NULL;
    if (s->block_n != 128) return MOE_ERR_SHAPE;
    const auto positive = [](float c) { return c > 0.f && c <= 3.0e38f; };
    if (!positive(nv->x_gscale) || !positive(nv->h_gscale)) return MOE_ERR_SHAPE;
    if (!aligned(nv->w1_gscale, 4) || !aligned(nv->w2_gscale, 4)) return MOE_ERR_ALIGN;
    return MOE_OK;
}
}  // namespace

int moe_layer_nvfp4(const moe_shape* s, const moe_nvfp4* nv, const float* logits, const uint16_t* shared_logit,
                    const uint16_t* x, const moe_weights* w, int32_t* topk_ids, float* topk_w, void* ws,
                    size_t ws_bytes, uint16_t* out, moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if ((rc = check_nvfp4(s, nv))) return rc;
    if (s->T > 0 && (!logits || !x || !topk_ids || !topk_w || !out || (s->num_shared > 0 && !shared_logit)))
        return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
    if ((rc = check_weights(w))) return rc;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((rc = run_route_sort(s, logits, shared_logit, topk_ids, topk_w, ws, st, nullptr, false, nullptr, nullptr)))
        return rc;
    return run_forward(s, x, w, topk_w, ws, out, st, true, nullptr, false, nv);
}

int moe_layer_nvfp4_events(const moe_shape* s, const moe_nvfp4* nv, const float* logits,
                           const uint16_t* shared_logit, const uint16_t* x, const moe_weights* w, int32_t* topk_ids,
                           float* topk_w, void* ws, size_t ws_bytes, uint16_t* out, void* const* events,
                           moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if ((rc = check_nvfp4(s, nv))) return rc;
    if (!events) return MOE_ERR_NULL;
    for (int i = 0; i < 7; ++i)
        if (!events[i]) return MOE_ERR_NULL;
    if (s->T > 0 && (!logits || !x || !topk_ids || !topk_w || !out || (s->num_shared > 0 && !shared_logit)))
        return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
    if ((rc = check_weights(w))) return rc;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!rec(events, 0, st)) return MOE_ERR_CUDA;
    if ((rc = run_route_sort(s, logits, shared_logit, topk_ids, topk_w, ws, st, events, false, nullptr, nullptr)))
        return rc;
    return run_forward(s, x, w, topk_w, ws, out, st, false, events, false, nv);
}

int moe_router(const moe_shape* s, const uint16_t* x, const uint16_t* wr, float* logits, void* ws, size_t ws_bytes,
               moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (s->T > 0 && (!x || !wr || !logits)) return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(wr, 16) || !aligned(logits, 16)) return MOE_ERR_ALIGN;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    return run_router(s, x, wr, logits, ws, reinterpret_cast<cudaStream_t>(stream));
}

int moe_layer_router(const moe_shape* s, const uint16_t* wr, const uint16_t* shared_logit, const uint16_t* x,
                     const moe_weights* w, float* logits, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
                     uint16_t* out, moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (s->T > 0 && (!wr || !logits || !x || !topk_ids || !topk_w || !out || (s->num_shared > 0 && !shared_logit)))
        return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(wr, 16) || !aligned(logits, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
    if ((rc = check_weights(w))) return rc;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((rc = run_router(s, x, wr, logits, ws, st))) return rc;
    bool gathered = false;
    if ((rc = run_route_sort(s, logits, shared_logit, topk_ids, topk_w, ws, st, nullptr, true, x, &gathered))) return rc;
    return run_forward(s, x, w, topk_w, ws, out, st, true, nullptr, gathered);
}

int moe_layer_events(const moe_shape* s, const float* logits, const uint16_t* shared_logit, const uint16_t* x,
                     const moe_weights* w, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, uint16_t* out,
                     void* const* events, moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!events) return MOE_ERR_NULL;
    for (int i = 0; i < 7; ++i)
        if (!events[i]) return MOE_ERR_NULL;
    if (s->T > 0 && (!logits || !x || !topk_ids || !topk_w || !out || (s->num_shared > 0 && !shared_logit)))
        return MOE_ERR_NULL;
    if (!aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
    if ((rc = check_weights(w))) return rc;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!rec(events, 0, st)) return MOE_ERR_CUDA;
    bool gathered = false;
    if ((rc = run_route_sort(s, logits, shared_logit, topk_ids, topk_w, ws, st, events, false, x, &gathered))) return rc;
    return run_forward(s, x, w, topk_w, ws, out, st, false, events, gathered);
}

// The copy streams and events of moe_layer_host's pipelined form, one set per
// device, created on first use; calls enqueue under the mutex, so each wait
// refers to the record its own call just made.  With one stream per
// direction, a call's output copies and the input copies of a call on
// another caller stream (with its own workspace) share the link instead of
// queueing behind each other.
struct HostPipeRes {
    cudaStream_t cs = nullptr, ds = nullptr;
    cudaEvent_t start = nullptr, logits_in = nullptr, done = nullptr;
    cudaEvent_t x_in[kHostChunks] = {}, out_ready[kHostChunks] = {};
};
constexpr int kMaxPipeDevices = 64;
HostPipeRes g_pipe[kMaxPipeDevices];
std::mutex g_pipe_mu;

int pipe_resources(HostPipeRes** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxPipeDevices) return MOE_ERR_CUDA;
    HostPipeRes& r = g_pipe[dev];
    if (!r.cs) {
        auto mk = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
        bool ok = cudaStreamCreateWithFlags(&r.cs, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&r.ds, cudaStreamNonBlocking) == cudaSuccess && mk(&r.start) &&
                  mk(&r.logits_in) && mk(&r.done);
        for (int c = 0; ok && c < kHostChunks; ++c) ok = mk(&r.x_in[c]) && mk(&r.out_ready[c]);
        if (!ok) {
            r.cs = r.ds = nullptr;
            return MOE_ERR_CUDA;
        }
    }
    *out = &r;
    return MOE_OK;
}

int moe_layer_host(const moe_shape* s, const float* logits_host, const uint16_t* shared_logit_host,
                   const uint16_t* x_host, const moe_weights* w, void* ws, size_t ws_bytes, uint16_t* out_host,
                   moe_stream_t stream) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (s->T > 0 && (!logits_host || !x_host || !out_host || (s->num_shared > 0 && !shared_logit_host)))
        return MOE_ERR_NULL;
    if ((rc = check_weights(w))) return rc;
    if ((rc = check_ws(s, ws, ws_bytes))) return rc;
    const Dims d = make_dims(*s);
    const Layout L = make_layout(d);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* lg = at<float>(ws, L.st_logits);
    uint16_t* sl = at<uint16_t>(ws, L.st_shared);
    uint16_t* xd = at<uint16_t>(ws, L.st_x);
    uint16_t* od = at<uint16_t>(ws, L.st_out);
    int32_t* ids = at<int32_t>(ws, L.st_ids);
    float* tw = at<float>(ws, L.st_w);
    bool gathered = false;
    const size_t row_bytes = size_t(d.H) * 2;
    if (d.mode == kModePrefill && d.T > 0) {
        // Long batches: logits, then x in token chunks, on the host-to-device
        // stream (after the caller's stream reaches this call); routing
        // starts when the logits land, each chunk's gather when its rows
        // land; each chunk's output leaves on the device-to-host stream when
        // it is combined.  The caller's stream waits for the last output
        // copy.
        std::lock_guard<std::mutex> lock(g_pipe_mu);
        HostPipeRes* r = nullptr;
        if ((rc = pipe_resources(&r))) return rc;
        HostPipe hp{r->cs, r->ds, {}, {}, out_host};
        for (int c = 0; c < kHostChunks; ++c) {
            hp.x_in[c] = r->x_in[c];
            hp.out_ready[c] = r->out_ready[c];
        }
        bool ok = cudaEventRecord(r->start, st) == cudaSuccess && cudaStreamWaitEvent(r->cs, r->start, 0) == cudaSuccess &&
                  cudaMemcpyAsync(lg, logits_host, size_t(d.T) * d.Eg * 4, cudaMemcpyHostToDevice, r->cs) ==
                      cudaSuccess &&
                  (d.S == 0 || cudaMemcpyAsync(sl, shared_logit_host, size_t(d.T) * d.S * 2, cudaMemcpyHostToDevice,
                                               r->cs) == cudaSuccess) &&
                  cudaEventRecord(r->logits_in, r->cs) == cudaSuccess;
        for (int c = 0; ok && c < kHostChunks; ++c) {
            const int t0 = chunk_begin(d.T, c), t1 = chunk_begin(d.T, c + 1);
            if (t1 > t0)
                ok = cudaMemcpyAsync(xd + size_t(t0) * d.H, x_host + size_t(t0) * d.H, size_t(t1 - t0) * row_bytes,
                                     cudaMemcpyHostToDevice, r->cs) == cudaSuccess;
            ok = ok && cudaEventRecord(r->x_in[c], r->cs) == cudaSuccess;
        }
        if (!ok || cudaStreamWaitEvent(st, r->logits_in, 0) != cudaSuccess) return MOE_ERR_CUDA;
        if ((rc = run_route_sort(s, lg, d.S > 0 ? sl : nullptr, ids, tw, ws, st, nullptr, false, nullptr, &gathered)))
            return rc;
        if ((rc = run_forward(s, xd, w, tw, ws, od, st, true, nullptr, false, nullptr, &hp))) return rc;
        if (cudaEventRecord(r->done, r->ds) != cudaSuccess || cudaStreamWaitEvent(st, r->done, 0) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (cudaMemcpyAsync(lg, logits_host, size_t(d.T) * d.Eg * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (d.S > 0 &&
        cudaMemcpyAsync(sl, shared_logit_host, size_t(d.T) * d.S * 2, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemcpyAsync(xd, x_host, size_t(d.T) * row_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if ((rc = run_route_sort(s, lg, d.S > 0 ? sl : nullptr, ids, tw, ws, st, nullptr, false, xd, &gathered))) return rc;
    if ((rc = run_forward(s, xd, w, tw, ws, od, st, true, nullptr, gathered))) return rc;
    if (cudaMemcpyAsync(out_host, od, size_t(d.T) * row_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_get_views(const moe_shape* s, void* ws, moe_views* v) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!ws || !v) return MOE_ERR_NULL;
    const Dims d = make_dims(*s);
    const Layout L = make_layout(d);
    v->header = at<int32_t>(ws, L.header);
    v->expert_counts = at<int32_t>(ws, L.counts);
    v->expert_offsets = at<int32_t>(ws, L.offsets);
    v->vinfo = at<int32_t>(ws, L.vinfo);
    v->a_map = at<int32_t>(ws, L.a_map);
    v->c_map = at<int32_t>(ws, L.c_map);
    v->xq = at<uint8_t>(ws, L.xq);
    v->xq_sf = at<uint8_t>(ws, L.xsf);
    v->act = at<uint8_t>(ws, L.act);
    v->act_sf = at<uint8_t>(ws, L.asf);
    v->y = at<void>(ws, L.y);
    v->max_v = d.V_max;
    v->rows_alloc = d.rows_alloc;
    v->y_is_bf16 = L.y_bf16;
    v->sf_tile_bytes_x = L.xsf_tile_bytes;
    v->x_token_order = L.x_token_order;
    v->sf_tile_bytes_act = L.asf_tile_bytes;
    return MOE_OK;
}

int moe_get_status(const void* ws, int32_t* status, int32_t* detail) {
    if (!ws || !status || !detail) return MOE_ERR_NULL;
    int32_t h[2];
    if (cudaMemcpy(h, static_cast<const int32_t*>(ws) + kHdrStatus, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    *status = h[0];
    *detail = h[1];
    return MOE_OK;
}

int moe_set_gemm2_path(int32_t path) {
    if (path != MOE_GEMM2_AUTO && path != MOE_GEMM2_SPLIT && path != MOE_GEMM2_DENSE) return MOE_ERR_SHAPE;
    g_gemm2_path.store(path);
    return MOE_OK;
}

int moe_test_set_stall(uint64_t stall_ns) {
    g_test_stall_ns.store(stall_ns);
    return MOE_OK;
}

int moe_num_sms(int32_t* n) {
    if (!n) return MOE_ERR_NULL;
    *n = num_sms_cached();
    return *n > 0 ? MOE_OK : MOE_ERR_CUDA;
}

int moe_layer_launch_count(const moe_shape* s, int32_t* count) {
    int rc = check_shape(s);
    if (rc) return rc;
    if (!count) return MOE_ERR_NULL;
    const Dims d = make_dims(*s);
    const bool fused = route_sort_fusable(d.T, d.kp);
    int n = fused ? 1 : 1 + (sort_tokens_ok(d.T, d.kp, d.Et) ? 1 : sort_launch_count(static_cast<int64_t>(d.T) * d.kp));
    // [gather,] FC1, FC2, combine (the GEMM2 gate is decided inside the
    // sort); the decode tilings' x quantisation rides on the fused route +
    // sort up to 64 tokens, on the route launch up to 512
    const bool x_done = d.mode == kModeDecode && (fused ? route_sort_fuses_x(d.T) : sort_tokens_ok(d.T, d.kp, d.Et));
    if (d.T > 0) n += x_done ? 3 : 4;
    *count = n;
    return MOE_OK;
}

}  // extern "C"
