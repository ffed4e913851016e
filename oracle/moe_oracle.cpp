/*
 * CPU oracle for the fused MXFP4 Mixture-of-Experts layer forward.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  The GPU library shares no code with it:
 * every format, rounding rule and loop below is written out here from the
 * definitions, in fp64, slowly and plainly.
 *
 * Sources (page titles from the reference pages):
 *   [P1] "[sglang] Kimi-K3.1 MXFP4 decode MoE kernel generalised to shape
 *        templates" -- sections 1 (virtual experts: chunks of kBlockN rows per
 *        touched expert, bound E + T*top-k/kBlockN), 5 (routing: ids outside
 *        [expert_offset, expert_offset + E) get no row and expanded index -1;
 *        rows of an expert ordered by ascending token id).
 *   [P3] "[SGLang] CUTLASS MoE" -- structure diagram (route -> map -> quant ->
 *        GEMM1 (m*topk,k)x(E,k,2n) -> SiLU&Mul -> GEMM2 (m*topk,n)x(E,n,k) ->
 *        shuffle*mul*sum -> (m,k)), section 1 (prepare_moe_input: a_map input
 *        reorder, c_map output restore, expert_offsets start rows), section 4
 *        (silu_and_mul: SiLU of the first half times the second half),
 *        section 5 (apply_shuffle_mul_sum: un-permute, multiply by the routing
 *        weight, sum over top-k).
 *   [P1] section 4 (the FC1 epilogue's activation as a parameter: SiTU with
 *        constants beta and linear_beta, whose fixed form at beta 4, lb 25 is
 *        printed there, and the clamped SwiGLU with a limit).
 *   [P5] "[sglang] SGLang MoE shared expert: fuse 3 kernels into 1" -- the
 *        appended shared expert id N_BASE + s and its weight
 *        sigmoid(fp32(logit)) * scale.
 *   The MX element formats E2M1 / E4M3 and the E8M0 scale, and the MX
 *   conversion rule (shared exponent floor(log2 amax) - emax, elements rounded
 *   to nearest even with saturation) follow the OCP Microscaling Formats (MX)
 *   v1.0 specification, which the layer's MXFP4 weights / MXFP8 activations
 *   name.
 *
 * Conventions of this implementation (the readings of unstated points):
 *   - E2M1 codes are packed two per byte, element 2i in the low nibble.
 *   - W1 of an expert is [2I, H] with rows [0, I) = gate and [I, 2I) = up;
 *     W2 is [H, I].  One E8M0 scale per 32 consecutive K elements of a row.
 *   - topk ids are global expert ids; the shared expert s has id E_global + s
 *     and local index E_local + s.
 *   - Ranks inside an expert follow ascending slot index t*k' + j, which is
 *     ascending token id when a token picks an expert at most once.
 *   - SiTU<beta, lb>(g, u) = beta tanh(g/beta) sigmoid(g) * lb tanh(u/lb):
 *     the printed fixed form 2 tanh(g/4) (1 + tanh(g/2)) * 25 tanh(u/25)
 *     with 1 + tanh(g/2) = 2 sigmoid(g) and the constants generalised.
 *   - Clamped SwiGLU<L>(g, u) = silu(min(g, L)) * clamp(u, -L, L): the gate
 *     is capped above, the up projection on both sides.
 */
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

enum { FMT_E2M1 = 0, FMT_E4M3 = 1 };

/* ---------------------------------------------------------------- formats */

/* E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is
 * subnormal; no inf / NaN. */
double e2m1_value(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0 is
 * subnormal; S.1111.111 is NaN; no inf. */
double e4m3_value(int code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return std::nan("");
    double mag = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* E8M0: unsigned exponent, bias 127; 255 is NaN. */
double e8m0_value(int code) {
    if (code == 255) return std::nan("");
    return std::ldexp(1.0, code - 127);
}

int fmt_emax(int fmt) { return fmt == FMT_E2M1 ? 2 : 8; }
int fmt_ncodes(int fmt) { return fmt == FMT_E2M1 ? 8 : 127; } /* non-negative finite codes 0..n-1 */
int fmt_sign_bit(int fmt) { return fmt == FMT_E2M1 ? 0x8 : 0x80; }
double fmt_value(int fmt, int code) { return fmt == FMT_E2M1 ? e2m1_value(code) : e4m3_value(code); }

/* Nearest non-negative finite code to |q| (q finite); ties go to the even
 * code, which is the one with the even mantissa LSB.  Values beyond the
 * largest finite magnitude land on it (saturation). */
int nearest_code(int fmt, double aq) {
    int best = 0;
    double best_d = std::fabs(aq - fmt_value(fmt, 0));
    for (int c = 1; c < fmt_ncodes(fmt); ++c) {
        double d = std::fabs(aq - fmt_value(fmt, c));
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return best;
}

/* MX conversion of one block of n values (exact fp64 inputs).
 * Shared exponent e = floor(log2(amax)) - emax, clamped to [-127, 127], stored
 * as E8M0 code e + 127; amax == 0 gives code 0.  Each element is v * 2^-e
 * rounded to nearest even on the element grid, saturating; the sign of a
 * zero result is kept. */
void mx_quantize_block(const double* v, int n, int fmt, uint8_t* codes, uint8_t* scale_code) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(v[i]));
    int e = -127;
    if (amax > 0.0) {
        int ex;
        std::frexp(amax, &ex); /* amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1 */
        e = (ex - 1) - fmt_emax(fmt);
        e = std::min(127, std::max(-127, e));
    }
    *scale_code = (uint8_t)(e + 127);
    for (int i = 0; i < n; ++i) {
        double q = std::ldexp(v[i], -e);
        int c = nearest_code(fmt, std::fabs(q));
        if (std::signbit(v[i])) c |= fmt_sign_bit(fmt);
        codes[i] = (uint8_t)c;
    }
}

/* fp64 -> bf16 bits, round to nearest even (one rounding, from the exact
 * value).  bf16: 8 significant bits, exponent range of fp32. */
uint16_t bf16_rne(double d) {
    if (std::isnan(d)) return 0x7FC0;
    double a = std::fabs(d);
    uint16_t sign = std::signbit(d) ? 0x8000 : 0;
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else {
        int ex;
        std::frexp(a, &ex);                 /* a in [2^(ex-1), 2^ex) */
        int q = std::max(ex - 8, -133);     /* quantum: 8 bits, or the subnormal step 2^-133 */
        r = std::nearbyint(std::ldexp(a, -q)); /* default rounding mode: to nearest even */
        r = std::ldexp(r, q);
        if (r > 0x1.FEp127) return (uint16_t)(sign | 0x7F80); /* overflow to inf */
    }
    float f = (float)r; /* exact: r is a bf16 value */
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

/* Local expert index of a global id, or -1.  Shared experts sit after the
 * routed ones. */
enum { ACT_SWIGLU = 0, ACT_SWIGLU_CLAMP = 1, ACT_SITU = 2 };

double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }

/* The FC1 activation h(gate, up) in fp64 ([P3] section 4 for SwiGLU, [P1]
 * section 4 for the variants). */
double activation(int act, double c0, double c1, double g, double u) {
    if (act == ACT_SWIGLU_CLAMP) {
        double gc = g < c0 ? g : c0;
        double uc = u < -c0 ? -c0 : (u > c0 ? c0 : u);
        return gc * sigmoid(gc) * uc;
    }
    if (act == ACT_SITU) return c0 * std::tanh(g / c0) * sigmoid(g) * (c1 * std::tanh(u / c1));
    return g * sigmoid(g) * u;
}

int local_expert(int32_t id, int E_global, int E_local, int expert_offset, int S) {
    if (id >= E_global && id < E_global + S) return E_local + (id - E_global);
    if (id >= expert_offset && id < expert_offset + E_local) return id - expert_offset;
    return -1;
}

int e2m1_code_at(const uint8_t* packed_row, int64_t k) {
    uint8_t b = packed_row[k >> 1];
    return (k & 1) ? (b >> 4) : (b & 0xF);
}

/* Decode tables, filled once from the value functions above. */
struct Tables {
    double e2m1[16], e4m3[256], e8m0[256];
    Tables() {
        for (int c = 0; c < 16; ++c) e2m1[c] = e2m1_value(c);
        for (int c = 0; c < 256; ++c) {
            e4m3[c] = e4m3_value(c);
            e8m0[c] = e8m0_value(c);
        }
    }
};
const Tables& tables() {
    static const Tables t;
    return t;
}

/* Decode one MXFP4 row of K elements into fp64. */
void decode_mxfp4_row(const uint8_t* codes, const uint8_t* scales, int64_t K, double* out) {
    const Tables& tb = tables();
    for (int64_t k = 0; k < K; ++k) out[k] = tb.e2m1[e2m1_code_at(codes, k)] * tb.e8m0[scales[k / 32]];
}

/* ---------------------------------------------------------------- NVFP4
 * The FP4 path of "[SGLang] CUTLASS MoE", section 6 (cutlass_moe_fp4): E2M1
 * elements scaled in blocks of 16, with a per-tensor scale correcting the
 * narrow E2M1 range (FLOAT4_E2M1_MAX = 6).  Here: one positive E4M3 block
 * scale per 16 consecutive K elements and one fp32 global scale gs per
 * tensor (per expert matrix for the weights); value = e2m1 * e4m3 / gs.
 * Quantising a block of 16 takes every decision in fp32, the precision the
 * GPU kernels compute in:
 *   s  = fp32(fp32(amax * gs) / 6),  sf = E4M3 code nearest to s (ties to
 *        even, saturating at 448);
 *   dec(sf) == 0 (s underflows E4M3): every element is +0 or -0 by its sign;
 *   else r = fp32(gs / dec(sf)), q_i = E2M1 code nearest to fp32(v_i * r)
 *        (ties to even, saturating at 6), the sign of v_i kept.
 * A weight matrix's global scale is gs = fp32(2688 / amax) (2688 = 448 * 6:
 * the largest block scale times the largest element), 1 for a zero matrix. */
constexpr float kNvfp4Range = 2688.0f;

void nvfp4_quantize_block(const float* v, float gs, uint8_t* codes, uint8_t* sf_code) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(v[i]));
    const float sv = (amax * gs) / 6.0f;
    const int sf = nearest_code(FMT_E4M3, (double)sv);
    *sf_code = (uint8_t)sf;
    const float dsf = (float)e4m3_value(sf);
    for (int i = 0; i < 16; ++i) {
        int c = 0;
        if (dsf > 0.0f) {
            const float r = gs / dsf;
            const float q = v[i] * r;
            c = nearest_code(FMT_E2M1, std::fabs((double)q));
        }
        if (std::signbit(v[i])) c |= 0x8;
        codes[i] = (uint8_t)c;
    }
}

float nvfp4_global_scale(const float* w, int64_t n) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) amax = std::max(amax, std::fabs(w[i]));
    return amax > 0.0f ? kNvfp4Range / amax : 1.0f;
}

/* Decode one NVFP4 row of K elements (packed codes, one E4M3 per 16) into fp64. */
void decode_nvfp4_row(const uint8_t* codes, const uint8_t* scales, int64_t K, float gs, double* out) {
    const Tables& tb = tables();
    for (int64_t k = 0; k < K; ++k) out[k] = tb.e2m1[e2m1_code_at(codes, k)] * tb.e4m3[scales[k / 16]] / (double)gs;
}

}  // namespace

extern "C" {

/* ------------------------------------------------------------- exported */

double oracle_e2m1_value(int code) { return e2m1_value(code); }
double oracle_e4m3_value(int code) { return e4m3_value(code); }
double oracle_e8m0_value(int code) { return e8m0_value(code); }
uint16_t oracle_bf16_rne(double d) { return bf16_rne(d); }
/* The FC1 activation: act 0 SwiGLU, 1 clamped SwiGLU (c0 = limit), 2 SiTU
 * (c0 = beta, c1 = linear beta). */
double oracle_activation(int act, double c0, double c1, double g, double u) { return activation(act, c0, c1, g, u); }

/* One MX block; fmt 0 = E2M1, 1 = E4M3.  codes are one byte per element. */
void oracle_mx_quantize_block(const double* v, int n, int fmt, uint8_t* codes, uint8_t* scale_code) {
    mx_quantize_block(v, n, fmt, codes, scale_code);
}

/* Rows of fp32 values [rows, K] to MXFP4: packed codes [rows, K/2] (element
 * 2i in the low nibble) and E8M0 scales [rows, K/32].  K % 32 == 0. */
void oracle_quantize_mxfp4(const float* w, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales) {
    std::vector<double> v(32);
    std::vector<uint8_t> c(32);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < K / 32; ++b) {
            for (int i = 0; i < 32; ++i) v[i] = (double)w[r * K + b * 32 + i];
            mx_quantize_block(v.data(), 32, FMT_E2M1, c.data(), &scales[r * (K / 32) + b]);
            for (int i = 0; i < 32; i += 2)
                codes[r * (K / 2) + b * 16 + i / 2] = (uint8_t)(c[i] | (c[i + 1] << 4));
        }
    }
}

/* bf16 rows [rows, K] to MXFP8 E4M3: codes [rows, K], scales [rows, K/32]. */
void oracle_quantize_mxfp8_bf16(const uint16_t* x, int64_t rows, int64_t K, uint8_t* codes, uint8_t* scales) {
    std::vector<double> v(32);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < K / 32; ++b) {
            for (int i = 0; i < 32; ++i) v[i] = bf16_to_double(x[r * K + b * 32 + i]);
            mx_quantize_block(v.data(), 32, FMT_E4M3, &codes[r * K + b * 32], &scales[r * (K / 32) + b]);
        }
}

/* NVFP4 (see nvfp4_quantize_block).  One block of 16 fp32 values; codes one
 * byte per element. */
void oracle_nvfp4_quantize_block(const float* v, float gs, uint8_t* codes, uint8_t* sf_code) {
    nvfp4_quantize_block(v, gs, codes, sf_code);
}

/* Global scale of a weight matrix of n fp32 values: fp32(2688 / amax). */
float oracle_nvfp4_global_scale(const float* w, int64_t n) { return nvfp4_global_scale(w, n); }

/* Rows of fp32 values [rows, K] to NVFP4 with global scale gs: packed codes
 * [rows, K/2] (element 2i in the low nibble), E4M3 scales [rows, K/16].
 * K % 16 == 0. */
void oracle_quantize_nvfp4(const float* w, int64_t rows, int64_t K, float gs, uint8_t* codes, uint8_t* scales) {
    uint8_t c[16];
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < K / 16; ++b) {
            nvfp4_quantize_block(w + r * K + b * 16, gs, c, &scales[r * (K / 16) + b]);
            for (int i = 0; i < 16; i += 2) codes[r * (K / 2) + b * 8 + i / 2] = (uint8_t)(c[i] | (c[i + 1] << 4));
        }
}

/* bf16 rows [rows, K] to NVFP4 with global scale gs: codes one byte per
 * element [rows, K], E4M3 scales [rows, K/16]. */
void oracle_quantize_nvfp4_bf16(const uint16_t* x, int64_t rows, int64_t K, float gs, uint8_t* codes,
                                uint8_t* scales) {
    float v[16];
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < K / 16; ++b) {
            for (int i = 0; i < 16; ++i) v[i] = (float)bf16_to_double(x[r * K + b * 16 + i]);
            nvfp4_quantize_block(v, gs, &codes[r * K + b * 16], &scales[r * (K / 16) + b]);
        }
}

/* Router logits: logits[t][e] = fp32( sum_h x[t][h] * wr[e][h] ) with x bf16
 * [T, H] and wr bf16 [E_global, H] (row e holds expert e's router weights).
 * The bf16 products are exact in fp64; the fp64 sum is rounded to fp32 once.
 * (The router GEMM ahead of the routing step, whose output the pages' kernels
 * take as given: "... MXFP4 decode MoE ... shape templates", section 5
 * starts from the logits' top-k ids.) */
void oracle_router_logits(int T, int H, int E_global, const uint16_t* x, const uint16_t* wr, float* logits) {
    std::vector<double> xr(H), wrow(H);
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) xr[h] = bf16_to_double(x[(int64_t)t * H + h]);
        for (int e = 0; e < E_global; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h) acc += xr[h] * bf16_to_double(wr[(int64_t)e * H + h]);
            logits[(int64_t)t * E_global + e] = static_cast<float>(acc);
        }
    }
}

/* Top-k routing.  Per token: the k largest fp32 logits in descending order,
 * ties to the lower expert id; weights exp(l_j - m) / sum_sel exp(l_i - m),
 * which is softmax over all experts followed by renormalisation over the
 * selected ones.  With S shared experts, slots k..k+S-1 hold id E_global + s
 * and weight sigmoid(fp32(bf16 logit)) * scale.  ids [T, k+S], w [T, k+S]. */
void oracle_route(int T, int E_global, int k, const float* logits, int S, const uint16_t* shared_logit,
                  double shared_scale, int32_t* ids, double* w) {
    int kp = k + S;
    std::vector<char> taken(E_global);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (int64_t)t * E_global;
        std::fill(taken.begin(), taken.end(), 0);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E_global; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict: equal keeps the lower id */
            }
            taken[best] = 1;
            ids[t * kp + j] = best;
        }
        double m = (double)l[ids[t * kp]];
        double sum = 0.0;
        for (int j = 0; j < k; ++j) sum += std::exp((double)l[ids[t * kp + j]] - m);
        for (int j = 0; j < k; ++j) w[t * kp + j] = std::exp((double)l[ids[t * kp + j]] - m) / sum;
        for (int s = 0; s < S; ++s) {
            double x = bf16_to_double(shared_logit[t * S + s]);
            ids[t * kp + k + s] = E_global + s;
            w[t * kp + k + s] = shared_scale / (1.0 + std::exp(-x));
        }
    }
}

/* Token-to-expert sort.
 *   counts[e], e in [0, E_local + S): slots whose id maps to local expert e.
 *   offsets[e] = sum_{e' < e} counts[e'], offsets[E_local + S] = total rows.
 *   row of slot s (expert e) = offsets[e] + #{s' < s : slot s' maps to e}.
 *   c_map[s] = row or -1; a_map[row] = s.
 *   vinfo[v] = {e, first_row, tokens, chunk} for each chunk of B rows of each
 *   expert, experts ascending, chunks ascending.
 * Returns the number of virtual experts. */
int oracle_sort(int T, int kp, const int32_t* ids, int E_global, int E_local, int expert_offset, int S, int B,
                int32_t* counts, int32_t* offsets, int32_t* a_map, int32_t* c_map, int32_t* vinfo) {
    int Et = E_local + S;
    int64_t n = (int64_t)T * kp;
    std::vector<int> loc(n);
    for (int e = 0; e < Et; ++e) counts[e] = 0;
    for (int64_t s = 0; s < n; ++s) {
        loc[s] = local_expert(ids[s], E_global, E_local, expert_offset, S);
        if (loc[s] >= 0) counts[loc[s]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < Et; ++e) offsets[e + 1] = offsets[e] + counts[e];
    std::vector<int> seen(Et, 0);
    for (int64_t s = 0; s < n; ++s) {
        if (loc[s] < 0) {
            c_map[s] = -1;
            continue;
        }
        int row = offsets[loc[s]] + seen[loc[s]]++;
        c_map[s] = row;
        a_map[row] = (int32_t)s;
    }
    int nv = 0;
    for (int e = 0; e < Et; ++e)
        for (int c = 0; c * B < counts[e]; ++c) {
            vinfo[nv * 4 + 0] = e;
            vinfo[nv * 4 + 1] = offsets[e] + c * B;
            vinfo[nv * 4 + 2] = std::min(B, counts[e] - c * B);
            vinfo[nv * 4 + 3] = c;
            ++nv;
        }
    return nv;
}

/* Layer forward for a list of tokens.
 *
 * Inputs: x bf16 [T, H]; ids [T, k'] and w [T, k'] from routing; weights of
 * the local experts (E_local + S of them) given as compact arrays with
 * wmap[e] = index into them (-1 = not supplied, an error if needed):
 *   w1 codes [n, 2I, H/2], w1 scales [n, 2I, H/32],
 *   w2 codes [n, H, I/2],  w2 scales [n, H, I/32].
 * For each token t in toks[0..ntok):
 *   xq = MXFP8(x[t]);  for each slot j with a local expert e:
 *     G[r] = sum_h dec(xq[h]) dec(W1[e][r][h]),  U[r] = same with row I + r
 *     h[r] = act(G[r], U[r])             (SwiGLU: silu(g) u, silu(g) = g / (1 + exp(-g));
 *                                         the variants as in activation())
 *     hq = MXFP8(h);  Y[n] = sum_i dec(hq[i]) dec(W2[e][n][i])
 *     acc[n] += w[t,j] * Y[n]             (j ascending)
 *   out_f64[t] = acc, out_bf16[t] = bf16_rne(acc).
 * Optional outputs (may be NULL): act codes [ntok, k', I] and act scales
 * [ntok, k', I/32] (zero for non-local slots); xq codes [ntok, H], xq scales
 * [ntok, H/32]; y_slot [ntok, k', H] = w[t,j] * Y of each slot (the rows the
 * un-permute step sums; zero for non-local slots).  Returns 0, or -1 when a
 * needed expert is missing. */
int oracle_forward(int T, int H, int I, int kp, int E_global, int E_local, int expert_offset, int S,
                   const uint16_t* x, const int32_t* ids, const double* w, const int32_t* wmap,
                   const uint8_t* w1, const uint8_t* w1s, const uint8_t* w2, const uint8_t* w2s, int ntok,
                   const int32_t* toks, double* out_f64, uint16_t* out_bf16, uint8_t* act_codes,
                   uint8_t* act_scales, uint8_t* xq_codes, uint8_t* xq_scales, int act, double act_c0,
                   double act_c1, double* y_slot) {
    (void)T;
    std::vector<uint8_t> xq(H), xs(H / 32), hq(I), hs(I / 32);
    std::vector<double> xd(H), G(I), U(I), hv(I), hd(I), acc(H), Y(H), wg(H), wu(H), w2r(I);
    const Tables& tb = tables();
    for (int it = 0; it < ntok; ++it) {
        int t = toks[it];
        oracle_quantize_mxfp8_bf16(x + (int64_t)t * H, 1, H, xq.data(), xs.data());
        if (xq_codes) std::memcpy(xq_codes + (int64_t)it * H, xq.data(), H);
        if (xq_scales) std::memcpy(xq_scales + (int64_t)it * (H / 32), xs.data(), H / 32);
        for (int h = 0; h < H; ++h) xd[h] = tb.e4m3[xq[h]] * tb.e8m0[xs[h / 32]];
        std::fill(acc.begin(), acc.end(), 0.0);
        for (int j = 0; j < kp; ++j) {
            int64_t slot = (int64_t)t * kp + j;
            int e = local_expert(ids[slot], E_global, E_local, expert_offset, S);
            uint8_t* ac = act_codes ? act_codes + ((int64_t)it * kp + j) * I : nullptr;
            uint8_t* as = act_scales ? act_scales + ((int64_t)it * kp + j) * (I / 32) : nullptr;
            double* ys = y_slot ? y_slot + ((int64_t)it * kp + j) * H : nullptr;
            if (e < 0) {
                if (ac) std::memset(ac, 0, I);
                if (as) std::memset(as, 0, I / 32);
                if (ys) std::fill(ys, ys + H, 0.0);
                continue;
            }
            int wi = wmap[e];
            if (wi < 0) return -1;
            const uint8_t* W1 = w1 + (int64_t)wi * 2 * I * (H / 2);
            const uint8_t* W1s = w1s + (int64_t)wi * 2 * I * (H / 32);
            const uint8_t* W2 = w2 + (int64_t)wi * H * (I / 2);
            const uint8_t* W2s = w2s + (int64_t)wi * H * (I / 32);
            for (int r = 0; r < I; ++r) {
                decode_mxfp4_row(W1 + (int64_t)r * (H / 2), W1s + (int64_t)r * (H / 32), H, wg.data());
                decode_mxfp4_row(W1 + (int64_t)(I + r) * (H / 2), W1s + (int64_t)(I + r) * (H / 32), H, wu.data());
                double g = 0.0, u = 0.0;
                for (int h = 0; h < H; ++h) {
                    g += xd[h] * wg[h];
                    u += xd[h] * wu[h];
                }
                G[r] = g;
                U[r] = u;
                hv[r] = activation(act, act_c0, act_c1, g, u);
            }
            for (int b = 0; b < I / 32; ++b) mx_quantize_block(&hv[b * 32], 32, FMT_E4M3, &hq[b * 32], &hs[b]);
            if (ac) std::memcpy(ac, hq.data(), I);
            if (as) std::memcpy(as, hs.data(), I / 32);
            for (int i = 0; i < I; ++i) hd[i] = tb.e4m3[hq[i]] * tb.e8m0[hs[i / 32]];
            for (int n = 0; n < H; ++n) {
                decode_mxfp4_row(W2 + (int64_t)n * (I / 2), W2s + (int64_t)n * (I / 32), I, w2r.data());
                double y = 0.0;
                for (int i = 0; i < I; ++i) y += hd[i] * w2r[i];
                Y[n] = y;
            }
            for (int n = 0; n < H; ++n) acc[n] += w[slot] * Y[n];
            if (ys)
                for (int n = 0; n < H; ++n) ys[n] = w[slot] * Y[n];
        }
        for (int n = 0; n < H; ++n) {
            if (out_f64) out_f64[(int64_t)it * H + n] = acc[n];
            if (out_bf16) out_bf16[(int64_t)it * H + n] = bf16_rne(acc[n]);
        }
    }
    return 0;
}

/* The layer forward of the NVFP4 variant ("[SGLang] CUTLASS MoE", section 6:
 * the activations quantised with a global scale, grouped FP4 GEMMs, per-expert
 * alphas).  As oracle_forward, with NVFP4 in place of MXFP8 / MXFP4:
 *   xq = NVFP4(x[t], gs_x);   W1[e], W2[e] NVFP4 with global scales gs_w1[e],
 *   gs_w2[e] (packed codes [n, N, K/2], E4M3 scales [n, N, K/16]);
 *   G, U = sum_h dec(xq) dec(W1) in fp64, dec(v) = e2m1 * e4m3 / gs;
 *   h = act(G, U), rounded to fp32, hq = NVFP4(h, gs_h);
 *   Y = sum_i dec(hq) dec(W2);  out = bf16(sum_j w_j Y_j).
 * Optional outputs as in oracle_forward, with scales per 16 elements (act
 * scales [ntok, k', I/16], xq scales [ntok, H/16]). */
int oracle_forward_nvfp4(int T, int H, int I, int kp, int E_global, int E_local, int expert_offset, int S,
                         const uint16_t* x, const int32_t* ids, const double* w, const int32_t* wmap,
                         const uint8_t* w1, const uint8_t* w1s, const float* w1gs, const uint8_t* w2,
                         const uint8_t* w2s, const float* w2gs, float gs_x, float gs_h, int ntok, const int32_t* toks,
                         double* out_f64, uint16_t* out_bf16, uint8_t* act_codes, uint8_t* act_scales,
                         uint8_t* xq_codes, uint8_t* xq_scales, int act, double act_c0, double act_c1, double* y_slot) {
    (void)T;
    std::vector<uint8_t> xq(H), xs(H / 16), hq(I), hs(I / 16);
    std::vector<double> xd(H), hd(I), acc(H), Y(H), wg(H), wu(H), w2r(I);
    std::vector<float> hv(I);
    const Tables& tb = tables();
    for (int it = 0; it < ntok; ++it) {
        int t = toks[it];
        oracle_quantize_nvfp4_bf16(x + (int64_t)t * H, 1, H, gs_x, xq.data(), xs.data());
        if (xq_codes) std::memcpy(xq_codes + (int64_t)it * H, xq.data(), H);
        if (xq_scales) std::memcpy(xq_scales + (int64_t)it * (H / 16), xs.data(), H / 16);
        for (int h = 0; h < H; ++h) xd[h] = tb.e2m1[xq[h]] * tb.e4m3[xs[h / 16]] / (double)gs_x;
        std::fill(acc.begin(), acc.end(), 0.0);
        for (int j = 0; j < kp; ++j) {
            int64_t slot = (int64_t)t * kp + j;
            int e = local_expert(ids[slot], E_global, E_local, expert_offset, S);
            uint8_t* ac = act_codes ? act_codes + ((int64_t)it * kp + j) * I : nullptr;
            uint8_t* as = act_scales ? act_scales + ((int64_t)it * kp + j) * (I / 16) : nullptr;
            double* ys = y_slot ? y_slot + ((int64_t)it * kp + j) * H : nullptr;
            if (e < 0) {
                if (ac) std::memset(ac, 0, I);
                if (as) std::memset(as, 0, I / 16);
                if (ys) std::fill(ys, ys + H, 0.0);
                continue;
            }
            int wi = wmap[e];
            if (wi < 0) return -1;
            const uint8_t* W1 = w1 + (int64_t)wi * 2 * I * (H / 2);
            const uint8_t* W1s = w1s + (int64_t)wi * 2 * I * (H / 16);
            const uint8_t* W2 = w2 + (int64_t)wi * H * (I / 2);
            const uint8_t* W2s = w2s + (int64_t)wi * H * (I / 16);
            for (int r = 0; r < I; ++r) {
                decode_nvfp4_row(W1 + (int64_t)r * (H / 2), W1s + (int64_t)r * (H / 16), H, w1gs[wi], wg.data());
                decode_nvfp4_row(W1 + (int64_t)(I + r) * (H / 2), W1s + (int64_t)(I + r) * (H / 16), H, w1gs[wi],
                                 wu.data());
                double g = 0.0, u = 0.0;
                for (int h = 0; h < H; ++h) {
                    g += xd[h] * wg[h];
                    u += xd[h] * wu[h];
                }
                hv[r] = (float)activation(act, act_c0, act_c1, g, u);
            }
            for (int b = 0; b < I / 16; ++b) nvfp4_quantize_block(&hv[b * 16], gs_h, &hq[b * 16], &hs[b]);
            if (ac) std::memcpy(ac, hq.data(), I);
            if (as) std::memcpy(as, hs.data(), I / 16);
            for (int i = 0; i < I; ++i) hd[i] = tb.e2m1[hq[i]] * tb.e4m3[hs[i / 16]] / (double)gs_h;
            for (int n = 0; n < H; ++n) {
                decode_nvfp4_row(W2 + (int64_t)n * (I / 2), W2s + (int64_t)n * (I / 16), I, w2gs[wi], w2r.data());
                double y = 0.0;
                for (int i = 0; i < I; ++i) y += hd[i] * w2r[i];
                Y[n] = y;
            }
            for (int n = 0; n < H; ++n) acc[n] += w[slot] * Y[n];
            if (ys)
                for (int n = 0; n < H; ++n) ys[n] = w[slot] * Y[n];
        }
        for (int n = 0; n < H; ++n) {
            if (out_f64) out_f64[(int64_t)it * H + n] = acc[n];
            if (out_bf16) out_bf16[(int64_t)it * H + n] = bf16_rne(acc[n]);
        }
    }
    return 0;
}

}  // extern "C"
