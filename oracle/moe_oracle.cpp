// moe_oracle.cpp -- CPU oracle of the fine-grained fp8 MoE decode / verify layer.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the bench's CPU
// baseline load this file's library.  It shares no code, header, table or
// constant generator with the CUDA path; it is a plain, slow, step-by-step
// restatement of what the layer computes.
//
// Sources (web pages, cited by title and section):
//   [P1] openinfer #610 "TP8 span row mapping -- single-user speculative decode
//        at 186 tok/s": sections "What", "How", "Gates" (8-row block = 1
//        committed + 7 drafts; expert union; fixed-order reductions; pad rows
//        zero-filled, no NaN leak).
//   [P2] mstar #388 "Speed up GLM-5.2 with fp8 kernels and one-graph MTP":
//        the commit on kernel switches (router kernel, fused fp8 MoE decode
//        chain, the partials reduced once, "reference" per-expert dequant loop),
//        the commit on FlashInfer's block-scale GEMM (activations quantised to
//        e4m3 per 128 columns), the commit moving NoAuxTcRouter's top-k op.
//   [P4] MoE-Infinity #140 "converge spec-decode stack": commit list
//        (e_score_correction_bias; FP8 block dequant; expert tensors
//        [gate_proj, up_proj, down_proj]; 128x128 routed FP8 block scales).
//   [P5] pypto-serving #223 "DSpark speculation (K=7)": "What this adds"
//        (router gate cast to FP32; idle rows carry -1; 8-row verify window).
//
// The pages print no formulas.  Where they are silent the plainest reading is
// taken; each such reading is marked READING below.
//
// Precision: every step whose floating-point result decides an integer (router
// logits -> expert ids, activation quantisation -> e4m3 codes) runs in IEEE
// fp32 with an explicitly specified operation order, so that an fp32 kernel
// following the same order reproduces it bit for bit.  The expert GEMMs,
// SiLU and the combine accumulate in fp64 (template parameter Acc; fp32 is
// available for comparison).  Build with -ffp-contract=off: no silent fusing.
//
// Parity pins (tests/test_oracle_*.py): e4m3 decode against its closed form for
// all 256 codes and against torch.float8_e4m3fn; encoder against brute-force
// nearest-value search; own exp against math.exp; router logits against an
// fp64 dot product within the fp32 rounding bound; top-k against a library
// sort; union against a brute-force scan; expert FFN against an fp64 numpy
// matmul on library-dequantised weights; combine against closed forms (equal
// experts, zero rows, pads).  End-to-end layer values are pinned only through
// those parts: the pages print no worked example ("parity unpinned" for the
// absolute layer values as a whole).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

struct Cfg {
    int32_t hidden, inter, n_experts, n_groups, topk_groups, topk, n_shared;
    float routed_scaling;
};

constexpr int QB = 128;  // quantisation block (128 columns; 128x128 weight blocks)

// ---------------------------------------------------------------- formats --

float bits_to_f32(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
uint32_t f32_to_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }

// bf16 is the upper half of an fp32: widening is exact.
float bf16_to_f32(uint16_t b) { return bits_to_f32(uint32_t(b) << 16); }

// Round a double to bf16, round-to-nearest-even, directly (no detour through
// fp32, so no double rounding).  bf16 keeps 8 significant bits and the fp32
// exponent range; its smallest subnormal is 2^-133.
uint16_t f64_to_bf16(double v) {
    if (std::isnan(v)) return 0x7FC0;
    if (v == 0.0) return std::signbit(v) ? 0x8000 : 0x0000;
    int e2;
    std::frexp(v, &e2);                       // |v| in [2^(e2-1), 2^e2)
    int qexp = std::max(e2 - 8, -133);        // weight of the last kept bit
    double quantum = std::ldexp(1.0, qexp);
    double r = std::nearbyint(v / quantum) * quantum;   // exact scaling; RNE
    const double bf16_max = std::ldexp(255.0, 120);     // (2 - 2^-7) * 2^127
    if (std::fabs(r) > bf16_max) return std::signbit(v) ? 0xFF80 : 0x7F80;
    float f = static_cast<float>(r);          // exact: r is a bf16 value
    return static_cast<uint16_t>(f32_to_bits(f) >> 16);
}

// OCP FP8 E4M3 ("e4m3fn"): sign, 4 exponent bits with bias 7, 3 mantissa
// bits, no infinities, S.1111.111 is NaN, largest finite 448.  Decoded from
// the closed form of the format definition.
float e4m3_decode(uint8_t q) {
    int s = q >> 7, e = (q >> 3) & 0xF, m = q & 7;
    if (e == 15 && m == 7) return std::nanf("");
    double mag = (e == 0) ? std::ldexp(double(m), -9)          // m/8 * 2^-6
                          : std::ldexp(double(8 + m), e - 10); // (1+m/8) * 2^(e-7)
    return static_cast<float>(s ? -mag : mag);
}

// Nearest e4m3 value to an fp32 input, ties to even mantissa, saturating to
// +-448 (the "satfinite" conversion).  NaN stays NaN.
uint8_t e4m3_encode(float v) {
    if (std::isnan(v)) return 0x7F;
    uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
    double a = std::fabs(double(v));
    if (a >= 448.0) return sign | 0x7E;
    // Grid spacing: 2^-9 below the smallest normal 2^-6, else 2^(e-3) in
    // [2^e, 2^(e+1)).
    double quantum;
    if (a < std::ldexp(1.0, -6)) {
        quantum = std::ldexp(1.0, -9);
    } else {
        int e2;
        std::frexp(a, &e2);                   // a in [2^(e2-1), 2^e2)
        quantum = std::ldexp(1.0, (e2 - 1) - 3);
    }
    double count = std::nearbyint(a / quantum);   // RNE on the grid count
    double r = count * quantum;
    if (r > 448.0) r = 448.0;                 // rounding up past the top saturates
    if (r == 0.0) return sign;
    // Encode r exactly.
    if (r < std::ldexp(1.0, -6)) {            // subnormal: r = m * 2^-9
        return sign | static_cast<uint8_t>(std::ldexp(r, 9));
    }
    int e2;
    double f = std::frexp(r, &e2);            // r = f * 2^e2, f in [0.5, 1)
    int ex = (e2 - 1) + 7;                    // biased exponent
    int m = static_cast<int>(f * 16.0) - 8;   // f*16 in [8, 16)
    return sign | static_cast<uint8_t>((ex << 3) | m);
}

// ------------------------------------------------------------ own exp ----
// exp(a) by Cody-Waite range reduction (W. J. Cody and W. Waite, "Software
// Manual for the Elementary Functions", 1980) and the Taylor series of e^r to
// degree 7 in Horner form.  a = n*ln2 + r, |r| <~ ln2/2, e^a = 2^n * e^r.
// LN2_HI is ln2 cut to 16 significant bits so that n*LN2_HI is exact for
// |n| < 256; LN2_LO is fp32(ln2 - LN2_HI).  Coefficients are fp32(1/k!).
// The op sequence is part of the routing contract: the GPU router performs
// the same IEEE fp32 operations in the same order.
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e4p-1f;
constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
constexpr float kC2 = 0x1p-1f, kC3 = 0x1.555556p-3f, kC4 = 0x1.555556p-5f,
                kC5 = 0x1.111112p-7f, kC6 = 0x1.6c16c2p-10f, kC7 = 0x1.a01a02p-13f;

float own_exp(float a) {
    if (a != a) return a;
    if (a > 87.0f) a = 87.0f;                 // keep 2^n a normal number
    if (a < -87.0f) a = -87.0f;
    float n = std::nearbyintf(a * kLog2e);    // fp32 product, rounded to even integer
    float r = std::fmaf(-n, kLn2Hi, a);
    r = std::fmaf(-n, kLn2Lo, r);
    float p = kC7;
    p = std::fmaf(p, r, kC6);
    p = std::fmaf(p, r, kC5);
    p = std::fmaf(p, r, kC4);
    p = std::fmaf(p, r, kC3);
    p = std::fmaf(p, r, kC2);
    p = std::fmaf(p, r, 1.0f);
    p = std::fmaf(p, r, 1.0f);
    float two_n = bits_to_f32(static_cast<uint32_t>(static_cast<int32_t>(n) + 127) << 23);
    return p * two_n;
}

// Router score: sigma(l) = 1 / (1 + e^-l), IEEE fp32 add and divide.
float own_sigmoid(float l) { return 1.0f / (1.0f + own_exp(-l)); }

// --------------------------------------------------------- router GEMV ----
// logits[r,e] = sum_h x[r,h] * Wr[e,h] in fp32 (router gate kept in FP32:
// [P5] "What this adds"; the x row widened exactly from bf16).  The reduction
// order is fixed so that a kernel can reproduce it (fixed-order reductions,
// [P1] "Gates"):
//   * h is cut into chunks of 1024 (the last chunk may be shorter);
//   * inside chunk c, lane l in 0..31 owns h = c*1024 + 128*i + 4*l + j
//     (i ascending, then j = 0..3) and accumulates p[c][l] = fma(x, w, p)
//     sequentially from 0;
//   * per lane, q[l] = p[0][l], then q[l] = q[l] + p[c][l] for c = 1, 2, ...;
//   * the 32 lane values are combined by the butterfly v[l] = v[l] + v[l^d]
//     for d = 16, 8, 4, 2, 1; the result is v[0].
float router_dot(const uint16_t* x, const float* w, int H) {
    const int kChunk = 1024;
    float q[32];
    int nchunks = (H + kChunk - 1) / kChunk;
    for (int c = 0; c < nchunks; ++c) {
        int h_end = std::min(H, (c + 1) * kChunk);
        for (int l = 0; l < 32; ++l) {
            float p = 0.0f;
            for (int h0 = c * kChunk; h0 < h_end; h0 += 128)
                for (int j = 0; j < 4; ++j) {
                    int h = h0 + 4 * l + j;
                    p = std::fmaf(bf16_to_f32(x[h]), w[h], p);
                }
            q[l] = (c == 0) ? p : q[l] + p;
        }
    }
    for (int d = 16; d >= 1; d >>= 1) {
        float v[32];
        for (int l = 0; l < 32; ++l) v[l] = q[l] + q[l ^ d];
        std::memcpy(q, v, sizeof(q));
    }
    return q[0];
}

// ------------------------------------------------- grouped top-k routing ----
// Sigmoid scoring with a correction bias and grouped top-k, in the noaux_tc
// style that the router name NoAuxTcRouter ([P2]) and the parameter
// e_score_correction_bias ([P4]) point to.  READINGS:
//   * s = sigma(logit); b = s + bias is used for selection only;
//   * group score = sum of the two largest b in the group (the largest alone
//     when a group holds one expert);
//   * the topk_groups best groups are kept (score descending, lower group id
//     first on ties); the topk best experts inside them are chosen by b
//     descending, lower expert id first on ties, and listed in that order;
//   * weights w_k = (s_k / (s_0 + s_1 + ... + s_{K-1})) * routed_scaling,
//     the denominator summed in k order, IEEE divide then multiply;
//   * a pad row ([P5] idle rows carry -1) gets ids -1 and weights 0.
void route_row_from_logits(const Cfg& c, const float* logits, const float* bias,
                           int32_t* ids, float* wts) {
    const int E = c.n_experts, G = c.n_groups, epg = E / G, K = c.topk;
    std::vector<float> s(E), b(E);
    for (int e = 0; e < E; ++e) {
        s[e] = own_sigmoid(logits[e]);
        b[e] = s[e] + bias[e];
    }
    std::vector<float> gscore(G);
    for (int g = 0; g < G; ++g) {
        std::vector<float> v(b.begin() + g * epg, b.begin() + (g + 1) * epg);
        std::sort(v.begin(), v.end(), [](float p, float q) { return p > q; });
        gscore[g] = (epg >= 2) ? v[0] + v[1] : v[0];
    }
    std::vector<int> gorder(G);
    for (int g = 0; g < G; ++g) gorder[g] = g;
    std::stable_sort(gorder.begin(), gorder.end(),
                     [&](int p, int q) { return gscore[p] > gscore[q]; });
    std::vector<int> cand;
    for (int t = 0; t < c.topk_groups; ++t)
        for (int e = gorder[t] * epg; e < (gorder[t] + 1) * epg; ++e) cand.push_back(e);
    std::sort(cand.begin(), cand.end(), [&](int p, int q) {
        if (b[p] != b[q]) return b[p] > b[q];
        return p < q;
    });
    float den = s[cand[0]];
    for (int k = 1; k < K; ++k) den = den + s[cand[k]];
    for (int k = 0; k < K; ++k) {
        ids[k] = cand[k];
        wts[k] = (s[cand[k]] / den) * c.routed_scaling;
    }
}

// ------------------------------------------------ activation quantisation ----
// Per row, per 128 columns: amax = max |v|; scale = amax / 448 (1 when the
// block is all zeros, so no NaN); code = e4m3_rn_sat(v / scale).  READING of
// "quantizes the activations to e4m3 per 128 columns" ([P2], FlashInfer
// commit); fp32 divide, as the kernel does.
void quant_1x128(const float* v, int n, uint8_t* q, float* scale) {
    for (int b0 = 0; b0 < n; b0 += QB) {
        float amax = 0.0f;
        for (int i = b0; i < b0 + QB; ++i) amax = std::max(amax, std::fabs(v[i]));
        float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
        scale[b0 / QB] = s;
        for (int i = b0; i < b0 + QB; ++i) q[i] = e4m3_encode(v[i] / s);
    }
}

// Table of e4m3_decode over all 256 codes (filled from the closed form once).
const float* decode_table() {
    static const std::vector<float> t = [] {
        std::vector<float> v(256);
        for (int i = 0; i < 256; ++i) v[i] = e4m3_decode(static_cast<uint8_t>(i));
        return v;
    }();
    return t.data();
}

// Dequantised weight element: e4m3 code times its 128x128 block scale, in
// fp32 (READING: the scale multiplies; [P4] FP8 block dequant).
inline float wdeq(const float* lut, const uint8_t* q, const float* s, int ncols, int n, int k) {
    return lut[q[size_t(n) * ncols + k]] * s[size_t(n / QB) * (ncols / QB) + k / QB];
}

// ------------------------------------------------------------ expert FFN ----
// One expert on one row: g = x.Wg^T, u = x.Wu^T, h = silu(g) * u, h quantised
// per 1x128 like the activations, o = h.Wd^T.  x arrives quantised (codes +
// per-128 scales) and is dequantised to fp32 first.  Weights: gate/up [I,H],
// down [H,I], output-major ([P4] "[gate_proj, up_proj, down_proj]").
template <typename Acc>
void expert_ffn(const Cfg& c, const uint8_t* xq, const float* xs,
                const uint8_t* wg, const float* sg, const uint8_t* wu, const float* su,
                const uint8_t* wd, const float* sd, double* out, uint8_t* hq_out,
                float* hs_out) {
    const int H = c.hidden, I = c.inter;
    const float* lut = decode_table();
    std::vector<float> xd(H);
    for (int h = 0; h < H; ++h) xd[h] = e4m3_decode(xq[h]) * xs[h / QB];
    std::vector<float> hv(I);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < I; ++n) {
        Acc g = 0, u = 0;
        for (int k = 0; k < H; ++k) {
            g += Acc(xd[k]) * Acc(wdeq(lut, wg, sg, H, n, k));
            u += Acc(xd[k]) * Acc(wdeq(lut, wu, su, H, n, k));
        }
        double gd = double(g);
        double silu = gd / (1.0 + std::exp(-gd));
        hv[n] = static_cast<float>(silu * double(u));
    }
    std::vector<uint8_t> hq(I);
    std::vector<float> hs(I / QB);
    quant_1x128(hv.data(), I, hq.data(), hs.data());
    std::vector<float> hd(I);
    for (int n = 0; n < I; ++n) hd[n] = e4m3_decode(hq[n]) * hs[n / QB];
#pragma omp parallel for schedule(static)
    for (int m = 0; m < H; ++m) {
        Acc o = 0;
        for (int k = 0; k < I; ++k) o += Acc(hd[k]) * Acc(wdeq(lut, wd, sd, I, m, k));
        out[m] = double(o);
    }
    if (hq_out) std::memcpy(hq_out, hq.data(), I);
    if (hs_out) std::memcpy(hs_out, hs.data(), sizeof(float) * (I / QB));
}

// One expert on one row with 16-bit activations ("w8a16": mstar #388, commit
// on kernel switches and the FlashInfer commit -- fp8 weights, bf16
// activations at decode sizes; the activations are not quantised).  x is the
// row's bf16 values.  round16 != 0 (the w8a16 variant, READING of "w8a16"):
// every weight is dequantised to bf16, bf16_rne(e4m3(q) * s) from the exact
// product, and h = silu(g) * u is rounded to bf16 before the down GEMM (the
// down GEMM's activations are 16-bit too).  round16 == 0: weights e4m3(q) * s
// and h exact in fp64 -- the layer without any activation or weight rounding,
// the yardstick both variants' quantisation error is measured against.
template <typename Acc>
void expert_ffn_a16(const Cfg& c, const float* x, const uint8_t* wg, const float* sg,
                    const uint8_t* wu, const float* su, const uint8_t* wd, const float* sd,
                    double* out, bool round16) {
    const int H = c.hidden, I = c.inter;
    const float* lut = decode_table();
    auto w_at = [&](const uint8_t* q, const float* sc, int ncols, int n, int k) -> double {
        const double v = double(lut[q[size_t(n) * ncols + k]]) *
                         double(sc[size_t(n / QB) * (ncols / QB) + k / QB]);
        return round16 ? double(bf16_to_f32(f64_to_bf16(v))) : v;
    };
    std::vector<double> hv(I);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < I; ++n) {
        Acc g = 0, u = 0;
        for (int k = 0; k < H; ++k) {
            g += Acc(x[k]) * Acc(w_at(wg, sg, H, n, k));
            u += Acc(x[k]) * Acc(w_at(wu, su, H, n, k));
        }
        const double gd = double(g);
        const double hval = gd / (1.0 + std::exp(-gd)) * double(u);
        hv[n] = round16 ? double(bf16_to_f32(f64_to_bf16(hval))) : hval;
    }
#pragma omp parallel for schedule(static)
    for (int m = 0; m < H; ++m) {
        Acc o = 0;
        for (int k = 0; k < I; ++k) o += Acc(hv[k]) * Acc(w_at(wd, sd, I, m, k));
        out[m] = double(o);
    }
}

}  // namespace

// =================================================================== C ABI ==
extern "C" {

typedef struct {
    int32_t hidden, inter, n_experts, n_groups, topk_groups, topk, n_shared;
    float routed_scaling;
} orc_config;

static Cfg to_cfg(const orc_config* p) {
    return Cfg{p->hidden, p->inter, p->n_experts, p->n_groups, p->topk_groups,
               p->topk, p->n_shared, p->routed_scaling};
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

float orc_e4m3_decode(uint8_t q) { return e4m3_decode(q); }
uint8_t orc_e4m3_encode(float v) { return e4m3_encode(v); }
float orc_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }
uint16_t orc_f64_to_bf16(double v) { return f64_to_bf16(v); }
float orc_exp(float a) { return own_exp(a); }
float orc_sigmoid(float l) { return own_sigmoid(l); }

void orc_e4m3_encode_n(const float* v, int64_t n, uint8_t* q) {
    for (int64_t i = 0; i < n; ++i) q[i] = e4m3_encode(v[i]);
}

void orc_quant_1x128(const float* v, int32_t n, uint8_t* q, float* scale) {
    quant_1x128(v, n, q, scale);
}

// logits [R,E] fp32 from x bf16 [R,H] and Wr fp32 [E,H].
void orc_router_logits(const orc_config* cfg, const uint16_t* x, const float* wr,
                       int32_t R, float* logits) {
    Cfg c = to_cfg(cfg);
#pragma omp parallel for schedule(static) collapse(2)
    for (int r = 0; r < R; ++r)
        for (int e = 0; e < c.n_experts; ++e)
            logits[size_t(r) * c.n_experts + e] =
                router_dot(x + size_t(r) * c.hidden, wr + size_t(e) * c.hidden, c.hidden);
}

// Routing from given logits; row_valid NULL = every row valid.
void orc_route_from_logits(const orc_config* cfg, const float* logits, const float* bias,
                           const uint8_t* row_valid, int32_t R, int32_t* ids, float* wts) {
    Cfg c = to_cfg(cfg);
    for (int r = 0; r < R; ++r) {
        int32_t* id = ids + size_t(r) * c.topk;
        float* w = wts + size_t(r) * c.topk;
        if (row_valid && !row_valid[r]) {
            for (int k = 0; k < c.topk; ++k) { id[k] = -1; w[k] = 0.0f; }
            continue;
        }
        route_row_from_logits(c, logits + size_t(r) * c.n_experts, bias, id, w);
    }
}

void orc_route(const orc_config* cfg, const uint16_t* x, const float* wr, const float* bias,
               const uint8_t* row_valid, int32_t R, int32_t* ids, float* wts, float* logits_out) {
    Cfg c = to_cfg(cfg);
    std::vector<float> logits(size_t(R) * c.n_experts, 0.0f);
#pragma omp parallel for schedule(static)
    for (int r = 0; r < R; ++r) {
        if (row_valid && !row_valid[r]) continue;   // a pad row is not routed
        for (int e = 0; e < c.n_experts; ++e)
            logits[size_t(r) * c.n_experts + e] =
                router_dot(x + size_t(r) * c.hidden, wr + size_t(e) * c.hidden, c.hidden);
    }
    orc_route_from_logits(cfg, logits.data(), bias, row_valid, R, ids, wts);
    if (logits_out) std::memcpy(logits_out, logits.data(), sizeof(float) * logits.size());
}

// Deduplicated expert union and dispatch order ([P1] "What": the union phase;
// the verify block's per-token union of routed experts, [P4]).  Definition:
//   counts[e]  = number of valid (row, k) slots routed to expert e, e < E;
//   counts[E]  = number of valid rows (the shared expert sees every one);
//   offsets    = exclusive prefix of counts, E+2 entries, experts ascending,
//                the shared expert last;
//   inside an expert, slots are placed in (row, k) order; shared rows in row
//   order;
//   pos[r*(K+1)+k] = gathered position of slot (r,k), k = K the shared slot;
//                -1 for pad rows;
//   src[p]     = r*(K+1)+k of gathered position p;
//   ulist      = experts with counts > 0, ascending, then E; *n_union = their
//                number (shared excluded).
void orc_build_union(const orc_config* cfg, const int32_t* ids, int32_t R, int32_t* counts,
                     int32_t* offsets, int32_t* ulist, int32_t* n_union, int32_t* pos,
                     int32_t* src) {
    Cfg c = to_cfg(cfg);
    const int E = c.n_experts, K = c.topk, KS = K + 1;
    std::vector<uint8_t> valid(R, 0);
    for (int r = 0; r < R; ++r) valid[r] = ids[size_t(r) * K] >= 0;
    for (int e = 0; e <= E; ++e) counts[e] = 0;
    for (int r = 0; r < R; ++r) {
        if (!valid[r]) continue;
        for (int k = 0; k < K; ++k) counts[ids[size_t(r) * K + k]] += 1;
        counts[E] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e <= E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    std::vector<int32_t> fill(offsets, offsets + E + 1);
    for (int r = 0; r < R; ++r) {
        for (int k = 0; k < KS; ++k) pos[size_t(r) * KS + k] = -1;
        if (!valid[r]) continue;
        for (int k = 0; k < K; ++k) {
            int e = ids[size_t(r) * K + k];
            int p = fill[e]++;
            pos[size_t(r) * KS + k] = p;
            src[p] = r * KS + k;
        }
    }
    for (int r = 0; r < R; ++r) {
        if (!valid[r]) continue;
        int p = fill[E]++;
        pos[size_t(r) * KS + K] = p;
        src[p] = r * KS + K;
    }
    int u = 0;
    for (int e = 0; e < E; ++e)
        if (counts[e] > 0) ulist[u++] = e;
    *n_union = u;
    ulist[u] = E;
}

// One expert on one row (see expert_ffn).  acc64 != 0: fp64 accumulation.
void orc_expert_ffn(const orc_config* cfg, const uint8_t* xq, const float* xs,
                    const uint8_t* wg, const float* sg, const uint8_t* wu, const float* su,
                    const uint8_t* wd, const float* sd, double* out, uint8_t* hq_out,
                    float* hs_out, int32_t acc64) {
    Cfg c = to_cfg(cfg);
    if (acc64)
        expert_ffn<double>(c, xq, xs, wg, sg, wu, su, wd, sd, out, hq_out, hs_out);
    else
        expert_ffn<float>(c, xq, xs, wg, sg, wu, su, wd, sd, out, hq_out, hs_out);
}

// One expert on one bf16 row with 16-bit activations (see expert_ffn_a16):
// round16 != 0 the w8a16 variant, 0 the unrounded yardstick.
void orc_expert_ffn_a16(const orc_config* cfg, const uint16_t* x_bf16, const uint8_t* wg,
                        const float* sg, const uint8_t* wu, const float* su, const uint8_t* wd,
                        const float* sd, double* out, int32_t round16, int32_t acc64) {
    Cfg c = to_cfg(cfg);
    std::vector<float> xf(c.hidden);
    for (int h = 0; h < c.hidden; ++h) xf[h] = bf16_to_f32(x_bf16[h]);
    if (acc64)
        expert_ffn_a16<double>(c, xf.data(), wg, sg, wu, su, wd, sd, out, round16 != 0);
    else
        expert_ffn_a16<float>(c, xf.data(), wg, sg, wu, su, wd, sd, out, round16 != 0);
}

// The whole layer on the rows listed in `rows` (all R rows when rows == NULL).
// Weights: routed gate/up [E,I,H] with scales [E,I/128,H/128], down [E,H,I]
// with scales [E,H/128,I/128]; the shared expert(s) in the same layout with
// n_shared in place of E.  Per row r:
//   1. route (ids, weights) from fp32 logits, as above;
//   2. quantise x[r] per 1x128 (the same codes feed every expert);
//   3. o_k = expert_ffn(ids[k]) for k = 0..K-1 and o_s = shared expert(s);
//   4. y = bf16_rne( ((w_0*o_0 + w_1*o_1) + ... + w_{K-1}*o_{K-1}) + o_s ),
//      the weighted sum in k order, the shared term(s) added last with
//      weight 1 ([P1] "fixed-order reductions"; [P2] routed and shared
//      experts of one layer);
//   5. a pad row (row_valid[r] == 0) gives +0.0 everywhere whatever x holds
//      ([P1] "Span pad ranks zero-fill ... no NaN leaks").
// Outputs: out_bf16 [R,H]; ids/wts [R,K]; y_acc [R,H] fp64 (nullable): the
// value before the bf16 rounding.
// variant: 0 = fp8 (the layer above), 1 = w8a16, 2 = no activation or weight
// rounding (see expert_ffn_a16); routing and combine are the same in all three.
void orc_moe_layer_variant(const orc_config* cfg, const uint16_t* x, const float* wr,
                           const float* bias, const uint8_t* w_gate, const float* s_gate,
                           const uint8_t* w_up, const float* s_up, const uint8_t* w_down,
                           const float* s_down, const uint8_t* sh_gate, const float* sh_s_gate,
                           const uint8_t* sh_up, const float* sh_s_up, const uint8_t* sh_down,
                           const float* sh_s_down, const uint8_t* row_valid, int32_t R,
                           const int32_t* rows, int32_t n_rows, uint16_t* out_bf16,
                           int32_t* ids_out, float* wts_out, double* y_acc, int32_t acc64,
                           int32_t variant) {
    Cfg c = to_cfg(cfg);
    const int H = c.hidden, I = c.inter, K = c.topk;
    const size_t gsz = size_t(I) * H;                    // elements per gate/up/down
    const size_t gss = size_t(I / QB) * (H / QB);        // scales per tensor
    std::vector<int32_t> all;
    if (!rows) {
        all.resize(R);
        for (int r = 0; r < R; ++r) all[r] = r;
        rows = all.data();
        n_rows = R;
    }
    std::vector<double> o(H), acc(H);
    std::vector<float> xf(H), xs(H / QB);
    std::vector<uint8_t> xq(H);
    for (int t = 0; t < n_rows; ++t) {
        const int r = rows[t];
        uint16_t* yrow = out_bf16 + size_t(r) * H;
        int32_t* id = ids_out + size_t(r) * K;
        float* w = wts_out + size_t(r) * K;
        if (row_valid && !row_valid[r]) {
            for (int h = 0; h < H; ++h) yrow[h] = 0x0000;
            for (int k = 0; k < K; ++k) { id[k] = -1; w[k] = 0.0f; }
            if (y_acc) for (int h = 0; h < H; ++h) y_acc[size_t(r) * H + h] = 0.0;
            continue;
        }
        const uint16_t* xr = x + size_t(r) * H;
        std::vector<float> logits(c.n_experts);
#pragma omp parallel for schedule(static)
        for (int e = 0; e < c.n_experts; ++e)
            logits[e] = router_dot(xr, wr + size_t(e) * H, H);
        route_row_from_logits(c, logits.data(), bias, id, w);
        for (int h = 0; h < H; ++h) xf[h] = bf16_to_f32(xr[h]);
        quant_1x128(xf.data(), H, xq.data(), xs.data());
        auto ffn = [&](const uint8_t* g_, const float* sg_, const uint8_t* u_, const float* su_,
                       const uint8_t* d_, const float* sd_) {
            if (variant == 0)
                orc_expert_ffn(cfg, xq.data(), xs.data(), g_, sg_, u_, su_, d_, sd_, o.data(),
                               nullptr, nullptr, acc64);
            else if (acc64)
                expert_ffn_a16<double>(c, xf.data(), g_, sg_, u_, su_, d_, sd_, o.data(),
                                       variant == 1);
            else
                expert_ffn_a16<float>(c, xf.data(), g_, sg_, u_, su_, d_, sd_, o.data(),
                                      variant == 1);
        };
        for (int k = 0; k < K; ++k) {
            const size_t e = size_t(id[k]);
            ffn(w_gate + e * gsz, s_gate + e * gss, w_up + e * gsz, s_up + e * gss,
                w_down + e * gsz, s_down + e * gss);
            for (int h = 0; h < H; ++h)
                acc[h] = (k == 0) ? double(w[k]) * o[h] : acc[h] + double(w[k]) * o[h];
        }
        for (int sidx = 0; sidx < c.n_shared; ++sidx) {
            const size_t e = size_t(sidx);
            ffn(sh_gate + e * gsz, sh_s_gate + e * gss, sh_up + e * gsz, sh_s_up + e * gss,
                sh_down + e * gsz, sh_s_down + e * gss);
            for (int h = 0; h < H; ++h) acc[h] = acc[h] + o[h];
        }
        for (int h = 0; h < H; ++h) yrow[h] = f64_to_bf16(acc[h]);
        if (y_acc) std::memcpy(y_acc + size_t(r) * H, acc.data(), sizeof(double) * H);
    }
}

void orc_moe_layer(const orc_config* cfg, const uint16_t* x, const float* wr, const float* bias,
                   const uint8_t* w_gate, const float* s_gate, const uint8_t* w_up,
                   const float* s_up, const uint8_t* w_down, const float* s_down,
                   const uint8_t* sh_gate, const float* sh_s_gate, const uint8_t* sh_up,
                   const float* sh_s_up, const uint8_t* sh_down, const float* sh_s_down,
                   const uint8_t* row_valid, int32_t R, const int32_t* rows, int32_t n_rows,
                   uint16_t* out_bf16, int32_t* ids_out, float* wts_out, double* y_acc,
                   int32_t acc64) {
    orc_moe_layer_variant(cfg, x, wr, bias, w_gate, s_gate, w_up, s_up, w_down, s_down, sh_gate,
                          sh_s_gate, sh_up, sh_s_up, sh_down, sh_s_down, row_valid, R, rows,
                          n_rows, out_bf16, ids_out, wts_out, y_acc, acc64, 0);
}

// ------------------------------------------------- greedy verify + accept ----
// Speculative verify of spans of 8 rows (openinfer #610 "What": 1 committed
// token + up to 7 drafts per span; pypto-serving #223 "What this adds": accept
// the longest matching prefix plus the bonus prediction, 1..8 tokens per step;
// mstar #388: greedy verify run on the device).  Span q covers rows
// 8q .. 8q+7; row 0 of the span holds the committed token's position, row j
// (1 <= j <= n_draft[q]) the j-th draft.  The target's greedy token at row j is
// argmax_v logits[8q+j, v] (ties to the lower index) and predicts the token
// after row j.  Draft j (draft[8q+j]) is accepted when every draft before it
// was and draft[8q+j] == argmax(row j-1).  With m drafts accepted the span
// emits draft_1 .. draft_m and then the bonus argmax(row m): accept_len = m+1
// tokens, out[8q .. 8q+m], the rest of the span's out set to -1.
// logits_is_bf16 != 0: logits are bf16 bit patterns, else fp32.
void orc_greedy_verify(const void* logits, int32_t logits_is_bf16, int32_t V,
                       const int32_t* draft, const int32_t* n_draft, int32_t n_span,
                       int32_t* accept_len, int32_t* out, int32_t* argmax_out) {
    const int S = 8;
    std::vector<int32_t> am(size_t(n_span) * S);
    // argmax: the first index of the largest value; NaN never wins (a row of
    // NaN gives index 0).  READING: the pages do not say how ties or NaN are
    // treated; the first maximal index is numpy's and torch's CPU convention.
    for (int r = 0; r < n_span * S; ++r) {
        int best = -1;
        float bv = 0.0f;
        for (int v = 0; v < V; ++v) {
            float x = logits_is_bf16
                          ? bf16_to_f32(static_cast<const uint16_t*>(logits)[size_t(r) * V + v])
                          : static_cast<const float*>(logits)[size_t(r) * V + v];
            if (std::isnan(x)) continue;
            if (best < 0 || x > bv) {
                bv = x;
                best = v;
            }
        }
        am[r] = best < 0 ? 0 : best;
        if (argmax_out) argmax_out[r] = am[r];
    }
    for (int q = 0; q < n_span; ++q) {
        const int nd = std::max(0, std::min(S - 1, int(n_draft[q])));
        int m = 0;
        while (m < nd && draft[q * S + m + 1] == am[q * S + m]) ++m;
        for (int j = 0; j < S; ++j) out[q * S + j] = -1;
        for (int j = 0; j < m; ++j) out[q * S + j] = draft[q * S + j + 1];
        out[q * S + m] = am[q * S + m];
        accept_len[q] = m + 1;
    }
}

// ------------------------------------------------ residual add + RMSNorm ----
// The MoE output feeds the next layer through the residual stream and its
// RMSNorm (mstar #388, commit on kernel switches: the MoE's partials reduced
// once, fused with the next add + RMSNorm; the decoder layer's
// residual + mlp(norm(...)) in the review thread).  READING, per valid row:
//   z = residual + y          (y the layer's combine sum before rounding)
//   residual_out = bf16_rne(z)
//   normed = bf16_rne(z / sqrt(mean_h(z^2) + eps) * gamma)
// computed in fp64 from the inputs; pad rows give +0.0 in both outputs.
void orc_add_rmsnorm(const double* y, const uint16_t* residual, const float* gamma, float eps,
                     const uint8_t* row_valid, int32_t R, int32_t H, uint16_t* residual_out,
                     uint16_t* normed) {
    std::vector<double> z(H);
    for (int r = 0; r < R; ++r) {
        uint16_t* ro = residual_out + size_t(r) * H;
        uint16_t* no = normed + size_t(r) * H;
        if (row_valid && !row_valid[r]) {
            for (int h = 0; h < H; ++h) ro[h] = no[h] = 0;
            continue;
        }
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            z[h] = double(bf16_to_f32(residual[size_t(r) * H + h])) + y[size_t(r) * H + h];
            ss += z[h] * z[h];
        }
        const double inv = 1.0 / std::sqrt(ss / H + double(eps));
        for (int h = 0; h < H; ++h) {
            ro[h] = f64_to_bf16(z[h]);
            no[h] = f64_to_bf16(z[h] * inv * double(gamma[h]));
        }
    }
}

}  // extern "C"
