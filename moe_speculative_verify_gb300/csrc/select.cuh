// select.cuh -- sigmoid scores and grouped top-k of one router row, one warp
// (sm_103a).  Included by the stand-alone selection kernel and by the fused
// selection + union kernel, so both take the same decisions by the same code.
//
// The router of a sigmoid-scored, bias-corrected, group-limited MoE (mstar
// #388 "Speed up GLM-5.2 with fp8 kernels and one-graph MTP", commit moving
// NoAuxTcRouter's top-k op; MoE-Infinity #140, e_score_correction_bias).
// Every floating-point step is an explicitly rounded IEEE fp32 operation; all
// reductions are exact comparisons, so their order does not matter.
#pragma once

#include "common.cuh"

namespace moe {

// exp by Cody-Waite range reduction (Cody and Waite, "Software Manual for the
// Elementary Functions", 1980): a = n*ln2 + r with ln2 split into a head of 16
// significant bits (n*head exact) and an fp32 tail, then the Taylor series of
// e^r to degree 7 in Horner form, then scaling by 2^n through the exponent
// field.  Argument clamped to [-87, 87] so 2^n stays a normal number.
__device__ __forceinline__ float cw_exp(float a) {
    const float kLog2e = 0x1.715476p+0f;
    const float kLn2Hi = 0x1.62e4p-1f;
    const float kLn2Lo = 0x1.7f7d1cp-20f;
    if (a != a) return a;
    if (a > 87.0f) a = 87.0f;
    if (a < -87.0f) a = -87.0f;
    const float n = rintf(__fmul_rn(a, kLog2e));
    float r = __fmaf_rn(-n, kLn2Hi, a);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = 0x1.a01a02p-13f;              // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);   // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);    // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);    // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);    // 1/3!
    p = __fmaf_rn(p, r, 0x1p-1f);           // 1/2!
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
    return __fmul_rn(p, two_n);
}

__device__ __forceinline__ float router_sigmoid(float l) {
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, cw_exp(-l)));
}

// Total order of fp32 values as unsigned keys (-0 folded onto +0).
__device__ __forceinline__ uint32_t ordered_key(float f) {
    if (f == 0.0f) f = 0.0f;
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Larger value first; on equal values the lower index wins.
__device__ __forceinline__ uint64_t rank_key(float v, int idx) {
    return (static_cast<uint64_t>(ordered_key(v)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

constexpr int kSelPer = MOE_MAX_EXPERTS / 32;   // experts per lane

// One warp selects the experts of one valid row.  `lrow` is the row's E
// logits, `sb` a shared-memory scratch of E floats owned by this warp.  On
// return lane k < K holds the k-th chosen expert (biased score descending,
// lower id first on ties) and its weight s_k / sum_j s_j * scaling, the sum
// taken in k order.
//
// Lane l keeps experts l, l + 32, ... (coalesced loads).  Group scores are
// computed by lpg lanes per group (lpg the largest power of two with
// lpg * G <= 32), each taking every lpg-th expert of its group, then merged
// by xor shuffles inside the lane group; the topk_groups groups are those of
// rank < topk_groups; the experts are K rounds of a warp maximum.
__device__ __forceinline__ void select_row(const float* __restrict__ lrow,
                                           const float* __restrict__ bias, int E, int G, int TG,
                                           int K, float scaling, float* sb, int lane, int* out_id,
                                           float* out_w) {
    const int epg = E / G;
    float sv[kSelPer];
    uint32_t vkey[kSelPer];
    {
        float lg[kSelPer], bi[kSelPer];
#pragma unroll
        for (int j = 0; j < kSelPer; ++j) {
            const int e = lane + 32 * j;
            lg[j] = (e < E) ? lrow[e] : 0.0f;
            bi[j] = (e < E) ? bias[e] : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kSelPer; ++j) {
            const int e = lane + 32 * j;
            sv[j] = router_sigmoid(lg[j]);
            const float b = __fadd_rn(sv[j], bi[j]);
            if (e < E) sb[e] = b;
            vkey[j] = ordered_key(b);
        }
    }
    __syncwarp();

    // group scores: the two largest biased scores of each group
    int lpg = 1;
    while (lpg * 2 * G <= 32) lpg *= 2;
    const int g = lane / lpg, sub = lane & (lpg - 1);
    float t1 = -INFINITY, t2 = -INFINITY;
    if (g < G) {
        for (int e = g * epg + sub; e < (g + 1) * epg; e += lpg) {
            const float v = sb[e];
            if (v > t1) {
                t2 = t1;
                t1 = v;
            } else if (v > t2) {
                t2 = v;
            }
        }
    }
    for (int d = lpg >> 1; d >= 1; d >>= 1) {
        const float o1 = __shfl_xor_sync(0xFFFFFFFFu, t1, d);
        const float o2 = __shfl_xor_sync(0xFFFFFFFFu, t2, d);
        const float hi = fmaxf(t1, o1), lo = fminf(t1, o1);
        t2 = fmaxf(lo, fmaxf(t2, o2));
        t1 = hi;
    }
    const float gs = (epg >= 2) ? __fadd_rn(t1, t2) : t1;
    // rank of each group among all groups (ties: lower group id first)
    const uint64_t gkey = (g < G) ? rank_key(gs, g) : 0ull;
    int grank = 0;
    for (int o = 0; o < G; ++o) grank += (__shfl_sync(0xFFFFFFFFu, gkey, o * lpg) > gkey) ? 1 : 0;
    const int my_group_rank = __shfl_sync(0xFFFFFFFFu, grank, (lane < G ? lane : 0) * lpg);
    const uint32_t gmask = __ballot_sync(0xFFFFFFFFu, lane < G && my_group_rank < TG);

    // candidates: experts of the kept groups
#pragma unroll
    for (int j = 0; j < kSelPer; ++j) {
        const int e = lane + 32 * j;
        if (e >= E || !((gmask >> (e / epg)) & 1u)) vkey[j] = 0u;
    }
    int my_id = -1;       // lane k keeps the k-th chosen expert
    float my_s = 0.0f;
    for (int k = 0; k < K; ++k) {
        uint32_t bk = 0u, bid = 0xFFFFFFFFu;
#pragma unroll
        for (int j = 0; j < kSelPer; ++j)
            if (vkey[j] > bk) {
                bk = vkey[j];
                bid = static_cast<uint32_t>(lane + 32 * j);
            }
        const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, bk);
        const uint32_t e = __reduce_min_sync(0xFFFFFFFFu, (bk == top) ? bid : 0xFFFFFFFFu);
        float s_e = 0.0f;
        if ((e & 31u) == static_cast<uint32_t>(lane)) {
#pragma unroll
            for (int j = 0; j < kSelPer; ++j)
                if (static_cast<uint32_t>(lane + 32 * j) == e) {
                    vkey[j] = 0u;
                    s_e = sv[j];
                }
        }
        s_e = __shfl_sync(0xFFFFFFFFu, s_e, static_cast<int>(e & 31u));
        if (lane == k) {
            my_id = static_cast<int>(e);
            my_s = s_e;
        }
    }
    // the denominator summed in k order
    float den = __shfl_sync(0xFFFFFFFFu, my_s, 0);
    for (int k = 1; k < K; ++k) den = __fadd_rn(den, __shfl_sync(0xFFFFFFFFu, my_s, k));
    *out_id = my_id;
    *out_w = __fmul_rn(__fdiv_rn(my_s, den), scaling);
    __syncwarp();   // sb may be reused for the warp's next row
}

}  // namespace moe
