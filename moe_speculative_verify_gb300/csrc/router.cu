// router.cu -- router logits and grouped top-k selection (sm_103a).
//
// The router of a sigmoid-scored, bias-corrected, group-limited MoE (mstar
// #388 "Speed up GLM-5.2 with fp8 kernels and one-graph MTP", commit moving
// NoAuxTcRouter's top-k op; MoE-Infinity #140, e_score_correction_bias;
// pypto-serving #223 "What this adds": router gate kept in FP32).
//
// Every floating-point step is an explicitly rounded IEEE fp32 operation in
// a fixed order (the order is part of the ABI contract in moe_verify.h), so
// the chosen expert ids do not depend on launch shape, batch slot or compiler
// contraction.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ------------------------------------------------------ router logits ----
// logits[r, e] for a tile of RT rows and EC experts per block.  Warp c of the
// block computes, for chunk c of the hidden dimension (1024 columns), the 32
// per-lane partial sums of every (row, expert) pair of the tile; the block then
// folds the chunks in ascending order per lane and finishes with the xor
// butterfly across lanes.
template <int RT, int EC>
__global__ void __launch_bounds__(512) router_logits_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ wr,
    const uint8_t* __restrict__ row_valid, int R, int H, int E, float* __restrict__ logits) {
    extern __shared__ float part[];  // [nchunks][EC][RT][32]
    pdl_wait();
    pdl_launch_dependents();
    const int nchunks = (H + 1023) / 1024;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * EC;
    const int r0 = blockIdx.y * RT;

    if (warp < nchunks) {
        const int c = warp;
        float p[EC][RT];
#pragma unroll
        for (int a = 0; a < EC; ++a)
#pragma unroll
            for (int b = 0; b < RT; ++b) p[a][b] = 0.0f;
        const int nsteps = min(8, (H - c * 1024) / 128);   // 128-column steps of this chunk
        // Loads of four steps are issued together, then consumed in column
        // order: the fma sequence per lane is unchanged.
#pragma unroll
        for (int s0 = 0; s0 < 8; s0 += 4) {
            float4 w4[4][EC];
            uint2 xv[4][RT];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                if (s0 + s < nsteps) {
                    const int h = c * 1024 + (s0 + s) * 128 + 4 * lane;
#pragma unroll
                    for (int a = 0; a < EC; ++a) {
                        const int e = min(e0 + a, E - 1);
                        w4[s][a] = __ldg(reinterpret_cast<const float4*>(wr + size_t(e) * H + h));
                    }
#pragma unroll
                    for (int b = 0; b < RT; ++b) {
                        const int r = min(r0 + b, R - 1);
                        xv[s][b] = __ldg(reinterpret_cast<const uint2*>(x + size_t(r) * H + h));
                    }
                }
            }
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                if (s0 + s < nsteps) {
#pragma unroll
                    for (int b = 0; b < RT; ++b) {
                        const float x0 = bf16_bits_to_f32(xv[s][b].x & 0xFFFFu);
                        const float x1 = bf16_bits_to_f32(xv[s][b].x >> 16);
                        const float x2 = bf16_bits_to_f32(xv[s][b].y & 0xFFFFu);
                        const float x3 = bf16_bits_to_f32(xv[s][b].y >> 16);
#pragma unroll
                        for (int a = 0; a < EC; ++a) {
                            float q = p[a][b];
                            q = __fmaf_rn(x0, w4[s][a].x, q);
                            q = __fmaf_rn(x1, w4[s][a].y, q);
                            q = __fmaf_rn(x2, w4[s][a].z, q);
                            q = __fmaf_rn(x3, w4[s][a].w, q);
                            p[a][b] = q;
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int a = 0; a < EC; ++a)
#pragma unroll
            for (int b = 0; b < RT; ++b) part[((c * EC + a) * RT + b) * 32 + lane] = p[a][b];
    }
    __syncthreads();

    const int nwarps = blockDim.x >> 5;
    for (int pair = warp; pair < EC * RT; pair += nwarps) {
        const int a = pair / RT, b = pair % RT;
        const int e = e0 + a, r = r0 + b;
        float q = part[((0 * EC + a) * RT + b) * 32 + lane];
        for (int c = 1; c < nchunks; ++c) q = __fadd_rn(q, part[((c * EC + a) * RT + b) * 32 + lane]);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) q = __fadd_rn(q, __shfl_xor_sync(0xFFFFFFFFu, q, d));
        if (lane == 0 && e < E && r < R && (row_valid == nullptr || row_valid[r] != 0))
            logits[size_t(r) * E + e] = q;
    }
}

// Large-R variant: a block computes a tile of 32 rows x 32 experts with 16
// warps; the warp (wr, we) owns rows 8*wr.. and experts 8*we.. (64 pairs) and
// lane l of the warp is lane l of the reduction tree for every one of them.
// Per 128-column step the block stages x (bf16) and w (fp32) in shared memory;
// a thread accumulates its 64 lane partials of the current 1024-column chunk in
// registers (fma in column order), folds them into the per-lane chunk sums in
// shared memory at the end of each chunk (q = p for the first chunk, then
// q = q + p), and the warp finishes every pair with the xor butterfly: the same
// IEEE operations in the same order as the small-R kernel.
constexpr int kTileR = 32, kTileE = 32, kTileThreads = 512;

__global__ void __launch_bounds__(kTileThreads, 1) router_logits_tiled_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ wr,
    const uint8_t* __restrict__ row_valid, int R, int H, int E, float* __restrict__ logits) {
    extern __shared__ __align__(16) uint8_t rsm[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(rsm);                          // [2][32][128]
    float* wsm = reinterpret_cast<float*>(rsm + 2 * kTileR * 128 * 2);        // [2][32][128]
    float* qsm = wsm + 2 * kTileE * 128;                                      // [16 warps][64][32]
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wrow = (warp >> 2) * 8, wexp = (warp & 3) * 8;
    const int r0 = blockIdx.y * kTileR, e0 = blockIdx.x * kTileE;
    const int steps = H / 128;

    auto stage = [&](int i, int buf) {
        // x tile: 32 rows x 128 bf16 = 512 x 16 bytes; w tile: 32 x 128 fp32 = 1024 x 16 bytes
        {
            const int row = tid >> 4, c = (tid & 15) * 8;
            const int r = min(r0 + row, R - 1);
            *reinterpret_cast<uint4*>(xs + (buf * kTileR + row) * 128 + c) =
                __ldg(reinterpret_cast<const uint4*>(x + size_t(r) * H + i * 128 + c));
        }
        for (int q = tid; q < kTileE * 32; q += kTileThreads) {
            const int ex = q >> 5, c = (q & 31) * 4;
            const int e = min(e0 + ex, E - 1);
            *reinterpret_cast<float4*>(wsm + (buf * kTileE + ex) * 128 + c) =
                __ldg(reinterpret_cast<const float4*>(wr + size_t(e) * H + i * 128 + c));
        }
    };

    float p[8][8];
    stage(0, 0);
    __syncthreads();
    for (int i = 0; i < steps; ++i) {
        const int buf = i & 1;
        if (i + 1 < steps) stage(i + 1, buf ^ 1);
        if ((i & 7) == 0) {
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) p[a][b] = 0.0f;
        }
        float4 wv[8];
#pragma unroll
        for (int b = 0; b < 8; ++b)
            wv[b] = *reinterpret_cast<const float4*>(wsm + (buf * kTileE + wexp + b) * 128 + 4 * lane);
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const uint2 xv =
                *reinterpret_cast<const uint2*>(xs + (buf * kTileR + wrow + a) * 128 + 4 * lane);
            const float x0 = bf16_bits_to_f32(xv.x & 0xFFFFu), x1 = bf16_bits_to_f32(xv.x >> 16);
            const float x2 = bf16_bits_to_f32(xv.y & 0xFFFFu), x3 = bf16_bits_to_f32(xv.y >> 16);
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                float q = p[a][b];
                q = __fmaf_rn(x0, wv[b].x, q);
                q = __fmaf_rn(x1, wv[b].y, q);
                q = __fmaf_rn(x2, wv[b].z, q);
                q = __fmaf_rn(x3, wv[b].w, q);
                p[a][b] = q;
            }
        }
        if ((i & 7) == 7 || i + 1 == steps) {   // end of a 1024-column chunk
            float* qw = qsm + size_t(warp) * 64 * 32;
            const bool first = (i < 8);
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    float* slot = qw + (a * 8 + b) * 32 + lane;
                    *slot = first ? p[a][b] : __fadd_rn(*slot, p[a][b]);
                }
        }
        __syncthreads();
    }
    const float* qw = qsm + size_t(warp) * 64 * 32;
    for (int pair = 0; pair < 64; ++pair) {
        float q = qw[pair * 32 + lane];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) q = __fadd_rn(q, __shfl_xor_sync(0xFFFFFFFFu, q, d));
        const int r = r0 + wrow + pair / 8, e = e0 + wexp + pair % 8;
        if (lane == 0 && r < R && e < E && (row_valid == nullptr || row_valid[r] != 0))
            logits[size_t(r) * E + e] = q;
    }
}

// -------------------------------------------------- sigmoid with own exp ----
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

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, v, d);
        v = o > v ? o : v;
    }
    return v;
}

// ------------------------------------------------------ grouped top-k ----
// One warp per row: sigmoid scores, biased scores, group scores (sum of the
// two largest biased scores), the topk_groups best groups, the topk best
// experts inside them, and the normalised weights.  Lane l holds experts
// l, l+32, l+64, ...; every reduction is over exact comparisons (no
// arithmetic), so its order does not matter.
constexpr int kSelWarps = 8;
constexpr int kPer = MOE_MAX_EXPERTS / 32;

__global__ void __launch_bounds__(kSelWarps * 32) route_select_kernel(
    const float* __restrict__ logits, const float* __restrict__ bias,
    const uint8_t* __restrict__ row_valid, int R, int E, int G, int TG, int K, float scaling,
    int32_t* __restrict__ ids, float* __restrict__ wts) {
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * kSelWarps + warp;
    if (r >= R) return;
    if (row_valid != nullptr && row_valid[r] == 0) {
        if (lane < K) {
            ids[size_t(r) * K + lane] = -1;
            wts[size_t(r) * K + lane] = 0.0f;
        }
        return;
    }
    const int epg = E / G;
    float sv[kPer], bv[kPer];
    float lg[kPer], bi[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = lane + 32 * j;
        lg[j] = (e < E) ? logits[size_t(r) * E + e] : 0.0f;
        bi[j] = (e < E) ? bias[e] : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        sv[j] = router_sigmoid(lg[j]);
        bv[j] = __fadd_rn(sv[j], bi[j]);
    }

    // group scores: per group, the two largest biased scores, merged over the warp
    float gscore_mine = -INFINITY;               // lane g keeps group g's score
    for (int g = 0; g < G; ++g) {
        float t1 = -INFINITY, t2 = -INFINITY;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int e = lane + 32 * j;
            if (e < E && e / epg == g) {
                const float v = bv[j];
                if (v > t1) {
                    t2 = t1;
                    t1 = v;
                } else if (v > t2) {
                    t2 = v;
                }
            }
        }
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) {
            const float o1 = __shfl_xor_sync(0xFFFFFFFFu, t1, d);
            const float o2 = __shfl_xor_sync(0xFFFFFFFFu, t2, d);
            const float hi = fmaxf(t1, o1), lo = fminf(t1, o1);
            t2 = fmaxf(lo, fmaxf(t2, o2));
            t1 = hi;
        }
        if (lane == g) gscore_mine = (epg >= 2) ? __fadd_rn(t1, t2) : t1;
    }
    // the topk_groups best groups: rank of each group among all (ties: lower id)
    const uint64_t gkey = (lane < G) ? rank_key(gscore_mine, lane) : 0ull;
    int grank = 0;
    for (int g = 0; g < G; ++g) grank += (__shfl_sync(0xFFFFFFFFu, gkey, g) > gkey) ? 1 : 0;
    const uint32_t gmask = __ballot_sync(0xFFFFFFFFu, lane < G && grank < TG);

    // the topk best experts of the kept groups: K rounds of a warp-wide max of
    // the ordered score, then the lowest id among the lanes holding it
    uint32_t vkey[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = lane + 32 * j;
        vkey[j] = (e < E && ((gmask >> (e / epg)) & 1u)) ? ordered_key(bv[j]) : 0u;
    }
    int my_id = -1;       // lane k keeps the k-th chosen expert
    float my_s = 0.0f;
    for (int k = 0; k < K; ++k) {
        uint32_t bk = 0u, bid = 0xFFFFFFFFu;
#pragma unroll
        for (int j = 0; j < kPer; ++j)
            if (vkey[j] > bk) {
                bk = vkey[j];
                bid = static_cast<uint32_t>(lane + 32 * j);
            }
        const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, bk);
        const uint32_t e = __reduce_min_sync(0xFFFFFFFFu, (bk == top) ? bid : 0xFFFFFFFFu);
        float s_e = 0.0f;
        if ((e & 31u) == static_cast<uint32_t>(lane)) {
#pragma unroll
            for (int j = 0; j < kPer; ++j)
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
    // weights: the denominator summed in k order, then every lane its own w_k
    float den = __shfl_sync(0xFFFFFFFFu, my_s, 0);
    for (int k = 1; k < K; ++k) den = __fadd_rn(den, __shfl_sync(0xFFFFFFFFu, my_s, k));
    if (lane < K) {
        ids[size_t(r) * K + lane] = my_id;
        wts[size_t(r) * K + lane] = __fmul_rn(__fdiv_rn(my_s, den), scaling);
    }
}

// ----------------------------------------------------------- launchers ----
cudaError_t launch_router(const uint16_t* x, const float* wr, const float* bias,
                          const uint8_t* row_valid, int R, int H, int E, int G, int TG, int K,
                          float scaling, int32_t* ids, float* wts, float* logits,
                          cudaStream_t stream) {
    const int nchunks = (H + 1023) / 1024;
    const int threads = max(32, nchunks * 32);
    if (R <= 64) {
        constexpr int RT = 8, EC = 1;
        dim3 grid(E / EC, (R + RT - 1) / RT);
        const size_t smem = size_t(nchunks) * EC * RT * 32 * sizeof(float);
        cudaError_t e = launch_pdl(router_logits_kernel<RT, EC>, grid, dim3(threads), smem, stream,
                                   x, wr, row_valid, R, H, E, logits);
        if (e != cudaSuccess) return e;
    } else {
        dim3 grid((E + kTileE - 1) / kTileE, (R + kTileR - 1) / kTileR);
        const size_t smem = size_t(2) * kTileR * 128 * 2 + size_t(2) * kTileE * 128 * 4 +
                            size_t(kTileThreads / 32) * 64 * 32 * 4;
        cudaError_t e = cudaFuncSetAttribute(router_logits_tiled_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        e = launch_pdl(router_logits_tiled_kernel, grid, dim3(kTileThreads), smem, stream, x, wr,
                       row_valid, R, H, E, logits);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_pdl(route_select_kernel, dim3((R + kSelWarps - 1) / kSelWarps), dim3(kSelWarps * 32),
                   0, stream, logits, bias, row_valid, R, E, G, TG, K, scaling, ids, wts);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
