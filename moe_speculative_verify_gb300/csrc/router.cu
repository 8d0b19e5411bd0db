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
#include "select.cuh"

namespace moe {

// ------------------------------------------------------ router logits ----
// logits[r, e] for a tile of RT rows and EC experts per block.  Warp c of the
// block computes, for chunk c of the hidden dimension (1024 columns), the 32
// per-lane partial sums of every (row, expert) pair of the tile; the block then
// folds the chunks in ascending order per lane and finishes with the xor
// butterfly across lanes.
template <int RT, int EC, int BS, int MAXT, int MINB>
__global__ void __launch_bounds__(MAXT, MINB) router_logits_kernel(
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
        // Loads of BS steps are issued together, then consumed in column
        // order: the fma sequence per lane is unchanged.
#pragma unroll
        for (int s0 = 0; s0 < 8; s0 += BS) {
            float4 w4[BS][EC];
            uint2 xv[BS][RT];
#pragma unroll
            for (int s = 0; s < BS; ++s) {
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
            for (int s = 0; s < BS; ++s) {
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

// Large-R variant: a block computes a tile of 32 rows x 32 experts; the warp
// (wr, we) owns rows 8*wr.. and PE experts from PE*we.. (8*PE pairs) and lane
// l of the warp is lane l of the reduction tree for every one of them.  Per
// 128-column step the block stages x (bf16) and w (fp32) in shared memory
// through a ring of kTileStages buffers filled by cp.async (kTileStages - 1
// steps in flight); a thread accumulates its lane partials of the current
// 1024-column chunk in registers (fma in column order), folds them into the
// per-lane chunk sums in shared memory at the end of each chunk (q = p for the
// first chunk, then q = q + p), and the warp finishes every pair with the xor
// butterfly: the same IEEE operations in the same order as the small-R kernel.
// A larger PE reads each x and w value from shared memory for more fmas:
// measured at 4096 rows, 16 experts a thread (8 warps, 220 registers) took
// the prefill layer from 4.597 to 4.522 ms against 8 (16 warps).
constexpr int kTileR = 32, kTileE = 32, kTileStages = 4;
constexpr int kTileXBytes = kTileR * 128 * 2, kTileWBytes = kTileE * 128 * 4;
constexpr int kTilePE = 16;   // experts per thread

template <int PE>
struct RouterTile {
    static constexpr int WARPS = 4 * (kTileE / PE);
    static constexpr int THREADS = 32 * WARPS;
    static constexpr size_t SMEM = size_t(kTileStages) * (kTileXBytes + kTileWBytes) +
                                   size_t(WARPS) * 8 * PE * 32 * 4;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int PE>
__global__ void __launch_bounds__(RouterTile<PE>::THREADS, 1) router_logits_tiled_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ wr,
    const uint8_t* __restrict__ row_valid, int R, int H, int E, float* __restrict__ logits) {
    constexpr int NTH = RouterTile<PE>::THREADS;
    constexpr int EG = kTileE / PE;   // expert groups of the warp grid
    extern __shared__ __align__(16) uint8_t rsm[];
    uint16_t* xs = reinterpret_cast<uint16_t*>(rsm);                                // [S][32][128]
    float* wsm = reinterpret_cast<float*>(rsm + kTileStages * kTileXBytes);         // [S][32][128]
    float* qsm = wsm + kTileStages * kTileE * 128;                                  // [warps][8*PE][32]
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wrow = (warp / EG) * 8, wexp = (warp % EG) * PE;
    const int r0 = blockIdx.y * kTileR, e0 = blockIdx.x * kTileE;
    const int steps = H / 128;

    // Step i's tiles into ring buffer i % kTileStages: x is 512 x 16 bytes, w
    // 1024 x 16 bytes, spread over the block's threads.
    auto issue = [&](int i) {
        if (i < steps) {
            const int buf = i % kTileStages;
#pragma unroll
            for (int u = 0; u < kTileR * 16 / NTH; ++u) {
                const int q = tid + u * NTH;
                const int xrow = q >> 4, xc = (q & 15) * 8;
                cp_async16(xs + (buf * kTileR + xrow) * 128 + xc,
                           x + size_t(min(r0 + xrow, R - 1)) * H + i * 128 + xc);
            }
#pragma unroll
            for (int u = 0; u < kTileE * 32 / NTH; ++u) {
                const int q = tid + u * NTH;
                const int ex = q >> 5, c = (q & 31) * 4;
                const int e = min(e0 + ex, E - 1);
                cp_async16(wsm + (buf * kTileE + ex) * 128 + c, wr + size_t(e) * H + i * 128 + c);
            }
        }
        cp_async_commit();   // one group per step, empty past the end: uniform counting
    };

    float p[8][PE];
#pragma unroll
    for (int i = 0; i < kTileStages - 1; ++i) issue(i);
    for (int i = 0; i < steps; ++i) {
        const int buf = i % kTileStages;
        cp_async_wait<kTileStages - 2>();   // this thread's copies of step i have landed
        __syncthreads();                    // everyone's have; step i-1's buffer is free
        issue(i + kTileStages - 1);
        if ((i & 7) == 0) {
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < PE; ++b) p[a][b] = 0.0f;
        }
        // all PE experts' columns held, each row's x read and widened once;
        // every pair's four fmas stay in column order
        float4 wv[PE];
#pragma unroll
        for (int b = 0; b < PE; ++b)
            wv[b] = *reinterpret_cast<const float4*>(wsm + (buf * kTileE + wexp + b) * 128 + 4 * lane);
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const uint2 xv =
                *reinterpret_cast<const uint2*>(xs + (buf * kTileR + wrow + a) * 128 + 4 * lane);
            const float x0 = bf16_bits_to_f32(xv.x & 0xFFFFu), x1 = bf16_bits_to_f32(xv.x >> 16);
            const float x2 = bf16_bits_to_f32(xv.y & 0xFFFFu), x3 = bf16_bits_to_f32(xv.y >> 16);
#pragma unroll
            for (int b = 0; b < PE; ++b) {
                float q = p[a][b];
                q = __fmaf_rn(x0, wv[b].x, q);
                q = __fmaf_rn(x1, wv[b].y, q);
                q = __fmaf_rn(x2, wv[b].z, q);
                q = __fmaf_rn(x3, wv[b].w, q);
                p[a][b] = q;
            }
        }
        if ((i & 7) == 7 || i + 1 == steps) {   // end of a 1024-column chunk
            float* qw = qsm + size_t(warp) * 8 * PE * 32;
            const bool first = (i < 8);
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < PE; ++b) {
                    float* slot = qw + (a * PE + b) * 32 + lane;
                    *slot = first ? p[a][b] : __fadd_rn(*slot, p[a][b]);
                }
        }
    }
    cp_async_wait<0>();
    const float* qw = qsm + size_t(warp) * 8 * PE * 32;
    for (int pair = 0; pair < 8 * PE; ++pair) {
        float q = qw[pair * 32 + lane];
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) q = __fadd_rn(q, __shfl_xor_sync(0xFFFFFFFFu, q, d));
        const int r = r0 + wrow + pair / PE, e = e0 + wexp + pair % PE;
        if (lane == 0 && r < R && e < E && (row_valid == nullptr || row_valid[r] != 0))
            logits[size_t(r) * E + e] = q;
    }
}

// ------------------------------------------------------ grouped top-k ----
// One warp per row (select.cuh); pad rows get ids -1 and weights 0.
constexpr int kSelWarps = 8;

__global__ void __launch_bounds__(kSelWarps * 32) route_select_kernel(
    const float* __restrict__ logits, const float* __restrict__ bias,
    const uint8_t* __restrict__ row_valid, int R, int E, int G, int TG, int K, float scaling,
    int32_t* __restrict__ ids, float* __restrict__ wts) {
    __shared__ float s_b[kSelWarps][MOE_MAX_EXPERTS];
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * kSelWarps + warp;
    if (r >= R) return;
    int id = -1;
    float w = 0.0f;
    if (row_valid == nullptr || row_valid[r] != 0)
        select_row(logits + size_t(r) * E, bias, E, G, TG, K, scaling, s_b[warp], lane, &id, &w);
    if (lane < K) {
        ids[size_t(r) * K + lane] = id;
        wts[size_t(r) * K + lane] = w;
    }
}

// ----------------------------------------------------------- launchers ----
cudaError_t launch_router_logits(const uint16_t* x, const float* wr, const uint8_t* row_valid,
                                 int R, int H, int E, float* logits, cudaStream_t stream) {
    const int nchunks = (H + 1023) / 1024;
    const int threads = max(32, nchunks * 32);
    if (R <= 64) {
        constexpr int RT = 8, EC = 1;
        dim3 grid(E / EC, (R + RT - 1) / RT);
        const size_t smem = size_t(nchunks) * EC * RT * 32 * sizeof(float);
        // up to 6 chunks (hidden <= 6144): all eight steps of a chunk in one
        // batch of loads, two blocks per SM; wider rows: batches of four
        cudaError_t e =
            (nchunks <= 6)
                ? launch_pdl(router_logits_kernel<RT, EC, 8, 192, 2>, grid, dim3(threads), smem,
                             stream, x, wr, row_valid, R, H, E, logits)
                : launch_pdl(router_logits_kernel<RT, EC, 4, 512, 1>, grid, dim3(threads), smem,
                             stream, x, wr, row_valid, R, H, E, logits);
        if (e != cudaSuccess) return e;
    } else {
        dim3 grid((E + kTileE - 1) / kTileE, (R + kTileR - 1) / kTileR);
        using T = RouterTile<kTilePE>;
        cudaError_t e = cudaFuncSetAttribute(router_logits_tiled_kernel<kTilePE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(T::SMEM));
        if (e != cudaSuccess) return e;
        e = launch_pdl(router_logits_tiled_kernel<kTilePE>, grid, dim3(T::THREADS), T::SMEM, stream,
                       x, wr, row_valid, R, H, E, logits);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_router(const uint16_t* x, const float* wr, const float* bias,
                          const uint8_t* row_valid, int R, int H, int E, int G, int TG, int K,
                          float scaling, int32_t* ids, float* wts, float* logits,
                          cudaStream_t stream) {
    cudaError_t e = launch_router_logits(x, wr, row_valid, R, H, E, logits, stream);
    if (e != cudaSuccess) return e;
    e = launch_pdl(route_select_kernel, dim3((R + kSelWarps - 1) / kSelWarps), dim3(kSelWarps * 32),
                   0, stream, logits, bias, row_valid, R, E, G, TG, K, scaling, ids, wts);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
