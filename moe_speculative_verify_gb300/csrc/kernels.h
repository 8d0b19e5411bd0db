// kernels.h -- launch entry points of the device kernels, used by the host ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "layout.h"

namespace moe {

// Host: cudaFuncSetAttribute(MaxDynamicSharedMemorySize) only when a launch
// needs more than the kernel already allows on the current device (a runtime
// call per launch otherwise, on the path of every layer).  The attribute
// belongs to the process, so the record is process-wide and the allowance
// only ever grows: a launch that needs less than another thread set runs
// under the larger allowance.
inline cudaError_t ensure_dyn_smem(const void* func, int bytes) {
    struct Entry {
        const void* f;
        int dev, bytes;
    };
    static std::mutex mu;
    static Entry tab[64];
    static int n = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    Entry* hit = nullptr;
    for (int i = 0; i < n && !hit; ++i)
        if (tab[i].f == func && tab[i].dev == dev) hit = &tab[i];
    if (hit && hit->bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (hit)
        hit->bytes = bytes;
    else if (n < 64)
        tab[n++] = Entry{func, dev, bytes};
    return cudaSuccess;
}

// Modes of the persistent expert-GEMM kernel (ffn.cu).
constexpr int kFfnGateUp = 0;   // gate/up GEMMs + SiLU*mul + h quantisation
constexpr int kFfnDown = 1;     // down GEMM
constexpr int kFfnFused = 2;    // both, one launch, one tile queue

// Tensor maps of the expert GEMMs: gate, up, shared gate, shared up, gathered
// rows x; down, shared down, quantised h.
struct FfnMaps {
    CUtensorMap g, u, sg, su, x, d, sd, h;
};

// Arguments of the persistent expert-GEMM kernel (ffn.cu).
struct FfnArgs {
    const int32_t* ub;         // union buffer
    UnionLayout ul;
    const float* s_gate;       // routed scales [E, I/128, H/128]
    const float* s_up;
    const float* sh_s_gate;    // shared-expert scales [S, I/128, H/128]
    const float* sh_s_up;
    const float* s_down;       // [E, H/128, I/128]
    const float* sh_s_down;
    const float* xs;           // gathered-row scales [rows, H/128]
    uint8_t* hq;               // quantised h [rows, I]
    float* hs;                 // h scales [rows, I/128]
    float* y_slots;            // [R*K, H]
    float* y_shared;           // [R, H]
    int out_vec;               // y_slots and y_shared 16-byte aligned: rows stored 16 bytes at a time
    int32_t* ready;            // [max_items] gate/up blocks of h finished (fused mode)
    int32_t* sched;            // [2] tile counter, CTAs done claiming (zero between launches)
    int32_t* err;              // device error word
    int R;                     // rows of the call
    int32_t ushape;            // union_shape_word of the call
    int H, I;
    int E, K, KS;
    int n_stages;
    int tiled;                 // weight codes in 16 KB blocks (else row-major)
    uint64_t timeout_ns;
};

// Arguments of the w8a16 expert-GEMM kernel (ffn16.cu).
struct Ffn16Args {
    const int32_t* ub;         // union buffer
    UnionLayout ul;
    const float* s_gate;       // routed scales [E, I/128, H/128]
    const float* s_up;
    const float* sh_s_gate;    // shared-expert scales [S, I/128, H/128]
    const float* sh_s_up;
    const float* s_down;       // [E, H/128, I/128]
    const float* sh_s_down;
    uint16_t* hb;              // bf16 h [rows, I]
    float* y_slots;            // [R*K, H]
    float* y_shared;           // [R, H]
    int32_t* ready;            // [max_items] gate/up blocks of h finished
    int32_t* sched;            // [2] tile counter, CTAs done claiming (zero between launches)
    int32_t* err;              // device error word
    int R;                     // rows of the call
    int32_t ushape;            // union_shape_word of the call
    int H, I;
    int E, K, KS;
    int n_wstages;
    int tiled;                 // weight codes in 16 KB blocks (else row-major)
    uint64_t timeout_ns;
};

cudaError_t launch_dispatch16(const uint16_t* x, const int32_t* ub, const UnionLayout& L, int R,
                              int H, int KS, int32_t ushape, uint16_t* xb, int32_t* ready,
                              int n_ready, int32_t* err, cudaStream_t stream);
cudaError_t launch_ffn16(const FfnMaps& mp, Ffn16Args args, int n_sms, int smem_limit,
                         cudaStream_t stream);
// Tensor maps of the large-R router logits kernel: x bf16 [R, H] in boxes of
// 4 * rt rows and the router weights fp32 [E, H] in boxes of 32 rows,
// unswizzled, kRouterStageCols columns wide; rt = rows of a consumer warp
// (router_rows_per_warp).
// Two 128-column blocks a stage: measured at 4096 rows, 410 -> 354 us
// against one (half as many barrier waits and releases per column).
constexpr int kRouterStageCols = 256;
struct RouterMaps {
    CUtensorMap x, w;
    int rt;
};

// Rows a consumer warp of the large-R router kernel takes per tile (tiles of
// 4x that many rows x 32 experts): 6, 7, 8 or 9, whichever makes the busiest
// of the n_sms CTAs finish first.  A CTA's time is its tile count times a
// tile's cost; measured at 4096 rows and 256 experts (bit-identical logits at
// every height), a wave of tiles took 36.2, 39.6, 43.6 and 49.2 us at 6, 7, 8
// and 9 rows a warp, the costs 45 : 50 : 55 : 62 below.  So 6 rows where the
// tiles fit in one wave (up to 456 rows at 256 experts), 7 at 512 and 1000
// rows (moe_route 57.3 -> 55.2 and 100.4 -> 92.2 us against 8), 9 at 2048 and
// 4096, where 912 tiles fill six waves of 152 exactly (182.3 -> 155.8 and
// 308.3 -> 295.4 us).
inline int router_rows_per_warp(int R, int E, int n_sms) {
    constexpr int kCost[4] = {45, 50, 55, 62};
    int best = 6;
    long long best_cost = -1;
    for (int rt = 6; rt <= 9; ++rt) {
        const long long tiles = static_cast<long long>((R + 4 * rt - 1) / (4 * rt)) * ((E + 31) / 32);
        const long long grid = tiles < n_sms ? tiles : (n_sms > 0 ? n_sms : 1);
        const long long c = ((tiles + grid - 1) / grid) * kCost[rt - 6];
        if (best_cost < 0 || c < best_cost) {
            best = rt;
            best_cost = c;
        }
    }
    return best;
}
// Above 64 rows `maps` is required; a wait that runs out records
// MOE_ERR_TIMEOUT in *err (when err is not null).
cudaError_t launch_router_logits(const uint16_t* x, const float* wr, const uint8_t* row_valid,
                                 int R, int H, int E, float* logits, const RouterMaps* maps,
                                 int n_sms, int32_t* err, uint64_t timeout_ns,
                                 cudaStream_t stream);
cudaError_t launch_router(const uint16_t* x, const float* wr, const float* bias,
                          const uint8_t* row_valid, int R, int H, int E, int G, int TG, int K,
                          float scaling, int32_t* ids, float* wts, float* logits,
                          const RouterMaps* maps, int n_sms, int32_t* err, uint64_t timeout_ns,
                          cudaStream_t stream);
cudaError_t launch_union(const int32_t* ids, int R, int E, int K, int S, int n_tile, int32_t* ub,
                         const UnionLayout& L, cudaStream_t stream);
// Selection and union in one launch for calls of at most kRouteUnionMaxRows
// rows (the logits come from launch_router's first kernel).
constexpr int kRouteUnionMaxRows = 64;
cudaError_t launch_route_union(const float* logits, const float* bias, const uint8_t* row_valid,
                               int R, int E, int G, int TG, int K, float scaling, int32_t* ids,
                               float* wts, int S, int n_tile, int32_t* ub, const UnionLayout& L,
                               cudaStream_t stream);
// Row-major [n, rows, cols] e4m3 codes into 16 KB 128x128 blocks (tile.cu).
cudaError_t launch_tile_weights(const uint8_t* src, uint8_t* dst, int64_t n, int rows, int cols,
                                cudaStream_t stream);
cudaError_t launch_dispatch(const uint16_t* x, const int32_t* ub, const UnionLayout& L, int R,
                            int H, int KS, int32_t ushape, uint8_t* xg, float* xs, int32_t* ready,
                            int n_ready, int32_t* err, cudaStream_t stream);
cudaError_t launch_ffn(int nt, int mode, const FfnMaps& mp, const FfnArgs& args, int n_sms,
                       int smem_limit, cudaStream_t stream);
// The combine kernels record a union built for another call in its word [5].
cudaError_t launch_combine(const float* y_slots, const float* y_shared, const float* wts,
                           int32_t* ub, const UnionLayout& L, int R, int E, int H, int K, int S,
                           uint16_t* out, cudaStream_t stream);
cudaError_t launch_combine_add_rmsnorm(const float* y_slots, const float* y_shared, const float* wts,
                                       int32_t* ub, const UnionLayout& L, int R, int E, int H,
                                       int K, int S, const uint16_t* residual, const float* gamma,
                                       float eps, uint16_t* residual_out, uint16_t* normed,
                                       cudaStream_t stream);
cudaError_t launch_wait_timeout(int32_t* err, uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_greedy_verify(const void* logits, bool bf16, int V, int R, const int32_t* draft,
                                 const int32_t* n_draft, int32_t* am, int32_t* accept_len,
                                 int32_t* out, cudaStream_t stream);

}  // namespace moe
