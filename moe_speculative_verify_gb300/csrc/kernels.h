// kernels.h -- launch entry points of the device kernels, used by the host ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"

namespace moe {

// Arguments of the persistent expert-GEMM kernel (ffn.cu).
struct FfnArgs {
    const int32_t* ub;         // union buffer
    UnionLayout ul;
    const float* s_a0;         // routed scales of A0 (gate or down) [E, M/128, Kd/128]
    const float* s_a1;         // routed scales of A1 (up)
    const float* sh_s_a0;      // shared-expert scales
    const float* sh_s_a1;
    const float* bs;           // row (B operand) scales [rows, Kd/128]
    uint8_t* hq;               // gate/up: quantised h [rows, M]
    float* hs;                 // gate/up: h scales [rows, M/128]
    float* y_slots;            // down: [R*K, M]
    float* y_shared;           // down: [R, M]
    int32_t* err;              // device error word
    int M;                     // output features per expert
    int Kd;                    // reduction length
    int E, K, KS;
    int n_stages;
    uint64_t timeout_ns;
};

cudaError_t launch_router(const uint16_t* x, const float* wr, const float* bias,
                          const uint8_t* row_valid, int R, int H, int E, int G, int TG, int K,
                          float scaling, int32_t* ids, float* wts, float* logits,
                          cudaStream_t stream);
cudaError_t launch_union(const int32_t* ids, int R, int E, int K, int S, int n_tile, int32_t* ub,
                         const UnionLayout& L, cudaStream_t stream);
cudaError_t launch_dispatch(const uint16_t* x, const int32_t* ub, const UnionLayout& L, int R,
                            int H, int KS, uint8_t* xg, float* xs, cudaStream_t stream);
cudaError_t launch_ffn(int nt, bool gate_up, const CUtensorMap& a0, const CUtensorMap& a1,
                       const CUtensorMap& sh0, const CUtensorMap& sh1, const CUtensorMap& b,
                       const FfnArgs& args, int n_sms, int max_tiles, int smem_limit,
                       cudaStream_t stream);
cudaError_t launch_combine(const float* y_slots, const float* y_shared, const float* wts,
                           const int32_t* ub, const UnionLayout& L, int R, int H, int K, int S,
                           uint16_t* out, cudaStream_t stream);
cudaError_t launch_wait_timeout(int32_t* err, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace moe
