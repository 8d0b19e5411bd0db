// noalloc.cu -- moe_layer for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: a plugin whose
// host framework owns every device allocation and gives plugins none, code on
// a latency-critical path that is not allowed to call cudaMalloc, or a caller
// that only learns the row count when the layer runs.  For them the layer's
// scratch lives in one fixed-size array in the library's own device memory.
// The array is reserved on every GPU that loads the library, for as long as the
// process runs, so it is kept modest: kStaticScratchBytes (32 MiB), enough for
// up to 109 rows at the GLM-5.2 layer shape (hidden 6144, inter 2048, 256
// experts, top-8, one shared expert).
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "layout.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;

// The layer's whole workspace (error word, routing, union, FFN scratch, slot
// outputs) for calls of moe_layer_noalloc.  Host code must not use this name
// as an address: it is resolved per device with cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Per device: the context the address was looked up in, and the address.  A
// context of its own (a driver context made current by the caller) or the
// primary context created again after cudaDeviceReset loads the library's
// device code anew, so the array may sit elsewhere: the address is looked up
// again whenever the current context is not the one it was found in.
struct ScratchAddr {
    CUcontext ctx = nullptr;
    void* addr = nullptr;
};
ScratchAddr g_addr[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 ctx_get_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    });
    return fn;
}

// Device address of the scratch array on the current device, looked up with
// that device current and cached per (device, context).
moe_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    auto get_ctx = ctx_get_current();
    CUcontext ctx = nullptr;
    if (get_ctx == nullptr || get_ctx(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchAddr& a = g_addr[dev];
    if (ctx == nullptr || a.addr == nullptr || a.ctx != ctx) {
        // (with no context current yet, the lookup makes the device's
        // primary context current)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        if (ctx == nullptr && (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr))
            return MOE_ERR_CUDA;
        a.ctx = ctx;
        a.addr = p;
    }
    *out = a.addr;
    return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_layer_noalloc(const moe_config_t* cfg, const void* x_bf16,
                                          const float* w_router, const float* bias,
                                          const moe_weights_t* w, const uint8_t* row_valid,
                                          int32_t R, void* out_bf16, int32_t* topk_ids_out,
                                          float* topk_w_out, int32_t* device_status,
                                          moe_stream_t stream) {
    if (cfg == nullptr) return MOE_ERR_INVALID_ARG;
    if (R < 0) return MOE_ERR_INVALID_ARG;
    if (R == 0) return MOE_OK;
    const size_t need = moe_workspace_bytes(cfg, R);
    if (need == 0) {
        // the shape or the row count is refused: report it as moe_layer would
        return moe_layer(cfg, x_bf16, w_router, bias, w, row_valid, R, out_bf16, topk_ids_out,
                         topk_w_out, nullptr, 0, stream);
    }
    if (need > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;
    if (device_status && (reinterpret_cast<uintptr_t>(device_status) % 4) != 0)
        return MOE_ERR_INVALID_ARG;
    void* scratch = nullptr;
    moe_status_t st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents; only the error word at its
    // head must start at zero (every other byte the layer reads it writes first).
    if (cudaMemsetAsync(scratch, 0, moe::kCtlBytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    st = moe_layer(cfg, x_bf16, w_router, bias, w, row_valid, R, out_bf16, topk_ids_out,
                   topk_w_out, scratch, kStaticScratchBytes, stream);
    if (st != MOE_OK) return st;
    if (device_status &&
        cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
