// combine.cu -- fixed-order weighted combine of the expert outputs plus the
// shared expert, pad rows zero-filled (sm_103a).
//
// openinfer #610 "TP8 span row mapping -- single-user speculative decode at
// 186 tok/s", sections "What" and "Gates": same fixed-order reductions
// whichever mapping carries a row; span pad ranks zero-fill their rows so no
// NaN leaks.  mstar #388 "Speed up GLM-5.2 with fp8 kernels and one-graph
// MTP": the MoE's partials reduced once, routed and shared experts together.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "layout.h"

namespace cg = cooperative_groups;

namespace moe {

// A union built for another call (row count or shape) is not read: the kernel
// writes nothing and records MOE_ERR_INVALID_ARG in the union's word [5].
__device__ __forceinline__ bool combine_union_ok(int32_t* ub, int R, int E, int K, int S) {
    if (union_fits(ub, R, union_shape_word(E, K, S))) return true;
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        atomicCAS(ub + 5, 0, MOE_ERR_INVALID_ARG);
    return false;
}

// One thread per (row, 4 columns).  acc = w0*o0, then fma over k = 1..K-1,
// then + shared, rounded once to bf16.  No atomics: the order is fixed.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y_slots,
                                                      const float* __restrict__ y_shared,
                                                      const float* __restrict__ wts,
                                                      int32_t* __restrict__ ub,
                                                      UnionLayout L, int R, int E, int H, int K,
                                                      int S, uint16_t* __restrict__ out) {
    pdl_wait();
    pdl_launch_dependents();
    const int r = blockIdx.x;
    const int h = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
    if (h >= H) return;
    const int KS = K + S;
    const float* w = wts + size_t(r) * K;
    // The union's shape words, the row's pad word, the shared row and the
    // first four slots are requested together (their addresses do not depend
    // on the union's contents and lie inside the call's buffers), then
    // checked: one memory round trip before the first fmas instead of three.
    const int pos0 = ub[L.pos + size_t(r) * KS];
    float4 ysh = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (S) ysh = __ldg(reinterpret_cast<const float4*>(y_shared + size_t(r) * H + h));
    float4 y[4];
    float wk[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        if (u < K) {
            y[u] = __ldg(reinterpret_cast<const float4*>(y_slots + (size_t(r) * K + u) * H + h));
            wk[u] = w[u];
        }
    }
    if (!combine_union_ok(ub, R, E, K, S)) return;
    uint2* dst = reinterpret_cast<uint2*>(out + size_t(r) * H + h);
    if (pos0 < 0) {
        *dst = make_uint2(0u, 0u);
        return;
    }
    // the K slots in k order, four rows requested at a time (few registers:
    // more blocks per SM keep more rows in flight)
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    for (int k0 = 0; k0 < K; k0 += 4) {
        if (k0 > 0) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (k0 + u < K) {
                    y[u] = __ldg(reinterpret_cast<const float4*>(y_slots + (size_t(r) * K + k0 + u) * H + h));
                    wk[u] = w[k0 + u];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + u;
            if (k >= K) break;
            if (k == 0) {
                a0 = __fmul_rn(wk[u], y[u].x);
                a1 = __fmul_rn(wk[u], y[u].y);
                a2 = __fmul_rn(wk[u], y[u].z);
                a3 = __fmul_rn(wk[u], y[u].w);
            } else {
                a0 = __fmaf_rn(wk[u], y[u].x, a0);
                a1 = __fmaf_rn(wk[u], y[u].y, a1);
                a2 = __fmaf_rn(wk[u], y[u].z, a2);
                a3 = __fmaf_rn(wk[u], y[u].w, a3);
            }
        }
    }
    if (S) {
        a0 = __fadd_rn(a0, ysh.x);
        a1 = __fadd_rn(a1, ysh.y);
        a2 = __fadd_rn(a2, ysh.z);
        a3 = __fadd_rn(a3, ysh.w);
    }
    const uint32_t b0 = __bfloat16_as_ushort(__float2bfloat16_rn(a0));
    const uint32_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(a1));
    const uint32_t b2 = __bfloat16_as_ushort(__float2bfloat16_rn(a2));
    const uint32_t b3 = __bfloat16_as_ushort(__float2bfloat16_rn(a3));
    *dst = make_uint2(b0 | (b1 << 16), b2 | (b3 << 16));
}

cudaError_t launch_combine(const float* y_slots, const float* y_shared, const float* wts,
                           int32_t* ub, const UnionLayout& L, int R, int E, int H, int K, int S,
                           uint16_t* out, cudaStream_t stream) {
    dim3 grid(R, (H / 4 + 255) / 256);
    cudaError_t e = launch_pdl(combine_kernel, grid, dim3(256), 0, stream, y_slots, y_shared, wts, ub,
                               L, R, E, H, K, S, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Combine fused with the residual add and the RMSNorm of the next layer
// (mstar #388 "Speed up GLM-5.2 with fp8 kernels and one-graph MTP", commit on
// kernel switches: the MoE's partials reduced once, fused with the next
// add + RMSNorm).  One cluster of kNormCluster CTAs per row, CTA c owning the
// c-th slice of H / kNormCluster columns:
//   acc = the fixed-order combine sum (as combine_kernel, before rounding);
//   z = residual + acc;  residual_out = bf16_rne(z);
//   normed = bf16_rne(z * rsqrt(sum(z^2) / H + eps) * gamma).
// The sum of squares is reduced in a fixed order: per thread over its columns
// in order, xor butterfly in the warp, warps in index order, then the CTAs'
// partial sums in rank order (read through distributed shared memory by every
// CTA), so a row's bits do not depend on the batch.  Pad rows give +0.0 in
// both outputs.
constexpr int kNormThreads = 128;
constexpr int kNormCluster = 8;
constexpr int kNormMaxChunks = 4;      // H / 4 / kNormCluster / kNormThreads, H <= 16384

__global__ void __launch_bounds__(kNormThreads) combine_add_rmsnorm_kernel(
    const float* __restrict__ y_slots, const float* __restrict__ y_shared,
    const float* __restrict__ wts, int32_t* __restrict__ ub, UnionLayout L, int R, int E, int H,
    int K, int S, const uint16_t* __restrict__ residual, const float* __restrict__ gamma, float eps,
    uint16_t* __restrict__ residual_out, uint16_t* __restrict__ normed) {
    __shared__ float s_warp[kNormThreads / 32];
    __shared__ float s_part;
    cg::cluster_group cl = cg::this_cluster();
    pdl_wait();
    pdl_launch_dependents();
    const int r = blockIdx.x / kNormCluster;
    const int rank = static_cast<int>(cl.block_rank());
    const int KS = K + S;
    const int nchunks = H / 4 / kNormCluster;                 // float4 chunks of this CTA
    const int c0 = rank * nchunks;
    const float* w = wts + size_t(r) * K;
    // chunk c's K slots, shared row and residual
    float4 y[MOE_MAX_TOPK + 1];
    uint2 rb = make_uint2(0u, 0u);
    auto load_chunk = [&](int c) {
        const int h = 4 * (c0 + c);
#pragma unroll
        for (int k = 0; k < MOE_MAX_TOPK; ++k)
            if (k < K) y[k] = __ldg(reinterpret_cast<const float4*>(y_slots + (size_t(r) * K + k) * H + h));
        if (S) y[MOE_MAX_TOPK] = __ldg(reinterpret_cast<const float4*>(y_shared + size_t(r) * H + h));
        rb = *reinterpret_cast<const uint2*>(residual + size_t(r) * H + h);
    };
    // The union's words, the row's pad word and the first chunk's rows are
    // requested together (their addresses do not depend on the union's
    // contents), then checked.
    const int pos0 = ub[L.pos + size_t(r) * KS];
    if (threadIdx.x < nchunks) load_chunk(threadIdx.x);
    // the same words for every CTA of every cluster: all leave here or none
    if (!combine_union_ok(ub, R, E, K, S)) return;
    // the same for every CTA of the cluster: all leave here or none
    const bool valid = pos0 >= 0;
    if (!valid) {
        for (int c = threadIdx.x; c < nchunks; c += kNormThreads) {
            reinterpret_cast<uint2*>(residual_out + size_t(r) * H)[c0 + c] = make_uint2(0u, 0u);
            reinterpret_cast<uint2*>(normed + size_t(r) * H)[c0 + c] = make_uint2(0u, 0u);
        }
        return;
    }
    float4 z[kNormMaxChunks];
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < kNormMaxChunks; ++i) {
        const int c = threadIdx.x + i * kNormThreads;
        if (c < nchunks) {
            const int h = 4 * (c0 + c);
            if (i > 0) load_chunk(c);
            const float w0 = w[0];
            float a0 = __fmul_rn(w0, y[0].x), a1 = __fmul_rn(w0, y[0].y),
                  a2 = __fmul_rn(w0, y[0].z), a3 = __fmul_rn(w0, y[0].w);
#pragma unroll
            for (int k = 1; k < MOE_MAX_TOPK; ++k) {
                if (k < K) {
                    const float wk = w[k];
                    a0 = __fmaf_rn(wk, y[k].x, a0);
                    a1 = __fmaf_rn(wk, y[k].y, a1);
                    a2 = __fmaf_rn(wk, y[k].z, a2);
                    a3 = __fmaf_rn(wk, y[k].w, a3);
                }
            }
            if (S) {
                a0 = __fadd_rn(a0, y[MOE_MAX_TOPK].x);
                a1 = __fadd_rn(a1, y[MOE_MAX_TOPK].y);
                a2 = __fadd_rn(a2, y[MOE_MAX_TOPK].z);
                a3 = __fadd_rn(a3, y[MOE_MAX_TOPK].w);
            }
            float4 zz;
            zz.x = __fadd_rn(bf16_bits_to_f32(rb.x & 0xFFFFu), a0);
            zz.y = __fadd_rn(bf16_bits_to_f32(rb.x >> 16), a1);
            zz.z = __fadd_rn(bf16_bits_to_f32(rb.y & 0xFFFFu), a2);
            zz.w = __fadd_rn(bf16_bits_to_f32(rb.y >> 16), a3);
            z[i] = zz;
            ss = __fmaf_rn(zz.x, zz.x, ss);
            ss = __fmaf_rn(zz.y, zz.y, ss);
            ss = __fmaf_rn(zz.z, zz.z, ss);
            ss = __fmaf_rn(zz.w, zz.w, ss);
            const uint32_t b0 = __bfloat16_as_ushort(__float2bfloat16_rn(zz.x));
            const uint32_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(zz.y));
            const uint32_t b2 = __bfloat16_as_ushort(__float2bfloat16_rn(zz.z));
            const uint32_t b3 = __bfloat16_as_ushort(__float2bfloat16_rn(zz.w));
            *reinterpret_cast<uint2*>(residual_out + size_t(r) * H + h) =
                make_uint2(b0 | (b1 << 16), b2 | (b3 << 16));
        }
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, d));
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = s_warp[0];
        for (int i = 1; i < kNormThreads / 32; ++i) t = __fadd_rn(t, s_warp[i]);
        s_part = t;
    }
    cl.sync();   // every CTA's partial sum is in its shared memory
    float t = *cl.map_shared_rank(&s_part, 0);
    for (int i = 1; i < kNormCluster; ++i) t = __fadd_rn(t, *cl.map_shared_rank(&s_part, i));
    const float inv = __frsqrt_rn(__fadd_rn(__fdiv_rn(t, static_cast<float>(H)), eps));
#pragma unroll
    for (int i = 0; i < kNormMaxChunks; ++i) {
        const int c = threadIdx.x + i * kNormThreads;
        if (c < nchunks) {
            const int h = 4 * (c0 + c);
            const float4 g = __ldg(reinterpret_cast<const float4*>(gamma + h));
            const uint32_t b0 = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__fmul_rn(z[i].x, inv), g.x)));
            const uint32_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__fmul_rn(z[i].y, inv), g.y)));
            const uint32_t b2 = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__fmul_rn(z[i].z, inv), g.z)));
            const uint32_t b3 = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(__fmul_rn(z[i].w, inv), g.w)));
            *reinterpret_cast<uint2*>(normed + size_t(r) * H + h) = make_uint2(b0 | (b1 << 16), b2 | (b3 << 16));
        }
    }
    cl.sync();   // no CTA leaves while another may still read its partial sum
}

cudaError_t launch_combine_add_rmsnorm(const float* y_slots, const float* y_shared, const float* wts,
                                       int32_t* ub, const UnionLayout& L, int R, int E, int H,
                                       int K, int S, const uint16_t* residual, const float* gamma,
                                       float eps, uint16_t* residual_out, uint16_t* normed,
                                       cudaStream_t stream) {
    if (H % (4 * kNormCluster) != 0 || H / 4 / kNormCluster > kNormMaxChunks * kNormThreads)
        return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl_cluster(combine_add_rmsnorm_kernel,
                                       dim3(static_cast<unsigned>(R) * kNormCluster),
                                       dim3(kNormThreads), kNormCluster, 0, stream, y_slots,
                                       y_shared, wts, ub, L, R, E, H, K, S, residual, gamma,
                                       eps, residual_out, normed);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Diagnostic: one block waits on a barrier nothing arrives on; the bounded
// wait gives up after timeout_ns and records MOE_ERR_TIMEOUT.
__global__ void wait_timeout_kernel(int32_t* err, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, err, timeout_ns);
}

cudaError_t launch_wait_timeout(int32_t* err, uint64_t timeout_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}

}  // namespace moe
