// verify.cu -- greedy speculative verify and acceptance on the device (sm_103a).
//
// openinfer #610 "TP8 span row mapping -- single-user speculative decode at
// 186 tok/s", section "What": a span of 8 rows holds 1 committed token and up
// to 7 drafts.  pypto-serving #223 "DSpark speculation (K=7)", "What this
// adds": accept the longest matching prefix plus the bonus prediction, 1..8
// tokens per step.  mstar #388 "Speed up GLM-5.2 with fp8 kernels and
// one-graph MTP": greedy verify runs on the device inside the step.
//
// Two kernels: the target's greedy token per row (argmax over the vocabulary,
// one cluster of CTAs per row), then the acceptance rule per span (one thread each).
// The argmax reduces 64-bit keys (ordered value, then the complement of the
// index): the largest value wins, the lowest index wins ties, NaN never wins.
// The key order is total, so the result does not depend on the reduction
// order or the launch shape.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int kArgmaxThreads = 512;
constexpr int kArgmaxCluster = 8;      // CTAs per row

__device__ __forceinline__ uint64_t argmax_key(float v, uint32_t idx) {
    uint32_t hi;
    if (v != v) {
        hi = 0u;                                   // NaN: below every number
    } else {
        if (v == 0.0f) v = 0.0f;                   // -0 and +0 are equal
        const uint32_t u = __float_as_uint(v);
        hi = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    return (static_cast<uint64_t>(hi) << 32) | (0xFFFFFFFFu - idx);
}

__device__ __forceinline__ uint64_t max64(uint64_t a, uint64_t b) { return a > b ? a : b; }

// A row is split over the kArgmaxCluster CTAs of one cluster, CTA c taking
// the c-th contiguous slice (in vectors of 16 bytes when the rows allow it);
// CTA 0 reduces the slices' keys through distributed shared memory.
template <bool BF16, bool VEC>
__global__ void __launch_bounds__(kArgmaxThreads) row_argmax_kernel(const void* __restrict__ logits,
                                                                   int V, int32_t* __restrict__ am) {
    __shared__ uint64_t s_red[kArgmaxThreads / 32];
    __shared__ uint64_t s_best;
    cg::cluster_group cl = cg::this_cluster();
    pdl_wait();
    pdl_launch_dependents();
    const int r = blockIdx.x / kArgmaxCluster;
    const int c = static_cast<int>(cl.block_rank());
    constexpr int PER = VEC ? (BF16 ? 8 : 4) : 1;          // elements per load
    const int n = V / PER;                                  // loads per row
    const int lo = static_cast<int>((int64_t(n) * c) / kArgmaxCluster);
    const int hi = static_cast<int>((int64_t(n) * (c + 1)) / kArgmaxCluster);
    uint64_t best = 0;
    if (BF16) {
        const uint16_t* row = static_cast<const uint16_t*>(logits) + size_t(r) * V;
        if (VEC) {
            const uint4* rv = reinterpret_cast<const uint4*>(row);
#pragma unroll 8
            for (int i = lo + threadIdx.x; i < hi; i += kArgmaxThreads) {
                const uint4 q = __ldg(rv + i);
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    best = max64(best, argmax_key(bf16_bits_to_f32(w[k] & 0xFFFFu), 8 * i + 2 * k));
                    best = max64(best, argmax_key(bf16_bits_to_f32(w[k] >> 16), 8 * i + 2 * k + 1));
                }
            }
        } else {
            for (int i = lo + threadIdx.x; i < hi; i += kArgmaxThreads)
                best = max64(best, argmax_key(bf16_bits_to_f32(row[i]), i));
        }
    } else {
        const float* row = static_cast<const float*>(logits) + size_t(r) * V;
        if (VEC) {
            const float4* rv = reinterpret_cast<const float4*>(row);
#pragma unroll 8
            for (int i = lo + threadIdx.x; i < hi; i += kArgmaxThreads) {
                const float4 q = __ldg(rv + i);
                best = max64(best, argmax_key(q.x, 4 * i));
                best = max64(best, argmax_key(q.y, 4 * i + 1));
                best = max64(best, argmax_key(q.z, 4 * i + 2));
                best = max64(best, argmax_key(q.w, 4 * i + 3));
            }
        } else {
            for (int i = lo + threadIdx.x; i < hi; i += kArgmaxThreads)
                best = max64(best, argmax_key(row[i], i));
        }
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) best = max64(best, __shfl_xor_sync(0xFFFFFFFFu, best, d));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x < 32) {
        best = (threadIdx.x < kArgmaxThreads / 32) ? s_red[threadIdx.x] : 0ull;
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) best = max64(best, __shfl_xor_sync(0xFFFFFFFFu, best, d));
        if (threadIdx.x == 0) s_best = best;
    }
    cl.sync();   // every slice's key is in its CTA's shared memory
    if (c == 0 && threadIdx.x < 32) {
        best = (threadIdx.x < kArgmaxCluster) ? *cl.map_shared_rank(&s_best, threadIdx.x) : 0ull;
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) best = max64(best, __shfl_xor_sync(0xFFFFFFFFu, best, d));
        if (threadIdx.x == 0)
            am[r] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(best & 0xFFFFFFFFu));
    }
    cl.sync();   // no CTA leaves while CTA 0 may still read its key
}

// Span q: draft j (1 <= j <= n_draft) is accepted while every earlier one was
// and it equals the target's token at row j-1; then the bonus token.
__global__ void accept_kernel(const int32_t* __restrict__ am, const int32_t* __restrict__ draft,
                              const int32_t* __restrict__ n_draft, int n_span,
                              int32_t* __restrict__ accept_len, int32_t* __restrict__ out) {
    pdl_wait();
    pdl_launch_dependents();
    const int q = blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= n_span) return;
    const int nd = max(0, min(7, n_draft[q]));
    const int32_t* a = am + size_t(q) * 8;
    const int32_t* d = draft + size_t(q) * 8;
    int m = 0;
    while (m < nd && d[m + 1] == a[m]) ++m;
    int32_t* o = out + size_t(q) * 8;
    for (int j = 0; j < 8; ++j) o[j] = (j < m) ? d[j + 1] : (j == m ? a[m] : -1);
    accept_len[q] = m + 1;
}

}  // namespace

cudaError_t launch_greedy_verify(const void* logits, bool bf16, int V, int R, const int32_t* draft,
                                 const int32_t* n_draft, int32_t* am, int32_t* accept_len,
                                 int32_t* out, cudaStream_t stream) {
    const size_t elem = bf16 ? 2 : 4;
    const bool vec = ((size_t(V) * elem) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    const dim3 grid(static_cast<unsigned>(R) * kArgmaxCluster), block(kArgmaxThreads);
    cudaError_t e;
    if (bf16)
        e = vec ? launch_pdl_cluster(row_argmax_kernel<true, true>, grid, block, kArgmaxCluster, 0,
                                     stream, logits, V, am)
                : launch_pdl_cluster(row_argmax_kernel<true, false>, grid, block, kArgmaxCluster, 0,
                                     stream, logits, V, am);
    else
        e = vec ? launch_pdl_cluster(row_argmax_kernel<false, true>, grid, block, kArgmaxCluster, 0,
                                     stream, logits, V, am)
                : launch_pdl_cluster(row_argmax_kernel<false, false>, grid, block, kArgmaxCluster,
                                     0, stream, logits, V, am);
    if (e != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int n_span = R / 8;
    e = launch_pdl(accept_kernel, dim3((n_span + 127) / 128), dim3(128), 0, stream, am, draft,
                   n_draft, n_span, accept_len, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
