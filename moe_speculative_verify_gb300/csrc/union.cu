// union.cu -- expert union of a batch and the dispatch of its rows (sm_103a).
//
// openinfer #610 "TP8 span row mapping -- single-user speculative decode at
// 186 tok/s", section "What": the union phase over the block's rows, mapping-
// agnostic, deterministic; MoE-Infinity #140, route-ahead prefetch: the
// per-token union of the verify block's routed experts.  mstar #388, FlashInfer
// commit: activations quantised to e4m3 per 128 columns before the fp8 GEMM.
//
// The union is integer work and fully deterministic: per-expert row sets are
// built as bitmaps (order-independent atomics), and positions are assigned by
// walking each bitmap in row order.
#include "common.cuh"
#include "kernels.h"
#include "layout.h"
#include "select.cuh"

namespace moe {

constexpr int kUnionThreads = 1024;

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
        int wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xFFFFFFFFu, wi, d);
            if (lane >= d) wi += o;
        }
        s_warp[lane] = wi - w;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    return s_warp[warp] + incl - v;
}

// Shared memory of the union build, in bytes.
__host__ __device__ inline size_t union_smem_bytes(int R, int E) {
    const size_t words = size_t(E) * (((R + 31) / 32) | 1);
    return words * 4 + ((words + 1) & ~size_t(1)) * 2 + ((R + 15) & ~15) + size_t(4 * E + 8) * 4;
}

// The union of one call, built by one block of kUnionThreads threads from the
// routed ids (global or shared memory); `sm` is union_smem_bytes of shared
// memory, 4-byte aligned.
__device__ void union_block(const int32_t* ids, int R, int E, int K, int S, int n_tile,
                            int32_t* __restrict__ ub, const UnionLayout& L, uint32_t* sm) {
    const int W = (R + 31) / 32;
    // an odd stride between experts: the lanes of a warp that touch word w of
    // different experts then fall on different shared-memory banks (with W a
    // multiple of 32 they all hit one bank)
    const int WS = W | 1;
    uint32_t* bm = sm;                                                   // [E][WS] row bitmaps
    uint16_t* wpre = reinterpret_cast<uint16_t*>(bm + size_t(E) * WS);   // [E][WS] rows before word
    uint8_t* s_valid = reinterpret_cast<uint8_t*>(wpre + ((size_t(E) * WS + 1) & ~size_t(1)));
    int* s_cnt = reinterpret_cast<int*>(s_valid + ((R + 15) & ~15));     // [E+1]
    int* s_off = s_cnt + (E + 1);                                        // [E+2]
    int* s_ioff = s_off + (E + 2);                                       // [E+1]
    __shared__ int s_warp[32];
    __shared__ int s_total, s_err, s_nvalid, s_items, s_nunion;
    const int tid = threadIdx.x;
    const int KS = K + S;

    for (int i = tid; i < E * WS; i += kUnionThreads) bm[i] = 0u;
    if (tid == 0) {
        s_err = 0;
        s_nvalid = 0;
    }
    __syncthreads();

    // 1. row validity: all -1 (pad), or K distinct ids in [0, E)
    for (int r = tid; r < R; r += kUnionThreads) {
        const int32_t* row = ids + size_t(r) * K;
        int rid[MOE_MAX_TOPK];
#pragma unroll
        for (int k = 0; k < MOE_MAX_TOPK; ++k) rid[k] = (k < K) ? row[k] : 0;
        bool pad = true, ok = true;
#pragma unroll
        for (int k = 0; k < MOE_MAX_TOPK; ++k) {
            if (k >= K) break;
            const int e = rid[k];
            if (e != -1) pad = false;
            if (e < 0 || e >= E) ok = false;
#pragma unroll
            for (int j = 0; j < k; ++j)
                if (rid[j] == e) ok = false;
        }
        if (!pad && !ok) atomicExch(&s_err, MOE_ERR_INVALID_ARG);
        const bool v = !pad && ok;
        s_valid[r] = v ? 1 : 0;
        if (v) atomicAdd(&s_nvalid, 1);
    }
    __syncthreads();

    // 2. per-expert row bitmaps (order-independent)
    for (int i = tid; i < R * K; i += kUnionThreads) {
        const int r = i / K;
        if (!s_valid[r]) continue;
        atomicOr(&bm[size_t(ids[i]) * WS + (r >> 5)], 1u << (r & 31));
    }
    __syncthreads();

    // 3. per-expert counts and per-word prefix counts, a thread per expert
    //    (the odd stride puts the experts' words on different banks; at 512
    //    and 4096 rows this measured faster than a warp per expert, 16.4 ->
    //    12.4 and 54.2 -> 51.2 us)
    for (int e = tid; e < E; e += kUnionThreads) {
        int c = 0;
        for (int w = 0; w < W; ++w) {
            wpre[size_t(e) * WS + w] = static_cast<uint16_t>(c);
            c += __popc(bm[size_t(e) * WS + w]);
        }
        s_cnt[e] = c;
    }
    if (tid == 0) s_cnt[E] = S ? s_nvalid : 0;
    __syncthreads();

    // 4. offsets (experts ascending, shared last), union list, item offsets
    //    (the shared entry's items first), by block scans
    const int cnt = (tid <= E) ? s_cnt[tid] : 0;
    const int off = block_exclusive_scan(cnt, s_warp, &s_total);
    if (tid <= E) s_off[tid] = off;
    if (tid == E) s_off[E + 1] = off + cnt;
    const int hit = (tid < E && cnt > 0) ? 1 : 0;
    const int upos = block_exclusive_scan(hit, s_warp, &s_nunion);
    if (hit) ub[L.ulist + upos] = tid;
    const int entry = (tid == 0) ? E : tid - 1;          // item order: shared, 0, 1, ...
    const int nit = (tid <= E) ? (s_cnt[entry] + n_tile - 1) / n_tile : 0;
    const int ioff = block_exclusive_scan(nit, s_warp, &s_items);
    if (tid <= E) s_ioff[entry] = ioff;
    __syncthreads();
    if (tid == 0) {
        ub[L.ulist + s_nunion] = E;
        ub[0] = s_nunion;
        ub[1] = s_nvalid;
        ub[2] = s_off[E + 1];
        ub[3] = s_items;
        ub[4] = n_tile;
        ub[5] = s_err;
        ub[6] = R;
        ub[7] = union_shape_word(E, K, S);
    }
    for (int e = tid; e <= E; e += kUnionThreads) ub[L.counts + e] = s_cnt[e];
    for (int e = tid; e <= E + 1; e += kUnionThreads) ub[L.offsets + e] = s_off[e];

    // 5. routed positions: slot (r, k) of expert e goes after every slot of e
    //    in an earlier row -- offsets[e] + (rows of e before r)
    for (int i = tid; i < R * K; i += kUnionThreads) {
        const int r = i / K, k = i - r * K;
        if (!s_valid[r]) continue;
        const int e = ids[i];
        const int w = r >> 5;
        const uint32_t below = bm[size_t(e) * WS + w] & ((1u << (r & 31)) - 1u);
        const int p = s_off[e] + wpre[size_t(e) * WS + w] + __popc(below);
        ub[L.pos + r * KS + k] = p;
        ub[L.src + p] = r * KS + k;
    }

    // 6. shared positions (valid rows in row order) and pad rows
    const int per = (R + kUnionThreads - 1) / kUnionThreads;
    const int rb = tid * per;
    int local = 0;
    for (int r = rb; r < min(R, rb + per); ++r) local += s_valid[r];
    int rank = block_exclusive_scan(local, s_warp, &s_total);
    for (int r = rb; r < min(R, rb + per); ++r) {
        if (!s_valid[r]) {
            for (int k = 0; k < KS; ++k) ub[L.pos + r * KS + k] = -1;
        } else if (S) {
            const int p = s_off[E] + rank;
            ub[L.pos + r * KS + K] = p;
            ub[L.src + p] = r * KS + K;
            ++rank;
        }
    }

    // 7. work items: rows of each entry in chunks of n_tile
    for (int e = tid; e <= E; e += kUnionThreads) {
        const int c = s_cnt[e];
        for (int j = 0; j * n_tile < c; ++j) {
            int4 item;
            item.x = e;
            item.y = s_off[e] + j * n_tile;
            item.z = min(n_tile, c - j * n_tile);
            // the entry's first item and item count, for the GEMM's tile order
            item.w = s_ioff[e] * 1024 + (c + n_tile - 1) / n_tile;
            reinterpret_cast<int4*>(ub + L.items)[s_ioff[e] + j] = item;
        }
    }
}

__global__ void __launch_bounds__(kUnionThreads) union_kernel(const int32_t* __restrict__ ids,
                                                              int R, int E, int K, int S,
                                                              int n_tile, int32_t* __restrict__ ub,
                                                              UnionLayout L) {
    extern __shared__ uint32_t sm[];
    pdl_wait();
    pdl_launch_dependents();
    union_block(ids, R, E, K, S, n_tile, ub, L, sm);
}

// Selection and union of a small call (R <= kRouteUnionMaxRows) in one block:
// warp w selects rows w, w + 32 (select.cuh), the ids stay in shared memory,
// and the block builds the union from them.  Same decisions and the same
// union buffer as route_select_kernel followed by union_kernel.
__global__ void __launch_bounds__(kUnionThreads) route_union_kernel(
    const float* __restrict__ logits, const float* __restrict__ bias,
    const uint8_t* __restrict__ row_valid, int R, int E, int G, int TG, int K, float scaling,
    int32_t* __restrict__ ids, float* __restrict__ wts, int S, int n_tile,
    int32_t* __restrict__ ub, UnionLayout L) {
    extern __shared__ uint32_t sm[];
    float* s_b = reinterpret_cast<float*>(sm);                         // [32][E]
    int32_t* s_ids = reinterpret_cast<int32_t*>(s_b + 32 * E);         // [R][K]
    uint32_t* s_un = reinterpret_cast<uint32_t*>(s_ids + ((R * K + 3) & ~3));
    pdl_wait();
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = warp; r < R; r += kUnionThreads / 32) {
        int id = -1;
        float w = 0.0f;
        if (row_valid == nullptr || row_valid[r] != 0)
            select_row(logits + size_t(r) * E, bias, E, G, TG, K, scaling, s_b + warp * E, lane,
                       &id, &w);
        if (lane < K) {
            s_ids[r * K + lane] = id;
            ids[size_t(r) * K + lane] = id;
            wts[size_t(r) * K + lane] = w;
        }
    }
    __syncthreads();
    union_block(s_ids, R, E, K, S, n_tile, ub, L, s_un);
}

// Quantise each valid row per 128 columns to e4m3 and write it to its gathered
// positions (K routed slots, then the shared slot).  One warp per (row, block).
__global__ void __launch_bounds__(256) dispatch_kernel(const uint16_t* __restrict__ x,
                                                       const int32_t* __restrict__ ub, UnionLayout L,
                                                       int R, int H, int KS, int32_t ushape,
                                                       uint8_t* __restrict__ xg,
                                                       float* __restrict__ xs,
                                                       int32_t* __restrict__ ready, int n_ready,
                                                       int32_t* __restrict__ err) {
    pdl_wait();
    pdl_launch_dependents();
    // the fused expert GEMM's per-item counters start at zero every call
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < n_ready; i += blockDim.x) ready[i] = 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x;
    const int HB = H / kBlock;
    const int b = blockIdx.y * 8 + warp;
    // the union's shape words, the row's first position and the x block are
    // requested together (none of their addresses depends on the union's
    // contents), then checked
    const int32_t* pos = ub + L.pos + size_t(r) * KS;
    const int p0 = (b < HB) ? pos[0] : -1;
    uint2 xv = make_uint2(0u, 0u);
    if (b < HB) xv = __ldg(reinterpret_cast<const uint2*>(x + size_t(r) * H + b * kBlock + 4 * lane));
    // a union built for another call: its positions may lie outside xg
    if (!union_fits(ub, R, ushape)) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            record_error(err, MOE_ERR_INVALID_ARG);
        return;
    }
    if (b >= HB || p0 < 0) return;  // past the row's blocks, or a pad row
    const float f0 = bf16_bits_to_f32(xv.x & 0xFFFFu), f1 = bf16_bits_to_f32(xv.x >> 16);
    const float f2 = bf16_bits_to_f32(xv.y & 0xFFFFu), f3 = bf16_bits_to_f32(xv.y >> 16);
    float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, d));
    const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
    const uint32_t q = to_e4m3x4(__fdiv_rn(f0, sc), __fdiv_rn(f1, sc), __fdiv_rn(f2, sc),
                                 __fdiv_rn(f3, sc));
    for (int k = 0; k < KS; ++k) {
        const int p = (k == 0) ? p0 : pos[k];
        reinterpret_cast<uint32_t*>(xg + size_t(p) * H + b * kBlock)[lane] = q;
        if (lane == 0) xs[size_t(p) * HB + b] = sc;
    }
}

cudaError_t launch_union(const int32_t* ids, int R, int E, int K, int S, int n_tile,
                         int32_t* ub, const UnionLayout& L, cudaStream_t stream) {
    const size_t smem = union_smem_bytes(R, E);
    cudaError_t e =
        ensure_dyn_smem(reinterpret_cast<const void*>(union_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_pdl(union_kernel, dim3(1), dim3(kUnionThreads), smem, stream, ids, R, E, K, S, n_tile,
                   ub, L);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_dispatch(const uint16_t* x, const int32_t* ub, const UnionLayout& L, int R,
                            int H, int KS, int32_t ushape, uint8_t* xg, float* xs, int32_t* ready,
                            int n_ready, int32_t* err, cudaStream_t stream) {
    const int HB = H / kBlock;
    dim3 grid(R, (HB + 7) / 8);
    cudaError_t e = launch_pdl(dispatch_kernel, grid, dim3(256), 0, stream, x, ub, L, R, H, KS,
                               ushape, xg, xs, ready, n_ready, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_route_union(const float* logits, const float* bias, const uint8_t* row_valid,
                               int R, int E, int G, int TG, int K, float scaling, int32_t* ids,
                               float* wts, int S, int n_tile, int32_t* ub, const UnionLayout& L,
                               cudaStream_t stream) {
    if (R > kRouteUnionMaxRows) return cudaErrorInvalidValue;
    const size_t smem = size_t(32) * E * 4 + size_t((R * K + 3) & ~3) * 4 + union_smem_bytes(R, E);
    cudaError_t e =
        ensure_dyn_smem(reinterpret_cast<const void*>(route_union_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = launch_pdl(route_union_kernel, dim3(1), dim3(kUnionThreads), smem, stream, logits, bias,
                   row_valid, R, E, G, TG, K, scaling, ids, wts, S, n_tile, ub, L);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
