// ffn.cu -- block-scaled e4m3 expert GEMMs on tcgen05 tensor cores (sm_103a).
//
// openinfer #610 "TP8 span row mapping -- single-user speculative decode at
// 186 tok/s", section "What": gate/up GEMM + SiLU, then the down GEMM, over
// the expert union, with fixed-order reductions.  mstar #388 "Speed up
// GLM-5.2 with fp8 kernels and one-graph MTP": fp8 experts (routed and
// shared) with 128x128 block scales; activations quantised to e4m3 per 128
// columns (FlashInfer commit).  MoE-Infinity #140: expert tensors
// [gate_proj, up_proj, down_proj], output-major.
//
// One persistent kernel per GEMM.  Work = (item, 128-row block of the output
// features); an item is up to NT gathered rows of one expert (union entry).
// Swap-AB: the weight tile is the MMA's A operand (M = 128 output features),
// the rows are the B operand (N = NT), so a verify batch of a few rows still
// fills the 128-row MMA.  Per 128-wide K-block the MMA writes a fresh fp32
// partial to tensor memory; the epilogue warps read it back and fold it into
// fp32 register accumulators with the block's weight scale times the row's
// activation scale (fp32 128x128 scales cannot be expressed in the MMA's own
// block-scale format).
//
// Warp roles (one CTA per SM):
//   warp 0 lane 0: TMA producer -- weight tiles (evict-first) and row tiles
//                  into an n_stages ring of shared-memory stages;
//   warp 1 lane 0: MMA issuer -- 4 x tcgen05.mma (K = 32) per operand per
//                  K-block into a ring of ACC_BUFS tensor-memory partials;
//   warps 2.. : epilogue -- 4 * NT/16 warps; warp w reads TMEM lanes
//                  32*(w%4).. and 16 columns, promotes the partials, then
//                  gate/up: h = silu(g) * u, per-row 1x128 e4m3 quantisation
//                  of h, coalesced row stores; down: fp32 rows to their slot.
// Every barrier wait is bounded; a timeout records MOE_ERR_TIMEOUT, winds the
// roles down, drains in-flight copies and MMAs, frees tensor memory, returns.
#include "common.cuh"
#include "kernels.h"
#include "layout.h"

namespace moe {

template <int NT, bool GU>
struct FfnCfg {
    static constexpr int NA = GU ? 2 : 1;            // weight operands per stage
    static constexpr int A_BYTES = 128 * 128;
    static constexpr int B_BYTES = NT * 128;
    static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
    static constexpr int CSPLIT = NT / 16;
    static constexpr int EPI_WARPS = 4 * CSPLIT;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int THREADS = 64 + EPI_THREADS;
    static constexpr int ACC_BUFS = 4;
    static constexpr int ACC_COLS = NA * NT;
    static constexpr int TMEM_COLS = (ACC_BUFS * ACC_COLS <= 32) ? 32
                                     : (ACC_BUFS * ACC_COLS <= 64) ? 64
                                     : (ACC_BUFS * ACC_COLS <= 128) ? 128
                                     : (ACC_BUFS * ACC_COLS <= 256) ? 256 : 512;
    static_assert(ACC_BUFS * ACC_COLS <= 512, "tensor memory");
};

// Shared-memory carve-up, identical on host (size) and device (pointers).
struct FfnSmem {
    int stages, sa, sw, red, tile, src, bars, tmem, flag, bytes;
};

__host__ __device__ inline FfnSmem ffn_smem(int nt, int na, int n_stages, int kb, int stage_bytes) {
    FfnSmem s;
    int b = 0;
    s.stages = b;
    b += n_stages * stage_bytes;
    s.sa = b;
    b += nt * kb * 4;
    s.sw = b;
    b += na * kb * 4;
    s.red = b;
    b += 4 * nt * 4;
    s.tile = b;
    b += nt * 128;
    s.src = b;
    b += nt * 4;
    b = (b + 7) & ~7;
    s.bars = b;
    b += (2 * n_stages + 2 * 8 + 1) * 8;
    s.tmem = b;
    b += 4;
    s.flag = b;
    b += 4;
    s.bytes = b + 1024;  // slack to align the base to 1024 bytes
    return s;
}

// AND of `ok` over the epilogue threads, at a named barrier.
__device__ __forceinline__ bool epi_bar_and(bool ok, int nthreads) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1 : 0), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <int NT, bool GU>
__global__ void __launch_bounds__(FfnCfg<NT, GU>::THREADS, 1)
    ffn_kernel(const __grid_constant__ CUtensorMap map_a0, const __grid_constant__ CUtensorMap map_a1,
               const __grid_constant__ CUtensorMap map_sh0,
               const __grid_constant__ CUtensorMap map_sh1,
               const __grid_constant__ CUtensorMap map_b, const FfnArgs p) {
    using C = FfnCfg<NT, GU>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int KB = p.Kd / kBlock;
    const int MB = p.M / kBlock;
    const FfnSmem L = ffn_smem(NT, C::NA, p.n_stages, KB, C::STAGE_BYTES);
    uint8_t* st_base = smem + L.stages;
    float* s_sa = reinterpret_cast<float*>(smem + L.sa);     // [NT][KB]
    float* s_sw = reinterpret_cast<float*>(smem + L.sw);     // [NA][KB]
    float* s_red = reinterpret_cast<float*>(smem + L.red);   // [4][NT]
    uint8_t* s_tile = smem + L.tile;                         // [NT][128]
    int* s_src = reinterpret_cast<int*>(smem + L.src);       // [NT]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + p.n_stages;
    uint64_t* acc_full = empty + p.n_stages;
    uint64_t* acc_empty = acc_full + 8;
    uint64_t* drain = acc_empty + 8;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.tmem);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.flag);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < C::ACC_BUFS; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], C::EPI_WARPS);
        }
        mbar_init(drain, 1);
        *s_abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&map_a0);
        prefetch_tensormap(&map_b);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // Items must have been cut to this kernel's row tile.
    const int n_items = (p.ub[4] == NT) ? p.ub[3] : 0;
    if (threadIdx.x == 0 && p.ub[4] != NT && p.ub[3] > 0) record_error(p.err, MOE_ERR_INVALID_ARG);
    const int n_tiles = n_items * MB;
    const int4* items = reinterpret_cast<const int4*>(p.ub + p.ul.items);
    uint32_t issued = 0;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            for (int t = blockIdx.x; t < n_tiles && !*s_abort; t += gridDim.x) {
                const int4 it = items[t / MB];
                const int mb = t % MB;
                const bool sh = it.x == p.E;
                const CUtensorMap* m0 = sh ? &map_sh0 : &map_a0;
                const CUtensorMap* m1 = sh ? &map_sh1 : &map_a1;
                const int arow = (sh ? 0 : it.x) * p.M + mb * kBlock;
                bool ok = true;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    uint8_t* st = st_base + stage * C::STAGE_BYTES;
                    tma_load_2d_hint(st, m0, &full[stage], kb * kBlock, arow, pol);
                    if (GU) tma_load_2d_hint(st + C::A_BYTES, m1, &full[stage], kb * kBlock, arow, pol);
                    tma_load_2d(st + C::NA * C::A_BYTES, &map_b, &full[stage], kb * kBlock, it.y);
                    ++issued;
                    if (++stage == p.n_stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) {
                    *s_abort = 1;
                    break;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------- MMA issuer
            constexpr uint32_t idesc = idesc_e4m3_f32(128, NT);
            int stage = 0, ab = 0;
            uint32_t phase = 0, aph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (*s_abort || !mbar_wait(&acc_empty[ab], aph ^ 1u, p.err, p.timeout_ns) ||
                        !mbar_wait(&full[stage], phase, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(st_base + stage * C::STAGE_BYTES);
                    const uint32_t bb = a0 + C::NA * C::A_BYTES;
                    const uint32_t d0 = tmem + ab * C::ACC_COLS;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mma_e4m3(d0, sdesc_k_sw128(a0 + 32 * k), sdesc_k_sw128(bb + 32 * k), idesc,
                                 k > 0);
                        if (GU)
                            mma_e4m3(d0 + NT, sdesc_k_sw128(a0 + C::A_BYTES + 32 * k),
                                     sdesc_k_sw128(bb + 32 * k), idesc, k > 0);
                    }
                    mma_commit(&empty[stage]);
                    mma_commit(&acc_full[ab]);
                    if (++stage == p.n_stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++ab == C::ACC_BUFS) {
                        ab = 0;
                        aph ^= 1u;
                    }
                }
            }
            if (!ok) *s_abort = 1;
        }
    } else {
        // ----------------------------------------------------- epilogue
        const int ew = warp - 2;
        const int q = warp & 3;          // TMEM lane quadrant this warp may access
        const int cg = ew >> 2;          // 16-column group
        const int m = 32 * q + lane;     // output feature inside the 128-row block
        const int et = threadIdx.x - 64; // 0 .. EPI_THREADS-1
        int ab = 0;
        uint32_t aph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            const int4 it = items[t / MB];
            const int mb = t % MB;
            const bool sh = it.x == p.E;
            const int ex = sh ? 0 : it.x;
            const int row0 = it.y, nrow = it.z;
            // previous tile's readers are done with the scale / tile buffers
            ok = epi_bar_and(ok, C::EPI_THREADS);
            if (!ok) break;
            for (int i = et; i < NT * KB; i += C::EPI_THREADS) {
                const int n = i / KB, kb = i - n * KB;
                s_sa[i] = (n < nrow) ? p.bs[size_t(row0 + n) * KB + kb] : 0.0f;
            }
            for (int i = et; i < C::NA * KB; i += C::EPI_THREADS) {
                const int a = i / KB, kb = i - a * KB;
                const float* sp = (a == 0) ? (sh ? p.sh_s_a0 : p.s_a0) : (sh ? p.sh_s_a1 : p.s_a1);
                s_sw[i] = sp[(size_t(ex) * MB + mb) * KB + kb];
            }
            if (!GU)
                for (int i = et; i < NT; i += C::EPI_THREADS)
                    s_src[i] = (i < nrow) ? p.ub[p.ul.src + row0 + i] : -1;
            ok = epi_bar_and(ok, C::EPI_THREADS);
            if (!ok) break;

            float acc0[16], acc1[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                acc0[j] = 0.0f;
                acc1[j] = 0.0f;
            }
            for (int kb = 0; kb < KB && ok; ++kb) {
                if (!mbar_wait(&acc_full[ab], aph, p.err, p.timeout_ns)) {
                    ok = false;
                    *s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                                    ab * C::ACC_COLS + cg * 16;
                float v0[16], v1[16];
                tmem_ld16(ta, v0);
                if (GU) tmem_ld16(ta + NT, v1);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
                const float w0 = s_sw[kb];
                const float w1 = GU ? s_sw[KB + kb] : 0.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float a = s_sa[(cg * 16 + j) * KB + kb];
                    acc0[j] = fmaf(v0[j], w0 * a, acc0[j]);
                    if (GU) acc1[j] = fmaf(v1[j], w1 * a, acc1[j]);
                }
                if (++ab == C::ACC_BUFS) {
                    ab = 0;
                    aph ^= 1u;
                }
            }
            if (GU) {
                // h = silu(g) * u; per-row amax over the 128 features
                float h[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = cg * 16 + j;
                    const float g = acc0[j];
                    h[j] = (c < nrow) ? (g / (1.0f + __expf(-g))) * acc1[j] : 0.0f;
                    float a = fabsf(h[j]);
#pragma unroll
                    for (int d = 16; d >= 1; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, d));
                    if (lane == 0) s_red[q * NT + c] = a;
                }
                ok = epi_bar_and(ok, C::EPI_THREADS);
                if (!ok) break;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = cg * 16 + j;
                    const float amax = fmaxf(fmaxf(s_red[c], s_red[NT + c]),
                                             fmaxf(s_red[2 * NT + c], s_red[3 * NT + c]));
                    const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
                    s_tile[c * 128 + m] = to_e4m3(__fdiv_rn(h[j], sc));
                    if (m == 0 && c < nrow) p.hs[size_t(row0 + c) * MB + mb] = sc;
                }
                ok = epi_bar_and(ok, C::EPI_THREADS);
                if (!ok) break;
                for (int i = et; i < nrow * 8; i += C::EPI_THREADS) {
                    const int c = i >> 3, ch = i & 7;
                    *reinterpret_cast<uint4*>(p.hq + size_t(row0 + c) * p.M + mb * kBlock + ch * 16) =
                        *reinterpret_cast<const uint4*>(s_tile + c * 128 + ch * 16);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = cg * 16 + j;
                    if (ok && c < nrow) {
                        const int slot = s_src[c];
                        const int r = slot / p.KS, k = slot - r * p.KS;
                        float* dst = (k < p.K) ? p.y_slots + (size_t(r) * p.K + k) * p.M
                                               : p.y_shared + size_t(r) * p.M;
                        dst[mb * kBlock + m] = acc0[j];
                    }
                }
            }
        }
        if (!ok) *s_abort = 1;
    }

    __syncthreads();
    if (*s_abort) {
        // Wind down: let every copy this CTA issued land and every MMA finish
        // before the CTA releases tensor memory and exits.
        if (threadIdx.x == 0) {
            const uint32_t first = issued > static_cast<uint32_t>(p.n_stages)
                                       ? issued - static_cast<uint32_t>(p.n_stages) : 0u;
            for (uint32_t i = first; i < issued; ++i)
                mbar_wait(&full[i % p.n_stages], (i / p.n_stages) & 1u, nullptr, p.timeout_ns);
        }
        if (threadIdx.x == 32) {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, p.timeout_ns);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------- launchers ----
template <int NT, bool GU>
static cudaError_t launch_ffn_t(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& sh0,
                                const CUtensorMap& sh1, const CUtensorMap& b, FfnArgs args,
                                int n_sms, int max_tiles, int smem_limit, cudaStream_t stream) {
    using C = FfnCfg<NT, GU>;
    const int KB = args.Kd / kBlock;
    int stages = 12;
    FfnSmem L = ffn_smem(NT, C::NA, stages, KB, C::STAGE_BYTES);
    while (stages > 2 && L.bytes > smem_limit) {
        --stages;
        L = ffn_smem(NT, C::NA, stages, KB, C::STAGE_BYTES);
    }
    if (L.bytes > smem_limit) return cudaErrorInvalidConfiguration;
    args.n_stages = stages;
    cudaError_t e = cudaFuncSetAttribute(ffn_kernel<NT, GU>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L.bytes);
    if (e != cudaSuccess) return e;
    const int grid = max(1, min(n_sms, max_tiles));
    ffn_kernel<NT, GU><<<grid, C::THREADS, L.bytes, stream>>>(a0, a1, sh0, sh1, b, args);
    return cudaGetLastError();
}

cudaError_t launch_ffn(int nt, bool gate_up, const CUtensorMap& a0, const CUtensorMap& a1,
                       const CUtensorMap& sh0, const CUtensorMap& sh1, const CUtensorMap& b,
                       const FfnArgs& args, int n_sms, int max_tiles, int smem_limit,
                       cudaStream_t stream) {
    if (gate_up) {
        switch (nt) {
            case 16: return launch_ffn_t<16, true>(a0, a1, sh0, sh1, b, args, n_sms, max_tiles, smem_limit, stream);
            case 32: return launch_ffn_t<32, true>(a0, a1, sh0, sh1, b, args, n_sms, max_tiles, smem_limit, stream);
            case 64: return launch_ffn_t<64, true>(a0, a1, sh0, sh1, b, args, n_sms, max_tiles, smem_limit, stream);
        }
    } else {
        switch (nt) {
            case 16: return launch_ffn_t<16, false>(a0, a1, sh0, sh1, b, args, n_sms, max_tiles, smem_limit, stream);
            case 32: return launch_ffn_t<32, false>(a0, a1, sh0, sh1, b, args, n_sms, max_tiles, smem_limit, stream);
            case 64: return launch_ffn_t<64, false>(a0, a1, sh0, sh1, b, args, n_sms, max_tiles, smem_limit, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
