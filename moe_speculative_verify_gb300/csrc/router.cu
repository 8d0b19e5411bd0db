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
#include <atomic>

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

// Large-R variant, persistent (one CTA per SM): tiles of LR = 4 * RT rows x
// kLE experts, tile t at rows (t / n_eb) * LR and experts (t % n_eb) * kLE,
// taken by the CTAs in turn.  Consumer warp w owns the tile's rows
// (w / 2) * RT .. +RT-1 and experts (w % 2) * 16 .. +15, and lane l of the
// warp is lane l of the reduction tree for those RT * 16 (row, expert) pairs:
// each row's x is widened from bf16 once for 16 experts (measured at 4096
// rows: 319.5 -> 309.2 us against 16 rows x 8 experts, at 25 % more
// shared-memory reads).  RT = 6 to 9 (24- to 36-row tiles), as
// router_rows_per_warp chooses.
//
// Per stage of kLCols columns, x [kLR][kLCols] bf16 and w [kLE][kLCols] fp32
// arrive by TMA in a ring of kLStages slots (a full and an empty barrier
// each).  Warpgroup 0 is the producer: its thread 0 waits for a slot's empty
// phase and refills it; the 8 consumer warps of warpgroups 1 and 2 only wait
// for full slots and arrive on empty ones (no round trip), so they drift apart
// instead of meeting at every stage.  The producer warpgroup gives up its
// registers (setmaxnreg: 40 a thread) to the consumers (232), whose RT x 16
// pair tiles need them: 4 x 32 x 40 + 8 x 32 x 232 = 384 x 168, the launch's.
// A thread forms its lane partials
// of the current 1024-column chunk in registers (fma in column order) and
// folds them at the chunk's end into the chunk sums held in tensor memory
// (q = p for the first chunk, q = q + p after): shared memory carries only x
// and w.  The last chunk's sums stay in registers and the warp finishes the
// tree by recursive halving: at distance d = 16 .. 1 each lane keeps half of
// its values and adds its partner's copy of them, which are the xor
// butterfly's additions (v[l] + v[l ^ d], IEEE addition commutes) with every
// value summed in one lane only; lane l ends with pairs RT*l/2 .. RT*l/2 + RT/2 - 1
// (for odd RT the last level's sums are formed in both lanes of a pair and
// stored alternately).  The same IEEE operations in the same order as the
// small-R kernel, at every RT.
constexpr int kLE = 32;
constexpr int kLPE = 16;                                    // experts of a thread
constexpr int kLWarps = 4 * (kLE / kLPE);                   // consumer warps
constexpr int kLThreads = 32 * (4 + kLWarps);              // + the producer warpgroup
constexpr int kLProdRegs = 40, kLConsRegs = 232, kLLaunchRegs = 65536 / kLThreads / 8 * 8;
static_assert(kLWarps == 8, "two consumer warpgroups");
static_assert(128 * kLProdRegs + 32 * kLWarps * kLConsRegs <= kLThreads * kLLaunchRegs,
              "register split within the launch's registers");
constexpr int kLCols = kRouterStageCols;                 // columns per stage
constexpr int kLBlk = kLCols / 128;                      // 128-column blocks per stage
constexpr int kLStages = 1024 / kLCols;                  // up to 192 KB of stages
constexpr int kLWBytes = kLE * kLCols * 4;
static_assert(kLBlk >= 1 && 8 % kLBlk == 0, "a stage holds whole blocks of one chunk");
template <int RT>
struct RouterTile {
    static constexpr int LR = 4 * RT;                    // rows of a tile
    static constexpr int NP = RT * kLPE;                 // pairs of a thread
    static constexpr int XBytes = LR * kLCols * 2;
    static constexpr int StageBytes = XBytes + kLWBytes;
    static constexpr size_t Smem = size_t(kLStages) * StageBytes + 256;
    // chunk sums: the two warps of a lane quarter at columns 0 and NPCols
    // (32-column aligned), in a power-of-two allocation
    static constexpr int NPCols = (NP + 31) / 32 * 32;
    static constexpr uint32_t TmemCols = ((kLWarps / 4) * NPCols <= 256) ? 256u : 512u;
    static_assert(NP % 16 == 0 && (kLWarps / 4) * NPCols <= int(TmemCols), "pairs per lane, TMEM");
    static_assert(XBytes % 128 == 0 && StageBytes % 128 == 0, "TMA destinations 128-byte aligned");
};

__device__ __forceinline__ void tmem_st32f(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
        "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
        "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
        "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16f(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
        "f"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One recursive-halving level over the first N values at xor distance D.
template <int M, int N, int D>
__device__ __forceinline__ void halve(float (&v)[M], int lane) {
    const bool upper = (lane & D) != 0;
#pragma unroll
    for (int j = 0; j < N / 2; ++j) {
        const float send = upper ? v[j] : v[j + N / 2];
        const float keep = upper ? v[j + N / 2] : v[j];
        v[j] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, D));
    }
}

template <int RT>
__global__ void __launch_bounds__(kLThreads, 1) router_logits_tma_kernel(
    const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
    const uint8_t* __restrict__ row_valid, int R, int H, int E, float* __restrict__ logits,
    int32_t* err, uint64_t timeout_ns) {
    using T = RouterTile<RT>;
    constexpr int kLR = T::LR, kLRT = RT, kLNP = T::NP;
    // the weight columns of a block held for 8 experts at a time (each x row
    // then widened twice), which frees 32 registers for the RT x 16
    // accumulators: measured at 4096 rows, 316.0 -> 295.4 us at RT = 9 and
    // 308.3 -> 305.1 at RT = 8; 2048 rows at RT = 7 170.0 -> 167.2 us
    constexpr int kEG = (RT >= 7) ? 2 : 1;
    constexpr int kLXBytes = T::XBytes, kLStageBytes = T::StageBytes;
    extern __shared__ __align__(1024) uint8_t lsm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(lsm + kLStages * kLStageBytes);
    uint64_t* empty = full + kLStages;                               // consumers done with it
    int32_t* last = reinterpret_cast<int32_t*>(empty + kLStages);    // last stage load issued
    uint32_t* tslot = reinterpret_cast<uint32_t*>(last + kLStages);
    volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_eb = (E + kLE - 1) / kLE;
    const int n_tiles = ((R + kLR - 1) / kLR) * n_eb;
    const int NB = H / 128;                       // 128-column blocks
    const int NSt = (NB + kLBlk - 1) / kLBlk;     // stages per tile
    const int my_tiles =
        static_cast<int>(blockIdx.x) < n_tiles ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int G = my_tiles * NSt;   // this CTA's stage loads, over all its tiles

    // load g into ring slot g % kLStages (one thread); columns past H read as 0
    auto issue = [&](int g) {
        const int st = g % kLStages, s = g % NSt;
        const int t = blockIdx.x + (g / NSt) * gridDim.x;
        uint8_t* base = lsm + st * kLStageBytes;
        last[st] = g;
        mbar_arrive_expect_tx(&full[st], kLStageBytes);
        tma_load_2d(base, &xmap, &full[st], s * kLCols, (t / n_eb) * kLR);
        tma_load_2d(base + kLXBytes, &wmap, &full[st], s * kLCols, (t % n_eb) * kLE);
    };

    if (tid == 0) {
        prefetch_tensormap(&xmap);
        prefetch_tensormap(&wmap);
        for (int i = 0; i < kLStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kLWarps);
            last[i] = -1;
        }
        *s_abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, T::TmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_wait();   // x may be written by the previous kernel
    pdl_launch_dependents();

    bool ok = true;
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLProdRegs));
        if (tid == 0) {
            // every stage load in order; slot reuse waits for its empty phase
            for (int n = 0; n < G && ok; ++n) {
                const int st = n % kLStages;
                if (n >= kLStages) {
                    const uint32_t par = ((n / kLStages) - 1) & 1;
                    uint64_t t0 = 0;
                    for (uint32_t it = 0; !mbar_try_wait<20000>(&empty[st], par); ++it) {
                        if (it == 0) t0 = globaltimer_ns();
                        if (*s_abort || globaltimer_ns() - t0 > timeout_ns || it >= (1u << 30)) {
                            if (!*s_abort) record_error(err, MOE_ERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                issue(n);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kLConsRegs));
        const int cw = warp - 4;   // consumer warp
        const int wrow = (cw / (kLE / kLPE)) * kLRT, wexp = (cw % (kLE / kLPE)) * kLPE;
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) +
                            static_cast<uint32_t>(cw >> 2) * T::NPCols;
        int g = 0;
        for (int ti = 0; ti < my_tiles && ok; ++ti) {
            const int t = blockIdx.x + ti * gridDim.x;
            float p[kLNP];   // pair k = kLPE * row + expert of the warp's kLRT x kLPE
            // p += the chunk sums held in tensor memory, 32 pairs a load and
            // two loads in flight per wait (a last 16 pairs where RT is odd)
            auto fold = [&](float (&pp)[kLNP]) {
#pragma unroll
                for (int j = 0; j < kLNP / 32; j += 2) {
                    float q0[32], q1[32];
                    tmem_ld32(tq + 32 * j, q0);
                    if (j + 1 < kLNP / 32) tmem_ld32(tq + 32 * (j + 1), q1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) pp[32 * j + i] = __fadd_rn(q0[i], pp[32 * j + i]);
                    if (j + 1 < kLNP / 32) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            pp[32 * (j + 1) + i] = __fadd_rn(q1[i], pp[32 * (j + 1) + i]);
                    }
                }
                if constexpr (kLNP % 32 != 0) {
                    constexpr int j0 = kLNP - 16;
                    float q0[16];
                    tmem_ld16(tq + j0, q0);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) pp[j0 + i] = __fadd_rn(q0[i], pp[j0 + i]);
                }
            };
            for (int s = 0; s < NSt; ++s, ++g) {
                const int st = g % kLStages;
                const uint32_t par = (g / kLStages) & 1;
                // the outcome is made uniform across the warp before use
                bool got = mbar_try_wait(&full[st], par);
                if (!got) got = !*s_abort && mbar_wait(&full[st], par, err, timeout_ns);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    ok = false;
                    break;
                }
                const uint16_t* xs = reinterpret_cast<const uint16_t*>(lsm + st * kLStageBytes);
                const float* ws = reinterpret_cast<const float*>(lsm + st * kLStageBytes + kLXBytes);
#pragma unroll
                for (int i = 0; i < kLBlk; ++i) {
                    const int blk = s * kLBlk + i;
                    if (blk < NB) {
                        if ((blk & 7) == 0) {
#pragma unroll
                            for (int k = 0; k < kLNP; ++k) p[k] = 0.0f;
                        }
#pragma unroll
                        for (int eg = 0; eg < kEG; ++eg) {
                            float4 wv[kLPE / kEG];
#pragma unroll
                            for (int b = 0; b < kLPE / kEG; ++b)
                                wv[b] = *reinterpret_cast<const float4*>(
                                    ws + (wexp + eg * (kLPE / kEG) + b) * kLCols + i * 128 + 4 * lane);
#pragma unroll
                            for (int a = 0; a < kLRT; ++a) {
                                const uint2 xv = *reinterpret_cast<const uint2*>(
                                    xs + (wrow + a) * kLCols + i * 128 + 4 * lane);
                                const float x0 = bf16_bits_to_f32(xv.x & 0xFFFFu);
                                const float x1 = bf16_bits_to_f32(xv.x >> 16);
                                const float x2 = bf16_bits_to_f32(xv.y & 0xFFFFu);
                                const float x3 = bf16_bits_to_f32(xv.y >> 16);
#pragma unroll
                                for (int b = 0; b < kLPE / kEG; ++b) {
                                    const int k = a * kLPE + eg * (kLPE / kEG) + b;
                                    float q = p[k];
                                    q = __fmaf_rn(x0, wv[b].x, q);
                                    q = __fmaf_rn(x1, wv[b].y, q);
                                    q = __fmaf_rn(x2, wv[b].z, q);
                                    q = __fmaf_rn(x3, wv[b].w, q);
                                    p[k] = q;
                                }
                            }
                        }
                    }
                }
                // this warp is done with the slot
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
                // a chunk's end before the tile's last block: q = p (first chunk)
                // or q = q + p, 32 pairs at a time
                const int lastblk = min(s * kLBlk + kLBlk, NB) - 1;
                if ((lastblk & 7) == 7 && lastblk != NB - 1) {
                    __syncwarp();
                    if (lastblk >= 8) fold(p);
#pragma unroll
                    for (int j = 0; j < kLNP / 32; ++j) tmem_st32f(tq + 32 * j, p + 32 * j);
                    if constexpr (kLNP % 32 != 0) tmem_st16f(tq + kLNP - 16, p + kLNP - 16);
                    tmem_wait_st();
                }
            }
            if (!ok) break;
            if (NB > 8) {   // the last chunk: q + p, kept in registers
                __syncwarp();
                fold(p);
            }
            halve<kLNP, kLNP, 16>(p, lane);
            halve<kLNP, kLNP / 2, 8>(p, lane);
            halve<kLNP, kLNP / 4, 4>(p, lane);
            halve<kLNP, kLNP / 8, 2>(p, lane);
            // lanes 2m and 2m+1 now hold the same RT pairs, RT*m .. RT*m + RT-1
            const int r0 = (t / n_eb) * kLR + wrow;
            const int e0 = (t % n_eb) * kLE + wexp;
            if constexpr (kLRT % 2 == 0) {
                halve<kLNP, kLRT, 1>(p, lane);
                // lane l holds pairs NL*l .. NL*l + NL-1 (NL = RT / 2), pair k
                // being row k / kLPE and expert k % kLPE of the warp's block
                constexpr int NL = kLRT / 2;
#pragma unroll
                for (int j = 0; j < NL; ++j) {
                    const int k = NL * lane + j;
                    const int r = r0 + k / kLPE, e = e0 + k % kLPE;
                    if (r < R && e < E && (row_valid == nullptr || row_valid[r] != 0))
                        logits[size_t(r) * E + e] = p[j];
                }
            } else {
                // RT pairs do not halve: both lanes of a pair form the last
                // level's sums (the same bits: IEEE addition commutes) and
                // store alternate ones
#pragma unroll
                for (int j = 0; j < kLRT; ++j) p[j] = __fadd_rn(p[j], __shfl_xor_sync(0xFFFFFFFFu, p[j], 1));
#pragma unroll
                for (int j = 0; j < kLRT; ++j) {
                    const int k = kLRT * (lane >> 1) + j;
                    const int r = r0 + k / kLPE, e = e0 + k % kLPE;
                    if ((j & 1) == (lane & 1) && r < R && e < E &&
                        (row_valid == nullptr || row_valid[r] != 0))
                        logits[size_t(r) * E + e] = p[j];
                }
            }
        }
    }
    if (!ok) *s_abort = 1;

    __syncthreads();
    if (*s_abort && tid == 0) {
        // let every copy issued land before the CTA exits (bounded)
        constexpr uint64_t kDrainNs = 2000000;
        const uint64_t t0 = globaltimer_ns();
        for (int i = 0; i < kLStages; ++i) {
            if (last[i] < 0) continue;
            const uint64_t used = globaltimer_ns() - t0;
            if (used >= kDrainNs) break;
            mbar_wait(&full[i], (last[i] / kLStages) & 1, nullptr, kDrainNs - used);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TmemCols);
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
template <int RT>
static cudaError_t launch_router_tma(const CUtensorMap& xmap, const CUtensorMap& wmap,
                                     const uint8_t* row_valid, int R, int H, int E, float* logits,
                                     int n_sms, int32_t* err, uint64_t timeout_ns,
                                     cudaStream_t stream) {
    using T = RouterTile<RT>;
    const int n_tiles = ((R + T::LR - 1) / T::LR) * ((E + kLE - 1) / kLE);
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(router_logits_tma_kernel<RT>),
                                    static_cast<int>(T::Smem));
    if (e != cudaSuccess) return e;
    // the warpgroups' register split needs the launch's full share (the
    // compiled count, read once)
    static std::atomic<int> regs{0};
    if (regs.load(std::memory_order_relaxed) == 0) {
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, router_logits_tma_kernel<RT>)) != cudaSuccess) return e;
        regs.store(fa.numRegs, std::memory_order_relaxed);
    }
    if (regs.load(std::memory_order_relaxed) < kLLaunchRegs) return cudaErrorInvalidConfiguration;
    return launch_pdl(router_logits_tma_kernel<RT>, dim3(min(n_tiles, max(n_sms, 1))),
                      dim3(kLThreads), T::Smem, stream, xmap, wmap, row_valid, R, H, E, logits,
                      err, timeout_ns);
}

cudaError_t launch_router_logits(const uint16_t* x, const float* wr, const uint8_t* row_valid,
                                 int R, int H, int E, float* logits, const RouterMaps* maps,
                                 int n_sms, int32_t* err, uint64_t timeout_ns,
                                 cudaStream_t stream) {
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
        if (maps == nullptr) return cudaErrorInvalidValue;
        cudaError_t e;
        switch (maps->rt) {
            case 6: e = launch_router_tma<6>(maps->x, maps->w, row_valid, R, H, E, logits, n_sms, err, timeout_ns, stream); break;
            case 7: e = launch_router_tma<7>(maps->x, maps->w, row_valid, R, H, E, logits, n_sms, err, timeout_ns, stream); break;
            case 8: e = launch_router_tma<8>(maps->x, maps->w, row_valid, R, H, E, logits, n_sms, err, timeout_ns, stream); break;
            case 9: e = launch_router_tma<9>(maps->x, maps->w, row_valid, R, H, E, logits, n_sms, err, timeout_ns, stream); break;
            default: return cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_router(const uint16_t* x, const float* wr, const float* bias,
                          const uint8_t* row_valid, int R, int H, int E, int G, int TG, int K,
                          float scaling, int32_t* ids, float* wts, float* logits,
                          const RouterMaps* maps, int n_sms, int32_t* err, uint64_t timeout_ns,
                          cudaStream_t stream) {
    cudaError_t e = launch_router_logits(x, wr, row_valid, R, H, E, logits, maps, n_sms, err,
                                         timeout_ns, stream);
    if (e != cudaSuccess) return e;
    e = launch_pdl(route_select_kernel, dim3((R + kSelWarps - 1) / kSelWarps), dim3(kSelWarps * 32),
                   0, stream, logits, bias, row_valid, R, E, G, TG, K, scaling, ids, wts);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
