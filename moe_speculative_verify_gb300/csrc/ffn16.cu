// ffn16.cu -- w8a16 expert GEMMs: e4m3 weights dequantised to bf16 in the
// kernel, bf16 activations, bf16 tcgen05 MMA (sm_103a).
//
// mstar #388 "Speed up GLM-5.2 with fp8 kernels and one-graph MTP", commit on
// kernel switches and the FlashInfer commit: fp8 linears run w8a16 at decode
// sizes -- fp8 weights with their 128x128 block scales, 16-bit activations
// that are not quantised.  The weight is dequantised as bf16_rne(e4m3 * scale)
// (one scale per 128x128 tile), the gathered rows and h stay bf16, and the
// MMA accumulates the whole K of a tile in fp32 tensor memory.
//
// One persistent kernel over the tile order of the fp8 path (gate/up tiles,
// then down tiles, entry-major; a down tile starts once every gate/up tile of
// its item has stored its block of h), for items of up to 16 rows, the tiles
// handed out at run time as in the fp8 GEMM.  Warp roles (one CTA per SM):
//   warp 0 lane 0: TMA producer -- claims the CTA's tiles and publishes them
//                  to the other roles; e4m3 weight tiles (16 KB) into a ring
//                  of staging buffers;
//   warps 1, 18 lane 0: MMA issuers, alternate steps -- 8 x tcgen05.mma
//                  kind::f16 (K = 16) per 128-wide K-block, A (the bf16 weight
//                  tile) from tensor memory, B (the rows) from shared memory,
//                  into the tile's accumulator: gate (even steps) and up (odd)
//                  side by side for a gate/up tile; for a down tile with an even
//                  number of K-blocks the even and odd K-blocks into the two
//                  halves, which the epilogue adds (one issuer for an odd
//                  number);
//   warps 2..13  : dequant, three groups of four taking turns -- a staged
//                  tile to bf16, written straight into a tensor-memory
//                  operand slot (tcgen05.st; the dequantised tile never
//                  touches shared memory);
//   warp 19 lane 0: row copies -- each step's 16 rows (bf16) into the
//                  slot's shared part once the slot is free (for a down tile
//                  once the item's h is complete);
//   warps 14..17 : epilogue -- gate/up: h = silu(g) * u rounded to bf16, row
//                  stores; down: fp32 rows to their slot.
// Every wait is bounded; a timeout records MOE_ERR_TIMEOUT and winds down.
#include "common.cuh"
#include "kernels.h"
#include "layout.h"

namespace moe {

namespace {

constexpr int kNT = kW8A16RowsPerItem;       // rows per item (MMA N)
constexpr int kDqGroupWarps = 4;
// three groups of four, each taking every third step (measured: with two
// groups the MMA issuers waited for converted tiles 45 % of the kernel)
constexpr int kDqGroups = 3;
constexpr int kDqWarps = kDqGroups * kDqGroupWarps;
constexpr int kEpiWarps = 4;
// warp 0 producer, warp 1 MMA issuer, dequant warps, epilogue warps, second
// MMA issuer (measured: one thread issuing these small-N MMAs was busy 60 % of
// the kernel, ~107 cycles per MMA, and set the pace), row-copy warp
constexpr int kMma2Warp = 2 + kDqWarps + kEpiWarps;
// row copies in a warp of their own (measured at 8 rows: 287.7 -> 285.7 us
// against one of the dequant warps taking each step's copies in turn)
constexpr int kBLoadWarp = kMma2Warp + 1;
constexpr int kThreads16 = 32 * (4 + kDqWarps + kEpiWarps);
// registers a thread for one block per SM: each SM sub-partition holds 16K
// registers and ceil(warps / 4) of the block's warps; in steps of 8
constexpr int kMaxRegs16 = (16384 / (((kThreads16 / 32 + 3) / 4) * 32)) / 8 * 8;
constexpr int kWBytes = 128 * 128;           // e4m3 weight tile
constexpr int kBBytes = kNT * 128 * 2;       // bf16 rows: two K halves of kNT x 128 B
constexpr int kSlotBytes = kBBytes;          // shared-memory part of an operand slot
constexpr int kSlots = 6;                    // operand slots (dequant -> MMA)
constexpr int kMaxWStages = 8;    // weight ring (measured at 8 rows: 12 stages 290.0 us, 10 289.4, 6-8 287.8)
constexpr int kAccCols = 2 * kNT;
constexpr int kAccBufs = 4;
constexpr int kACols = 64;                   // a bf16 128x128 tile in TMEM: 2 per 32-bit column
constexpr int kAColBase = kAccBufs * kAccCols;
constexpr int kTmemCols = 512;
static_assert(kAColBase + kSlots * kACols <= kTmemCols, "tensor memory");
// every dequant group owns its own operand slots (step n uses slot
// n % kSlots, group g the steps g, g + kDqGroups, ...), so a slot's uses come
// in order from one group that finishes each before it starts the next, and
// a parity wait on the slot's barriers never has more than one phase pending.
// With slots shared between groups a group can run two uses ahead of a
// pending one, and its parity wait then passes on the older phase (a variant
// with 4 slots and 3 groups faulted on the GPU).
static_assert(kSlots % kDqGroups == 0, "operand slots a multiple of the dequant groups");
static_assert(kSlotBytes % 1024 == 0, "operand slots stay 1024-byte aligned");

// Tiles are handed out at run time, as in the fp8 GEMM: a CTA's first tile
// is its block index, every further one the producer claims from a global
// counter one tile ahead and publishes into entry k % kTq16 of a shared-memory
// queue (completing tq_full[k % kTq16]); the other roles read the entries in
// order.  No role trails the producer by more than the weight ring, the
// operand slots and the accumulators together (every tile has at least one
// step), far below kTq16, so an entry is read before it is rewritten.
constexpr int kTq16 = 64;

struct TileEntry16 {
    int t;               // tile index (>= the tile count: no more tiles)
    int item, blk, gu;
};

struct Smem16 {
    int slots, wst, tq, bars, tmem, flag, bytes;
};

__host__ __device__ inline Smem16 smem16(int n_w) {
    Smem16 s;
    int b = 0;
    s.slots = b;
    b += kSlots * kSlotBytes;
    s.wst = b;
    b += n_w * kWBytes;
    s.tq = b;
    b += kTq16 * static_cast<int>(sizeof(TileEntry16));
    s.bars = b;
    b += (2 * n_w + 2 * kSlots + 2 * kAccBufs + 1 + kTq16) * 8;
    s.tmem = b;
    b += 4;
    s.flag = b;
    b += 4;
    s.bytes = b + 1024;
    return s;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major, N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A (128 x 16 bf16) read from tensor
// memory, lane m = row m, two K elements per 32-bit column.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (32x32b shape).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ int ld_acquire16(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool wait_ready(const int32_t* ctr, int target, int32_t* err,
                                           uint64_t timeout_ns, volatile int* abort_flag) {
    if (ld_acquire16(ctr) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        __nanosleep(32);
        if (ld_acquire16(ctr) >= target) return true;
        if ((it & 31u) == 31u && (*abort_flag || globaltimer_ns() - t0 > timeout_ns)) break;
    }
    record_error(err, MOE_ERR_TIMEOUT);
    return false;
}

// Four e4m3 codes (one 32-bit word, lowest byte first) times `s`, rounded to
// bf16, as two packed bf16x2 words.
__device__ __forceinline__ uint2 dequant4(uint32_t w, float s) {
    uint32_t h01, h23;
    const uint16_t lo = static_cast<uint16_t>(w & 0xFFFFu), hi = static_cast<uint16_t>(w >> 16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(lo));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(hi));
    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
    // code x scale, two per packed instruction (each an IEEE fp32 product)
    float p0, p1, p2, p3;
    mul2(p0, p1, f01.x, f01.y, s, s);
    mul2(p2, p3, f23.x, f23.y, s, s);
    uint2 r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r.x) : "f"(p1), "f"(p0));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r.y) : "f"(p3), "f"(p2));
    return r;
}

struct Tile16 {
    int item, blk;
    bool gu;
};

__device__ __forceinline__ Tile16 tile16_of(int t, int n_gu, int mb_i, int mb_h,
                                            const int4* __restrict__ items) {
    Tile16 x;
    int mb;
    if (t < n_gu) {
        mb = mb_i;
        x.gu = true;
    } else {
        t -= n_gu;
        mb = mb_h;
        x.gu = false;
    }
    const int w = __ldg(&items[t / mb].w);
    const int first = w >> 10, n = w & 1023;
    const int local = t - first * mb;
    x.blk = local / n;
    x.item = first + (local - x.blk * n);
    return x;
}

__global__ void __maxnreg__(kMaxRegs16)
    ffn16_kernel(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_u,
                 const __grid_constant__ CUtensorMap map_sg, const __grid_constant__ CUtensorMap map_su,
                 const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_d,
                 const __grid_constant__ CUtensorMap map_sd, const __grid_constant__ CUtensorMap map_h,
                 const Ffn16Args p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int KB_H = p.H / kBlock, KB_I = p.I / kBlock;
    const int MB_I = p.I / kBlock, MB_H = p.H / kBlock;
    const int NW = p.n_wstages;
    const Smem16 L = smem16(NW);
    uint8_t* slots = smem + L.slots;
    uint8_t* wst = smem + L.wst;
    uint64_t* w_full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* w_empty = w_full + NW;
    uint64_t* a_full = w_empty + NW;
    uint64_t* a_empty = a_full + kSlots;
    uint64_t* acc_full = a_empty + kSlots;
    uint64_t* acc_empty = acc_full + kAccBufs;
    uint64_t* drain = acc_empty + kAccBufs;
    uint64_t* tq_full = drain + 1;             // [kTq16] tile-queue entry written
    TileEntry16* tq = reinterpret_cast<TileEntry16*>(smem + L.tq);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.tmem);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.flag);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NW; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], kDqGroupWarps);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&a_full[s], kDqGroupWarps + 1);
            mbar_init(&a_empty[s], 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&acc_full[b], 2);   // one commit from each MMA issuer
            mbar_init(&acc_empty[b], kEpiWarps);
        }
        mbar_init(drain, 2);
        for (int b = 0; b < kTq16; ++b) mbar_init(&tq_full[b], 1);
        *s_abort = 0;
        fence_barrier_init();
        prefetch_tensormap(&map_g);
        prefetch_tensormap(&map_d);
        prefetch_tensormap(&map_x);
        prefetch_tensormap(&map_h);
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // The union buffer comes from a kernel at least two launches back: it is
    // complete when this kernel starts.  Items must have been cut to 16 rows.
    // a union built for another call (row count, shape or row tile) runs nothing
    const bool fits = union_fits(p.ub, p.R, p.ushape) && p.ub[4] == kNT;
    const int n_items = fits ? p.ub[3] : 0;
    if (threadIdx.x == 0 && !fits) record_error(p.err, MOE_ERR_INVALID_ARG);
    const int n_gu = n_items * MB_I;
    const int n_tiles = n_gu + n_items * MB_H;
    const int4* items = reinterpret_cast<const int4*>(p.ub + p.ul.items);

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol = policy_evict_first();
            int ws = 0;
            uint32_t wph = 0;
            bool ok = true;
            auto publish = [&](uint32_t k, int t) {
                TileEntry16& en = tq[k % kTq16];
                en.t = t;
                if (t < n_tiles) {
                    const Tile16 tl = tile16_of(t, n_gu, MB_I, MB_H, items);
                    en.item = tl.item;
                    en.blk = tl.blk;
                    en.gu = tl.gu ? 1 : 0;
                }
                mbar_arrive(&tq_full[k % kTq16]);
            };
            // one tile's weight steps j0 .. j1-1 into the ring
            auto load_steps = [&](int t, int j0, int j1) {
                const Tile16 tl = tile16_of(t, n_gu, MB_I, MB_H, items);
                const int4 it = items[tl.item];
                const bool sh = it.x == p.E;
                const int ex = sh ? 0 : it.x;
                for (int j = j0; j < j1; ++j) {
                    if (*s_abort || !mbar_wait(&w_empty[ws], wph ^ 1u, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&w_full[ws], kWBytes);
                    uint8_t* dst = wst + ws * kWBytes;
                    if (tl.gu) {
                        const CUtensorMap* m = (j & 1) ? (sh ? &map_su : &map_u) : (sh ? &map_sg : &map_g);
                        const int2 c = wbox(p.tiled, ex * p.I + tl.blk * kBlock, j >> 1,
                                            p.H / kBlock);
                        tma_load_2d_hint(dst, m, &w_full[ws], c.x, c.y, pol);
                    } else {
                        const int2 c = wbox(p.tiled, ex * p.H + tl.blk * kBlock, j,
                                            p.I / kBlock);
                        tma_load_2d_hint(dst, sh ? &map_sd : &map_d, &w_full[ws], c.x, c.y, pol);
                    }
                    if (++ws == NW) {
                        ws = 0;
                        wph ^= 1u;
                    }
                }
            };
            const int t0 = blockIdx.x;
            publish(0, t0);
            // weights are inputs of the layer: the first tile's first ring of
            // them is requested before the wait on the previous kernel (the
            // tile counter is that kernel's output: tiles are claimed after)
            int pre = 0;
            if (t0 < n_tiles) {
                const int NS0 = (t0 < n_gu) ? 2 * KB_H : KB_I;
                pre = NS0 < NW ? NS0 : NW;
                load_steps(t0, 0, pre);
            }
            pdl_wait();
            pdl_launch_dependents();
            uint32_t kq = 0;
            for (int t = t0; t < n_tiles && ok && !*s_abort; ++kq) {
                const int tn = atomicAdd(p.sched, 1) + static_cast<int>(gridDim.x);
                publish(kq + 1, tn);
                const int NS = (t < n_gu) ? 2 * KB_H : KB_I;
                load_steps(t, (kq == 0) ? pre : 0, NS);
                t = tn;
            }
            // This CTA claims no more tiles; the last CTA to get here resets
            // the counter (and this count) for the next launch on the workspace.
            __threadfence();
            if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
                __threadfence();
                atomicExch(p.sched, 0);
                atomicExch(p.sched + 1, 0);
            }
            if (!ok) *s_abort = 1;
        }
    } else if (warp == 1 || warp == kMma2Warp) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuers
            // Both walk every step (slot positions); each waits for, issues
            // and commits its own steps (a commit covers its thread's MMAs).
            // The issuers' latency per step sets the kernel's pace, so they
            // do not read the abort flag before their waits: every wait is
            // bounded, and after another role's failure they leave at the end
            // of one more timeout (measured at 8 rows: 285.7 -> 273.0 us).
            // A step's eight B descriptors are its first one plus the byte
            // offset / 16: shared memory lies below 256 KB, so the 14-bit
            // address field cannot carry (273.0 -> 271.0 us).
            constexpr uint32_t idesc = idesc_bf16_f32(128, kNT);
            const int mine = (warp == 1) ? 0 : 1;
            int slot = 0, ab = 0;
            uint32_t sph = 0, aph = 0;
            bool ok = true;
            for (uint32_t kq = 0; ok; ++kq) {
                if (!mbar_wait(&tq_full[kq % kTq16], (kq / kTq16) & 1u, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const TileEntry16 en = tq[kq % kTq16];
                if (en.t >= n_tiles) break;
                const bool gu = en.gu != 0;
                const int NS = gu ? 2 * KB_H : KB_I;
                if (!mbar_wait(&acc_empty[ab], aph ^ 1u, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t d0 = tmem + ab * kAccCols;
                // steps split by parity over the two halves of the accumulator
                const bool split = gu || (NS % 2) == 0;
                for (int j = 0; j < NS; ++j) {
                    const int s_cur = slot;
                    const uint32_t ph = sph;
                    if (++slot == kSlots) {
                        slot = 0;
                        sph ^= 1u;
                    }
                    if (split ? ((j & 1) != mine) : (mine != 0)) continue;
                    if (!mbar_wait(&a_full[s_cur], ph, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = tmem + kAColBase + s_cur * kACols;
                    const uint32_t b0 = smem_u32(slots + s_cur * kSlotBytes);
                    const uint32_t d = d0 + (split ? (j & 1) * kNT : 0);
                    const bool first = split ? (j < 2) : (j == 0);
                    const uint64_t bd0 = sdesc_k_sw128(b0);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t half = static_cast<uint32_t>(k >> 2), kk = k & 3;
                        mma_bf16_ts(d, a0 + 8 * k, bd0 + ((half * (kBBytes / 2) + 32 * kk) >> 4),
                                    idesc, (first && k == 0) ? 0u : 1u);
                    }
                    mma_commit(&a_empty[s_cur]);
                }
                if (!ok) break;
                mma_commit(&acc_full[ab]);
                if (++ab == kAccBufs) {
                    ab = 0;
                    aph ^= 1u;
                }
            }
            if (!ok) *s_abort = 1;
        }
    } else if (warp == kBLoadWarp) {
        if (lane == 0) {
            // ---------------------------------------------- row copies
            int slot = 0;
            uint32_t sph = 0;
            bool ok = true;
            pdl_wait();   // gathered rows and the counters belong to the previous kernel
            for (uint32_t kq = 0; ok; ++kq) {
                if (*s_abort ||
                    !mbar_wait(&tq_full[kq % kTq16], (kq / kTq16) & 1u, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const TileEntry16 en = tq[kq % kTq16];
                if (en.t >= n_tiles) break;
                const bool gu = en.gu != 0;
                const int4 it = items[en.item];
                const int NS = gu ? 2 * KB_H : KB_I;
                bool h_ready = gu;
                for (int j = 0; j < NS; ++j) {
                    const int s_cur = slot;
                    const uint32_t ph = sph;
                    if (++slot == kSlots) {
                        slot = 0;
                        sph ^= 1u;
                    }
                    if (*s_abort || !mbar_wait(&a_empty[s_cur], ph ^ 1u, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    if (!h_ready) {
                        // h of this item comes from this launch's gate/up tiles
                        if (!wait_ready(p.ready + en.item, MB_I, p.err, p.timeout_ns, s_abort)) {
                            ok = false;
                            break;
                        }
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        h_ready = true;
                    }
                    const int kb = gu ? (j >> 1) : j;
                    const CUtensorMap* bm = gu ? &map_x : &map_h;
                    uint8_t* sl = slots + s_cur * kSlotBytes;
                    mbar_arrive_expect_tx(&a_full[s_cur], kBBytes);
                    tma_load_2d(sl, bm, &a_full[s_cur], kb * kBlock, it.y);
                    tma_load_2d(sl + kBBytes / 2, bm, &a_full[s_cur], kb * kBlock + 64, it.y);
                }
            }
            if (!ok) *s_abort = 1;
        }
    } else if (warp < 2 + kDqWarps) {
        // --------------------------------------------------------- dequant
        // kDqGroups groups of four warps take turns over the CTA's step
        // sequence (group g the steps g, g + kDqGroups, ...), so that many
        // staged tiles are converted at once.  In a group,
        // warp w converts rows 32*(w%4) .. +31 (the TMEM lanes it may access)
        // of the tile: per thread the 128 codes of its row, read from the
        // swizzled stage, written as 64 bf16x2 columns.
        const int dw = warp - 2;
        const int grp = dw / kDqGroupWarps;
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        uint32_t n = 0;              // the CTA's step counter (every group counts every step)
        bool ok = true;
        // nothing here reads the previous kernel's outputs; the wait only
        // keeps the roles together (converting before it measured the same)
        pdl_wait();
        for (uint32_t kq = 0; ok; ++kq) {
            bool got = !*s_abort &&
                       mbar_wait(&tq_full[kq % kTq16], (kq / kTq16) & 1u, p.err, p.timeout_ns);
            if (!__all_sync(0xFFFFFFFFu, got)) {
                ok = false;
                break;
            }
            const TileEntry16 en = tq[kq % kTq16];
            if (en.t >= n_tiles) break;
            const Tile16 tl{en.item, en.blk, en.gu != 0};
            const int4 it = items[tl.item];
            const bool sh = it.x == p.E;
            const int ex = sh ? 0 : it.x;
            const int NS = tl.gu ? 2 * KB_H : KB_I;
            const int KB = tl.gu ? KB_H : KB_I;
            const int MB = tl.gu ? MB_I : MB_H;
            const float* sg = sh ? p.sh_s_gate : p.s_gate;
            const float* su = sh ? p.sh_s_up : p.s_up;
            const float* sd = sh ? p.sh_s_down : p.s_down;
            const size_t sbase = (size_t(ex) * MB + tl.blk) * KB;
            auto scale_of = [&](int j) -> float {
                return tl.gu ? __ldg(((j & 1) ? su : sg) + sbase + (j >> 1)) : __ldg(sd + sbase + j);
            };
            // this group's first step of the tile
            const int j0 = (grp - static_cast<int>(n % kDqGroups) + kDqGroups) % kDqGroups;
            float s_next = (j0 < NS) ? scale_of(j0) : 0.0f;
            // weight stage and phase of the group's step: divided out once
            // per tile, then advanced kDqGroups steps at a time
            uint32_t nj = n + static_cast<uint32_t>(j0);
            int ws = static_cast<int>(nj % static_cast<uint32_t>(NW));
            uint32_t wph = (nj / static_cast<uint32_t>(NW)) & 1u;
            for (int j = j0; j < NS; j += kDqGroups, nj += kDqGroups) {
                const int slot = static_cast<int>(nj % kSlots);
                const uint32_t sph = (nj / kSlots) & 1u;
                const float s = s_next;
                if (j + kDqGroups < NS) s_next = scale_of(j + kDqGroups);
                // every wait's outcome is made uniform across the warp before use;
                // no abort-flag read before these bounded waits (as in the MMA
                // threads; measured 270.6 -> 267.2 us at 8 rows)
                bool got = mbar_wait(&a_empty[slot], sph ^ 1u, p.err, p.timeout_ns);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                got = mbar_wait(&w_full[ws], wph, p.err, p.timeout_ns);
                if (!__all_sync(0xFFFFFFFFu, got)) {
                    ok = false;
                    break;
                }
                const uint8_t* src = wst + ws * kWBytes + row * 128;
                uint4 q[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    q[c] = *reinterpret_cast<const uint4*>(src + ((c ^ (row & 7)) << 4));
                // the stage is read: hand it back before converting
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[ws]);
                __syncwarp();   // tcgen05.st is warp-wide: the whole warp, converged
                const uint32_t ta = tmem + (static_cast<uint32_t>(32 * qd) << 16) + kAColBase +
                                    slot * kACols;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    uint32_t o[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v = q[4 * h2 + c];
                        const uint2 o0 = dequant4(v.x, s), o1 = dequant4(v.y, s);
                        const uint2 o2 = dequant4(v.z, s), o3 = dequant4(v.w, s);
                        o[8 * c + 0] = o0.x;
                        o[8 * c + 1] = o0.y;
                        o[8 * c + 2] = o1.x;
                        o[8 * c + 3] = o1.y;
                        o[8 * c + 4] = o2.x;
                        o[8 * c + 5] = o2.y;
                        o[8 * c + 6] = o3.x;
                        o[8 * c + 7] = o3.y;
                    }
                    tmem_st32(ta + 32 * h2, o);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[slot]);
                ws += kDqGroups;   // NW >= kDqGroups
                if (ws >= NW) {
                    ws -= NW;
                    wph ^= 1u;
                }
            }
            n += static_cast<uint32_t>(NS);
        }
        if (!ok) *s_abort = 1;
    } else {
        // ----------------------------------------------------- epilogue
        const int q = warp & 3;            // TMEM lane quadrant this warp may access
        const int m = 32 * q + lane;       // output feature inside the 128-row block
        const int et = threadIdx.x - 32 * (2 + kDqWarps);
        int ab = 0;
        uint32_t aph = 0;
        bool ok = true;
        pdl_wait();
        for (uint32_t kq = 0; ok; ++kq) {
            const bool got_t = __all_sync(0xFFFFFFFFu, !*s_abort &&
                mbar_wait(&tq_full[kq % kTq16], (kq / kTq16) & 1u, p.err, p.timeout_ns));
            if (!bar_and(1, got_t, 32 * kEpiWarps)) {
                ok = false;
                break;
            }
            const TileEntry16 en = tq[kq % kTq16];
            if (en.t >= n_tiles) break;
            const Tile16 tl{en.item, en.blk, en.gu != 0};
            const int4 it = items[tl.item];
            const int row0 = it.y, nrow = it.z;
            // all four epilogue warps learn of a failed wait together
            const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(&acc_full[ab], aph, p.err,
                                                                 p.timeout_ns));
            if (!bar_and(1, got, 32 * kEpiWarps)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + ab * kAccCols;
            // gate and up, or a down tile's even- and odd-K-block halves
            const bool split = tl.gu || (KB_I % 2) == 0;
            float g[kNT], u[kNT];
            tmem_ld16(ta, g);
            if (split) tmem_ld16(ta + kNT, u);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
            if (++ab == kAccBufs) {
                ab = 0;
                aph ^= 1u;
            }
            if (tl.gu) {
#pragma unroll
                for (int c = 0; c < kNT; ++c) {
                    if (c < nrow) {
                        const float h = (g[c] / (1.0f + __expf(-g[c]))) * u[c];
                        p.hb[size_t(row0 + c) * p.I + tl.blk * kBlock + m] =
                            __bfloat16_as_ushort(__float2bfloat16_rn(h));
                    }
                }
                // release this block of h to the item's down tiles
                (void)bar_and(1, true, 32 * kEpiWarps);
                if (et == 0) {
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __threadfence();
                    atomicAdd(p.ready + tl.item, 1);
                }
            } else {
#pragma unroll
                for (int c = 0; c < kNT; ++c) {
                    if (c < nrow) {
                        const int slot = __ldg(p.ub + p.ul.src + row0 + c);
                        const int r = slot / p.KS, k = slot - r * p.KS;
                        float* dst = (k < p.K) ? p.y_slots + (size_t(r) * p.K + k) * p.H
                                               : p.y_shared + size_t(r) * p.H;
                        dst[tl.blk * kBlock + m] = split ? __fadd_rn(g[c], u[c]) : g[c];
                    }
                }
            }
        }
        if (!ok) *s_abort = 1;
    }

    __syncthreads();
    if (*s_abort) {
        // Wind down: copies already issued land within microseconds; give them
        // a fixed budget, then let every issued MMA finish before tensor
        // memory is released.
        constexpr uint64_t kDrainNs = 1000000;   // 1 ms
        if (threadIdx.x == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < kDrainNs) __nanosleep(1000);
        }
        if (threadIdx.x == 32 * kMma2Warp) mma_commit(drain);
        if (threadIdx.x == 32) {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, kDrainNs);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Gathered bf16 rows: each valid row copied to its K + S positions; one warp
// per (row, 128 columns).  Clears the per-item counters of the GEMM.
__global__ void __launch_bounds__(256) dispatch16_kernel(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ ub,
                                                         UnionLayout L, int R, int H, int KS,
                                                         int32_t ushape,
                                                         uint16_t* __restrict__ xb,
                                                         int32_t* __restrict__ ready, int n_ready,
                                                         int32_t* __restrict__ err) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < n_ready; i += blockDim.x) ready[i] = 0;
    if (!union_fits(ub, R, ushape)) {   // built for another call
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            record_error(err, MOE_ERR_INVALID_ARG);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x;
    const int b = blockIdx.y * 8 + warp;
    if (b >= H / kBlock) return;
    const int32_t* pos = ub + L.pos + size_t(r) * KS;
    if (pos[0] < 0) return;   // pad row
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + size_t(r) * H + b * kBlock + 4 * lane));
    for (int k = 0; k < KS; ++k)
        reinterpret_cast<uint2*>(xb + size_t(pos[k]) * H + b * kBlock)[lane] = v;
}

}  // namespace

cudaError_t launch_dispatch16(const uint16_t* x, const int32_t* ub, const UnionLayout& L, int R,
                              int H, int KS, int32_t ushape, uint16_t* xb, int32_t* ready,
                              int n_ready, int32_t* err, cudaStream_t stream) {
    dim3 grid(R, (H / kBlock + 7) / 8);
    cudaError_t e = launch_pdl(dispatch16_kernel, grid, dim3(256), 0, stream, x, ub, L, R, H, KS,
                               ushape, xb, ready, n_ready, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_ffn16(const FfnMaps& mp, Ffn16Args args, int n_sms, int smem_limit,
                         cudaStream_t stream) {
    int nw = kMaxWStages;
    Smem16 L = smem16(nw);
    while (nw > kDqGroups && L.bytes > smem_limit) L = smem16(--nw);
    if (L.bytes > smem_limit) return cudaErrorInvalidConfiguration;
    args.n_wstages = nw;
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(ffn16_kernel), L.bytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl(ffn16_kernel, dim3(max(1, n_sms)), dim3(kThreads16), L.bytes, stream, mp.g, mp.u,
                   mp.sg, mp.su, mp.x, mp.d, mp.sd, mp.h, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
