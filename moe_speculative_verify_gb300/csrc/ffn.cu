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
// One persistent kernel, three modes: the gate/up GEMM alone, the down GEMM
// alone, or both in one launch (Fused) over a single tile queue -- every
// gate/up tile first, then every down tile -- so the SMs that finish their
// gate/up work early go on with down tiles instead of idling.  A down tile
// needs the whole h of its item: the item's gate/up tiles each release a
// per-item counter after storing their block of h, and the down tile's
// producer and epilogue acquire it (a bounded wait) before reading h.
//
// Work unit = (item, 128-row block of the output features); an item is up to
// NT gathered rows of one expert (union entry).  Swap-AB: the weight tile is
// the MMA's A operand (M = 128 output features), the rows are the B operand
// (N = NT), so a verify batch of a few rows still fills the 128-row MMA.  Per
// 128-wide K-block the MMA writes a fresh fp32 partial to tensor memory; the
// epilogue warps read it back and fold it into fp32 register accumulators with
// the block's weight scale times the row's activation scale (fp32 128x128
// scales cannot be expressed in the MMA's own block-scale format).
//
// Warp roles (one CTA per SM):
//   warp 0 lane 0: TMA producer -- weight tiles (evict-first) and row tiles
//                  into an n_stages ring of shared-memory stages;
//   warps 1, 2 lane 0: MMA issuers, alternate K-blocks -- 4 x tcgen05.mma
//                  (K = 32) per operand per K-block into a ring of ACC_BUFS
//                  tensor-memory partials, then one tcgen05.commit per K-block
//                  that frees its stages and hands its partial to the epilogue;
//   warps 3.. : epilogue -- 4 * NT/CW warps; warp w reads TMEM lanes
//                  32*(w%4).. and CW columns (16, or 8 at 32-row tiles),
//                  promotes the partials, then
//                  gate/up: h = silu(g) * u, per-row 1x128 e4m3 quantisation
//                  of h, coalesced row stores; down: fp32 rows to their slot.
// Every wait is bounded; a timeout records MOE_ERR_TIMEOUT, winds the roles
// down, drains in-flight copies and MMAs, frees tensor memory and returns.
#include "common.cuh"
#include "kernels.h"
#include "layout.h"

namespace moe {

template <int NT, int MODE>
struct FfnCfg {
    // One stage = one 128x128 weight tile + the item's 128-column row tile; a
    // gate/up K-block takes two stages (gate, then up), a down K-block one, so
    // both phases share one uniform ring.
    static constexpr int NA = (MODE == kFfnDown) ? 1 : 2;   // weight operands per K-block (max)
    static constexpr int A_BYTES = 128 * 128;
    static constexpr int B_OFF = A_BYTES;
    static constexpr int B_BYTES = NT * 128;
    static constexpr int STAGE_BYTES = B_OFF + B_BYTES;
    // a down tile's rows leave through shared memory as 16-byte stores at
    // 16-row tiles (measured in one run: verify8's GEMM 0.2264 -> 0.2253 ms,
    // verify64's 0.874 -> 0.872; at 64-row tiles the extra barrier cost more
    // than the scattered stores, +0.8 %)
    static constexpr bool STAGED_OUT = (NT == 16 && MODE != kFfnGateUp);
    // shared-memory tile at a tile's end: h codes, and a down tile's fp32 rows
    static constexpr int TILE_BYTES = STAGED_OUT ? NT * 128 * 4 : NT * 128;
    // columns per epilogue warp: 16 at 16- and 64-row tiles, 8 at 32-row
    // tiles (16 epilogue warps at 32 and 64 rows: the per-K-block promotion
    // is spread over as many warps as the block can hold)
    static constexpr int CW = (NT == 32) ? 8 : 16;
    static constexpr int CSPLIT = NT / CW;
    static constexpr int EPI_WARPS = 4 * CSPLIT;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int THREADS = 96 + EPI_THREADS;   // producer, two MMA issuers, epilogue
    // registers per thread for one block per SM: each of the four SM
    // sub-partitions holds 16K registers and ceil(warps / 4) of the block's
    // warps; in steps of 8, at most 255
    static constexpr int WARPS_PER_SMSP = (THREADS / 32 + 3) / 4;
    static constexpr int MAX_REGS_RAW = (16384 / (WARPS_PER_SMSP * 32)) / 8 * 8;
    static constexpr int MAX_REGS = MAX_REGS_RAW > 255 ? 255 : MAX_REGS_RAW;
    static constexpr int ACC_COLS = NA * NT;
    // as many tensor-memory partials as fit (at most 16): the MMA may run that
    // many K-blocks ahead of the epilogue across its tile transitions
    static constexpr int ACC_BUFS = (512 / ACC_COLS) < 16 ? (512 / ACC_COLS) : 16;
    static constexpr int TMEM_COLS = (ACC_BUFS * ACC_COLS <= 32) ? 32
                                     : (ACC_BUFS * ACC_COLS <= 64) ? 64
                                     : (ACC_BUFS * ACC_COLS <= 128) ? 128
                                     : (ACC_BUFS * ACC_COLS <= 256) ? 256 : 512;
    static_assert(ACC_BUFS * ACC_COLS <= 512, "tensor memory");
    // suspend-time hint of the producer's and MMA issuers' barrier waits: at
    // 32- and 64-row tiles waiting warps then leave their issue slots to the
    // epilogue warps
    // (measured: decode512's GEMMs 1.259 -> 1.220 ms, prefill4096's 4.09 ->
    // 4.02); at 16-row tiles, where the HBM stream bounds the kernel, none
    static constexpr uint32_t WAIT_HINT_NS = (NT >= 32) ? 20000u : 0u;
    static_assert(ACC_BUFS % 2 == 0, "the MMA checks TMEM partials in pairs");
};

constexpr int kMaxStages = 16;
constexpr int kStagesNt16 = 10;   // ring depth where the weight stream counts (see launch_ffn_t)
constexpr int kStagesWide = 6;        // ring depth of the separate kernels at 64-row tiles ...
constexpr int kStagesWideDecode = 7;  // ... and in calls of at most 512 rows
// Per K-block (not per stage) synchronisation, on two rings of barriers
// indexed by the CTA's K-block counter j:
//   kbfull[j % kKbRing] -- the K-block's operands have landed: the producer
//       arms it once with the bytes of all the K-block's stages, every TMA
//       copy of those stages completes on it;
//   kbrel[j % kKbRing]  -- one tcgen05.commit after the K-block's MMAs: its
//       stages are free for the producer and its partial is ready for the
//       epilogue.
// A barrier wait or a commit costs about as much as several small-N MMAs, so
// the MMA thread waits once for data and commits once per K-block.  The rings
// outlast the producer's and the epilogue's lead over the MMA (at most
// kMaxStages, resp. 16 K-blocks), so a parity wait never aliases.
constexpr int kKbRing = 32;

// Tiles are handed out at run time: a CTA's first tile is its block index,
// every further one comes from a global counter (claimed by the producer one
// tile ahead), so CTAs that finish early take more of the small down tiles and
// all end within about one tile of each other.  The producer writes the CTA's
// k-th tile into entry k % kTq of a shared-memory queue and completes
// tq_full[k % kTq]; the MMA issuers and the epilogue read the entries in
// order.  No role trails the producer by more than kMaxStages + 16 tiles
// (every tile has at least one stage and one K-block), so an entry is read
// before it is rewritten.
constexpr int kTq = 64;

struct TileEntry {
    int t;               // tile index (>= the tile count: no more tiles)
    int item, blk;       // the Tile fields
    int flags;           // 1: gate/up tile, 2: shared weight tile
    int4 it;             // the item record
};

// Shared-memory carve-up, identical on host (size) and device (pointers).
struct FfnSmem {
    int stages, sc, red, tile, src, tq, bars, tmem, flag, bytes;
};

// tile_bytes: the h tile of a gate/up tile (nt x 128 e4m3 codes) or, in a
// kernel with down tiles, the fp32 output tile (nt x 128 x 4 bytes).
__host__ __device__ inline FfnSmem ffn_smem(int nt, int n_stages, int kbmax, int stage_bytes,
                                             int tile_bytes) {
    FfnSmem s;
    int b = 0;
    s.stages = b;
    b += n_stages * stage_bytes;
    s.sc = b;
    b += 2 * kbmax * nt * 4;
    s.red = b;
    b += 5 * nt * 4;
    s.tile = b;
    b += tile_bytes;
    s.src = b;
    b += nt * 4;
    b = (b + 15) & ~15;
    s.tq = b;
    b += kTq * static_cast<int>(sizeof(TileEntry));
    s.bars = b;
    b += (2 * kKbRing + 16 + 1 + kTq) * 8;
    s.tmem = b;
    b += 4;
    s.flag = b;
    b += 4;
    s.bytes = b + 1024;  // slack to align the base to 1024 bytes
    return s;
}

// AND of `ok` over the epilogue threads (named barrier 1).
__device__ __forceinline__ bool epi_bar_and(bool ok, int nthreads) {
    return bar_and(1, ok, nthreads);
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until *ctr >= target (acquire).  False on timeout.
__device__ __forceinline__ bool wait_counter(const int32_t* ctr, int target, int32_t* err,
                                             uint64_t timeout_ns, volatile int* abort_flag) {
    if (ld_acquire(ctr) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        __nanosleep(32);
        if (ld_acquire(ctr) >= target) return true;
        if ((it & 31u) == 31u && (*abort_flag || globaltimer_ns() - t0 > timeout_ns)) break;
    }
    record_error(err, MOE_ERR_TIMEOUT);
    return false;
}

struct Tile {
    int item, blk;
    bool gu;
    bool shared_w;   // the weight tile is read by several items (row chunks)
};

// Tile t of the queue: gate/up tiles first, then down tiles.  Within a phase
// the order is entry-major, then output block, then row chunk: every row chunk
// of an expert that uses the same weight tile sits on adjacent tiles, so they
// run at the same time on neighbouring CTAs and the weight tile comes from
// DRAM once.  An item's w word holds its entry's first item * 1024 + items.
__device__ __forceinline__ Tile tile_of(int t, int n_gu, int mb_i, int mb_h,
                                        const int4* __restrict__ items) {
    Tile x;
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
    x.shared_w = n > 1;
    return x;
}

template <int NT, int MODE>
__global__ void __maxnreg__((FfnCfg<NT, MODE>::MAX_REGS))
    ffn_kernel(const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_u,
               const __grid_constant__ CUtensorMap map_sg, const __grid_constant__ CUtensorMap map_su,
               const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_d,
               const __grid_constant__ CUtensorMap map_sd, const __grid_constant__ CUtensorMap map_h,
               const FfnArgs p) {
    using C = FfnCfg<NT, MODE>;
    constexpr bool kFused = (MODE == kFfnFused);
    // Measured: the scale table from 16-byte loads is faster in every kernel
    // but the fused one at 64-row tiles (code generation), SiLU with the fast
    // division faster at every width.
    constexpr bool kVecTable = NT <= 32 || MODE != kFfnFused;
    constexpr bool kFastSilu = true;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int KB_H = p.H / kBlock, KB_I = p.I / kBlock;   // K-blocks of gate/up, of down
    const int MB_I = p.I / kBlock, MB_H = p.H / kBlock;   // output blocks of gate/up, of down
    const int KBMAX = (MODE == kFfnGateUp) ? KB_H : (MODE == kFfnDown) ? KB_I : max(KB_H, KB_I);
    const FfnSmem L = ffn_smem(NT, p.n_stages, KBMAX, C::STAGE_BYTES, C::TILE_BYTES);
    uint8_t* st_base = smem + L.stages;
    // per-tile scale table: weight block scale x row scale, [operand][kb][n]
    float* s_sc = reinterpret_cast<float*>(smem + L.sc);
    float* s_red = reinterpret_cast<float*>(smem + L.red);   // [4][NT] amax parts, [NT] h scales
    uint8_t* s_tile = smem + L.tile;                         // [NT][128] codes or fp32
    int* s_src = reinterpret_cast<int*>(smem + L.src);       // [NT]
    uint64_t* kbfull = reinterpret_cast<uint64_t*>(smem + L.bars);   // [kKbRing] operands landed
    uint64_t* kbrel = kbfull + kKbRing;        // [kKbRing] K-block done (stages free, partial ready)
    uint64_t* acc_empty = kbrel + kKbRing;     // [16] epilogue done with a TMEM partial
    uint64_t* drain = acc_empty + 16;
    uint64_t* tq_full = drain + 1;             // [kTq] tile-queue entry written
    TileEntry* tq = reinterpret_cast<TileEntry*>(smem + L.tq);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L.tmem);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L.flag);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // producer (thread 0): used_by[s] = the CTA's K-block index that reads
    // stage s (none yet: ~0); before a stage is refilled, that K-block must
    // be done, and on a wind-down its copies are waited for
    uint32_t used_by[kMaxStages];
    for (int q = 0; q < kMaxStages; ++q) used_by[q] = ~0u;

    if (threadIdx.x == 0) {
        for (int b = 0; b < kKbRing; ++b) {
            mbar_init(&kbfull[b], 1);
            mbar_init(&kbrel[b], 1);
        }
        for (int b = 0; b < C::ACC_BUFS; ++b) mbar_init(&acc_empty[b], C::EPI_WARPS);
        mbar_init(drain, 2);   // one commit from each MMA issuer
        for (int b = 0; b < kTq; ++b) mbar_init(&tq_full[b], 1);
        *s_abort = 0;
        fence_barrier_init();
        if (MODE != kFfnDown) {
            prefetch_tensormap(&map_g);
            prefetch_tensormap(&map_x);
        }
        if (MODE != kFfnGateUp) {
            prefetch_tensormap(&map_d);
            prefetch_tensormap(&map_h);
        }
    }
    if (warp == 1) {
        tmem_alloc(s_tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // The union buffer comes from a kernel at least two launches back: it is
    // complete when this kernel starts (see pdl_wait).  Items must have been
    // cut to this kernel's row tile.
    // a union built for another call (row count, shape or row tile) runs nothing
    const bool fits = union_fits(p.ub, p.R, p.ushape) && p.ub[4] == NT;
    const int n_items = fits ? p.ub[3] : 0;
    if (threadIdx.x == 0 && !fits) record_error(p.err, MOE_ERR_INVALID_ARG);
    const int n_gu = (MODE == kFfnDown) ? 0 : n_items * MB_I;
    const int n_tiles = n_gu + ((MODE == kFfnGateUp) ? 0 : n_items * MB_H);
    const int4* items = reinterpret_cast<const int4*>(p.ub + p.ul.items);
    uint32_t issued = 0;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_once = policy_evict_first();   // a weight tile read once
            const uint64_t pol_shared = policy_evict_last();  // read by several row chunks
            int stage = 0;
            uint32_t phase = 0;
            // Stage j of a tile: gate/up tiles alternate gate and up weight
            // tiles per K-block (j = 2*kb + {0, 1}); down tiles one per K-block.
            // stage j of a tile belongs to the CTA's K-block kbj; its first
            // stage arms the K-block's barrier with the bytes of all its
            // stages.  A gate/up K-block's row tile is loaded once, into its
            // gate stage, and both of its MMAs read it there.
            auto a_load = [&](const Tile& tl, const int4& it, int j, int s, uint32_t kbj) {
                const bool sh = it.x == p.E;
                const int ex = sh ? 0 : it.x;
                uint8_t* st = st_base + s * C::STAGE_BYTES;
                const uint64_t pol = tl.shared_w ? pol_shared : pol_once;
                uint64_t* bar = &kbfull[kbj % kKbRing];
                if (!tl.gu || (j & 1) == 0)
                    mbar_arrive_expect_tx(bar, tl.gu ? 2 * C::A_BYTES + C::B_BYTES : C::STAGE_BYTES);
                if (tl.gu) {
                    const CUtensorMap* m = (j & 1) ? (sh ? &map_su : &map_u) : (sh ? &map_sg : &map_g);
                    const int2 c = wbox(p.tiled, ex * p.I + tl.blk * kBlock, j >> 1, p.H / kBlock);
                    tma_load_2d_hint(st, m, bar, c.x, c.y, pol);
                } else {
                    const int2 c = wbox(p.tiled, ex * p.H + tl.blk * kBlock, j, p.I / kBlock);
                    tma_load_2d_hint(st, sh ? &map_sd : &map_d, bar, c.x, c.y, pol);
                }
            };
            auto b_load = [&](const Tile& tl, const int4& it, int j, int s, uint32_t kbj) {
                if (tl.gu && (j & 1)) return;   // the up stage reads the gate stage's rows
                const int kb = tl.gu ? (j >> 1) : j;
                tma_load_2d(st_base + s * C::STAGE_BYTES + C::B_OFF, tl.gu ? &map_x : &map_h,
                            &kbfull[kbj % kKbRing], kb * kBlock, it.y);
            };
            auto next_stage = [&]() {
                if (++stage == p.n_stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            auto wait_free = [&](int s) -> bool {
                const uint32_t jj = used_by[s];
                return jj == ~0u ||
                       mbar_wait<C::WAIT_HINT_NS>(&kbrel[jj % kKbRing], (jj / kKbRing) & 1u, p.err, p.timeout_ns);
            };
            auto publish = [&](uint32_t k, int t, const Tile& tl, const int4& it) {
                TileEntry& en = tq[k % kTq];
                en.t = t;
                en.item = tl.item;
                en.blk = tl.blk;
                en.flags = (tl.gu ? 1 : 0) | (tl.shared_w ? 2 : 0);
                en.it = it;
                mbar_arrive(&tq_full[k % kTq]);
            };
            uint32_t kb_base = 0;   // K-blocks of the CTA's earlier tiles
            // Weights are inputs of the layer, not outputs of the previous
            // kernel: the first tile's first weight tiles are requested before
            // the wait on that kernel, its row tiles after.
            const int t0 = blockIdx.x;
            int pre = 0;
            Tile tl0{0, 0, true, false};
            int4 it0 = make_int4(0, 0, 0, 0);
            if (t0 < n_tiles) {
                tl0 = tile_of(t0, n_gu, MB_I, MB_H, items);
                it0 = items[tl0.item];
                pre = min(tl0.gu ? 2 * KB_H : KB_I, p.n_stages);
                for (int j = 0; j < pre; ++j) {
                    used_by[j] = static_cast<uint32_t>(tl0.gu ? (j >> 1) : j);
                    a_load(tl0, it0, j, j, used_by[j]);
                }
            }
            publish(0, t0, tl0, it0);
            pdl_wait();
            pdl_launch_dependents();
            bool ok = true;
            if (kFused && t0 < n_tiles && !tl0.gu) {
                // the first tile is a down tile: its h comes from this launch
                ok = wait_counter(p.ready + tl0.item, MB_I, p.err, p.timeout_ns, s_abort);
                fence_proxy_async_global();
            }
            for (int j = 0; j < pre && ok; ++j) b_load(tl0, it0, j, j, used_by[j]);
            issued = static_cast<uint32_t>(pre);
            stage = pre % p.n_stages;
            phase = (pre == p.n_stages) ? 1u : 0u;
            // the next tile is claimed, and its item fetched, one tile ahead
            Tile tl_next = tl0;
            int4 it_next = it0;
            uint32_t kq = 0;   // queue entry of the current tile
            for (int t = t0; t < n_tiles && ok && !*s_abort; ++kq) {
                const Tile tl = tl_next;
                const int4 it = it_next;
                const int tn = atomicAdd(p.sched, 1) + static_cast<int>(gridDim.x);
                if (tn < n_tiles) {
                    tl_next = tile_of(tn, n_gu, MB_I, MB_H, items);
                    it_next = items[tl_next.item];
                }
                publish(kq + 1, tn, tl_next, it_next);
                const int NS = tl.gu ? 2 * KB_H : KB_I;
                int j = (kq == 0) ? pre : 0;
                if (kFused && !tl.gu && kq != 0) {
                    // h of this item comes from other tiles of this launch: request
                    // up to a ring of weight tiles, then wait for h, then its rows.
                    int nd = 0, dst[kMaxStages];
                    if (ld_acquire(p.ready + tl.item) < MB_I) {
                        while (nd < NS && nd < p.n_stages) {
                            if (!wait_free(stage)) {
                                ok = false;
                                break;
                            }
                            used_by[stage] = kb_base + static_cast<uint32_t>(nd);
                            a_load(tl, it, nd, stage, used_by[stage]);
                            dst[nd++] = stage;
                            ++issued;
                            next_stage();
                        }
                        if (ok && !wait_counter(p.ready + tl.item, MB_I, p.err, p.timeout_ns, s_abort))
                            ok = false;
                    }
                    fence_proxy_async_global();
                    for (int q = 0; q < nd && ok; ++q) b_load(tl, it, q, dst[q], used_by[dst[q]]);
                    j = nd;
                }
                for (; j < NS && ok; ++j) {
                    if (!wait_free(stage)) {
                        ok = false;
                        break;
                    }
                    used_by[stage] = kb_base + static_cast<uint32_t>(tl.gu ? (j >> 1) : j);
                    a_load(tl, it, j, stage, used_by[stage]);
                    b_load(tl, it, j, stage, used_by[stage]);
                    ++issued;
                    next_stage();
                }
                kb_base += static_cast<uint32_t>(tl.gu ? KB_H : KB_I);
                t = tn;
            }
            // This CTA claims no more tiles; the last CTA to get here resets
            // the counter (and this count) for the next launch on the
            // workspace.
            __threadfence();
            if (atomicAdd(p.sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
                __threadfence();
                atomicExch(p.sched, 0);
                atomicExch(p.sched + 1, 0);
            }
            if (!ok) *s_abort = 1;
        }
    } else if (warp == 1 || warp == 2) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuers
            // Two threads (warps 1 and 2) issue the MMAs of alternate
            // K-blocks: one thread issues small-N MMAs at barely more than
            // half the rate two can.  Each walks every K-block to keep the
            // stage position, and for its own ones waits for the TMEM partial
            // to be free and the operands to land, issues the MMAs and
            // commits (a commit covers its issuing thread's MMAs only).
            constexpr uint32_t idesc = idesc_e4m3_f32(128, NT);
            const uint32_t mine = static_cast<uint32_t>(warp - 1);
            int stage = 0;
            uint32_t jk = 0;   // the CTA's K-block counter
            bool ok = true;
            for (uint32_t kq = 0; ok; ++kq) {
                if (*s_abort ||
                    !mbar_wait<C::WAIT_HINT_NS>(&tq_full[kq % kTq], (kq / kTq) & 1u, p.err, p.timeout_ns)) {
                    ok = false;
                    break;
                }
                const int t = tq[kq % kTq].t;
                if (t >= n_tiles) break;
                const bool gu = t < n_gu;
                const int KB = gu ? KB_H : KB_I;
                const int nst = gu ? 2 : 1;
                for (int kb = 0; kb < KB && ok; ++kb, ++jk) {
                    const int s0 = stage;
                    stage += nst;
                    if (stage >= p.n_stages) stage -= p.n_stages;
                    if ((jk & 1u) != mine) continue;
                    const uint32_t ab = jk % C::ACC_BUFS;
                    if (*s_abort ||
                        !mbar_wait<C::WAIT_HINT_NS>(&acc_empty[ab], ((jk / C::ACC_BUFS) & 1u) ^ 1u, p.err,
                                   p.timeout_ns) ||
                        !mbar_wait<C::WAIT_HINT_NS>(&kbfull[jk % kKbRing], (jk / kKbRing) & 1u, p.err, p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d0 = tmem + ab * C::ACC_COLS;
                    int st = s0;
                    // the K-block's row tile sits in its first stage
                    const uint32_t bb = smem_u32(st_base + s0 * C::STAGE_BYTES) + C::B_OFF;
                    for (int op = 0; op < nst; ++op) {
                        const uint32_t a0 = smem_u32(st_base + st * C::STAGE_BYTES);
                        const uint32_t d = d0 + op * NT;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_e4m3(d, sdesc_k_sw128(a0 + 32 * k), sdesc_k_sw128(bb + 32 * k), idesc,
                                     k > 0);
                        if (++st == p.n_stages) st = 0;
                    }
                    mma_commit(&kbrel[jk % kKbRing]);   // stages free + partial ready
                }
            }
            if (!ok) *s_abort = 1;
        }
    } else {
        // ----------------------------------------------------- epilogue
        const int ew = warp - 3;
        const int q = warp & 3;          // TMEM lane quadrant this warp may access
        const int cg = ew >> 2;          // CW-column group
        const int m = 32 * q + lane;     // output feature inside the 128-row block
        const int et = threadIdx.x - 96; // 0 .. EPI_THREADS-1
        int ab = 0;
        uint32_t je = 0;   // the CTA's K-block counter
        bool ok = true;
        pdl_wait();   // row scales and outputs belong to the previous kernel
        for (uint32_t kq = 0;; ++kq) {
            // the tile's queue entry, then: the previous tile's readers are
            // done with the scale / tile buffers
            if (ok && !mbar_wait<C::WAIT_HINT_NS>(&tq_full[kq % kTq], (kq / kTq) & 1u, p.err, p.timeout_ns))
                ok = false;
            ok = epi_bar_and(ok, C::EPI_THREADS);
            if (!ok) break;
            const TileEntry en = tq[kq % kTq];
            if (en.t >= n_tiles) break;
            const Tile tl{en.item, en.blk, (en.flags & 1) != 0, (en.flags & 2) != 0};
            const int4 it = en.it;
            const bool sh = it.x == p.E;
            const int ex = sh ? 0 : it.x;
            const int row0 = it.y, nrow = it.z;
            const int KB = tl.gu ? KB_H : KB_I;
            const int MB = tl.gu ? MB_I : MB_H;
            if (kFused && !tl.gu) {
                // h and its scales come from this launch's gate/up tiles
                if (et == 0 && !wait_counter(p.ready + tl.item, MB_I, p.err, p.timeout_ns, s_abort))
                    ok = false;
                ok = epi_bar_and(ok, C::EPI_THREADS);
                if (!ok) break;
                (void)ld_acquire(p.ready + tl.item);
            }
            const float* bs = tl.gu ? p.xs : p.hs;
            const int na = tl.gu ? 2 : 1;
            // the row block's weight block scales, one per K-block (operand 0:
            // gate or down, 1: up)
            const size_t wrow = (size_t(ex) * MB + tl.blk) * KB;
            const float* sw0 = (tl.gu ? (sh ? p.sh_s_gate : p.s_gate) : (sh ? p.sh_s_down : p.s_down)) + wrow;
            const float* sw1 = (sh ? p.sh_s_up : p.s_up) + wrow;
            // table [operand][kb][n] = weight block scale x row scale; rows are
            // read kb fastest (coalesced), four K-blocks per 16-byte load when
            // the rows allow it.  Row scales are read with plain loads: h's
            // come from this launch (acquired above).
            if (kVecTable && (KB & 3) == 0 &&
                ((reinterpret_cast<uintptr_t>(sw0) | reinterpret_cast<uintptr_t>(sw1) |
                  reinterpret_cast<uintptr_t>(bs)) & 15) == 0) {
                const int K4 = KB >> 2;
                if (MODE != kFfnFused) {
                    // consecutive threads on consecutive rows: conflict-free
                    // stores and no runtime division (measured a little faster
                    // in these kernels, not in the fused one)
                    for (int a = 0; a < na; ++a) {
                        const float4* w4 = reinterpret_cast<const float4*>(a ? sw1 : sw0);
                        for (int i = et; i < K4 * NT; i += C::EPI_THREADS) {
                            const int n = i % NT, k4 = i / NT;
                            const bool live = n < nrow;
                            const float4 w = __ldg(w4 + k4);
                            float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                            if (live)
                                x = reinterpret_cast<const float4*>(bs + size_t(row0 + n) * KB)[k4];
                            float* d = s_sc + (a * KB + 4 * k4) * NT + n;
                            d[0] = live ? w.x * x.x : 0.0f;
                            d[NT] = live ? w.y * x.y : 0.0f;
                            d[2 * NT] = live ? w.z * x.z : 0.0f;
                            d[3 * NT] = live ? w.w * x.w : 0.0f;
                        }
                    }
                } else {
                    for (int i = et; i < na * NT * K4; i += C::EPI_THREADS) {
                        const int a = i / (NT * K4), rem = i - a * (NT * K4);
                        const int n = rem / K4, k4 = rem - n * K4;
                        const float4 w = __ldg(reinterpret_cast<const float4*>(a ? sw1 : sw0) + k4);
                        float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        if (n < nrow)
                            x = reinterpret_cast<const float4*>(bs + size_t(row0 + n) * KB)[k4];
                        float* d = s_sc + (a * KB + 4 * k4) * NT + n;
                        const bool live = n < nrow;
                        d[0] = live ? w.x * x.x : 0.0f;
                        d[NT] = live ? w.y * x.y : 0.0f;
                        d[2 * NT] = live ? w.z * x.z : 0.0f;
                        d[3 * NT] = live ? w.w * x.w : 0.0f;
                    }
                }
            } else {
                for (int i = et; i < na * NT * KB; i += C::EPI_THREADS) {
                    const int a = i / (NT * KB), rem = i - a * (NT * KB);
                    const int n = rem / KB, kb = rem - n * KB;
                    const float w = (a ? sw1 : sw0)[kb];
                    s_sc[(a * KB + kb) * NT + n] =
                        (n < nrow) ? w * bs[size_t(row0 + n) * KB + kb] : 0.0f;
                }
            }
            if (!tl.gu)
                // each gathered row's output row: y_slots row r*K + k (>= 0)
                // or y_shared row r (stored as -1 - r)
                for (int i = et; i < NT; i += C::EPI_THREADS) {
                    int d = -1;
                    if (i < nrow) {
                        const int slot = p.ub[p.ul.src + row0 + i];
                        const int r = slot / p.KS, k = slot - r * p.KS;
                        d = (k < p.K) ? r * p.K + k : -1 - r;
                    }
                    s_src[i] = d;
                }
            ok = epi_bar_and(ok, C::EPI_THREADS);
            if (!ok) break;

            constexpr int CW = C::CW;
            // columns per TMEM load: 8 in the 18-warp blocks (96 registers a
            // thread), else up to 16
            float acc0[CW], acc1[CW];
#pragma unroll
            for (int j = 0; j < CW; ++j) {
                acc0[j] = 0.0f;
                acc1[j] = 0.0f;
            }
            // in the 32- and 64-row tiles a warp whose CW columns all lie past
            // the item's rows (a cold expert's short item) reads no partial and
            // computes nothing; it still hands each partial back and meets every
            // barrier (measured at 512 rows: GEMM 1.122 -> 1.093 ms; the 16-row
            // tile keeps the plain loop, 1% faster there)
            const bool live = NT == 16 || cg * CW < nrow;
            for (int kb = 0; kb < KB && ok; ++kb) {
                // a failed wait is acted on by the whole warp (tcgen05.ld is warp-wide).
                // No suspend hint here: the epilogue releases the partials the
                // MMA waits for, so it polls (measured: prefill4096's GEMMs
                // 3.788 -> 3.721 ms, decode512's 1.097 -> 1.089; the producer and
                // the MMA issuers keep the hint, and a sleep between their polls
                // was slower still)
                if (!__all_sync(0xFFFFFFFFu, mbar_wait<0>(
                                                 &kbrel[je % kKbRing], (je / kKbRing) & 1u, p.err,
                                                 p.timeout_ns))) {
                    ok = false;
                    *s_abort = 1;
                    break;
                }
                tc_fence_after();
                // the warp's CW columns of the partial(s) in one round trip to
                // tensor memory; the partial is handed back to the MMA as soon
                // as it sits in registers, before the FMAs
                const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                                    ab * C::ACC_COLS + cg * CW;
                float v0[CW], v1[CW];
                if (live) {
                    tmem_ld<CW>(ta, v0);
                    if (C::NA == 2 && tl.gu) tmem_ld<CW>(ta + NT, v1);
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[ab]);
                // acc = fma(partial, weight scale x row scale, acc), two
                // columns per packed instruction (each an IEEE fma)
                const float4* q0 = reinterpret_cast<const float4*>(s_sc + kb * NT + cg * CW);
                if (!live) {
                } else if (C::NA == 2 && tl.gu) {
                    const float4* q1 = reinterpret_cast<const float4*>(s_sc + (KB + kb) * NT + cg * CW);
#pragma unroll
                    for (int v = 0; v < CW / 4; ++v) {
                        const float4 a4 = q0[v], b4 = q1[v];
                        float* a0p = &acc0[4 * v];
                        float* a1p = &acc1[4 * v];
                        fma2(a0p[0], a0p[1], v0[4 * v], v0[4 * v + 1], a4.x, a4.y);
                        fma2(a0p[2], a0p[3], v0[4 * v + 2], v0[4 * v + 3], a4.z, a4.w);
                        fma2(a1p[0], a1p[1], v1[4 * v], v1[4 * v + 1], b4.x, b4.y);
                        fma2(a1p[2], a1p[3], v1[4 * v + 2], v1[4 * v + 3], b4.z, b4.w);
                    }
                } else {
#pragma unroll
                    for (int v = 0; v < CW / 4; ++v) {
                        const float4 a4 = q0[v];
                        float* a0p = &acc0[4 * v];
                        fma2(a0p[0], a0p[1], v0[4 * v], v0[4 * v + 1], a4.x, a4.y);
                        fma2(a0p[2], a0p[3], v0[4 * v + 2], v0[4 * v + 3], a4.z, a4.w);
                    }
                }
                ++je;
                if (++ab == C::ACC_BUFS) ab = 0;
            }
            if (C::NA == 2 && tl.gu) {
                // h = silu(g) * u; per-row amax over the 128 features
                float h[CW];
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    const int c = cg * CW + j;
                    const float g = acc0[j];
                    const float sg = kFastSilu ? __fdividef(g, 1.0f + __expf(-g))
                                               : g / (1.0f + __expf(-g));
                    h[j] = (c < nrow) ? sg * acc1[j] : 0.0f;
                    // amax over the warp's 32 features in one instruction:
                    // non-negative floats order as their bit patterns (a NaN
                    // counts as 0, as fmaxf would skip it)
                    const float ah = fabsf(h[j]);
                    const float a = __uint_as_float(__reduce_max_sync(
                        0xFFFFFFFFu, (ah == ah) ? __float_as_uint(ah) : 0u));
                    if (lane == 0) s_red[q * NT + c] = a;
                }
                ok = epi_bar_and(ok, C::EPI_THREADS);
                if (!ok) break;
                // each row's scale once: amax over the four lane quarters, / 448
                if (et < NT) {
                    const float amax = fmaxf(fmaxf(s_red[et], s_red[NT + et]),
                                             fmaxf(s_red[2 * NT + et], s_red[3 * NT + et]));
                    const float sc = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
                    s_red[4 * NT + et] = sc;
                    if (et < nrow) p.hs[size_t(row0 + et) * MB + tl.blk] = sc;
                }
                ok = epi_bar_and(ok, C::EPI_THREADS);
                if (!ok) break;
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    const int c = cg * CW + j;
                    s_tile[c * 128 + m] = to_e4m3(__fdiv_rn(h[j], s_red[4 * NT + c]));
                }
                ok = epi_bar_and(ok, C::EPI_THREADS);
                if (!ok) break;
                for (int i = et; i < nrow * 8; i += C::EPI_THREADS) {
                    const int c = i >> 3, ch = i & 7;
                    *reinterpret_cast<uint4*>(p.hq + size_t(row0 + c) * p.I + tl.blk * kBlock + ch * 16) =
                        *reinterpret_cast<const uint4*>(s_tile + c * 128 + ch * 16);
                }
                if (kFused) {
                    // release this block of h to the item's down tiles
                    ok = epi_bar_and(ok, C::EPI_THREADS);
                    if (!ok) break;
                    if (et == 0) {
                        fence_proxy_async_global();
                        __threadfence();
                        atomicAdd(p.ready + tl.item, 1);
                    }
                }
            } else if (C::STAGED_OUT && p.out_vec) {
                // the tile's rows through shared memory, then out as 16-byte
                // stores, a row's 512 bytes by 32 consecutive threads
                float* stg = reinterpret_cast<float*>(s_tile);   // [NT][128]
#pragma unroll
                for (int j = 0; j < CW; ++j) stg[(cg * CW + j) * kBlock + m] = acc0[j];
                ok = epi_bar_and(ok, C::EPI_THREADS);
                if (!ok) break;
                for (int i = et; i < nrow * 32; i += C::EPI_THREADS) {
                    const int c = i >> 5, v = i & 31;
                    const int d = s_src[c];
                    float* dst = (d >= 0) ? p.y_slots + size_t(d) * p.H
                                          : p.y_shared + size_t(-1 - d) * p.H;
                    reinterpret_cast<float4*>(dst + tl.blk * kBlock)[v] =
                        reinterpret_cast<const float4*>(stg + c * kBlock)[v];
                }
            } else {
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    const int c = cg * CW + j;
                    if (ok && c < nrow) {
                        const int d = s_src[c];
                        float* dst = (d >= 0) ? p.y_slots + size_t(d) * p.H
                                              : p.y_shared + size_t(-1 - d) * p.H;
                        dst[tl.blk * kBlock + m] = acc0[j];
                    }
                }
            }
        }
        if (!ok) *s_abort = 1;
    }

    __syncthreads();
    if (*s_abort) {
        // Wind down: let every copy this CTA issued land and every MMA finish
        // before the CTA releases tensor memory and exits.  A stage whose row
        // tile was never requested cannot complete its barrier, so the copies
        // get one shared budget of kDrainNs (they land within microseconds).
        constexpr uint64_t kDrainNs = 2000000;   // 2 ms
        if (threadIdx.x == 0) {
            // the K-blocks of the stages last filled (a K-block whose copies
            // were not all requested never completes: the budget ends it)
            const uint64_t t0 = globaltimer_ns();
            for (int q = 0; q < p.n_stages && issued > 0; ++q) {
                const uint32_t jj = used_by[q];
                if (jj == ~0u) continue;
                const uint64_t used = globaltimer_ns() - t0;
                if (used >= kDrainNs) break;
                mbar_wait(&kbfull[jj % kKbRing], (jj / kKbRing) & 1u, nullptr, kDrainNs - used);
            }
            while (globaltimer_ns() - t0 < kDrainNs / 4) __nanosleep(1000);
        }
        if (threadIdx.x == 64) mma_commit(drain);
        if (threadIdx.x == 32) {
            mma_commit(drain);
            mbar_wait(drain, 0, nullptr, kDrainNs);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ----------------------------------------------------------- launchers ----
template <int NT, int MODE>
static cudaError_t launch_ffn_t(const FfnMaps& mp, FfnArgs args, int n_sms, int smem_limit,
                                cudaStream_t stream) {
    using C = FfnCfg<NT, MODE>;
    const int KB_H = args.H / kBlock, KB_I = args.I / kBlock;
    const int kbmax = (MODE == kFfnGateUp) ? KB_H : (MODE == kFfnDown) ? KB_I : max(KB_H, KB_I);
    // HBM streams 16 KB tiles fastest with about 8 of them in flight per SM
    // (a TMA probe: 7.2 TB/s at 6-8, 6.5 at 12).  Measured: 10 stages at
    // 16-row tiles and in the separate gate/up and down kernels at 32 rows
    // (verify8's layer 0.2439 -> 0.2415 ms against 8, the same from 10 to 14:
    // the first tile requests more weights before its dependent-launch wait);
    // in those at 64 rows 7 up to 512 rows (decode512's GEMMs 1.141 -> 1.125
    // ms) and 6 above (prefill4096's 3.92 -> 3.82 ms); the fused kernel at 32
    // and 64 rows keeps every stage that fits.
    int stages = kMaxStages;
    if (NT == 16 || (MODE != kFfnFused && NT == 32)) stages = kStagesNt16;
    if (MODE != kFfnFused && NT == 64) stages = (args.R <= 512) ? kStagesWideDecode : kStagesWide;
    FfnSmem L = ffn_smem(NT, stages, kbmax, C::STAGE_BYTES, C::TILE_BYTES);
    while (stages > 2 && L.bytes > smem_limit) {
        --stages;
        L = ffn_smem(NT, stages, kbmax, C::STAGE_BYTES, C::TILE_BYTES);
    }
    if (L.bytes > smem_limit) return cudaErrorInvalidConfiguration;
    args.n_stages = stages;
    cudaError_t e =
        ensure_dyn_smem(reinterpret_cast<const void*>(ffn_kernel<NT, MODE>), L.bytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl(ffn_kernel<NT, MODE>, dim3(max(1, n_sms)), dim3(C::THREADS), L.bytes, stream,
                   mp.g, mp.u, mp.sg, mp.su, mp.x, mp.d, mp.sd, mp.h, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int MODE>
static cudaError_t launch_ffn_mode(int nt, const FfnMaps& mp, const FfnArgs& args, int n_sms,
                                   int smem_limit, cudaStream_t stream) {
    switch (nt) {
        case 16: return launch_ffn_t<16, MODE>(mp, args, n_sms, smem_limit, stream);
        case 32: return launch_ffn_t<32, MODE>(mp, args, n_sms, smem_limit, stream);
        case 64: return launch_ffn_t<64, MODE>(mp, args, n_sms, smem_limit, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_ffn(int nt, int mode, const FfnMaps& mp, const FfnArgs& args, int n_sms,
                       int smem_limit, cudaStream_t stream) {
    switch (mode) {
        case kFfnGateUp: return launch_ffn_mode<kFfnGateUp>(nt, mp, args, n_sms, smem_limit, stream);
        case kFfnDown: return launch_ffn_mode<kFfnDown>(nt, mp, args, n_sms, smem_limit, stream);
        case kFfnFused: return launch_ffn_mode<kFfnFused>(nt, mp, args, n_sms, smem_limit, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
