// layout.h -- word offsets of the union buffer and byte offsets of the
// workspaces, computed identically on the host (sizes, launches) and passed
// to the kernels by value.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace moe {

// Word offsets inside the int32 union buffer (see moe_build_union).
struct UnionLayout {
    int32_t counts, offsets, ulist, pos, src, items, max_items, words;
};

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Rows per GEMM work item: the MMA N dimension, fixed by the row count of the
// call (a graph captured at R always replays the same kernels).  Above 256
// rows the 64-row tile: experts hit by hundreds of rows (Zipf-skewed decode
// batches) are cut into half as many items, each of which streams the
// expert's weights to its SM again (measured at 512 rows: layer 1.331 ->
// 1.284 ms against 32-row tiles).
inline int rows_per_item(int32_t R) {
    if (R <= 64) return 16;
    if (R <= 256) return 32;
    return 64;
}

inline UnionLayout union_layout(int32_t E, int32_t K, int32_t S, int32_t R) {
    UnionLayout L;
    const int64_t KS = K + S;
    int64_t w = 8;
    L.counts = static_cast<int32_t>(w);
    w += E + 1;
    L.offsets = static_cast<int32_t>(w);
    w += E + 2;
    L.ulist = static_cast<int32_t>(w);
    w += E + 1;
    L.pos = static_cast<int32_t>(w);
    w += int64_t(R) * KS;
    L.src = static_cast<int32_t>(w);
    w += int64_t(R) * KS;
    w = round_up(w, 4);
    L.items = static_cast<int32_t>(w);
    // sum over entries of ceil(count / n) <= (R*KS)/n + (number of entries)
    const int64_t entries = (E < int64_t(R) * K ? E : int64_t(R) * K) + S;
    L.max_items = static_cast<int32_t>(int64_t(R) * KS / 16 + entries + 1);
    w += int64_t(L.max_items) * 4;
    L.words = static_cast<int32_t>(round_up(w, 64));
    return L;
}

// The w8a16 variant: calls of at most kW8A16MaxRows rows, items of
// kW8A16RowsPerItem rows (the fp8 path's item size at these row counts).
constexpr int32_t kW8A16MaxRows = 64;
constexpr int32_t kW8A16RowsPerItem = 16;

// Scratch of the expert FFN stage (byte offsets from the workspace base).
// The w8a16 variant's bf16 rows (xb) and bf16 h (hb) reuse the fp8 path's
// region from xg on; they exist only for R <= kW8A16MaxRows (else -1).
// Words of the expert GEMM's tile scheduler (counter, CTAs done) after the
// per-item counters; the dispatch kernels zero both regions.
constexpr int32_t kSchedWords = 2;

struct FfnLayout {
    int64_t ctl, ready, sched, xg, xs, hq, hs, xb, hb, bytes;
    int64_t rows;       // capacity in gathered rows
    int32_t n_ready;    // per-item counters of the fused GEMM
};

inline FfnLayout ffn_layout(int32_t H, int32_t I, int32_t E, int32_t K, int32_t S, int32_t R) {
    FfnLayout L;
    L.rows = round_up(int64_t(R) * (K + S), 64) + 64;
    L.n_ready = union_layout(E, K, S, R).max_items;
    int64_t b = 0;
    L.ctl = b;
    b += 256;
    L.ready = b;
    L.sched = b + int64_t(L.n_ready) * 4;   // right after ready: zeroed with it
    b = round_up(L.sched + kSchedWords * 4, 256);
    L.xg = b;
    b = round_up(b + L.rows * H, 256);
    L.xs = b;
    b = round_up(b + L.rows * (H / 128) * 4, 256);
    L.hq = b;
    b = round_up(b + L.rows * I, 256);
    L.hs = b;
    b = round_up(b + L.rows * (I / 128) * 4, 256);
    L.bytes = b;
    L.xb = L.hb = -1;
    if (R <= kW8A16MaxRows) {
        L.xb = L.xg;
        L.hb = round_up(L.xb + L.rows * H * 2, 256);
        const int64_t end = round_up(L.hb + L.rows * I * 2, 256);
        if (end > L.bytes) L.bytes = end;
    }
    return L;
}

// Workspace of the fused layer: the FFN scratch first (so the error word sits
// at the head of the workspace), then routing, union and slot outputs.
struct LayerLayout {
    FfnLayout ffn;
    UnionLayout un;
    int64_t logits, ids, wts, ubuf, y_slots, y_shared, bytes;
};

inline LayerLayout layer_layout(int32_t H, int32_t I, int32_t E, int32_t K, int32_t S,
                                int32_t R) {
    LayerLayout L;
    L.ffn = ffn_layout(H, I, E, K, S, R);
    L.un = union_layout(E, K, S, R);
    int64_t b = L.ffn.bytes;
    L.logits = b;
    b = round_up(b + int64_t(R) * E * 4, 256);
    L.ids = b;
    b = round_up(b + int64_t(R) * K * 4, 256);
    L.wts = b;
    b = round_up(b + int64_t(R) * K * 4, 256);
    L.ubuf = b;
    b = round_up(b + int64_t(L.un.words) * 4, 256);
    L.y_slots = b;
    b = round_up(b + int64_t(R) * K * H * 4, 256);
    L.y_shared = b;
    b = round_up(b + int64_t(R) * H * 4, 256);
    L.bytes = b;
    return L;
}

}  // namespace moe
