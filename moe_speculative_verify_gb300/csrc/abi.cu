// abi.cu -- host side of the C ABI declared in include/moe_verify.h:
// argument validation, workspace carving, TMA tensor maps and kernel
// launches.  No allocation, no state between calls beyond cached device
// attributes and the driver entry point, no host synchronisation except in
// moe_get_device_error.
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "layout.h"

namespace {

using moe::FfnLayout;
using moe::LayerLayout;
using moe::UnionLayout;

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks: malformed shapes are invalid; well-formed ones beyond the
// compiled limits are unsupported.
moe_status_t check_cfg(const moe_config_t* c) {
    if (c == nullptr) return MOE_ERR_INVALID_ARG;
    if (c->hidden <= 0 || c->inter <= 0 || c->hidden % MOE_BLOCK || c->inter % MOE_BLOCK)
        return MOE_ERR_INVALID_ARG;
    if (c->n_experts <= 0 || c->n_groups <= 0 || c->n_experts % c->n_groups) return MOE_ERR_INVALID_ARG;
    if (c->topk_groups <= 0 || c->topk_groups > c->n_groups) return MOE_ERR_INVALID_ARG;
    if (c->topk <= 0 || c->topk > c->topk_groups * (c->n_experts / c->n_groups))
        return MOE_ERR_INVALID_ARG;
    if (c->n_shared < 0 || !std::isfinite(c->routed_scaling)) return MOE_ERR_INVALID_ARG;
    if (c->hidden > 16384 || c->inter > 16384 || c->n_experts > MOE_MAX_EXPERTS ||
        c->n_groups > MOE_MAX_GROUPS || c->topk > MOE_MAX_TOPK || c->n_shared > 1)
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status_t check_rows(int32_t R) {
    if (R < 0) return MOE_ERR_INVALID_ARG;
    if (R > MOE_MAX_ROWS) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

uint64_t timeout_ns(const moe_config_t* c) {
    return static_cast<uint64_t>(c->wait_timeout_us ? c->wait_timeout_us : 2000000u) * 1000ull;
}

struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;
};

DeviceInfo device_info() {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DeviceInfo{};
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sms == 0) {
        DeviceInfo d;
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cache[dev] = d;
    }
    return cache[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D uint8 tensor [rows, cols] (cols contiguous), 128-byte-swizzled boxes of
// 128 columns x box_rows rows; out-of-range rows read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

moe_status_t check_weights(const moe_config_t* c, const moe_weights_t* w) {
    if (w == nullptr) return MOE_ERR_INVALID_ARG;
    if (w->layout != MOE_LAYOUT_ROW_MAJOR && w->layout != MOE_LAYOUT_TILED)
        return MOE_ERR_INVALID_ARG;
    const void* codes[3] = {w->w_gate, w->w_up, w->w_down};
    const float* scales[3] = {w->s_gate, w->s_up, w->s_down};
    for (int i = 0; i < 3; ++i) {
        if (!codes[i] || !scales[i] || !aligned(codes[i], 16) || !aligned(scales[i], 4))
            return MOE_ERR_INVALID_ARG;
    }
    if (c->n_shared > 0) {
        const void* sc[3] = {w->sh_gate, w->sh_up, w->sh_down};
        const float* ss[3] = {w->sh_s_gate, w->sh_s_up, w->sh_s_down};
        for (int i = 0; i < 3; ++i)
            if (!sc[i] || !ss[i] || !aligned(sc[i], 16) || !aligned(ss[i], 4))
                return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

// The large-R router's maps: x bf16 [R, H] and w fp32 [E, H], boxes of
// kRouterStageCols columns x 32 rows, unswizzled; rows and columns past the
// end read as zero.
// The last few tensor-map sets built on this thread, keyed by everything
// that goes into them (pointers, sizes, boxes, layout): a call on the same
// buffers reuses them instead of encoding them again (each encoding is a
// host call on the path of every layer).  Keys are compared bytewise and
// built from zeroed memory.
template <typename Key, typename Val, int N = 4>
struct MapCache {
    Key key[N];
    Val val[N];
    bool used[N] = {};
    int next = 0;
    const Val* find(const Key& k) const {
        for (int i = 0; i < N; ++i)
            if (used[i] && std::memcmp(&key[i], &k, sizeof(Key)) == 0) return &val[i];
        return nullptr;
    }
    void put(const Key& k, const Val& v) {
        key[next] = k;
        val[next] = v;
        used[next] = true;
        next = (next + 1) % N;
    }
};

struct RouterMapKey {
    const void* x;
    const void* wr;
    int R, H, E, n_sms;
};

bool make_router_maps(const void* x, const float* wr, int R, int H, int E, int n_sms,
                      moe::RouterMaps* m) {
    RouterMapKey k;
    std::memset(&k, 0, sizeof(k));
    k.x = x;
    k.wr = wr;
    k.R = R;
    k.H = H;
    k.E = E;
    k.n_sms = n_sms;
    thread_local MapCache<RouterMapKey, moe::RouterMaps> cache;
    if (const moe::RouterMaps* hit = cache.find(k)) {
        *m = *hit;
        return true;
    }
    auto fn = encode_fn();
    if (!fn) return false;
    m->rt = moe::router_rows_per_warp(R, E, n_sms);
    const cuuint32_t xbox[2] = {cuuint32_t(moe::kRouterStageCols), cuuint32_t(4 * m->rt)};
    const cuuint32_t box[2] = {cuuint32_t(moe::kRouterStageCols), 32};
    const cuuint32_t es[2] = {1, 1};
    const cuuint64_t xd[2] = {cuuint64_t(H), cuuint64_t(R)}, xs[1] = {cuuint64_t(H) * 2};
    const cuuint64_t wd[2] = {cuuint64_t(H), cuuint64_t(E)}, wst[1] = {cuuint64_t(H) * 4};
    return fn(&m->x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), xd, xs, xbox, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
               CUDA_SUCCESS &&
           fn(&m->w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(wr), wd, wst, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
               CUDA_SUCCESS &&
           (cache.put(k, *m), true);
}

moe_status_t route_impl(const moe_config_t* c, const void* x, const float* wr, const float* bias,
                        const uint8_t* valid, int32_t R, int32_t* ids, float* wts, float* logits,
                        int32_t* err, cudaStream_t s) {
    moe::RouterMaps maps;
    const int sms = device_info().sms;
    if (R > moe::kRouteUnionMaxRows &&
        !make_router_maps(x, wr, R, c->hidden, c->n_experts, sms, &maps))
        return MOE_ERR_CUDA;
    return cuda_status(moe::launch_router(static_cast<const uint16_t*>(x), wr, bias, valid, R,
                                          c->hidden, c->n_experts, c->n_groups, c->topk_groups,
                                          c->topk, c->routed_scaling, ids, wts, logits, &maps,
                                          sms, err, timeout_ns(c), s));
}

moe_status_t union_impl(const moe_config_t* c, const int32_t* ids, int32_t R, int32_t* ub,
                        cudaStream_t s) {
    const UnionLayout L = moe::union_layout(c->n_experts, c->topk, c->n_shared, R);
    return cuda_status(moe::launch_union(ids, R, c->n_experts, c->topk, c->n_shared,
                                         moe::rows_per_item(R), ub, L, s));
}

// Pointers into the FFN workspace of one call.
struct FfnCall {
    FfnLayout FL;
    UnionLayout UL;
    int32_t* err;
    int32_t* ready;
    int32_t* sched;
    uint8_t* xg;
    float* xs;
    uint8_t* hq;
    float* hs;
    int nt;
};

FfnCall ffn_call(const moe_config_t* c, int32_t R, void* ws) {
    FfnCall f;
    f.FL = moe::ffn_layout(c->hidden, c->inter, c->n_experts, c->topk, c->n_shared, R);
    f.UL = moe::union_layout(c->n_experts, c->topk, c->n_shared, R);
    uint8_t* base = static_cast<uint8_t*>(ws);
    f.err = reinterpret_cast<int32_t*>(base + f.FL.ctl);
    f.ready = reinterpret_cast<int32_t*>(base + f.FL.ready);
    f.sched = reinterpret_cast<int32_t*>(base + f.FL.sched);
    f.xg = base + f.FL.xg;
    f.xs = reinterpret_cast<float*>(base + f.FL.xs);
    f.hq = base + f.FL.hq;
    f.hs = reinterpret_cast<float*>(base + f.FL.hs);
    f.nt = moe::rows_per_item(R);
    return f;
}

// 2-D bf16 tensor [rows, cols]: 128-byte-swizzled boxes of 64 columns x
// box_rows rows; out-of-range rows read as zero.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weight codes of matrices stacked to [rows, cols] (rows = matrices x their
// rows): 128x128 boxes, in either layout.  A tiled tensor is a column of
// 16 KB blocks, so its map is [rows * cols/128, 128]: block (rb, kb) of the
// stack is the box at row (rb * cols/128 + kb) * 128.
bool make_wmap(CUtensorMap* m, const void* base, int layout, uint64_t rows, uint64_t cols) {
    return layout == MOE_LAYOUT_TILED ? make_map(m, base, rows * (cols / 128), 128, 128)
                                      : make_map(m, base, rows, cols, 128);
}

struct FfnMapKey {
    const void* p[8];
    int64_t rows;
    int H, I, E, S, layout, nt;
};

// The eight tensor maps of the expert GEMMs.  Shared-expert maps fall back to
// the routed tensors when there is no shared expert (never read then).
bool make_maps(const moe_config_t* c, const moe_weights_t* w, const FfnCall& f, moe::FfnMaps* mp) {
    const int H = c->hidden, I = c->inter, E = c->n_experts, S = c->n_shared;
    FfnMapKey k;
    std::memset(&k, 0, sizeof(k));
    const void* ps[8] = {w->w_gate, w->w_up, S ? w->sh_gate : w->w_gate, S ? w->sh_up : w->w_up,
                         f.xg, w->w_down, S ? w->sh_down : w->w_down, f.hq};
    for (int i = 0; i < 8; ++i) k.p[i] = ps[i];
    k.rows = f.FL.rows;
    k.H = H;
    k.I = I;
    k.E = E;
    k.S = S;
    k.layout = w->layout;
    k.nt = f.nt;
    thread_local MapCache<FfnMapKey, moe::FfnMaps> cache;
    if (const moe::FfnMaps* hit = cache.find(k)) {
        *mp = *hit;
        return true;
    }
    const uint64_t srows = S ? uint64_t(S) : 1ull;
    const int lo = w->layout;
    const bool ok = make_wmap(&mp->g, w->w_gate, lo, uint64_t(E) * I, H) &&
                    make_wmap(&mp->u, w->w_up, lo, uint64_t(E) * I, H) &&
                    make_wmap(&mp->sg, ps[2], lo, srows * I, H) &&
                    make_wmap(&mp->su, ps[3], lo, srows * I, H) &&
                    make_map(&mp->x, f.xg, f.FL.rows, H, f.nt) &&
                    make_wmap(&mp->d, w->w_down, lo, uint64_t(E) * H, I) &&
                    make_wmap(&mp->sd, ps[6], lo, srows * H, I) &&
                    make_map(&mp->h, f.hq, f.FL.rows, I, f.nt);
    if (ok) cache.put(k, *mp);
    return ok;
}

moe::FfnArgs ffn_args(const moe_config_t* c, const moe_weights_t* w, const int32_t* ub, int32_t R,
                      const FfnCall& f, float* y_slots, float* y_shared) {
    const int S = c->n_shared;
    moe::FfnArgs a{};
    a.ub = ub;
    a.ul = f.UL;
    a.s_gate = w->s_gate;
    a.s_up = w->s_up;
    a.sh_s_gate = S ? w->sh_s_gate : w->s_gate;
    a.sh_s_up = S ? w->sh_s_up : w->s_up;
    a.s_down = w->s_down;
    a.sh_s_down = S ? w->sh_s_down : w->s_down;
    a.xs = f.xs;
    a.hq = f.hq;
    a.hs = f.hs;
    a.y_slots = y_slots;
    a.y_shared = y_shared;
    a.out_vec = aligned(y_slots, 16) && (y_shared == nullptr || aligned(y_shared, 16));
    a.ready = f.ready;
    a.sched = f.sched;
    a.err = f.err;
    a.R = R;
    a.ushape = moe::union_shape_word(c->n_experts, c->topk, c->n_shared);
    a.H = c->hidden;
    a.I = c->inter;
    a.E = c->n_experts;
    a.K = c->topk;
    a.KS = c->topk + S;
    a.tiled = w->layout == MOE_LAYOUT_TILED;
    a.timeout_ns = timeout_ns(c);
    return a;
}

moe_status_t dispatch_impl(const moe_config_t* c, const void* x, const int32_t* ub, int32_t R,
                           void* ws, cudaStream_t s) {
    const FfnCall f = ffn_call(c, R, ws);
    return cuda_status(moe::launch_dispatch(
        static_cast<const uint16_t*>(x), ub, f.UL, R, c->hidden, c->topk + c->n_shared,
        moe::union_shape_word(c->n_experts, c->topk, c->n_shared), f.xg, f.xs, f.ready,
        f.FL.n_ready + moe::kSchedWords, f.err, s));
}

// One of the three expert-GEMM modes (gate/up, down, or both fused).
moe_status_t gemm_impl(int mode, const moe_config_t* c, const moe_weights_t* w, const int32_t* ub,
                       int32_t R, float* y_slots, float* y_shared, void* ws, cudaStream_t s) {
    const FfnCall f = ffn_call(c, R, ws);
    const DeviceInfo dev = device_info();
    if (dev.sms <= 0) return MOE_ERR_CUDA;
    moe::FfnMaps mp;
    if (!make_maps(c, w, f, &mp)) return MOE_ERR_CUDA;
    return cuda_status(moe::launch_ffn(f.nt, mode, mp, ffn_args(c, w, ub, R, f, y_slots, y_shared),
                                       dev.sms, dev.smem_optin, s));
}

moe_status_t ffn_impl(const moe_config_t* c, const void* x, const moe_weights_t* w,
                      const int32_t* ub, int32_t R, float* y_slots, float* y_shared, void* ws,
                      cudaStream_t s) {
    moe_status_t st = dispatch_impl(c, x, ub, R, ws, s);
    if (st != MOE_OK) return st;
    // One fused launch at 16-row tiles (up to 64 rows).  At wider tiles the
    // gate/up and down launches measured faster (prefill 5.12 -> 4.46 ms,
    // decode512 1.37 -> 1.27 ms for the GEMMs): the down kernel keeps twice as
    // many tensor-memory partials, and with hundreds of tiles per SM the wave
    // tail between the launches costs little.  Same values either way.
    if (moe::rows_per_item(R) == 16)
        return gemm_impl(moe::kFfnFused, c, w, ub, R, y_slots, y_shared, ws, s);
    if ((st = gemm_impl(moe::kFfnGateUp, c, w, ub, R, nullptr, nullptr, ws, s)) != MOE_OK)
        return st;
    return gemm_impl(moe::kFfnDown, c, w, ub, R, y_slots, y_shared, ws, s);
}

// The w8a16 variant: bf16 rows gathered, then the dequantising GEMM kernel.
moe_status_t ffn16_impl(const moe_config_t* c, const void* x, const moe_weights_t* w,
                        const int32_t* ub, int32_t R, float* y_slots, float* y_shared, void* ws,
                        cudaStream_t s) {
    const FfnCall f = ffn_call(c, R, ws);
    if (f.FL.xb < 0 || f.nt != moe::kW8A16RowsPerItem) return MOE_ERR_UNSUPPORTED;
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint16_t* xb = reinterpret_cast<uint16_t*>(base + f.FL.xb);
    uint16_t* hb = reinterpret_cast<uint16_t*>(base + f.FL.hb);
    const int H = c->hidden, I = c->inter, E = c->n_experts, S = c->n_shared;
    moe_status_t st = cuda_status(moe::launch_dispatch16(
        static_cast<const uint16_t*>(x), ub, f.UL, R, H, c->topk + S,
        moe::union_shape_word(E, c->topk, S), xb, f.ready, f.FL.n_ready + moe::kSchedWords, f.err,
        s));
    if (st != MOE_OK) return st;
    const DeviceInfo dev = device_info();
    if (dev.sms <= 0) return MOE_ERR_CUDA;
    moe::FfnMaps mp;
    const uint64_t srows = S ? uint64_t(S) : 1ull;
    const int lo = w->layout;
    if (!(make_wmap(&mp.g, w->w_gate, lo, uint64_t(E) * I, H) &&
          make_wmap(&mp.u, w->w_up, lo, uint64_t(E) * I, H) &&
          make_wmap(&mp.sg, S ? w->sh_gate : w->w_gate, lo, srows * I, H) &&
          make_wmap(&mp.su, S ? w->sh_up : w->w_up, lo, srows * I, H) &&
          make_map_bf16(&mp.x, xb, f.FL.rows, H, moe::kW8A16RowsPerItem) &&
          make_wmap(&mp.d, w->w_down, lo, uint64_t(E) * H, I) &&
          make_wmap(&mp.sd, S ? w->sh_down : w->w_down, lo, srows * H, I) &&
          make_map_bf16(&mp.h, hb, f.FL.rows, I, moe::kW8A16RowsPerItem)))
        return MOE_ERR_CUDA;
    moe::Ffn16Args a{};
    a.ub = ub;
    a.ul = f.UL;
    a.s_gate = w->s_gate;
    a.s_up = w->s_up;
    a.sh_s_gate = S ? w->sh_s_gate : w->s_gate;
    a.sh_s_up = S ? w->sh_s_up : w->s_up;
    a.s_down = w->s_down;
    a.sh_s_down = S ? w->sh_s_down : w->s_down;
    a.hb = hb;
    a.y_slots = y_slots;
    a.y_shared = y_shared;
    a.ready = f.ready;
    a.sched = f.sched;
    a.err = f.err;
    a.R = R;
    a.ushape = moe::union_shape_word(E, c->topk, S);
    a.H = H;
    a.I = I;
    a.E = E;
    a.K = c->topk;
    a.KS = c->topk + S;
    a.tiled = w->layout == MOE_LAYOUT_TILED;
    a.timeout_ns = timeout_ns(c);
    return cuda_status(moe::launch_ffn16(mp, a, dev.sms, dev.smem_optin, s));
}

moe_status_t combine_impl(const moe_config_t* c, const float* y_slots, const float* y_shared,
                          const float* wts, const int32_t* ub, int32_t R, void* out,
                          cudaStream_t s) {
    const UnionLayout UL = moe::union_layout(c->n_experts, c->topk, c->n_shared, R);
    return cuda_status(moe::launch_combine(y_slots, y_shared, wts, const_cast<int32_t*>(ub), UL, R,
                                           c->n_experts, c->hidden, c->topk, c->n_shared,
                                           static_cast<uint16_t*>(out), s));
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    }
    return "MOE_ERR_UNKNOWN";
}

size_t moe_union_bytes(const moe_config_t* cfg, int32_t max_rows) {
    if (check_cfg(cfg) != MOE_OK || check_rows(max_rows) != MOE_OK) return 0;
    return size_t(moe::union_layout(cfg->n_experts, cfg->topk, cfg->n_shared, max_rows).words) * 4;
}

size_t moe_ffn_workspace_bytes(const moe_config_t* cfg, int32_t max_rows) {
    if (check_cfg(cfg) != MOE_OK || check_rows(max_rows) != MOE_OK) return 0;
    return size_t(moe::ffn_layout(cfg->hidden, cfg->inter, cfg->n_experts, cfg->topk, cfg->n_shared,
                                  max_rows)
                      .bytes);
}

size_t moe_workspace_bytes(const moe_config_t* cfg, int32_t max_rows) {
    if (check_cfg(cfg) != MOE_OK || check_rows(max_rows) != MOE_OK) return 0;
    return size_t(moe::layer_layout(cfg->hidden, cfg->inter, cfg->n_experts, cfg->topk,
                                    cfg->n_shared, max_rows)
                      .bytes);
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, int32_t max_rows, size_t* bytes) {
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    *bytes = 0;
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(max_rows)) != MOE_OK) return st;
    *bytes = moe_workspace_bytes(cfg, max_rows);
    return MOE_OK;
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x_bf16, const float* w_router,
                       const float* bias, const uint8_t* row_valid, int32_t R, int32_t* topk_ids,
                       float* topk_w, float* logits, moe_stream_t stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(R)) != MOE_OK) return st;
    if (R == 0) return MOE_OK;  // nothing to do; empty arrays may be NULL
    if (!x_bf16 || !w_router || !bias || !topk_ids || !topk_w || !logits) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(w_router, 16) || !aligned(bias, 4) ||
        !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(logits, 4))
        return MOE_ERR_INVALID_ARG;
    return route_impl(cfg, x_bf16, w_router, bias, row_valid, R, topk_ids, topk_w, logits,
                      nullptr, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_build_union(const moe_config_t* cfg, const int32_t* topk_ids, int32_t R,
                             int32_t* union_buf, size_t union_bytes, moe_stream_t stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(R)) != MOE_OK) return st;
    if (R == 0) return MOE_OK;  // nothing to do; empty arrays may be NULL
    if (!topk_ids || !union_buf || !aligned(topk_ids, 4) || !aligned(union_buf, 16))
        return MOE_ERR_INVALID_ARG;
    if (union_bytes < moe_union_bytes(cfg, R)) return MOE_ERR_WORKSPACE;
    return union_impl(cfg, topk_ids, R, union_buf, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn_fp8(const moe_config_t* cfg, const void* x_bf16,
                                const moe_weights_t* w, const int32_t* union_buf, int32_t R,
                                float* y_slots, float* y_shared, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(R)) != MOE_OK) return st;
    if (R == 0) return MOE_OK;  // nothing to do; empty arrays may be NULL
    if ((st = check_weights(cfg, w)) != MOE_OK) return st;
    if (!x_bf16 || !union_buf || !y_slots || !ws) return MOE_ERR_INVALID_ARG;
    if (cfg->n_shared > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(union_buf, 16) || !aligned(y_slots, 4) ||
        (y_shared && !aligned(y_shared, 4)) || !aligned(ws, 256))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_ffn_workspace_bytes(cfg, R)) return MOE_ERR_WORKSPACE;
    return ffn_impl(cfg, x_bf16, w, union_buf, R, y_slots, y_shared, ws,
                    reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn_w8a16(const moe_config_t* cfg, const void* x_bf16,
                                  const moe_weights_t* w, const int32_t* union_buf, int32_t R,
                                  float* y_slots, float* y_shared, void* ws, size_t ws_bytes,
                                  moe_stream_t stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(R)) != MOE_OK) return st;
    if (R > MOE_W8A16_MAX_ROWS) return MOE_ERR_UNSUPPORTED;
    if (R == 0) return MOE_OK;
    if ((st = check_weights(cfg, w)) != MOE_OK) return st;
    if (!x_bf16 || !union_buf || !y_slots || !ws) return MOE_ERR_INVALID_ARG;
    if (cfg->n_shared > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(union_buf, 16) || !aligned(y_slots, 4) ||
        (y_shared && !aligned(y_shared, 4)) || !aligned(ws, 256))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_ffn_workspace_bytes(cfg, R)) return MOE_ERR_WORKSPACE;
    return ffn16_impl(cfg, x_bf16, w, union_buf, R, y_slots, y_shared, ws,
                      reinterpret_cast<cudaStream_t>(stream));
}

// Common checks of the FFN-stage entry points.
static moe_status_t check_ffn_call(const moe_config_t* cfg, const int32_t* union_buf, int32_t R,
                                   void* ws, size_t ws_bytes) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(R)) != MOE_OK) return st;
    if (R == 0) return MOE_OK;
    if (!union_buf || !ws || !aligned(union_buf, 16) || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_ffn_workspace_bytes(cfg, R)) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x_bf16, const int32_t* union_buf,
                          int32_t R, void* ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status_t st = check_ffn_call(cfg, union_buf, R, ws, ws_bytes);
    if (st != MOE_OK || R == 0) return st;
    if (!x_bf16 || !aligned(x_bf16, 16)) return MOE_ERR_INVALID_ARG;
    return dispatch_impl(cfg, x_bf16, union_buf, R, ws, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_gate_up_fp8(const moe_config_t* cfg, const moe_weights_t* w,
                             const int32_t* union_buf, int32_t R, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
    moe_status_t st = check_ffn_call(cfg, union_buf, R, ws, ws_bytes);
    if (st != MOE_OK || R == 0) return st;
    if ((st = check_weights(cfg, w)) != MOE_OK) return st;
    return gemm_impl(moe::kFfnGateUp, cfg, w, union_buf, R, nullptr, nullptr, ws,
                     reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_down_fp8(const moe_config_t* cfg, const moe_weights_t* w,
                          const int32_t* union_buf, int32_t R, float* y_slots, float* y_shared,
                          void* ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status_t st = check_ffn_call(cfg, union_buf, R, ws, ws_bytes);
    if (st != MOE_OK || R == 0) return st;
    if ((st = check_weights(cfg, w)) != MOE_OK) return st;
    if (!y_slots || !aligned(y_slots, 4) || (cfg->n_shared > 0 && (!y_shared || !aligned(y_shared, 4))))
        return MOE_ERR_INVALID_ARG;
    return gemm_impl(moe::kFfnDown, cfg, w, union_buf, R, y_slots, y_shared, ws,
                     reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_gemms_fp8(const moe_config_t* cfg, const moe_weights_t* w,
                                  const int32_t* union_buf, int32_t R, float* y_slots,
                                  float* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status_t st = check_ffn_call(cfg, union_buf, R, ws, ws_bytes);
    if (st != MOE_OK || R == 0) return st;
    if ((st = check_weights(cfg, w)) != MOE_OK) return st;
    if (!y_slots || !aligned(y_slots, 4) || (cfg->n_shared > 0 && (!y_shared || !aligned(y_shared, 4))))
        return MOE_ERR_INVALID_ARG;
    return gemm_impl(moe::kFfnFused, cfg, w, union_buf, R, y_slots, y_shared, ws,
                     reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine(const moe_config_t* cfg, const float* y_slots, const float* y_shared,
                         const float* topk_w, const int32_t* union_buf, int32_t R, void* out_bf16,
                         moe_stream_t stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(R)) != MOE_OK) return st;
    if (R == 0) return MOE_OK;  // nothing to do; empty arrays may be NULL
    if (!y_slots || !topk_w || !union_buf || !out_bf16) return MOE_ERR_INVALID_ARG;
    if (cfg->n_shared > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
    if (!aligned(y_slots, 16) || (y_shared && !aligned(y_shared, 16)) || !aligned(topk_w, 4) ||
        !aligned(union_buf, 16) || !aligned(out_bf16, 16))
        return MOE_ERR_INVALID_ARG;
    return combine_impl(cfg, y_slots, y_shared, topk_w, union_buf, R, out_bf16,
                        reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine_add_rmsnorm(const moe_config_t* cfg, const float* y_slots,
                                     const float* y_shared, const float* topk_w,
                                     const int32_t* union_buf, int32_t R, const void* residual_bf16,
                                     const float* gamma, float eps, void* residual_out_bf16,
                                     void* normed_bf16, moe_stream_t stream) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(R)) != MOE_OK) return st;
    if (R == 0) return MOE_OK;
    if (!y_slots || !topk_w || !union_buf || !residual_bf16 || !gamma || !residual_out_bf16 ||
        !normed_bf16 || !(eps >= 0.0f))
        return MOE_ERR_INVALID_ARG;
    if (cfg->n_shared > 0 && !y_shared) return MOE_ERR_INVALID_ARG;
    if (!aligned(y_slots, 16) || (y_shared && !aligned(y_shared, 16)) || !aligned(topk_w, 4) ||
        !aligned(union_buf, 16) || !aligned(residual_bf16, 16) || !aligned(gamma, 16) ||
        !aligned(residual_out_bf16, 16) || !aligned(normed_bf16, 16))
        return MOE_ERR_INVALID_ARG;
    const UnionLayout UL = moe::union_layout(cfg->n_experts, cfg->topk, cfg->n_shared, R);
    return cuda_status(moe::launch_combine_add_rmsnorm(
        y_slots, y_shared, topk_w, const_cast<int32_t*>(union_buf), UL, R, cfg->n_experts,
        cfg->hidden, cfg->topk, cfg->n_shared,
        static_cast<const uint16_t*>(residual_bf16), gamma, eps,
        static_cast<uint16_t*>(residual_out_bf16), static_cast<uint16_t*>(normed_bf16),
        reinterpret_cast<cudaStream_t>(stream)));
}

static moe_status_t layer_impl(const moe_config_t* cfg, const void* x_bf16,
                               const float* w_router, const float* bias, const moe_weights_t* w,
                               const uint8_t* row_valid, int32_t R, void* out_bf16,
                               int32_t* topk_ids_out, float* topk_w_out, void* ws,
                               size_t ws_bytes, moe_stream_t stream, bool w8a16) {
    moe_status_t st = check_cfg(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_rows(R)) != MOE_OK) return st;
    if (w8a16 && R > MOE_W8A16_MAX_ROWS) return MOE_ERR_UNSUPPORTED;
    if (R == 0) return MOE_OK;  // nothing to do; empty arrays may be NULL
    if ((st = check_weights(cfg, w)) != MOE_OK) return st;
    if (!x_bf16 || !w_router || !bias || !out_bf16 || !ws) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(w_router, 16) || !aligned(bias, 4) ||
        !aligned(out_bf16, 16) || !aligned(ws, 256) ||
        (topk_ids_out && !aligned(topk_ids_out, 4)) || (topk_w_out && !aligned(topk_w_out, 4)))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_workspace_bytes(cfg, R)) return MOE_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const LayerLayout L = moe::layer_layout(cfg->hidden, cfg->inter, cfg->n_experts, cfg->topk,
                                            cfg->n_shared, R);
    uint8_t* base = static_cast<uint8_t*>(ws);
    float* logits = reinterpret_cast<float*>(base + L.logits);
    int32_t* ids = topk_ids_out ? topk_ids_out : reinterpret_cast<int32_t*>(base + L.ids);
    float* wts = topk_w_out ? topk_w_out : reinterpret_cast<float*>(base + L.wts);
    int32_t* ub = reinterpret_cast<int32_t*>(base + L.ubuf);
    float* y_slots = reinterpret_cast<float*>(base + L.y_slots);
    float* y_shared = reinterpret_cast<float*>(base + L.y_shared);
    if (R <= moe::kRouteUnionMaxRows) {
        // logits, then selection and union in one block
        if ((st = cuda_status(moe::launch_router_logits(
                 static_cast<const uint16_t*>(x_bf16), w_router, row_valid, R, cfg->hidden,
                 cfg->n_experts, logits, nullptr, 0, nullptr, 0, s))) != MOE_OK)
            return st;
        if ((st = cuda_status(moe::launch_route_union(
                 logits, bias, row_valid, R, cfg->n_experts, cfg->n_groups, cfg->topk_groups,
                 cfg->topk, cfg->routed_scaling, ids, wts, cfg->n_shared, moe::rows_per_item(R), ub,
                 L.un, s))) != MOE_OK)
            return st;
    } else {
        if ((st = route_impl(cfg, x_bf16, w_router, bias, row_valid, R, ids, wts, logits,
                             static_cast<int32_t*>(ws), s)) != MOE_OK)
            return st;
        if ((st = union_impl(cfg, ids, R, ub, s)) != MOE_OK) return st;
    }
    st = w8a16 ? ffn16_impl(cfg, x_bf16, w, ub, R, y_slots, y_shared, ws, s)
               : ffn_impl(cfg, x_bf16, w, ub, R, y_slots, y_shared, ws, s);
    if (st != MOE_OK) return st;
    return combine_impl(cfg, y_slots, y_shared, wts, ub, R, out_bf16, s);
}

moe_status_t moe_layer(const moe_config_t* cfg, const void* x_bf16, const float* w_router,
                       const float* bias, const moe_weights_t* w, const uint8_t* row_valid,
                       int32_t R, void* out_bf16, int32_t* topk_ids_out, float* topk_w_out,
                       void* ws, size_t ws_bytes, moe_stream_t stream) {
    return layer_impl(cfg, x_bf16, w_router, bias, w, row_valid, R, out_bf16, topk_ids_out,
                      topk_w_out, ws, ws_bytes, stream, false);
}

moe_status_t moe_layer_w8a16(const moe_config_t* cfg, const void* x_bf16, const float* w_router,
                             const float* bias, const moe_weights_t* w, const uint8_t* row_valid,
                             int32_t R, void* out_bf16, int32_t* topk_ids_out, float* topk_w_out,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
    return layer_impl(cfg, x_bf16, w_router, bias, w, row_valid, R, out_bf16, topk_ids_out,
                      topk_w_out, ws, ws_bytes, stream, true);
}

moe_status_t moe_greedy_verify(const void* logits, int32_t logits_bf16, int32_t V, int32_t R,
                               const int32_t* draft, const int32_t* n_draft, int32_t* argmax_out,
                               int32_t* accept_len, int32_t* out_tokens, moe_stream_t stream) {
    if (R < 0 || (R % 8) != 0 || V < 1) return MOE_ERR_INVALID_ARG;
    if (R > 65536) return MOE_ERR_UNSUPPORTED;
    if (R == 0) return MOE_OK;
    if (!logits || !draft || !n_draft || !argmax_out || !accept_len || !out_tokens)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(logits, logits_bf16 ? 2 : 4) || !aligned(draft, 4) || !aligned(n_draft, 4) ||
        !aligned(argmax_out, 4) || !aligned(accept_len, 4) || !aligned(out_tokens, 4))
        return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_greedy_verify(logits, logits_bf16 != 0, V, R, draft, n_draft,
                                                 argmax_out, accept_len, out_tokens,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_tile_weights(const uint8_t* src, uint8_t* dst, int64_t n, int32_t rows,
                              int32_t cols, moe_stream_t stream) {
    if (n < 0 || rows <= 0 || cols <= 0 || rows % 128 || cols % 128 || rows > 16384 ||
        cols > 16384)
        return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!src || !dst || !aligned(src, 16) || !aligned(dst, 16)) return MOE_ERR_INVALID_ARG;
    const uintptr_t bytes = uintptr_t(n) * uintptr_t(rows) * uintptr_t(cols);
    const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(dst);
    if (a < b + bytes && b < a + bytes) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_tile_weights(src, dst, n, rows, cols,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_get_device_error(void* ws, int32_t clear, moe_stream_t stream) {
    if (!ws || !aligned(ws, 4)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t err = 0;
    if (cudaMemcpyAsync(&err, ws, sizeof(err), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (clear && err != 0) {
        if (cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (err < 0 || err > MOE_ERR_WORKSPACE) return MOE_ERR_CUDA;
    return static_cast<moe_status_t>(err);
}

moe_status_t moe_diag_wait_timeout(void* ws, uint32_t timeout_us, moe_stream_t stream) {
    if (!ws || !aligned(ws, 4) || timeout_us == 0 || timeout_us > 10000000u) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_wait_timeout(static_cast<int32_t*>(ws),
                                                uint64_t(timeout_us) * 1000ull,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
