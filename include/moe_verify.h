/*
 * moe_verify.h -- C ABI of the fine-grained fp8 MoE layer for decode and
 * speculative verify on one GB300 (sm_103a).
 *
 * The problem, as the source pages state it:
 *   - openinfer #610 "TP8 span row mapping -- single-user speculative decode at
 *     186 tok/s", section "What": an 8-row block holds 1 committed token and up
 *     to 7 speculative drafts; the MoE phases are an expert union, a gate/up
 *     GEMM with SiLU and a down GEMM, with fixed-order reductions; pad rows are
 *     zero-filled so no NaN leaks (section "Gates": the same rows through any
 *     mapping must be bit-identical).
 *   - mstar #388 "Speed up GLM-5.2 with fp8 kernels and one-graph MTP", commit
 *     on kernel switches: the router kernel (NoAuxTcRouter's top-k op), the
 *     fused fp8 MoE decode chain over routed and shared experts, the MoE's
 *     partials reduced once; commit on FlashInfer's block-scale GEMM:
 *     activations quantised to e4m3 per 128 columns.
 *   - MoE-Infinity #140 "converge spec-decode stack", commit list: the sigmoid
 *     router's e_score_correction_bias; expert tensors [gate_proj, up_proj,
 *     down_proj] stored e4m3 with 128x128 FP8 block scales.
 *   - pypto-serving #223 "DSpark speculation (K=7)", "What this adds": the
 *     router gate kept in FP32; idle (pad) rows carry -1 and produce nothing.
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller owns
 *     every buffer and every stream.  The library allocates nothing and never
 *     synchronises the stream except in moe_get_device_error; apart from
 *     moe_layer_noalloc (see its own notes) it holds no state between calls.
 *     Calls are asynchronous on `stream`; the entry points that take their
 *     scratch from the caller can be captured in a CUDA graph.
 *   - Refusals are synchronous: a NULL required pointer, a misaligned pointer
 *     (16 bytes for bf16 / e4m3 / output arrays, 4 bytes for fp32 / int32), an
 *     unsupported shape or a short buffer returns an error code and launches
 *     nothing.  R == 0 returns MOE_OK and launches nothing.  R above
 *     MOE_MAX_ROWS returns MOE_ERR_UNSUPPORTED (no silent truncation).
 *   - A launch failure is read back with cudaGetLastError right after the
 *     launch and returned as MOE_ERR_CUDA, so it never surfaces in a later,
 *     unrelated kernel.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     start while the previous kernel on the stream finishes; it waits for
 *     that kernel's completion before reading its outputs or writing anything
 *     but may fetch read-only weights early.  Stream order is preserved.
 *   - A pad row (row_valid[r] == 0) may hold NaN in x.  It is not routed
 *     (ids -1, weights 0), takes no place in the union, and its output row is
 *     +0.0 in every column.
 *   - For a fixed R the kernel configuration is fixed, and no reduction depends
 *     on which slot of the batch a row occupies: a row's outputs are bit-
 *     identical wherever it sits and whatever its neighbours hold.
 *   - The expert GEMM kernels are persistent (one CTA per SM) and their CTAs
 *     wait on one another: a down tile starts once the gate/up tiles of its
 *     rows have stored their h, and the first tile of every CTA is fixed by
 *     its index.  They expect every SM to be free for them; while kernels of
 *     other streams hold SMs, some of their CTAs start late and the others
 *     wait.  Every such wait is bounded by wait_timeout_us: past it the call
 *     stops and records MOE_ERR_TIMEOUT (read with moe_get_device_error); it
 *     never hangs.
 */
#ifndef MOE_VERIFY_H
#define MOE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL / misaligned pointer, bad shape or ids   */
    MOE_ERR_UNSUPPORTED = 2,   /* shape or row count beyond the compiled limits */
    MOE_ERR_CUDA = 3,          /* a CUDA runtime or launch error                */
    MOE_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out            */
    MOE_ERR_WORKSPACE = 5      /* workspace or buffer smaller than required     */
} moe_status_t;

/* Compiled limits. */
#define MOE_MAX_ROWS 4096      /* rows per call                                   */
#define MOE_W8A16_MAX_ROWS 64  /* rows per call of the w8a16 variant              */
#define MOE_MAX_EXPERTS 256    /* routed experts                                  */
#define MOE_MAX_TOPK 16        /* experts per row                                 */
#define MOE_MAX_GROUPS 32      /* expert groups                                   */
#define MOE_BLOCK 128          /* quantisation block: 1x128 activations, 128x128 weights */

/*
 * Layer shape.  hidden (H) and inter (I) are multiples of 128 (128..16384);
 * n_experts (E) <= 256 is a multiple of n_groups (G <= 32); topk_groups (TG)
 * <= G; topk (K) <= min(16, TG*E/G); n_shared (S) is 0 or 1; routed_scaling
 * multiplies the normalised routing weights (2.5 for GLM-5.2-class layers).
 * wait_timeout_us bounds every device-side wait (0 = 2 000 000 us).
 */
typedef struct {
    int32_t hidden;
    int32_t inter;
    int32_t n_experts;
    int32_t n_groups;
    int32_t topk_groups;
    int32_t topk;
    int32_t n_shared;
    float routed_scaling;
    uint32_t wait_timeout_us;
} moe_config_t;

/*
 * Expert weights: e4m3 (OCP e4m3fn) codes, output-major (K contiguous), with
 * one fp32 scale per 128x128 block; the dequantised weight is code * scale.
 *   w_gate, w_up : uint8 [E, I, H]      s_gate, s_up : fp32 [E, I/128, H/128]
 *   w_down       : uint8 [E, H, I]      s_down       : fp32 [E, H/128, I/128]
 *   sh_*         : the shared expert, same layouts with S in place of E
 *                  (ignored when n_shared == 0).
 * Device memory, read only; 16-byte aligned codes, 4-byte aligned scales.
 *
 * layout says how the codes of each [rows, cols] matrix lie in memory (the
 * scales are always as above):
 *   MOE_LAYOUT_ROW_MAJOR (0): row-major, cols contiguous, as listed above;
 *   MOE_LAYOUT_TILED (1): the 128x128 blocks that the scales cover, each
 *     stored as 16 KB of its own (its 128 rows of 128 codes one after the
 *     other), blocks in row-block-major order: block (rb, kb) of matrix n at
 *     byte ((n * rows/128 + rb) * cols/128 + kb) * 16384.  The expert GEMMs
 *     stream every block once, along K, so this layout turns each of their
 *     weight streams into sequential 16 KB reads.  moe_tile_weights converts.
 * A zero-initialised layout field selects the row-major layout.
 */
#define MOE_LAYOUT_ROW_MAJOR 0
#define MOE_LAYOUT_TILED 1

typedef struct {
    const uint8_t* w_gate;
    const uint8_t* w_up;
    const uint8_t* w_down;
    const float* s_gate;
    const float* s_up;
    const float* s_down;
    const uint8_t* sh_gate;
    const uint8_t* sh_up;
    const uint8_t* sh_down;
    const float* sh_s_gate;
    const float* sh_s_up;
    const float* sh_s_down;
    int32_t layout;   /* MOE_LAYOUT_ROW_MAJOR or MOE_LAYOUT_TILED (all six code tensors) */
} moe_weights_t;

/*
 * moe_route -- router logits, sigmoid scores with correction bias, grouped
 * top-k and weight normalisation (mstar #388, NoAuxTcRouter; MoE-Infinity
 * #140, e_score_correction_bias; pypto-serving #223, router gate in FP32).
 *
 *   x_bf16    bf16 [R, H] row-major          w_router fp32 [E, H] (16-byte aligned)
 *   bias      fp32 [E]                        row_valid uint8 [R] or NULL (all valid)
 *   topk_ids  int32 [R, K]  (out)             topk_w   fp32 [R, K] (out)
 *   logits    fp32 [R, E]   (out, required: also the scratch between the
 *                            logits and the selection kernels)
 *
 * Definition (all IEEE fp32, fixed order, so a CPU restatement reproduces the
 * ids bit for bit):
 *   logit[r,e] = sum_h x[r,h] * w_router[e,h] reduced as follows: h is cut
 *     into chunks of 1024 (the last may be shorter); inside chunk c, lane
 *     l = 0..31 owns h = c*1024 + 128*i + 4*l + j (i ascending, j = 0..3) and
 *     forms p = fma(x, w, p) from p = 0; per lane q = p(chunk 0), then
 *     q = q + p(chunk c) for c = 1, 2, ...; the 32 lane values are combined by
 *     the butterfly v[l] = v[l] + v[l ^ d], d = 16, 8, 4, 2, 1.
 *   s = 1 / (1 + exp(-logit)) with exp evaluated by Cody-Waite reduction
 *     (ln2 split into a 16-significant-bit head and an fp32 tail) and the
 *     degree-7 Taylor series in Horner form, argument clamped to [-87, 87];
 *   b = s + bias[e];
 *   group score = the sum of the two largest b of the group (the largest
 *     alone for single-expert groups); the TG best groups are kept, ties to
 *     the lower group id;
 *   the K best experts of the kept groups by b, ties to the lower expert id,
 *     listed by b descending;
 *   w_k = (s_k / (s_0 + ... + s_{K-1})) * routed_scaling, the sum in k order.
 *   Pad rows: ids -1, weights 0, logits untouched.
 * Above 64 rows the logits kernel streams x and w_router through shared
 * memory by TMA and waits on its own copies with bounded waits
 * (wait_timeout_us); should one run out (the copies never landing), the
 * kernel leaves the logits of its unfinished tiles unwritten.  moe_route has
 * no error word to record that in; moe_layer records MOE_ERR_TIMEOUT in its
 * workspace's.
 */
moe_status_t moe_route(const moe_config_t* cfg, const void* x_bf16, const float* w_router,
                       const float* bias, const uint8_t* row_valid, int32_t R,
                       int32_t* topk_ids, float* topk_w, float* logits, moe_stream_t stream);

/*
 * moe_build_union -- the deduplicated expert union of the batch and its
 * dispatch order (openinfer #610, "What": the union phase; MoE-Infinity #140:
 * the per-token union of the verify block's routed experts).
 *
 *   topk_ids   int32 [R, K]: per valid row K distinct ids in [0, E); a pad row
 *              holds -1 in every slot.  A row breaking this is treated as a pad
 *              row and union_buf[5] is set to MOE_ERR_INVALID_ARG.
 *   union_buf  int32, at least moe_union_bytes(cfg, R) bytes (out).
 *
 * union_buf layout (int32 words; KS = K + S slots per row):
 *   [0] U  number of distinct routed experts hit    [1] R_v valid rows
 *   [2] T  gathered slots = R_v * KS                [3] GEMM work items
 *   [4] rows per work item                          [5] error code (0 = OK)
 *   [6] R, the row count it was built for           [7] shape word (E << 8) | (K << 1) | S
 *   counts  [E+1]   at word 8: slots per expert; counts[E] = R_v * S
 *   offsets [E+2]   exclusive prefix of counts (experts ascending, shared last)
 *   ulist   [E+1]   the U experts hit, ascending, then E (the shared entry)
 *   pos     [R*KS]  gathered position of slot (r, k); k = K is the shared
 *                   slot; -1 for pad rows
 *   src     [R*KS]  r*KS + k of gathered position p (p < T)
 *   items   [.. *4] work items (entry, first gathered row, row count, 0)
 * Inside an expert, slots are placed in (row, k) order; shared rows in row
 * order.  Word offsets of each array follow from E, K, S and R as listed.
 *
 * Every call that reads a union (moe_dispatch, the expert GEMM calls,
 * moe_expert_ffn_fp8 / _w8a16, moe_combine, moe_combine_add_rmsnorm) first
 * compares words [6] and [7] with its own R and shape.  A union built for
 * another call is not indexed: the call computes nothing and records
 * MOE_ERR_INVALID_ARG -- in the workspace error word (read it with
 * moe_get_device_error) for the calls that take a workspace, in the union's
 * own word [5] for the two combine calls (the only union word they write).
 */
size_t moe_union_bytes(const moe_config_t* cfg, int32_t max_rows);
moe_status_t moe_build_union(const moe_config_t* cfg, const int32_t* topk_ids, int32_t R,
                             int32_t* union_buf, size_t union_bytes, moe_stream_t stream);

/*
 * moe_expert_ffn_fp8 -- dispatch and the expert FFNs of the union
 * (openinfer #610, "What": union / GEMM / SiLU phases; mstar #388: fused fp8
 * MoE over routed and shared experts; FlashInfer commit: activations to e4m3
 * per 128 columns).  For every gathered slot (row r, expert e):
 *   x is quantised per row and 128 columns: scale = amax/448 (1 for an
 *     all-zero block), code = e4m3_rn_satfinite(x / scale) (fp32 divide);
 *   g = x^.Wg^T, u = x^.Wu^T with fp32 accumulation; h = silu(g) * u;
 *   h is quantised per 128 columns by the same rule;
 *   o = h^.Wd^T with fp32 accumulation.
 * Every GEMM runs on tcgen05 fp8 tensor cores with the 128x128 block scales
 * applied to each 128-wide K-block partial (fp32 scales are not expressible
 * in the MMA's own block-scale format).
 *
 *   x_bf16    bf16 [R, H]                     union_buf from moe_build_union
 *   y_slots   fp32 [R*K, H] (out): o of slot (r, k) at row r*K + k
 *   y_shared  fp32 [R, H]   (out): the shared expert's o (NULL if S == 0)
 *   ws        device scratch of at least moe_ffn_workspace_bytes(cfg, R) bytes,
 *             256-byte aligned; its first 256 bytes hold the device error word,
 *             which the caller zeroes once before first use (errors stay
 *             recorded until moe_get_device_error clears them).
 * Rows of y_* that belong to pad rows are left untouched.
 */
size_t moe_ffn_workspace_bytes(const moe_config_t* cfg, int32_t max_rows);
moe_status_t moe_expert_ffn_fp8(const moe_config_t* cfg, const void* x_bf16,
                                const moe_weights_t* w, const int32_t* union_buf, int32_t R,
                                float* y_slots, float* y_shared, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/*
 * moe_expert_ffn_w8a16 -- the expert FFNs of the union with 16-bit activations
 * (mstar #388, commit on kernel switches and the FlashInfer commit: fp8 linears
 * run w8a16 at decode sizes, fp8 weights with bf16 activations).  Per gathered
 * slot (row r, expert e), with no activation quantisation:
 *   every weight is dequantised to bf16: bf16_rne(e4m3(q) * s_block) (the
 *     product in fp32);
 *   g = x.Wg^T, u = x.Wu^T with x bf16 and fp32 accumulation over all of K;
 *   h = silu(g) * u rounded to bf16;  o = h.Wd^T with fp32 accumulation.
 * The GEMMs run on tcgen05 bf16 tensor cores (kind::f16); the dequantisation
 * happens in shared memory, inside the GEMM kernel.
 * Arguments, outputs and workspace as moe_expert_ffn_fp8 (the union built for
 * the same R).  R <= MOE_W8A16_MAX_ROWS, else MOE_ERR_UNSUPPORTED.
 */
moe_status_t moe_expert_ffn_w8a16(const moe_config_t* cfg, const void* x_bf16,
                                  const moe_weights_t* w, const int32_t* union_buf, int32_t R,
                                  float* y_slots, float* y_shared, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/*
 * The steps of moe_expert_ffn_fp8, callable one by one (same arguments, same
 * workspace).  moe_expert_ffn_fp8 (and moe_layer) is moe_dispatch followed by
 * moe_expert_gemms_fp8 for R <= 64 and by moe_gate_up_fp8 + moe_down_fp8 above
 * (measured faster there); moe_gate_up_fp8 followed by moe_down_fp8 computes
 * the same values as moe_expert_gemms_fp8 in two launches.
 *   moe_dispatch          quantise each valid row per 1x128 and write it to its
 *                         K+S gathered positions (workspace); clears the fused
 *                         GEMM's per-item counters;
 *   moe_expert_gemms_fp8  gate/up GEMMs + SiLU*mul + h quantisation and the down
 *                         GEMM in one persistent launch (a down tile starts once
 *                         every gate/up tile of its rows has stored its h);
 *   moe_gate_up_fp8       g and u GEMMs, h = silu(g) * u, h quantised per 1x128
 *                         (workspace);
 *   moe_down_fp8          the down GEMM, fp32 rows to y_slots / y_shared.
 * Order: each GEMM call must come after moe_dispatch of the same call on the
 * same stream, with no other launch of this library in between except
 * moe_gate_up_fp8 before moe_down_fp8 (kernels start while their predecessor
 * finishes, see the launch note below).
 */
moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x_bf16, const int32_t* union_buf,
                          int32_t R, void* ws, size_t ws_bytes, moe_stream_t stream);
moe_status_t moe_gate_up_fp8(const moe_config_t* cfg, const moe_weights_t* w,
                             const int32_t* union_buf, int32_t R, void* ws, size_t ws_bytes,
                             moe_stream_t stream);
moe_status_t moe_down_fp8(const moe_config_t* cfg, const moe_weights_t* w,
                          const int32_t* union_buf, int32_t R, float* y_slots, float* y_shared,
                          void* ws, size_t ws_bytes, moe_stream_t stream);
moe_status_t moe_expert_gemms_fp8(const moe_config_t* cfg, const moe_weights_t* w,
                                  const int32_t* union_buf, int32_t R, float* y_slots,
                                  float* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_combine -- fixed-order weighted combine plus the shared expert, pads
 * zero-filled (openinfer #610, "What"/"Gates": same fixed-order reductions,
 * pad rows zero-filled with no NaN leak; mstar #388: the MoE's partials
 * reduced once):
 *   acc = w_0 * o_0; acc = fma(w_k, o_k, acc) for k = 1..K-1;
 *   acc = acc + o_shared (weight 1); out = bf16_rne(acc); pad rows: +0.0.
 *   topk_w fp32 [R, K]; out_bf16 bf16 [R, H] (out).
 */
moe_status_t moe_combine(const moe_config_t* cfg, const float* y_slots, const float* y_shared,
                         const float* topk_w, const int32_t* union_buf, int32_t R,
                         void* out_bf16, moe_stream_t stream);

/*
 * moe_combine_add_rmsnorm -- moe_combine fused with the next layer's residual
 * add and RMSNorm (mstar #388, commit on kernel switches: the MoE's partials
 * reduced once, fused with the next add + RMSNorm).  Per valid row:
 *   acc = the combine sum of moe_combine, before its rounding;
 *   z = residual + acc;   residual_out = bf16_rne(z);
 *   normed = bf16_rne(z * rsqrt(sum_h(z^2) / H + eps) * gamma)
 * (sum of squares reduced in a fixed order; pad rows: +0.0 in both outputs).
 *   residual_bf16 bf16 [R, H]; gamma fp32 [H]; eps >= 0;
 *   residual_out_bf16, normed_bf16 bf16 [R, H] (out).  All 16-byte aligned.
 */
moe_status_t moe_combine_add_rmsnorm(const moe_config_t* cfg, const float* y_slots,
                                     const float* y_shared, const float* topk_w,
                                     const int32_t* union_buf, int32_t R, const void* residual_bf16,
                                     const float* gamma, float eps, void* residual_out_bf16,
                                     void* normed_bf16, moe_stream_t stream);

/*
 * moe_layer -- the whole layer: moe_route, moe_build_union,
 * moe_expert_ffn_fp8 and moe_combine on one stream, intermediates in `ws`.
 * Arguments follow the problem statement of openinfer #610 ("What"): R rows
 * (1 committed + up to 7 drafts per request, 8-row blocks, pads marked in
 * row_valid).
 *   out_bf16      bf16 [R, H] (out)
 *   topk_ids_out  int32 [R, K] or NULL;  topk_w_out fp32 [R, K] or NULL
 *   ws            at least moe_workspace_bytes(cfg, R) bytes, 256-byte aligned.
 */
size_t moe_workspace_bytes(const moe_config_t* cfg, int32_t max_rows);

/*
 * moe_workspace_size -- the same size as a status-returning query: *bytes is
 * set to moe_workspace_bytes(cfg, max_rows), which also covers the union
 * buffer (moe_union_bytes) and the FFN workspace (moe_ffn_workspace_bytes) of
 * a call of up to max_rows rows, so one buffer of this size serves any entry
 * point.  MOE_ERR_INVALID_ARG for a NULL pointer, a malformed shape or
 * max_rows < 0; MOE_ERR_UNSUPPORTED beyond the compiled limits (*bytes = 0).
 */
moe_status_t moe_workspace_size(const moe_config_t* cfg, int32_t max_rows, size_t* bytes);

moe_status_t moe_layer(const moe_config_t* cfg, const void* x_bf16, const float* w_router,
                       const float* bias, const moe_weights_t* w, const uint8_t* row_valid,
                       int32_t R, void* out_bf16, int32_t* topk_ids_out, float* topk_w_out,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_layer_w8a16 -- moe_layer with the expert FFNs of moe_expert_ffn_w8a16
 * (routing, union and combine unchanged).  Same arguments and workspace size;
 * R <= MOE_W8A16_MAX_ROWS, else MOE_ERR_UNSUPPORTED.
 */
moe_status_t moe_layer_w8a16(const moe_config_t* cfg, const void* x_bf16, const float* w_router,
                             const float* bias, const moe_weights_t* w, const uint8_t* row_valid,
                             int32_t R, void* out_bf16, int32_t* topk_ids_out, float* topk_w_out,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_layer_noalloc -- moe_layer without a caller-provided workspace.  The
 * source pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate device memory: a plugin whose host framework owns every
 * device allocation and hands out no scratch, code on a path that must not call
 * cudaMalloc, or a caller that cannot size a workspace ahead of the call.
 *
 * The layer's scratch is one array of 32 MiB (33 554 432 bytes) compiled into
 * this library; every GPU that loads the library holds it until the process
 * exits.  A call whose moe_workspace_bytes(cfg, R) exceeds it is refused with
 * MOE_ERR_UNSUPPORTED (at the GLM-5.2 shape -- H 6144, I 2048, E 256, K 8,
 * one shared expert -- up to 109 rows fit, e.g. a 64-row batched verify).  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library call.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress) and caches it per device and CUDA
 * context; make that first call outside any stream capture.  A call made in
 * another context than the cached one (a context of the caller's own, or the
 * primary context created again after cudaDeviceReset) looks the address up
 * again, so make the first call after such a change outside capture too.  Every call shares the one array and leaves its
 * contents behind; the call clears the error word at its head itself.  Calls
 * that overlap on the GPU (concurrent streams, or several host threads) race on
 * the array and corrupt each other: serialise them.
 *
 * Arguments as moe_layer, without ws / ws_bytes, plus:
 *   device_status  int32 device word or NULL: receives the layer's device error
 *                  code (MOE_OK, MOE_ERR_TIMEOUT, ...) in stream order.
 */
moe_status_t moe_layer_noalloc(const moe_config_t* cfg, const void* x_bf16,
                               const float* w_router, const float* bias, const moe_weights_t* w,
                               const uint8_t* row_valid, int32_t R, void* out_bf16,
                               int32_t* topk_ids_out, float* topk_w_out, int32_t* device_status,
                               moe_stream_t stream);

/*
 * moe_tile_weights -- copy n row-major e4m3 matrices [rows, cols] into the
 * MOE_LAYOUT_TILED layout (see moe_weights_t): a pure permutation of bytes,
 * done once when the weights are loaded.  For a set of expert weights call it
 * once per code tensor: w_gate and w_up with (E, I, H), w_down with (E, H, I),
 * and the shared expert's with S in place of E.  The layout is this library's
 * (for its HBM streams); the block-scaled e4m3 format itself is unchanged.
 *
 *   src  uint8 [n, rows, cols] device, 16-byte aligned (read only)
 *   dst  uint8, n*rows*cols bytes, device, 16-byte aligned, not overlapping src
 *   rows, cols  multiples of 128 (1 .. 16384 / 128 blocks each); n >= 0
 *
 * Asynchronous on stream.  MOE_ERR_INVALID_ARG: NULL or misaligned pointer,
 * overlap, n < 0, rows or cols not a positive multiple of 128 or above 16384.
 */
moe_status_t moe_tile_weights(const uint8_t* src, uint8_t* dst, int64_t n, int32_t rows,
                              int32_t cols, moe_stream_t stream);

/*
 * moe_greedy_verify -- greedy verify and acceptance of speculative spans on
 * the device (openinfer #610 "What": spans of 8 rows, 1 committed token + up to
 * 7 drafts; pypto-serving #223 "What this adds": accept the longest matching
 * prefix plus the bonus prediction, 1..8 tokens per step; mstar #388: the
 * verify runs on the device inside the step).
 *   logits       fp32 (logits_bf16 == 0) or bf16 [R, V]: the target model's
 *                logits at every row of every span
 *   R            rows, a multiple of 8 (span q = rows 8q .. 8q+7), <= 65536
 *   draft        int32 [R]: draft[8q + j] is span q's draft j (1 <= j <= 7);
 *                row 0's entry of a span is not read
 *   n_draft      int32 [R/8]: drafts present in span q (clamped to 0..7)
 *   argmax_out   int32 [R] (out): the target's greedy token of every row --
 *                the largest logit, the lowest index on ties, NaN never chosen
 *                (a row of NaN gives 0)
 *   accept_len   int32 [R/8] (out): 1 + the number of accepted drafts
 *   out_tokens   int32 [R] (out): per span the accepted drafts, then the bonus
 *                token, then -1 in the remaining slots
 * Draft j is accepted when every draft before it was and it equals the greedy
 * token of row j-1; the bonus is the greedy token of the row after the last
 * accepted draft.  V >= 1; pointers 4-byte aligned (logits 16-byte aligned
 * rows are read with vector loads when V * element size is a multiple of 16).
 */
moe_status_t moe_greedy_verify(const void* logits, int32_t logits_bf16, int32_t V, int32_t R,
                               const int32_t* draft, const int32_t* n_draft, int32_t* argmax_out,
                               int32_t* accept_len, int32_t* out_tokens, moe_stream_t stream);

/*
 * moe_get_device_error -- synchronises `stream`, then reads (and clears when
 * `clear` != 0) the device error word at the start of a workspace given to
 * moe_expert_ffn_fp8 or moe_layer.  Returns MOE_OK, MOE_ERR_TIMEOUT (a bounded
 * wait ran out: the kernel stopped, released its tensor memory and returned)
 * or MOE_ERR_CUDA.
 */
moe_status_t moe_get_device_error(void* ws, int32_t clear, moe_stream_t stream);

/*
 * moe_diag_wait_timeout -- diagnostic: launches one block that waits, with the
 * library's bounded wait, on a barrier nothing ever arrives on, for at most
 * timeout_us microseconds; it then records MOE_ERR_TIMEOUT in the error word
 * of `ws` (>= 256 bytes) and returns.  Exercises the timeout path without any
 * fault.
 */
moe_status_t moe_diag_wait_timeout(void* ws, uint32_t timeout_us, moe_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_VERIFY_H */
