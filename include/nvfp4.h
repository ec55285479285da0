/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 block-scaled MoE expert path.
 *
 * NVFP4 tensors: 4-bit E2M1 codes, two per byte (element 2j in the low nibble),
 * one unsigned E4M3 scale per 16 consecutive elements along K, and one FP32
 * global multiplier.  A value decodes as e2m1(code) * e4m3(scale) * global
 * (nvfp4-megamoe-kernel commit log, page 2 = commit efe63ca, single_shot_inference.py:
 * the weight_scale_2 fix, i.e. the NVFP4 dequantisation formula).  Activations carry
 * gs = amax / (6 * 448) as their global multiplier (page 3 = commit 4c6464e, vllm: the
 * activation global-scale passage); weights carry ws2 = weight_scale_2 and nothing else
 * (page 2: the input_scale passage, which keeps the checkpoint input_scale out of the
 * weight side).  A GEMM therefore computes
 * y = (gs * ws2) * sum_k e2m1(a) e4m3(sa) e2m1(b) e4m3(sb)
 * (page 1: the scale-semantics passage, y = (x * scale_a * gsa) @ (w * scale_b * gsb)).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated otherwise;
 *    the library keeps no reference after the call returns and never
 *    allocates device memory.  Calls that need scratch take a caller-owned
 *    workspace (ws, ws_bytes, 256-byte aligned) whose size the matching
 *    *_workspace_bytes query returns; its contents need no initialisation.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously; no call synchronises the host
 *    except nvfp4_get_device_error.  Kernels use programmatic dependent launch:
 *    a kernel may start while the previous kernel on the stream finishes, and
 *    reads its inputs only after that kernel completed.  The one exception is
 *    that the GEMMs of nvfp4_linear and of the MoE stages read the weights and
 *    the routing arrays one launch early (the one-token MoE forward also the
 *    token x and its top-k ids and weights).  Those must therefore be final
 *    before the call that opens the chain (nvfp4_linear, nvfp4_moe_forward or
 *    nvfp4_moe_dispatch) is enqueued, which ordinary stream order gives.
 *  - bf16 tensors are passed as void* to raw bf16 storage (row-major).
 *  - Scale-factor buffers in the "swizzled" tensor-core layout hold
 *    nvfp4_sf_bytes(rows, K) bytes: rows padded to a multiple of 128 and scale
 *    columns (K/16) to a multiple of 4, grouped into 512-byte blocks of
 *    128 rows x 4 columns stored row-group-major; the four scales of row r sit
 *    at byte 16*(r%32) + 4*((r%128)/32) of their block (page 3: the grouped-GEMM
 *    launch contract, A-side scales padded and swizzled).
 *  - Errors: argument problems are detected on the host and returned before
 *    anything is enqueued; nothing throws across the ABI.  A detail string for
 *    the last failing call on the calling thread is available from
 *    nvfp4_last_error_string().  Faults detected on the device (an expert id
 *    out of range, a pipeline wait that timed out) set a per-device flag word
 *    that nvfp4_get_device_error reads.
 *  - Shape rules: K % 64 == 0; GEMM output widths N % 16 == 0 for the dense
 *    linear and GEMM, N % 128 == 0 for the grouped linear and the MoE; all
 *    pointers 16-byte aligned; bf16 row strides a multiple of 8 elements.  Violations
 *    return NVFP4_ERR_UNSUPPORTED_SHAPE or NVFP4_ERR_MISALIGNED.
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_ABI_VERSION 6

/* Exported symbols: the library builds with hidden visibility by default. */
#if defined(NVFP4_BUILD) && defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad enum value     */
  NVFP4_ERR_UNSUPPORTED_SHAPE = 2,   /* K % 64, N % 16 / 128, E or topk out of range    */
  NVFP4_ERR_MISALIGNED = 3,          /* a pointer not 16-byte aligned, bad row stride   */
  NVFP4_ERR_WORKSPACE = 4,           /* ws_bytes below the size the query returns       */
  NVFP4_ERR_CUDA = 5,                /* a CUDA runtime call or launch failed            */
  NVFP4_ERR_DEVICE_FAULT = 6,        /* nvfp4_get_device_error: bad data seen on device */
  NVFP4_ERR_TIMEOUT = 7,             /* nvfp4_get_device_error: a bounded wait ran out  */
  NVFP4_ERR_UNSUPPORTED_DEVICE = 8   /* the current device is not sm_103                */
} nvfp4_status;

/* global-scale modes */
#define NVFP4_GS_DYNAMIC 0  /* compute gs = fl32(amax / 2688) over the whole input, write *gs */
#define NVFP4_GS_STATIC 1   /* read gs from *gs (warm-up calibrated value, page 3)          */

/* scale-factor output layouts of nvfp4_quantize_act */
#define NVFP4_SF_SWIZZLED 0 /* tensor-core layout described above                         */
#define NVFP4_SF_LINEAR 1   /* row-major (M, K/16), the checkpoint layout                 */

/* nvfp4_prepare_weights flags */
#define NVFP4_PREP_PLAIN 0
#define NVFP4_PREP_W13_INTERLEAVE 1 /* rows [0,N/2) gate, [N/2,N) up -> 64 gate + 64 up per 128 */

/* device fault flags returned by nvfp4_get_device_error */
#define NVFP4_DEVERR_BAD_EXPERT_ID 1  /* a top-k id outside [0, E); the entry was dropped  */
#define NVFP4_DEVERR_PIPELINE_TIMEOUT 2 /* a GEMM pipeline wait exceeded its limit        */
#define NVFP4_DEVERR_INTERNAL 4         /* a kernel invariant failed (a library bug)      */

NVFP4_API int nvfp4_abi_version(void);
NVFP4_API const char *nvfp4_status_string(nvfp4_status s);
/* Detail of the last non-OK status returned on the calling thread ("" if none). */
NVFP4_API const char *nvfp4_last_error_string(void);

/* Synchronises `stream`, ORs the device fault flags of the current device into
 * *flags and clears them.  Returns NVFP4_ERR_TIMEOUT if the timeout flag is
 * set, NVFP4_ERR_DEVICE_FAULT for any other flag, NVFP4_OK when clear. */
NVFP4_API nvfp4_status nvfp4_get_device_error(void *stream, int32_t *flags);

/* Bytes of a swizzled scale buffer for `rows` rows of K elements. */
NVFP4_API size_t nvfp4_sf_bytes(int64_t rows, int64_t K);

/* ---------------------------------------------------------------- (a) quantize
 * BF16 (M, K) with row stride ldx (elements) -> NVFP4 codes q (M, K/2) and
 * E4M3 block scales sf (swizzled: nvfp4_sf_bytes(M, K) bytes, padding written
 * as 0; linear: M*K/16 bytes).  Per 16-element block b with amax_b = max|x|:
 *   s = fl32(amax_b / fl32(6*gs)), sf = E4M3_rne_satfinite(s),
 *   d = fl32(e4m3(sf) * gs), q_i = E2M1_rne_satfinite(fl32(x_i * fl32(1/d)))
 * with the sign of x_i kept on zero codes, and all codes 0 when d == 0 or 1/d
 * overflows.  gs_mode NVFP4_GS_DYNAMIC computes gs = fl32(amax / 2688) over
 * all M*K elements (two launches: block-max partials, then quantize) and
 * stores it to *gs; NVFP4_GS_STATIC reads *gs.  Workspace: amax partials.
 * With M == 0 only gs is used (dynamic mode writes 0); x, q and sf may be NULL. */
NVFP4_API size_t nvfp4_quantize_workspace_bytes(int64_t M, int64_t K);
NVFP4_API nvfp4_status nvfp4_quantize_act(const void *x, int64_t M, int64_t K, int64_t ldx, int gs_mode,
                                float *gs, uint8_t *q, uint8_t *sf, int sf_layout, void *ws,
                                size_t ws_bytes, void *stream);

/* -------------------------------------------------- RMSNorm -> quantize
 * RMSNorm feeding the activation quantiser (the fused "P4" path of page 1 = commit
 * 1121cd7, single_shot_inference.py: the fused-RMSNorm A/B passage, whose harness compares
 * x_normed, the global scale, the FP4 data and the GEMM outputs of the fused and unfused
 * paths).  Per row r:
 *   inv_r = 1 / sqrt(fl32(sum_k x^2) / K + eps)        (correctly rounded sqrt, divide)
 *   x_normed[r,k] = bf16(fl32(fl32(x[r,k] * inv_r) * gamma[k]))
 * gamma is a bf16 vector of K.  nvfp4_rmsnorm writes x_normed (M, K) bf16 (the unfused
 * path; quantise it with nvfp4_quantize_act).  nvfp4_rmsnorm_quantize quantises x_normed
 * without a round trip through memory, with the same arguments and results as
 * nvfp4_quantize_act applied to nvfp4_rmsnorm's output (codes, scales and dynamic gs
 * bit-identical); x_normed, if not NULL, also receives the normalised rows.  Two launches.
 * Workspace: amax partials and the per-row inv_r. */
NVFP4_API size_t nvfp4_rmsnorm_quantize_workspace_bytes(int64_t M, int64_t K);
NVFP4_API nvfp4_status nvfp4_rmsnorm(const void *x, int64_t M, int64_t K, int64_t ldx, const void *gamma,
                                     float eps, void *y, void *stream);
NVFP4_API nvfp4_status nvfp4_rmsnorm_quantize(const void *x, int64_t M, int64_t K, int64_t ldx,
                                              const void *gamma, float eps, int gs_mode, float *gs,
                                              uint8_t *q, uint8_t *sf, int sf_layout, void *x_normed,
                                              void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------ weight prepare
 * Checkpoint-layout weights of G groups (experts): codes w (G, N, K/2) and
 * row-major E4M3 scales sf (G, N, K/16) used as stored, no transpose (page 2: the
 * checkpoint-layout fix, N-major codes and untransposed scales).  Writes w_out
 * (nvfp4_prepared_weight_bytes(G, N, K) bytes) and sf_out (G blocks of
 * nvfp4_sf_bytes(N, K)).  The prepared codes are tile-major: for group g, 128-row tile t
 * and 128-byte column slab s of the K/2 code bytes, block ((g * N/128 + t) * S + s),
 * S = ceil(K/256), holds the tile's 128 rows x 128 bytes contiguously (row r at byte
 * 128 r of the 16 KiB block); slab bytes past K/2 are zero codes.  A GEMM stage reads one
 * such block.  NVFP4_PREP_W13_INTERLEAVE reorders the rows of a fused gate/up projection so
 * that every 128-row tile holds 64 gate rows followed by the 64 matching up rows.
 * K % 64 == 0, N % 128 == 0; with G == 1 and no interleave N % 16 == 0 suffices, the
 * last tile's rows from N on then being zero codes and zero scales (sf_out holds
 * nvfp4_sf_bytes(N, K) bytes, which covers them).  Run once at load time; w and w_out
 * must not overlap.
 * Every w / w13 / w2 / sh_* weight argument below is such a prepared buffer. */
NVFP4_API size_t nvfp4_prepared_weight_bytes(int64_t G, int64_t N, int64_t K);
NVFP4_API nvfp4_status nvfp4_prepare_weights(const uint8_t *w, const uint8_t *sf, int64_t G, int64_t N,
                                   int64_t K, int flags, uint8_t *w_out, uint8_t *sf_out,
                                   void *stream);

/* ------------------------------------------------------------ (e) dense linear
 * y (M, N) bf16 = alpha * deq(xq) @ deq(W)^T with alpha = gs * ws2, where xq is
 * x (M, K) bf16 quantised at run time (gs_mode as for nvfp4_quantize_act,
 * *gs written in dynamic mode) and W is a prepared (N, K/2) + swizzled sf
 * weight with device scalar ws2 (Nvfp4Linear, page 2: the ws2-folding fixes).
 * K % 64 == 0, N % 16 == 0 (an N that is not a multiple of 128 ends in a partial tile of
 * the prepared weight; only the first N output columns are written).  Workspace:
 * quantised x + scales + partials. */
NVFP4_API size_t nvfp4_linear_workspace_bytes(int64_t M, int64_t K);
NVFP4_API nvfp4_status nvfp4_linear(const void *x, int64_t M, int64_t K, int64_t N, const uint8_t *w,
                          const uint8_t *w_sf, const float *ws2, int gs_mode, float *gs, void *y,
                          void *ws, size_t ws_bytes, void *stream);

/* Dense linear that allocates nothing and takes no workspace.  (No counterpart
 * on the pages: this entry point exists for callers, not for the method.)
 *
 * Some callers cannot allocate device memory at the point where they run the
 * linear.  Examples are a plugin inside a host inference engine that owns all
 * device memory and forbids allocation while it enqueues work, or a serving
 * loop that reserved a fixed memory budget at start-up and must not touch an
 * allocator per request.  Such a caller may also have no workspace to lend.
 *
 * This variant computes exactly what nvfp4_linear computes, with the same
 * arguments minus (ws, ws_bytes).  Its scratch (the quantised activations, their
 * scales and the amax partials) lives in one file-scope device array of
 * NVFP4_LINEAR_NOALLOC_MAX_BYTES bytes.  Every GPU that loads the library
 * holds that array until the process exits.
 *  - Limit: nvfp4_linear_workspace_bytes(M, K) must not exceed the array size.
 *    For K = 7168 that is M <= 1025; for K = 1536 it is M <= 4848.  Larger
 *    calls return NVFP4_ERR_WORKSPACE before anything is enqueued.
 *  - Set-up: the first call on each device resolves the array's device
 *    address, with that device current.  Make that first call before any
 *    stream capture begins.
 *  - Sharing: all calls on a device use the same array.  It keeps the contents
 *    of the last call, and nothing in it needs to start at zero, because every
 *    byte the GEMM reads is rewritten by the call's own quantise step.  Calls
 *    that overlap on the GPU (different streams without ordering between
 *    them) race on the array and give wrong results: serialise them.
 *  - It calls no cudaMalloc, cudaFree or allocating library routine. */
#define NVFP4_LINEAR_NOALLOC_MAX_BYTES (4u << 20)
NVFP4_API nvfp4_status nvfp4_linear_noalloc(const void *x, int64_t M, int64_t K, int64_t N,
                                            const uint8_t *w, const uint8_t *w_sf,
                                            const float *ws2, int gs_mode, float *gs, void *y,
                                            void *stream);

/* GEMM alone on already-quantised activations: xq (M, K/2) codes with
 * swizzled scales xsf (nvfp4_sf_bytes(M, K)) and device scalar gs; W and ws2
 * as for nvfp4_linear.  y (M, N) bf16. */
NVFP4_API nvfp4_status nvfp4_gemm(const uint8_t *xq, const uint8_t *xsf, const float *gs, int64_t M,
                        int64_t K, int64_t N, const uint8_t *w, const uint8_t *w_sf,
                        const float *ws2, void *y, void *stream);

/* ----------------------------------------------------- fixed-group linear
 * The input features of x (M, G*K) bf16 split into G equal groups of K; group g
 * multiplies its K columns by its own NVFP4 weight W_g (N, K/2) with ws2[g]:
 *   y[:, g*N:(g+1)*N] = (gs * ws2[g]) * deq(xq[:, g*K:(g+1)*K]) @ deq(W_g)^T
 * with one activation gs over all of x (gs_mode as for nvfp4_quantize_act).
 * This is the grouped o-projection of page 3 (the wo_a o-projection passage: a per-group
 * BMM with in_features 4096; the ScaledGroupedGemm passage: an NVFP4 grouped linear with
 * n_local_groups = 8).  w is
 * (G, N, K/2) prepared with NVFP4_PREP_PLAIN and w_sf G blocks of
 * nvfp4_sf_bytes(N, K); ws2 (G) fp32; y (M, G*N) bf16.  K % 64 == 0, N % 128 == 0. */
NVFP4_API size_t nvfp4_grouped_linear_workspace_bytes(int64_t M, int64_t G, int64_t K);
NVFP4_API nvfp4_status nvfp4_grouped_linear(const void *x, int64_t M, int64_t G, int64_t K, int64_t N,
                                            const uint8_t *w, const uint8_t *w_sf, const float *ws2,
                                            int gs_mode, float *gs, void *y, void *ws,
                                            size_t ws_bytes, void *stream);

/* --------------------------------------------------------------- router gate
 * The dense router of page 1 (the router-gate FP8 round-trip passage): the NVFP4 gate
 * weight (E, H/2) codes with row-major scales (E, H/16) and device scalar ws2 is
 * dequantised to bf16, quantised to FP8-E4M3 with one per-tensor scale s = amax / 448 and
 * dequantised back to bf16 (nvfp4_router_prepare, once):
 *   w = bf16(fl32(fl32(e2m1 * e4m3) * ws2)),  q = E4M3(fl32(w * fl32(1/s))),
 *   wg = bf16(fl32(e4m3(q) * s))                       (wg all zero when s == 0)
 * Per call (nvfp4_router): logits = x (T, H) bf16 @ wg^T in fp32, softmax over the E
 * experts, the topk largest probabilities (lower expert id first on ties) as ids (T, topk)
 * int32 and weights (T, topk) fp32 renormalised to sum 1 -- the inputs of the routing
 * stage.  The logits run on the tensor cores split over H; the workspace
 * (nvfp4_router_workspace_bytes, always required) holds the splits' fp32 partials, which
 * are summed in a fixed order, so repeated calls give identical logits.  logits (T, E) fp32,
 * if not NULL, receives the summed logits.  E <= 1024, topk <= min(32, E), H % 64 == 0,
 * T and H below 2^24.  Two launches. */
NVFP4_API size_t nvfp4_router_prepare_workspace_bytes(int64_t E, int64_t H);
NVFP4_API nvfp4_status nvfp4_router_prepare(const uint8_t *w, const uint8_t *w_sf, const float *ws2, int64_t E,
                                            int64_t H, void *wg, void *ws, size_t ws_bytes, void *stream);
NVFP4_API size_t nvfp4_router_workspace_bytes(int64_t T, int64_t E);
NVFP4_API nvfp4_status nvfp4_router(const void *x, int64_t T, int64_t H, const void *wg, int64_t E, int topk,
                                    int32_t *ids, float *weights, float *logits, void *ws, size_t ws_bytes,
                                    void *stream);

/* -------------------------------------------------------------- (b) routing
 * Groups the T*topk flat entries f = t*topk + j of ids (T, topk) int32 by
 * expert: counts[e] (E), offsets (E+1, exclusive prefix sum, int32 as the
 * grouped GEMM wants: page 3, the grouped-GEMM launch contract),
 * sorted_idx (T*topk) = the flat indices ordered by expert, increasing f
 * within an expert, and inv_idx (T*topk) = position of f in sorted_idx.
 * Ids outside [0, E) are dropped (inv_idx = -1) and raise
 * NVFP4_DEVERR_BAD_EXPERT_ID.  1 <= E <= 1024, 1 <= topk <= 32. */
NVFP4_API nvfp4_status nvfp4_moe_route(const int32_t *ids, int64_t T, int topk, int64_t E,
                             int32_t *counts, int32_t *offsets, int32_t *sorted_idx,
                             int32_t *inv_idx, void *stream);

/* ---------------------------------------------------------------- MoE layer
 * Routed experts e in [0, E) plus an optional always-active shared expert
 * (group E).  Weights are prepared with nvfp4_prepare_weights:
 *   w13 (E, 2I, H/2) + sf, NVFP4_PREP_W13_INTERLEAVE (checkpoint rows [0,I)
 *       gate, [I,2I) up), w13_ws2 (E) fp32;
 *   w2  (E, H, I/2) + sf, NVFP4_PREP_PLAIN, w2_ws2 (E) fp32;
 *   sh_w13 / sh_w2 the same for one expert, sh_ws2 = {w13 ws2, w2 ws2};
 *   pass sh_w13 == NULL for no shared expert.
 * For every token t:
 *   y[t] = sum_j topk_w[t,j] * E_{ids[t,j]}(x[t]) + E_shared(x[t]),
 *   E_e(x) = W2_e . requant(SiLU(gate_e(xq)) * up_e(xq); a2_gs[e])
 * with xq = x quantised with one global scale over all T tokens (a1_gs_mode as
 * above, *a1_gs written in dynamic mode) and a2_gs (E+1 entries, last = shared
 * expert) the static global scales of the re-quantised intermediate h
 * (warm-up calibrated, page 3: the warm-up calibration passage).
 * y (T, H) bf16; the output width is H (page 3: the MoE shape-rules passage).  H % 128 == 0, I % 64 == 0.
 * nvfp4_moe_forward with one token (T = 1, topk <= 8, H <= 7168) runs as routing, one GEMM
 * launch and the conversion of y: the GEMM CTAs quantise the token themselves, take their
 * tiles from the ids and add each tile's share of the down projection (its 64 columns of
 * the re-quantised h times that K step of w2) into the fp32 accumulator; the workspace's xq,
 * xsf and amax_partials are then left untouched.  The re-quantised h rows (hq, hsf) are the
 * ones the stage-by-stage calls produce; y agrees within fp32 summation order. */
typedef struct nvfp4_moe_ws_layout {
  /* byte offsets into the workspace */
  size_t counts;        /* int32 [G]        rows per group (G = E + has_shared)     */
  size_t offsets;       /* int32 [G+1]      exclusive scan of counts                 */
  size_t pad_offsets;   /* int32 [G+1]      exclusive scan of counts rounded to 128  */
  size_t tile_offsets;  /* int32 [G+1]      exclusive scan of ceil(counts / R), R the
                           m-tile height: 32 when T <= 128, else 128                */
  size_t sorted_idx;    /* int32 [T*topk]                                            */
  size_t inv_idx;       /* int32 [T*topk]                                            */
  size_t dest_rows;     /* int32 [T*topk]   permuted row of each flat entry (-1 dropped) */
  size_t tile_table;    /* int32x4 [rows_capacity/32] per R-row tile of the permuted
                           buffers, in tile order: group, tile index inside the group
                           (bit 30 set when the group spans several tiles), live rows
                           (1..R), first permuted row                                */
  size_t amax_partials; /* uint32 [1024]    block maxima of |x| as bf16 bits         */
  size_t xq;            /* uint8 [rows_capacity, H/2]  x quantised, permuted rows    */
  size_t xsf;           /* uint8 nvfp4_sf_bytes(rows_capacity, H)                    */
  size_t hq;            /* uint8 [rows_capacity, I/2]  h re-quantised                */
  size_t hsf;           /* uint8 nvfp4_sf_bytes(rows_capacity, I)                    */
  size_t y_acc;         /* float [T, H]     fp32 accumulator of the scatter-add      */
  size_t total;         /* bytes                                                     */
  int64_t rows_capacity; /* padded-row capacity of the permuted buffers              */
  /* row of group g, segment row i in xq/xsf/hq/hsf: pad_offsets[g] + i; routed
   * segment row i of expert e holds flat entry sorted_idx[offsets[e] + i];
   * shared segment row i holds token i. */
} nvfp4_moe_ws_layout;

NVFP4_API nvfp4_status nvfp4_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                                        int has_shared, nvfp4_moe_ws_layout *out);
NVFP4_API size_t nvfp4_moe_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                                 int has_shared);

NVFP4_API nvfp4_status nvfp4_moe_forward(const void *x, int64_t T, int64_t H, int64_t I, int64_t E,
                               int topk, const int32_t *topk_ids, const float *topk_w,
                               const uint8_t *w13, const uint8_t *w13_sf, const float *w13_ws2,
                               const uint8_t *w2, const uint8_t *w2_sf, const float *w2_ws2,
                               const uint8_t *sh_w13, const uint8_t *sh_w13_sf,
                               const uint8_t *sh_w2, const uint8_t *sh_w2_sf,
                               const float *sh_ws2, int a1_gs_mode, float *a1_gs,
                               const float *a2_gs, void *y, void *ws, size_t ws_bytes,
                               void *stream);

/* The four stages nvfp4_moe_forward enqueues, exposed for stage-wise checks
 * and timing.  Same arguments as nvfp4_moe_forward; they communicate through
 * the workspace (layout above) and must run in this order on one stream. */

/* (a)+(b): routing, global scale, quantisation of x into the permuted rows,
 * zeroing of the fp32 accumulator.  Three launches. */
NVFP4_API nvfp4_status nvfp4_moe_dispatch(const void *x, int64_t T, int64_t H, int64_t I, int64_t E,
                                int topk, const int32_t *topk_ids, int has_shared,
                                int a1_gs_mode, float *a1_gs, void *ws, size_t ws_bytes,
                                void *stream);
/* (c): grouped w13 GEMM, SiLU(gate)*up, NVFP4 re-quantisation into hq/hsf.
 * h_debug, if not NULL, receives the fp32 h rows (rows_capacity, I). */
NVFP4_API nvfp4_status nvfp4_moe_w13(int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                           const uint8_t *w13, const uint8_t *w13_sf, const float *w13_ws2,
                           const uint8_t *sh_w13, const uint8_t *sh_w13_sf, const float *sh_ws2,
                           const float *a1_gs, const float *a2_gs, float *h_debug, void *ws,
                           size_t ws_bytes, void *stream);
/* (d): grouped w2 GEMM with the top-k weighted fp32 scatter-add into y_acc. */
NVFP4_API nvfp4_status nvfp4_moe_w2(int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                          const float *topk_w, const uint8_t *w2, const uint8_t *w2_sf,
                          const float *w2_ws2, const uint8_t *sh_w2, const uint8_t *sh_w2_sf,
                          const float *sh_ws2, const float *a2_gs, void *ws, size_t ws_bytes,
                          void *stream);
/* y (T, H) bf16 = round-to-nearest-even(y_acc). */
NVFP4_API nvfp4_status nvfp4_moe_finalize(int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                                int has_shared, void *y, void *ws, size_t ws_bytes,
                                void *stream);

/* ------------------------------------------------------------ diagnostics
 * Runs one CTA that waits on a shared-memory barrier nothing arrives at, with
 * the same bounded-wait helper the GEMM pipeline uses and a limit of
 * timeout_us; it must give up, raise NVFP4_DEVERR_PIPELINE_TIMEOUT and return.
 * Used to test the timeout path without a fault. */
NVFP4_API nvfp4_status nvfp4_debug_wait_timeout(uint32_t timeout_us, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_GB300_H */
