// Internal declarations shared by the translation units of the library (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

constexpr int kMaxPartials = 1024;      // block-max partials of the amax reduction
constexpr int kMaxExperts = 1024;       // routing limit (E)
constexpr int kMaxTopk = 32;
constexpr uint64_t kPipelineTimeoutNs = 2000000000ull;  // 2 s: no healthy wait comes close

// GEMM tile geometry: two persistent CTAs per SM, each with its own pipeline.  Two
// CTAs double the MMA issue rate per SM and the two pipelines overlap each other's
// epilogues.  The block scales reach TMEM through tcgen05.st from the epilogue
// warps, so the tensor pipe runs only the 4 MMAs (128x128x64) of a stage.
constexpr int kBlockM = 128;            // UMMA M
constexpr int kBlockN = 128;            // UMMA N and output tile width
constexpr int kStageK = 256;            // FP4 elements per pipeline stage (128 bytes per row)
constexpr int kUmmaK = 64;              // K per tcgen05.mma (kind::mxf4nvf4, scale_vec::4X)
#ifndef NVFP4_GEMM_STAGES
#define NVFP4_GEMM_STAGES 3
#endif
constexpr int kStages = NVFP4_GEMM_STAGES;
constexpr int kCtasPerSm = 2;
constexpr int kAccBufs = 1;             // TMEM accumulators per CTA
constexpr int kABoxRows = 32;           // A rows per TMA box (only boxes with live rows load)
constexpr int kTileBytesA = kBlockM * kStageK / 2;   // 16 KiB
constexpr int kTileBytesB = kBlockN * kStageK / 2;   // 16 KiB
constexpr int kSfBytesPerKStep = 512;   // 128 rows x 4 scales
constexpr int kSfBytesStage = kSfBytesPerKStep * (kStageK / kUmmaK);  // 2 KiB
constexpr int kGemmThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr uint32_t kTmemAccCols = kAccBufs * kBlockN;
constexpr uint32_t kTmemSfCols = 32;                 // per stage: 16 SFA + 16 SFB columns
constexpr uint32_t kTmemCols = 256;                  // per CTA: 128 accumulator + 96 scale columns
static_assert(kCtasPerSm * kTmemCols <= 512, "two CTAs share the SM's 512 TMEM columns");

// full, empty, sf_ready per stage; two tfull/tempty; drain; h_full/h_empty; TMEM address; abort flag
constexpr size_t kGemmBarrierBytes = 256;

// The stage ring in shared memory.  The regular ring holds kStages stages with a
// 128-row A slot.  When no tile can have more than 32 live rows (decode-sized MoE
// calls, M <= 32), the A slot shrinks to one 32-row box and 4 stages fit in less
// shared memory: a third more weight bytes in flight per CTA.
// With kQuantA (dense linear, M <= 32, K <= kQuantMaxK) the CTA quantises the bf16
// activations itself: every K stage's A box and its rows' scale words stay resident (written
// once by the epilogue warps), and a ring of kQuantStages stages carries the weights only.
// One CTA per SM, owning all 512 TMEM columns.
constexpr int kQuantMaxK = 4096;
// Every CTA quantises all of x: the fused path pays off while x is small.
constexpr int64_t kQuantMaxElems = 16384;
constexpr int kQuantStages = 7;

// Small-A MoE tiles keep their (at most 32) rows in the first TMEM lane quarter, so one
// warp reads the whole accumulator.  It leaves the tile's h = SiLU(gate) * up in shared
// memory (rows of kHRowFloats fp32, padded so that row-strided float4 accesses cover all
// banks) and the four epilogue warps re-quantise it together.
constexpr int kHRowFloats = 68;

// One-token MoE calls (T = 1, top-k <= kTok1MaxTopk, H <= kTok1MaxK): every group's A is
// the same token row, so the w13 CTAs quantise it themselves into one resident 8-row
// swizzle atom per K stage (the row repeated: a token that lists an expert more than once
// fills that many rows) and take their tile schedule from the top-k ids.  They start
// streaming weights as soon as the routing kernel has started.
constexpr int kTok1MaxK = 7168;
constexpr int kTok1MaxTopk = 8;
constexpr int kTok1SchedBytes = 256;  // group entries (int4) + the group count

template <bool kSmallA, bool kQuantA = false, bool kTok1 = false>
struct Ring {
  static constexpr int kStagesR = kTok1 ? 4 : (kQuantA ? kQuantStages : (kSmallA ? 4 : kStages));
  static constexpr int kABytes = kTok1 ? 1024 : (kSmallA ? kABoxRows * kStageK / 2 : kTileBytesA);
  static constexpr int kASlots =
      kTok1 ? kTok1MaxK / kStageK : (kQuantA ? kQuantMaxK / kStageK : kStagesR);  // A slots
  // SFA: one 2 KB block per A slot; kQuantA: the (at most 32) rows' scale words only, 128 bytes
  // per K step; kTok1: the token row's four scale words per K stage
  static constexpr int kSfaBytes = kTok1 ? 512 : (kQuantA ? kASlots * 4 * 128 : kASlots * kSfBytesStage);
  static constexpr uint32_t kTmemColsR = (kQuantA && !kTok1) ? 512 : kTmemCols;
  // MMA issuing threads.  One tcgen05.mma holds its issuing thread ~100 ns whatever its N,
  // while issuers in different warps run side by side.  The one-tile-per-CTA linears
  // (kQuantA) are chains of such issues: they swap the operands (the weight tile is the
  // MMA's 128 rows, the at most 32 tokens its N), so that an accumulator is 32 columns, and
  // four issuers take the K stages round-robin into an accumulator each; the epilogue adds
  // them, every warp for 32 output features.
  static constexpr bool kSwapAB = kQuantA && !kTok1;
  static constexpr int kIssuers = kSwapAB ? 4 : 1;
  static constexpr uint32_t kAccColsR = kSwapAB ? kIssuers * kABoxRows : kTmemAccCols;  // scale columns follow
  static constexpr int kThreads = kGemmThreads + (kIssuers - 1) * 32;  // warps 6.. : the further issuers
  static constexpr int kHBytes = kSmallA && (!kQuantA || kTok1) ? kABoxRows * kHRowFloats * 4 : 0;  // h of a tile
  static constexpr int kSchedBytes = kTok1 ? kTok1SchedBytes : 0;
  // kTok1: the re-quantised h of a tile as the fused down projection's B operand (32 rows of
  // 32 bytes, 32-byte swizzle) and its rows' scale words
  static constexpr int kP2Bytes = kTok1 ? 32 * 32 + 32 * 4 + 4 * 8 : 0;  // + p2_full[2], p2_empty[2]
  static constexpr size_t kBarBytes = (3 * kStagesR + 7) * 8 + 8 + 24 <= kGemmBarrierBytes ? kGemmBarrierBytes : 512;
  static constexpr size_t kSmem = 1024 /* alignment slack */ + static_cast<size_t>(kASlots) * kABytes + kSfaBytes +
                                  static_cast<size_t>(kStagesR) * (kTileBytesB + kSfBytesStage) +
                                  kBarBytes + kHBytes + kSchedBytes + kP2Bytes;
  // Requested (not used) by launches that want one CTA per SM: two of these do not fit.
  static constexpr size_t kSmemSolo = (kQuantA && !kTok1) ? kSmem : 2 * kSmem;
  static_assert(!kQuantA || kSmallA, "the resident A holds one 32-row box per K stage");
  static_assert(kAccColsR + kStagesR * kTmemSfCols <= kTmemColsR, "TMEM budget");
  static_assert((3 * kStagesR + 7) * 8 + 8 + 24 <= kBarBytes, "barrier region and scratch");
  static_assert(kSmemSolo <= 232448, "per-block shared memory limit");
  static_assert((kQuantA && !kTok1) || 2 * (kSmem + 1024) <= 233472, "two CTAs per SM");
  static_assert(kABytes % 1024 == 0, "128-byte swizzle atoms stay 1024-byte aligned");
  static_assert(kSfaBytes % 512 == 0, "the B ring stays 512-byte aligned");
  static_assert(!kTok1 || (kTok1MaxK / 16) <= kSfaBytes, "one scale byte per 16 elements of the token row");
};

enum class Epi : int { kLinear = 0, kW13 = 1, kW2 = 2 };

struct GemmArgs {
  // problem
  int G;              // groups (1 for a dense GEMM)
  int N;              // output width per group: a multiple of 128 (of 16 for one group, last tile partial)
  int K;              // reduction length, multiple of 64
  int dense_M;        // rows of every group when counts == nullptr (dense / uniform groups)
  // grouped segments (device arrays written by the routing kernel)
  const int *counts;        // [G]
  const int *offsets;       // [G+1] unpadded (sorted order)
  const int *pad_offsets;   // [G+1]
  const int *tile_offsets;  // [G+1]
  const int4 *tile_table;   // per m tile in tile order: group, m tile in group (| kTileMulti
                            // when the group spans several), live rows, first A row (written
                            // by the routing kernel; the tiles are kABoxRows high in the
                            // small-A ring, else kBlockM); null: every group has dense_M rows
  int shared_group;         // group using the *_shared weights, or -1
  // scale factors
  const uint8_t *a_sf;      // swizzled, 128-row blocks aligned with the A rows
  const uint8_t *b_sf;      // G blocks of N*K/16 bytes
  const uint8_t *b_sf_shared;
  // epilogue
  const float *gs_a;        // activation global scale (device scalar)
  const float *ws2;         // per-group weight scale (G entries, or 1 for dense)
  const float *ws2_shared;  // shared-expert weight scale
  const float *gs_out;      // W13: static global scale of h per group (G entries)
  void *out;                // Linear: bf16 y (dense_M, N); W13: hq codes; W2: fp32 y_acc
  uint8_t *out_sf;          // W13: hsf (swizzled)
  float *h_debug;           // W13 optional fp32 h
  int out_ld;               // Linear: N; W13: I/2 bytes; W2: H floats
  const int *sorted_idx;    // W2
  const float *topk_w;      // W2
  int topk;                 // W2
  uint32_t *err;            // device fault flags
  int a_kc_total;           // 64-element K steps per row in A's scale layout (>= K/64)
  int a_group_koff;         // K steps of A skipped per group index (uniform groups splitting
                            // A's columns); 0 when groups own separate A rows
  int out_group_cols;       // Linear: output columns skipped per group index
  int early_b;              // 1: B tiles and the tile schedule may be read before the
                            // previous kernel completes (the caller's chain guarantees
                            // they were written two or more launches back)
  // kQuantA: the bf16 activations (dense_M rows of qa_ld = G*K elements; group g uses
  // columns g*K..), the static scale (null: dynamic amax/2688 over all columns) and
  // where CTA 0 writes the dynamic scale.  The tiles of a CTA all belong to one group.
  const void *qa_x;
  int64_t qa_ld;
  const float *qa_gs_static;
  float *qa_gs_out;
  // kTok1 (one-token MoE w13): the top-k ids of the token (the routing kernel reads the
  // same array) and the number of routed experts E; the groups are the distinct valid ids
  // in increasing order, then the shared group.
  const int32_t *tok1_ids;
  int tok1_E;
  // early_b: stages of the first tile's weights prefetched into L2 beyond the ring
  int early_l2;
  // One-token w13 with the down projection fused (p2_acc set; p2_N = H, p2_K = I): after a
  // w13 tile (h columns 64 nt .. 64 nt + 63 of group g) the CTA multiplies its re-quantised
  // h by that 64-wide K step of all H rows of the group's w2 (split K over I; the w2 codes
  // through the slice maps, p2_sf / p2_sf_shared their scales, p2_ws2 / p2_ws2_shared the
  // weight scales) and adds the products, times the group's routing weight (tok1_ids,
  // p2_topk_w; 1 for the shared group) and the static scale of h, into p2_acc (H fp32).
  float *p2_acc;
  int p2_N;
  int p2_K;
  const uint8_t *p2_sf;
  const uint8_t *p2_sf_shared;
  const float *p2_ws2;
  const float *p2_ws2_shared;
  const float *p2_topk_w;
};


// Launch with programmatic dependent launch allowed: the kernel may start while the
// previous kernel on the stream is finishing.  Every kernel of the library therefore
// runs griddepcontrol.wait before it reads any global input, and triggers its own
// dependents at its start.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launchers (return cudaError_t of the launch)
// Grid of the streaming kernels (quantisers): kStreamCtasPerSm CTAs of 256 threads per SM,
// each walking its share of the blocks.
constexpr int kStreamCtasPerSm = 4;
int stream_grid_cap();
cudaError_t launch_amax_partials(const void *x, int64_t M, int64_t K, int64_t ldx,
                                 uint32_t *partials, int nparts, cudaStream_t s);
int amax_partial_count(int64_t M, int64_t K);
cudaError_t launch_quantize(const void *x, int64_t M, int64_t K, int64_t ldx,
                            const uint32_t *partials, int nparts, const float *gs_static,
                            float *gs_out, uint8_t *q, uint8_t *sf, int sf_layout,
                            cudaStream_t s);
// Activation quantisation with a dynamic (amax/2688) or static gs.  Dynamic inputs of at most
// kInlineAmaxElems elements take one launch (each quantise block reduces x itself); larger ones
// an amax-partials launch first (partials: amax_partial_count(M, K) words of workspace).
constexpr int64_t kInlineAmaxElems = 32768;
cudaError_t launch_act_quant(const void *x, int64_t M, int64_t K, int64_t ldx, bool dynamic, uint32_t *partials,
                             const float *gs_static, float *gs_out, uint8_t *q, uint8_t *sf, int sf_layout,
                             cudaStream_t s);
cudaError_t launch_rmsnorm_stats(const void *x, int64_t M, int64_t K, int64_t ldx, const void *gamma, float eps,
                                 float *inv_rms, uint32_t *partials, int nparts, void *y, cudaStream_t s);
cudaError_t launch_rmsnorm_quantize(const void *x, int64_t M, int64_t K, int64_t ldx, const void *gamma,
                                    const float *inv_rms, const uint32_t *partials, int nparts,
                                    const float *gs_static, float *gs_out, uint8_t *q, uint8_t *sf, int sf_layout,
                                    cudaStream_t s);
int router_partial_count(int64_t nblocks);
cudaError_t launch_router_prepare(const uint8_t *w, const uint8_t *sf, const float *ws2, int64_t E, int64_t H,
                                  uint32_t *partials, void *wg, cudaStream_t s);
// Router logits on the tensor cores, split over K into router_splits(T, E, H) fp32 partials
// (partial: splits x T x E floats), then softmax + top-k over their sum.  tm_x / tm_w: byte
// tensor maps of x (T rows of 2H bytes) and wg (E rows) with 128-byte x 128-row boxes.
constexpr int64_t kRouterTargetCtas = 144;  // tiles x splits aimed for
constexpr int64_t kRouterMaxSplits = 48;
int router_splits(int64_t T, int64_t E, int64_t H);
cudaError_t launch_router(const CUtensorMap &tm_x, const CUtensorMap &tm_w, int64_t T, int64_t H, int64_t E, int topk,
                          int32_t *ids, float *weights, float *logits, float *partial, uint32_t *err, cudaStream_t s);
cudaError_t launch_prepare(const uint8_t *w, const uint8_t *sf, int64_t G, int64_t N, int64_t K,
                           int flags, uint8_t *w_out, uint8_t *sf_out, cudaStream_t s);

struct RouteBufs {
  int *counts, *offsets, *pad_offsets, *tile_offsets, *sorted_idx, *inv_idx, *dest_rows;
  int4 *tile_table;  // per tile: group, tile in group | kTileMulti, live rows, first row (or null)
  int tile_shift;    // log2 of the tile height: moe_tile_rows(T)
};

// Height of the MoE GEMMs' m tiles.  Up to kSmallTileMaxT tokens (a decode batch or a
// 128-token prefill chunk) the groups are cut into kABoxRows-row tiles, so every tile
// fits one A box and the GEMMs take the small-A ring with its fourth stage.  Most groups
// then hold one tile; the few with more rows (the shared expert, popular experts, or an
// expert listed twice by a token) span several, which run concurrently and share their
// weights through L2.  Larger batches, where popular experts hold thousands of rows,
// use kBlockM-row tiles.
constexpr int64_t kSmallTileMaxT = 128;
// Flag in a tile-table entry's second field (tile index inside the group): the group
// spans more than one tile.
constexpr int kTileMulti = 1 << 30;
inline int moe_tile_rows(int64_t T) { return T <= kSmallTileMaxT ? kABoxRows : kBlockM; }
inline int moe_tile_shift(int64_t T) { return T <= kSmallTileMaxT ? 5 : 7; }
static_assert((1 << 5) == kABoxRows && (1 << 7) == kBlockM, "tile shifts");
cudaError_t launch_route_amax(const int32_t *ids, int T, int topk, int E, int has_shared,
                              RouteBufs rb, const void *x, int64_t H, uint32_t *partials,
                              int nparts, float *y_acc, uint32_t *err, cudaStream_t s);
cudaError_t launch_dispatch_quant(const void *x, int T, int64_t H, int topk, int E,
                                  int has_shared, const int32_t *ids, RouteBufs rb,
                                  const uint32_t *partials, int nparts, const float *gs_static,
                                  float *gs_out, uint8_t *xq, uint8_t *xsf, cudaStream_t s);
cudaError_t launch_finalize(const float *y_acc, int64_t n, void *y, cudaStream_t s);
// small_a: every tile has at most kABoxRows live rows (the caller guarantees it; the
// kernel raises NVFP4_DEVERR_INTERNAL otherwise).
cudaError_t launch_gemm(Epi epi, const CUtensorMap &ta, const CUtensorMap &tb,
                        const CUtensorMap &tbs, const GemmArgs &args, int grid, bool one_per_sm,
                        bool small_a, cudaStream_t s);
// Dense or fixed-group linear with the activation quantisation fused (kQuantA): 1 <= M <= 32,
// K <= kQuantMaxK, grid = tiles <= SM count (one tile per CTA).
cudaError_t launch_gemm_quant_a(const CUtensorMap &tb, const GemmArgs &args, int grid, cudaStream_t s);
// One-token MoE w13 (T = 1): the CTAs quantise the token (args.qa_*) and derive the tile
// schedule from args.tok1_ids; two CTAs per SM.
cudaError_t launch_gemm_tok1(const CUtensorMap &tb, const CUtensorMap &tbs, const CUtensorMap &t2,
                             const CUtensorMap &t2s, const GemmArgs &args, int grid, cudaStream_t s);
// Dense GEMM on CTA pairs (256 x 256 tiles, tcgen05 cta_group::2): N % 256 == 0, A read
// through a tensor map with 128-row boxes.  gemm_pair_max_clusters: clusters of 2 that fit
// on the current device at once (0 if the query fails).
constexpr int64_t kPairMinM = 512;   // fewer rows: the one-SM tiles spread over more SMs
int gemm_pair_max_clusters();
cudaError_t launch_gemm_pair(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args, int clusters,
                             cudaStream_t s);
cudaError_t launch_wait_timeout_probe(uint32_t timeout_us, uint32_t *err, cudaStream_t s);

}  // namespace nvfp4
