// Dense NVFP4 block-scaled GEMM on CTA pairs (tcgen05 cta_group::2), for the tensor-bound
// linears (many rows, N a multiple of 256).
//
//   y[m, n] = bf16(gs * ws2 * sum_k e2m1(A[m,k]) e4m3(SFA[m,k/16]) e2m1(B[n,k]) e4m3(SFB[n,k/16]))
//
// An output tile is 256 x 256.  The two CTAs of a cluster each stage 128 rows of A and 128
// rows of B (the operand halves of one M = 256, N = 256 MMA), and each holds its 128 output
// rows x 256 columns in its own tensor memory.  Per byte staged in shared memory this does
// twice the MMA work of a 128 x 128 tile on one SM, which halves the L2 -> SM operand
// traffic that bounds the one-SM tiles at these shapes.
//
// One CTA per SM (192 KB of shared memory: a 5-stage ring of 256 K elements per stage),
// 15 warps per CTA:
//   warp 0       TMA producer: this CTA's A and B boxes (128 rows each) and scale blocks;
//   warp 1       owns the pair's tensor memory; in the even CTA, one lane issues the MMAs
//                of every other stage for both CTAs and commits them to the barriers of
//                both; warp 14's first lane issues the stages in between (into the same
//                accumulator, handing the turn on through the turn barriers);
//   warps 2..5   scale staging: each stage's A scales (this CTA's 128 rows) and the B scales
//                of all 256 B rows of the tile (the pair MMA reads B's scales for every N
//                row from each CTA's own tensor memory: 8 columns per K step, column c
//                holding rows 32 c .. 32 c + 31), shared memory -> this CTA's tensor memory
//                (tcgen05.st, one lane quarter per warp), then an arrival on the even CTA's
//                sf_ready barrier (the MMA issuer waits for all 8 warps);
//   warps 6..13  epilogue: 128 rows x 256 columns, two warps per lane quarter (128 columns
//                each); they hand the accumulator back to the even CTA's issuer (tempty).
// Every wait is bounded (kPipelineTimeoutNs).  A role that gives up raises
// NVFP4_DEVERR_PIPELINE_TIMEOUT and leaves its loop; the producer lets its copies in flight
// land, the issuer drains its MMAs, and every thread of both CTAs then meets at the final
// cluster barrier before the pair frees its tensor memory.
#include "common.cuh"

namespace nvfp4 {

namespace {

constexpr int kPM = 256;              // output tile rows (128 per CTA)
constexpr int kPN = 256;              // output tile columns (128 B rows staged per CTA)
constexpr int kPHalf = 128;
constexpr int kPStages = 5;
constexpr int kPScaleWarps = 4;
constexpr int kPEpiWarps = 8;
// MMA issuers of the even CTA: warp 1 and warps kPIssuerWarp0.. take the launch's stages in turn
constexpr int kPIssuers = 2;
constexpr int kPIssuerWarp0 = 2 + kPScaleWarps + kPEpiWarps;
constexpr int kPThreads = (2 + kPScaleWarps + kPEpiWarps + kPIssuers - 1) * 32;
constexpr int kPTileA = kPHalf * kStageK / 2;    // 16 KiB: 128 rows x 128 bytes
constexpr int kPTileB = kPHalf * kStageK / 2;    // 16 KiB
constexpr int kPSfbBytes = 2 * kSfBytesStage;     // B scales of both 128-row halves
constexpr int kPStageBytes = kPTileA + kPTileB + kSfBytesStage + kPSfbBytes;
constexpr uint32_t kPSfCols = 16 + 32;           // per stage: 4 K steps x (4 SFA + 8 SFB) columns
constexpr size_t kPSmem = 1024 + static_cast<size_t>(kPStages) * kPStageBytes + kGemmBarrierBytes;
constexpr uint32_t kPTmemCols = 512;
constexpr uint32_t kPAccCols = kPN;              // fp32 accumulator: 128 lanes x 256 columns
static_assert(kPAccCols + kPStages * kPSfCols <= kPTmemCols, "TMEM budget");
static_assert(kPSmem <= 232448, "per-block shared memory limit");
static_assert((4 * kPStages + 3 + kPIssuers) * 8 + 16 <= kGemmBarrierBytes, "barrier region");
// An issuer's previous own stage is g - kPIssuers, issued (in turn order) after every
// stage before it.  The slot of its next stage g has therefore landed stage g - kPStages,
// i.e. its barriers are at most one phase behind, only if kPIssuers <= kPStages; with more
// issuers a parity wait on that slot could match a phase two behind and pass too early.
static_assert(kPIssuers <= kPStages, "turn-taking issuers: at most one per ring stage");

// E2M1 x E2M1, UE4M3 scales, K-major A and B, M = 256 (the pair), N = 256.
constexpr uint32_t kPIdesc = (1u << 7) | (1u << 10) | ((uint32_t(kPN) >> 3) << 17) | ((uint32_t(kPM) >> 4) << 24);

__global__ void __launch_bounds__(kPThreads, 1)
    nvfp4_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = sA + kPStages * kPTileA;
  uint8_t *sSFA = sB + kPStages * kPTileB;
  uint8_t *sSFB = sSFA + kPStages * kSfBytesStage;
  uint64_t *full = reinterpret_cast<uint64_t *>(sSFB + kPStages * kPSfbBytes);
  uint64_t *empty = full + kPStages;
  uint64_t *sf_ready = empty + kPStages;  // used in the even CTA
  uint64_t *tfull = sf_ready + kPStages;
  uint64_t *tempty = tfull + 1;           // used in the even CTA
  uint64_t *drain = tempty + 1;
  uint64_t *turn = drain + 1;             // turn[i]: issuer i may issue its next stage (even CTA)
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(turn + kPIssuers);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 2 * kPScaleWarps);
    }
    mbar_init(tfull, kPIssuers);
    mbar_init(tempty, 2 * kPEpiWarps);
    mbar_init(drain, kPIssuers);
    for (int i = 0; i < kPIssuers; ++i) mbar_init(&turn[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised and tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  pdl_wait();
  pdl_trigger();

  const int M = args.dense_M;
  const int n_tiles = args.N / kPN;
  const int k_steps = args.K / kUmmaK;
  const int k_stages = (k_steps + 3) / 4;
  const int total_tiles = ((M + kPM - 1) / kPM) * n_tiles;
  const int a_rows_padded = (M + 127) / 128 * 128;  // rows of A's scale layout
  const int clusters = static_cast<int>(gridDim.x) / 2;
  const int cluster_id = static_cast<int>(blockIdx.x) / 2;
  // balanced grid: every wave of tiles (the last included) is (nearly) full
  const int waves = (total_tiles + clusters - 1) / clusters;
  const int active = waves > 0 ? (total_tiles + waves - 1) / waves : clusters;
  const int first = cluster_id < active ? cluster_id : total_tiles;
  // the leader's barriers, as the peer reaches them
  const uint32_t sf_ready_leader = cluster_addr(sf_ready, 0);
  const uint32_t tempty_leader = cluster_addr(tempty, 0);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_b = policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // bit s: stage s has a load in flight with parity bit (s + 8)
      bool ok = true;
      for (int idx = first; ok && idx < total_tiles; idx += active) {
        const int mt = idx / n_tiles, nt = idx - (idx / n_tiles) * n_tiles;
        const int a_row = mt * kPM + static_cast<int>(rank) * kPHalf;
        const int b_row = nt * kPN + static_cast<int>(rank) * kPHalf;
        const bool sfa_live = a_row < a_rows_padded;  // this half holds rows of A
        const uint8_t *sfa = args.a_sf + static_cast<size_t>(a_row / 128) * args.a_kc_total * kSfBytesPerKStep;
        // the B scales of both halves of the tile's 256 B rows
        const uint8_t *sfb = args.b_sf + static_cast<size_t>(nt * 2) * k_steps * kSfBytesPerKStep;
        for (int ks = 0; ks < k_stages; ++ks) {
          const int kv = min(4, k_steps - 4 * ks);
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, args.err, kPipelineTimeoutNs)) {
            ok = false;
            break;
          }
          const uint32_t bytes = kPTileA + kPTileB + (sfa_live ? kv * kSfBytesPerKStep : 0) + 2 * kv * kSfBytesPerKStep;
          mbar_arrive_expect_tx(&full[stage], bytes);
          // rows of A beyond M read as zeros (out-of-range box rows); their outputs are dropped
          tma_load_2d(sA + stage * kPTileA, &tmA, ks * (kStageK / 2), a_row, &full[stage], pol_a);
          // tile-major weights: block (128-row tile, stage) is contiguous
          tma_load_2d(sB + stage * kPTileB, &tmB, 0, (b_row / kPHalf * k_stages + ks) * kPHalf, &full[stage], pol_b);
          if (sfa_live)
            bulk_load(sSFA + stage * kSfBytesStage, sfa + static_cast<size_t>(ks) * kSfBytesStage,
                      kv * kSfBytesPerKStep, &full[stage], pol_a);
          for (int h = 0; h < 2; ++h)
            bulk_load(sSFB + stage * kPSfbBytes + h * kSfBytesStage,
                      sfb + (static_cast<size_t>(h) * k_steps + 4 * ks) * kSfBytesPerKStep, kv * kSfBytesPerKStep,
                      &full[stage], pol_b);
          issued = (issued & ~(0x101u << stage)) | (1u << stage) | (phase << (stage + 8));
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // let the copies in flight land before the CTA leaves (bounded by its own 100 ms)
        volatile int never = 0;
        for (int s = 0; s < kPStages; ++s)
          if (issued & (1u << s)) mbar_wait_bounded(&full[s], (issued >> (s + 8)) & 1u, &never, nullptr, 100000000ull);
      }
    }
  } else if (warp == 1 || warp >= kPIssuerWarp0) {
    if (leader && lane == 0) {
      // ------------------------------------------------------------ MMA issuers (even CTA)
      // Stage g of the launch (counted over all tiles) is issued by issuer g % kPIssuers, into the one
      // accumulator.  One tcgen05.mma holds its issuing thread about its own execution time;
      // with several issuers, one thread's waits for its next stage (scales staged, operands
      // landed) and its commits overlap the others' MMAs.  The hand-off orders the accumulator's
      // updates: after its stage, an issuer fences (tcgen05.fence::before_thread_sync) and
      // arrives on the next issuer's turn barrier; that one waits on it and fences
      // (::after_thread_sync) before its MMAs.  The turns go round in order, so a turn barrier
      // never runs a phase ahead of its waiter.
      const int iss = warp == 1 ? 0 : warp - kPIssuerWarp0 + 1;
      const int pred = (iss + kPIssuers - 1) % kPIssuers;  // the issuer of the stage before ours
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      int g = 0;  // stages of the launch so far
      bool ok = true;
      const uint32_t sA0 = smem_u32(sA), sB0 = smem_u32(sB);
      for (int idx = first; ok && idx < total_tiles; idx += active, ++it) {
        for (int ks = 0; ks < k_stages; ++ks, ++g) {
          const int kv = min(4, k_steps - 4 * ks);
          if (g % kPIssuers == iss) {
            // the tile's first stage waits for the epilogue to have read the previous tile
            if (ks == 0 && !mbar_wait_bounded_cluster(tempty, (it & 1) ^ 1, abort_flag, args.err, kPipelineTimeoutNs)) {
              ok = false;
              break;
            }
            // both CTAs' operands of the stage have landed and their scales are in tensor memory
            if (!mbar_wait_bounded_cluster(&sf_ready[stage], phase, abort_flag, args.err, kPipelineTimeoutNs) ||
                (g > 0 &&
                 !mbar_wait_bounded(&turn[iss], ((g - 1 - pred) / kPIssuers) & 1, abort_flag, args.err, kPipelineTimeoutNs))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sf_col = tmem_base + kPAccCols + stage * kPSfCols;
            const uint64_t adesc = smem_desc(sA0 + stage * kPTileA, 16, 1024, 2);
            const uint64_t bdesc = smem_desc(sB0 + stage * kPTileB, 16, 1024, 2);
            for (int j = 0; j < kv; ++j)
              tc_mma_nvf4_pair(tmem_base, adesc + 2 * j, bdesc + 2 * j, kPIdesc, sf_col + j * 4, sf_col + 16 + j * 8,
                               (ks | j) != 0);
            tc_fence_before();
            mbar_arrive(&turn[(iss + 1) % kPIssuers]);  // the next issuer takes stage g + 1
            tc_commit_pair(&empty[stage], 0x3);
          }
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair(tfull, 0x3);  // each issuer: its MMAs of the tile (tfull counts both)
      }
      // every MMA issued has completed before the pair frees its tensor memory
      volatile int never = 0;
      tc_commit_pair(drain, 0x1);
      mbar_wait_bounded(drain, 0, &never, nullptr, 100000000ull);
    }
  } else if (warp < 2 + kPScaleWarps) {
    // -------------------------------------------------------------- scale staging
    // Each K step's 512-byte block holds, at 16 r + 4 c, the four scales (64 K) of operand row
    // 32 c + r of a 128-row half; every 32-lane quarter of tensor memory gets the same copy
    // (lane 32 q + r, column + c), the arrangement the MMA reads.  B's two halves sit side by
    // side (columns 8 j + c and 8 j + 4 + c of K step j).  This warp writes its own quarter.
    const int quarter = warp & 3;
    const uint32_t sf_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + kPAccCols;
    const int sf_off = lane * 16;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int idx = first; ok && idx < total_tiles; idx += active) {
      const int mt = idx / n_tiles;
      const bool sfa_live = mt * kPM + static_cast<int>(rank) * kPHalf < a_rows_padded;
      for (int ks = 0; ks < k_stages; ++ks) {
        const int kv = min(4, k_steps - 4 * ks);
        ok = mbar_wait_bounded(&full[stage], phase, abort_flag, args.err, kPipelineTimeoutNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint8_t *pa = sSFA + stage * kSfBytesStage + sf_off;
        const uint8_t *pb = sSFB + stage * kPSfbBytes + sf_off;
        uint32_t ra[16], rb0[16], rb1[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 wa = (j < kv && sfa_live) ? *reinterpret_cast<const uint4 *>(pa + j * kSfBytesPerKStep)
                                                : make_uint4(0u, 0u, 0u, 0u);
          ra[4 * j] = wa.x, ra[4 * j + 1] = wa.y, ra[4 * j + 2] = wa.z, ra[4 * j + 3] = wa.w;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 wb = j < kv ? *reinterpret_cast<const uint4 *>(pb + h * kSfBytesStage + j * kSfBytesPerKStep)
                                    : make_uint4(0u, 0u, 0u, 0u);
            uint32_t *rb = (j < 2) ? rb0 : rb1;  // K steps 0, 1 -> columns 16..31; 2, 3 -> 32..47
            const int c = (j & 1) * 8 + h * 4;
            rb[c] = wb.x, rb[c + 1] = wb.y, rb[c + 2] = wb.z, rb[c + 3] = wb.w;
          }
        }
        tmem_st16(sf_lane + stage * kPSfCols, ra);
        tmem_st16(sf_lane + stage * kPSfCols + 16, rb0);
        tmem_st16(sf_lane + stage * kPSfCols + 32, rb1);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(sf_ready_leader + stage * 8);
        if (++stage == kPStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;             // tensor-memory lanes [32 quarter, 32 quarter + 32)
    const int half = (warp - 2 - kPScaleWarps) >> 2;  // columns [128 half, 128 half + 128)
    const float alpha = __ldg(args.gs_a) * __ldg(args.ws2);
    const bool out32 = (reinterpret_cast<uintptr_t>(args.out) & 31u) == 0;
    int it = 0;
    for (int idx = first; idx < total_tiles; idx += active, ++it) {
      const int mt = idx / n_tiles, nt = idx - (idx / n_tiles) * n_tiles;
      const int row0 = mt * kPM + static_cast<int>(rank) * kPHalf + quarter * 32;
      bool ok = mbar_wait_bounded(tfull, it & 1, abort_flag, args.err, kPipelineTimeoutNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader);
      };
      if (row0 >= M) {  // all 32 rows of this warp are past the end of A
        release();
        continue;
      }
      const int row = row0 + lane;
      const bool row_ok = row < M;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(half * 128);
      __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(args.out) + static_cast<int64_t>(row) * args.out_ld +
                         nt * kPN + half * 128;
      // two batches of 64 columns, one tensor-memory wait each: the accumulator goes back to
      // the issuer after two load round trips instead of eight
#pragma unroll 1
      for (int b = 0; b < 2; ++b) {
        uint32_t r[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tbase + b * 64 + q * 16, r[q]);
        tmem_ld_wait();
        if (b == 1) release();
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[q][2 * i]) * alpha,
                                                             __uint_as_float(r[q][2 * i + 1]) * alpha);
              packed[i] = *reinterpret_cast<const uint32_t *>(&v);
            }
            __nv_bfloat16 *dst = y + b * 64 + q * 16;
            if (out32) {
              st_global_v8(dst, packed);
            } else {
              uint4 *d4 = reinterpret_cast<uint4 *>(dst);
              d4[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
              d4[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair's MMAs have drained and both epilogues have read their accumulators
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kPTmemCols);
}

}  // namespace

// Clusters of the pair kernel that fit on the device at once (cached per device).
int gemm_pair_max_clusters() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(nvfp4_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kPSmem)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, nvfp4_gemm_pair_kernel, &cfg) != cudaSuccess) return 0;
  cached[dev] = n;
  return n;
}

cudaError_t launch_gemm_pair(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args, int clusters,
                             cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(nvfp4_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPSmem));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, nvfp4_gemm_pair_kernel, ta, tb, args);
}

}  // namespace nvfp4
