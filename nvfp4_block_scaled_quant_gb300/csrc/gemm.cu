// Grouped NVFP4 block-scaled GEMM on the 5th-generation tensor cores.
//
//   D[m, n] = sum_k e2m1(A[m,k]) e4m3(SFA[m,k/16]) e2m1(B[n,k]) e4m3(SFB[n,k/16])
//
// with one fp32 accumulator tile of 128 x 128 in TMEM per output tile
// (tcgen05.mma kind::mxf4nvf4, scale_vec::4X, K = 64 per instruction), operands
// staged in shared memory by TMA (128-byte swizzle, 256 FP4 elements of K per
// stage) and the block scales written to TMEM with tcgen05.st by the epilogue
// warps, which leaves the tensor pipe to the MMAs alone.  Two persistent CTAs
// per SM walk the tiles of all groups:
//   warp 0      TMA producer (one lane): A box rows only as far as the group's
//               live rows reach, B tile, A/B scale blocks (bulk copies);
//   warp 1      MMA issuer (one lane), owns the TMEM allocation;
//   warps 2..5  scale staging for every stage of a tile (each warp its TMEM
//               lane quarter: A and B scales of rows 32q..32q+31), then the
//               epilogue, one accumulator row per thread.
// The two CTAs of an SM overlap each other's epilogues and keep two MMA
// issuers busy (one accumulator buffer each).  The linears that quantise their own
// activations (one CTA per SM, at most 32 tokens) swap the operands instead: the
// weight tile is the MMA's 128 rows and the tokens its N, and warps 6..8 join warp 1
// as MMA issuers, each taking every fourth K stage into its own 32-column
// accumulator (one issuing thread is held ~100 ns per MMA; issuers in different
// warps overlap).  Every wait is bounded (kPipelineTimeoutNs); a role that gives up
// sets a shared abort flag, the others drain and the CTA frees TMEM and exits
// with NVFP4_DEVERR_PIPELINE_TIMEOUT raised.
//
// Epilogues (the fused steps of the MoE expert path):
//   kLinear  y = bf16(gs * ws2 * D)                       (Nvfp4Linear)
//   kW13     h = SiLU(a * D_gate) * (a * D_up), a = gs * ws2_e, then h is
//            re-quantised to NVFP4 with the static scale gs2_e into the
//            permuted rows of the w2 input                 (gate/up projection)
//   kW2      y_acc[t] += topk_w * gs2_e * ws2_e * D        (down projection,
//            top-k weighted scatter-add in fp32)
#include <type_traits>

#include "common.cuh"

namespace nvfp4 {

namespace {

struct Tile {
  int g;       // group
  int mt;      // m tile inside the group
  int nt;      // n tile
  int rows;    // live rows of this m tile (1..128)
  int a_row0;  // first A row (permuted/padded row index)
  bool multi;  // the group spans several m tiles, which read the same weights
};

// Schedule entry of m tile mtg: group, m tile inside the group, live rows, first A row.
// Grouped problems read the table the routing kernel wrote; uniform groups compute it.
// Callers fetch the entry of their next tile one tile ahead, so the load's latency
// overlaps the current tile.
__device__ __forceinline__ int4 tile_entry(const GemmArgs &a, int mtg) {
  if (a.tile_table != nullptr) return __ldg(a.tile_table + mtg);
  const int mt_per_group = (a.dense_M + kBlockM - 1) / kBlockM;
  const int g = mtg / mt_per_group;
  const int mt = mtg - g * mt_per_group;
  return make_int4(g, mt | (a.dense_M > kBlockM ? kTileMulti : 0), min(kBlockM, a.dense_M - mt * kBlockM),
                   mt * kBlockM);
}

__device__ __forceinline__ Tile make_tile(const int4 e, int idx, int n_tiles) {
  Tile t;
  t.g = e.x;
  t.mt = e.y & ~kTileMulti;
  t.multi = (e.y & kTileMulti) != 0;
  t.rows = e.z;
  t.a_row0 = e.w;
  t.nt = idx - (idx / n_tiles) * n_tiles;
  return t;
}

// Word c of the result is word (c + j) & 3 of v.  A 32-row tile whose first row is
// 32 j into its 128-row scale block needs the scales of its rows, which sit in word j
// of each 16-byte chunk, where the MMA reads the scales of rows 0..31: word 0.
__device__ __forceinline__ uint4 rotate_words(uint4 v, int j) {
  if (j & 2) v = make_uint4(v.z, v.w, v.x, v.y);
  if (j & 1) v = make_uint4(v.y, v.z, v.w, v.x);
  return v;
}

// instruction descriptor: E2M1 x E2M1, UE4M3 scales, K-major A and B, M=128, N=128
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t(kBlockN) >> 3) << 17) |
                            ((uint32_t(kBlockM) >> 4) << 24);

// Swapped-operand linears (weights M = 128, tokens N = 32)
constexpr uint32_t kIdescSwap = (1u << 7) | (1u << 10) | ((uint32_t(kABoxRows) >> 3) << 17) |
                                ((uint32_t(kBlockM) >> 4) << 24);

// The one-token kernel's fused down projection: per stage kP2RowTiles w2 row tiles of 128
// rows x one 64-element K step (32 bytes, 32-byte swizzle), each one MMA of M = 128 (w2 rows)
// by N = kP2N (rows of the re-quantised h: the token's copies, at most kTok1MaxTopk) into its
// own slot of one of two 64-column accumulator buffers, so that a stage's MMAs run while the
// epilogue reads the previous stage's.
constexpr int kP2RowTiles = 4;
constexpr int kP2N = 16;
constexpr int kP2TileBytes = kBlockN * 32;
constexpr uint32_t kIdescP2 = (1u << 7) | (1u << 10) | ((uint32_t(kP2N) >> 3) << 17) | ((uint32_t(kBlockM) >> 4) << 24);
static_assert(kP2RowTiles * kP2TileBytes <= kTileBytesB && kP2RowTiles * kSfBytesPerKStep <= kSfBytesStage,
              "a fused-down-projection stage fits a ring slot");
static_assert(2 * kP2RowTiles * kP2N <= kBlockN && kTok1MaxTopk <= kP2N, "two slot buffers fit the accumulator");

// SiLU(g) * u with the fast exponential and divide (relative error ~1e-6; for g below
// about -88, exp(-g) is +inf and the quotient is 0).
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Fused activation quantisation (dense_M <= 32 rows): the four epilogue warps (tid
// 0..127, named barrier 1) take gs = fl32(amax / 2688) over all qa_ld columns of x (or
// the static scale), then encode the K columns of group g (columns g*K .. g*K+K-1; g = 0
// for a dense linear) with the activation quantiser's arithmetic into the resident A
// boxes (one 32-row, 128-byte-swizzled 4 KB box per 256-element K stage: 16-byte chunk
// c of row r sits at chunk c ^ (r & 7)) and their scale words (row r's four scales of a
// 64-element K step at 4 r in that step's 128 bytes).  CTA 0 writes gs out; every CTA
// returns the same gs.
__device__ float quantize_resident_a(const GemmArgs &a, int g, uint8_t *sA, uint8_t *sSFA, uint32_t *scratch,
                                     int tid) {
  const int64_t M = a.dense_M, K = a.K, ld = a.qa_ld;
  const uint16_t *x = static_cast<const uint16_t *>(a.qa_x);
  const int warp = tid >> 5, lane = tid & 31;
  float gs;
  if (a.qa_gs_static == nullptr) {
    uint32_t m = 0;
    // the M x ld inputs are contiguous (row stride ld): U 16-byte loads in flight per thread,
    // 32 when x is large enough that 8 would take several round trips (the 8 x 4096 inputs
    // of a grouped o-projection token take one)
    const int n = static_cast<int>(M * (ld / 8));
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    auto reduce = [&](auto U) {
      constexpr int kU = decltype(U)::value;
      for (int i0 = tid; i0 < n; i0 += kU * 128) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int i = i0 + u * 128;
          v[u] = i < n ? __ldg(xv + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
        }
      }
    };
    if (n > 8 * 128)
      reduce(std::integral_constant<int, 32>());
    else
      reduce(std::integral_constant<int, 8>());
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) scratch[warp] = m;
    named_barrier_sync(1, 128);
    m = max(max(scratch[0], scratch[1]), max(scratch[2], scratch[3]));
    gs = __fdiv_rn(__uint_as_float(m << 16), 2688.0f);
  } else {
    gs = __ldg(a.qa_gs_static);
  }
  if (blockIdx.x == 0 && tid == 0 && a.qa_gs_out != nullptr) *a.qa_gs_out = gs;
  const float six_gs = __fmul_rn(6.0f, gs);
  const int64_t kb = K / 16;
#pragma unroll 2
  for (int i = tid; i < static_cast<int>(M * kb); i += 128) {
    const int r = i / static_cast<int>(kb), c = i - r * static_cast<int>(kb);  // row, 16-element block of the group
    const uint4 *src = reinterpret_cast<const uint4 *>(x + r * ld + static_cast<int64_t>(g) * K + c * 16);
    const uint4 p = __ldg(src), q = __ldg(src + 1);
    const uint32_t w[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
    uint32_t codes[2];
    const uint32_t sfb = encode_block16_bf16(w, gs, six_gs, codes);
    const int st = static_cast<int>(c >> 4), j = static_cast<int>(c & 15), rr = static_cast<int>(r);
    const int chunk = (j >> 1) ^ (rr & 7);
    *reinterpret_cast<uint2 *>(sA + st * (kABoxRows * kStageK / 2) + rr * 128 + chunk * 16 + (j & 1) * 8) =
        make_uint2(codes[0], codes[1]);
    sSFA[(st * 4 + ((j >> 2) & 3)) * 128 + rr * 4 + (j & 3)] = static_cast<uint8_t>(sfb);  // K step, row, block
  }
  fence_proxy_async_shared();  // the MMAs read the boxes through the async proxy
  named_barrier_sync(1, 128);
  return gs;
}

// One-token MoE w13 (T = 1): the four epilogue warps (tid 0..127, named barrier 1) take gs
// (dynamic: fl32(amax / 2688) over the token's K elements; static: read; CTA 0 writes a
// dynamic one out), encode the row with the activation quantiser's arithmetic and write its
// codes into all eight rows of the resident atom of every K stage (the atom of stage s is the
// 1 KB at s * 1024; 16-byte chunk c of row r sits at chunk c ^ r) and the row's scale bytes,
// one per 16 elements in K order, into sfa (four per 64-element K step: one 32-bit word).
__device__ float quantize_token_a(const GemmArgs &a, uint8_t *sA, uint8_t *sfa, uint32_t *scratch, int tid) {
  const int64_t K = a.K;
  const uint16_t *x = static_cast<const uint16_t *>(a.qa_x);
  const int warp = tid >> 5, lane = tid & 31;
  float gs;
  if (a.qa_gs_static == nullptr) {
    uint32_t m = 0;
    for (int64_t c = tid; c < K / 8; c += 128) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x) + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) m = max(m, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) scratch[warp] = m;
    named_barrier_sync(1, 128);
    m = max(max(scratch[0], scratch[1]), max(scratch[2], scratch[3]));
    gs = __fdiv_rn(__uint_as_float(m << 16), 2688.0f);
  } else {
    gs = __ldg(a.qa_gs_static);
  }
  if (blockIdx.x == 0 && tid == 0 && a.qa_gs_out != nullptr) *a.qa_gs_out = gs;
  const float six_gs = __fmul_rn(6.0f, gs);
  for (int64_t c = tid; c < K / 16; c += 128) {  // 16-element block c of the row
    const uint4 *src = reinterpret_cast<const uint4 *>(x + c * 16);
    const uint4 p = __ldg(src), q = __ldg(src + 1);
    const uint32_t w[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
    uint32_t codes[2];
    const uint32_t sfb = encode_block16_bf16(w, gs, six_gs, codes);
    const int st = static_cast<int>(c >> 4), j = static_cast<int>(c & 15);
#pragma unroll
    for (int r = 0; r < 8; ++r)
      *reinterpret_cast<uint2 *>(sA + st * 1024 + r * 128 + (((j >> 1) ^ r) * 16) + (j & 1) * 8) =
          make_uint2(codes[0], codes[1]);
    sfa[c] = static_cast<uint8_t>(sfb);
  }
  fence_proxy_async_shared();  // the MMAs read the atoms through the async proxy
  named_barrier_sync(1, 128);
  return gs;
}

// One-token MoE w13: the schedule the routing kernel writes, derived from the token's top-k
// ids by warp 0 (every lane calls this; topk <= 32).  The groups are the distinct valid ids
// in increasing order, each one 32-row tile of as many rows as the id occurs (padded
// segments of 128 rows: group i starts at row 128 i), then the shared group with the one
// token.  Entry i = (group, m tile 0, rows, first row); sched[15].x = the group count.
__device__ void tok1_schedule(const GemmArgs &a, int4 *sched, int lane) {
  int id = lane < a.topk ? __ldg(a.tok1_ids + lane) : -1;
  if (id < 0 || id >= a.tok1_E) id = -1;  // dropped, as the routing kernel drops it
  const unsigned same = __match_any_sync(0xffffffffu, id);
  const bool leader = id >= 0 && __ffs(same) - 1 == lane;
  const unsigned lead = __ballot_sync(0xffffffffu, leader);
  int rank = 0;  // distinct valid ids below this one
  for (unsigned m = lead; m; m &= m - 1) rank += __shfl_sync(0xffffffffu, id, __ffs(m) - 1) < id;
  if (leader) sched[rank] = make_int4(id, 0, __popc(same), kBlockM * rank);
  const int nd = __popc(lead);
  if (lane == 0) {
    if (a.shared_group >= 0) sched[nd] = make_int4(a.shared_group, 0, 1, kBlockM * nd);
    sched[15] = make_int4(nd + (a.shared_group >= 0 ? 1 : 0), 0, 0, 0);
  }
}

template <int kEpi, bool kSmallA, bool kQuantA>
__global__ void __launch_bounds__(Ring<kSmallA, kQuantA, kQuantA && kEpi == static_cast<int>(Epi::kW13)>::kThreads,
                                  (kQuantA && kEpi != static_cast<int>(Epi::kW13)) ? 1 : kCtasPerSm)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmBs,
                      const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  // kQuantA with the W13 epilogue: the one-token MoE w13 (resident token atoms, schedule from ids)
  constexpr bool kTok1 = kQuantA && kEpi == static_cast<int>(Epi::kW13);
  using R = Ring<kSmallA, kQuantA, kTok1>;
  constexpr int S = R::kStagesR;    // stages in the ring
  constexpr int kAB = R::kABytes;   // A slot per stage (kQuantA: per K stage, resident)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = sA + R::kASlots * kAB;
  uint8_t *sSFA = sB + S * kTileBytesB;
  uint8_t *sSFB = sSFA + R::kSfaBytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(sSFB + S * kSfBytesStage);
  uint64_t *empty = full + S;
  uint64_t *tfull = empty + S;
  uint64_t *tempty = tfull + 2;
  uint64_t *sf_ready = tempty + 2;
  uint64_t *drain = sf_ready + S;
  uint64_t *h_full = drain + 1;   // small-A W13: the tile's h is in h_s
  uint64_t *h_empty = drain + 2;  // small-A W13: the four epilogue warps have read h_s
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 3);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  uint32_t *q_scratch = reinterpret_cast<uint32_t *>(tmem_holder + 2);  // kQuantA: 5 words
  float *h_s = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(full) + R::kBarBytes);  // R::kHBytes
  int4 *sched = reinterpret_cast<int4 *>(reinterpret_cast<uint8_t *>(h_s) + R::kHBytes);  // kTok1
  uint8_t *p2_tile = reinterpret_cast<uint8_t *>(sched) + R::kSchedBytes;             // kTok1: h rows, B of the
  uint32_t *p2_sfw = reinterpret_cast<uint32_t *>(p2_tile + 32 * 32);                 // fused w2; their scales
  uint64_t *p2_full = reinterpret_cast<uint64_t *>(p2_sfw + 32);  // kTok1: a slot buffer holds MMA results
  uint64_t *p2_empty = p2_full + 2;                               // kTok1: the epilogue has read a buffer
  // (kTok1) the w2 codes of the fused down projection come through tmA (routed experts)
  // and tmC (the shared expert)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], R::kIssuers);
      mbar_init(&tempty[i], 4);
    }
    mbar_init(drain, R::kIssuers);
    mbar_init(h_full, 1);
    mbar_init(h_empty, 4);
    if constexpr (kTok1) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(&p2_full[i], 1);
        mbar_init(&p2_empty[i], 4);
      }
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_shared();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (args.shared_group >= 0) prefetch_tensormap(&tmBs);
    if (kTok1 && args.p2_acc != nullptr && args.shared_group >= 0) prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, R::kTmemColsR);
    tmem_relinquish();
  }
  if constexpr (kTok1) {
    if (warp == 0) tok1_schedule(args, sched, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Everything above overlaps the previous kernel.  Its outputs (the A operand, the
  // activation scale) are read only after pdl_wait; with early_b the producer first
  // streams the weights of its first stages, which the calling chain wrote earlier.
  // kTok1 reads nothing the previous kernel (the routing) writes: one idle lane waits for it
  // below, so that the next launch (and this grid's completion) still follow it.
  if (!kTok1 && (!args.early_b || threadIdx.x != 0)) {
    pdl_wait();
    pdl_trigger();
  }
  auto entry = [&](int mtg) { return kTok1 ? sched[mtg] : tile_entry(args, mtg); };

  const int n_tiles = (args.N + kBlockN - 1) / kBlockN;  // (a dense linear's N may end mid-tile)
  const int k_steps = args.K / kUmmaK;
  const int k_stages = (k_steps + 3) / 4;
  const int total_mtiles = kTok1 ? sched[15].x
                           : args.counts ? __ldg(args.tile_offsets + args.G)
                                         : args.G * ((args.dense_M + kBlockM - 1) / kBlockM);
  const int total_tiles = total_mtiles * n_tiles;
  // The tiles of a launch cost the same, so the CTAs taking part are trimmed to
  // ceil(tiles / waves): every wave, the last included, is (nearly) full instead of
  // leaving the last fraction of the run to a fraction of the CTAs.  CTAs beyond take none.
  const int waves = (total_tiles + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  const int grid = waves > 0 ? (total_tiles + waves - 1) / waves : static_cast<int>(gridDim.x);
  const int first = static_cast<int>(blockIdx.x) < grid ? static_cast<int>(blockIdx.x) : total_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      const uint64_t pol_stream = policy_evict_first();  // weights of a single-m-tile group: read once
      const uint64_t pol_reuse = policy_evict_normal();  // weights re-read by later m tiles
      const uint64_t pol_a = policy_evict_last();        // activations are re-read per n tile
      // Weight location of (tile, k stage): tensor map, first row, scale bytes.
      auto b_src = [&](const Tile &t, const CUtensorMap *&mb, int &b_row0, const uint8_t *&sfb) {
        const bool sh = t.g == args.shared_group;
        mb = sh ? &tmBs : &tmB;
        b_row0 = (sh ? 0 : t.g * args.N) + t.nt * kBlockN;
        sfb = (sh ? args.b_sf_shared : args.b_sf + static_cast<size_t>(t.g) * args.N * (args.K / 16)) +
              static_cast<size_t>(t.nt) * k_steps * kSfBytesPerKStep;
      };
      // Weights of a group whose other m tiles read them too stay in L2 (evict_normal);
      // the weights of a single-tile group stream with evict_first.
      auto weight_policy = [&](const Tile &t) { return t.multi ? pol_reuse : pol_stream; };
      // Weights of the first stages of this CTA's first tile, before the previous kernel ends.
      int early = 0;
      if (args.early_b) {
        if (first < total_tiles) {
          const Tile t = make_tile(entry(first / n_tiles), first, n_tiles);
          const CUtensorMap *mb;
          int b_row0;
          const uint8_t *sfb;
          b_src(t, mb, b_row0, sfb);
          const uint64_t pol_w = weight_policy(t);
          early = min(S, k_stages);
          for (int s = 0; s < early; ++s) {
            const int kv = min(4, k_steps - 4 * s);
            mbar_expect_tx(&full[s], kTileBytesB + kv * kSfBytesPerKStep);
            tma_load_2d(sB + s * kTileBytesB, mb, 0, (b_row0 / kBlockN * k_stages + s) * kBlockN, &full[s], pol_w);
            bulk_load(sSFB + s * kSfBytesStage, sfb + static_cast<size_t>(s) * kSfBytesStage,
                      kv * kSfBytesPerKStep, &full[s], pol_w);
          }
          // the next stages of the tile into L2, while the previous kernel finishes
          const int l2_end = min(k_stages, early + args.early_l2);
          for (int s = early; s < l2_end; ++s) {
            tma_prefetch_l2_2d(mb, 0, (b_row0 / kBlockN * k_stages + s) * kBlockN);
            bulk_prefetch_l2(sfb + static_cast<size_t>(s) * kSfBytesStage, min(4, k_steps - 4 * s) * kSfBytesPerKStep);
          }
        }
        pdl_wait();
        pdl_trigger();
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // bit s: stage s has a load in flight with parity bit (s+8)
      int n_issued = 0;     // stages issued so far (the first `early` already hold their B)
      bool ok = true;
      int4 next = first < total_tiles ? entry(first / n_tiles) : make_int4(0, 0, 0, 0);
      for (int idx = first; ok && idx < total_tiles; idx += grid) {
        const Tile t = make_tile(next, idx, n_tiles);
        if (idx + grid < total_tiles) next = entry((idx + grid) / n_tiles);
        const CUtensorMap *mb;
        int b_row0;
        const uint8_t *sfb;
        b_src(t, mb, b_row0, sfb);
        const uint64_t pol_w = weight_policy(t);
        const uint8_t *sfa =
            args.a_sf + (static_cast<size_t>(t.a_row0 / kBlockM) * args.a_kc_total +
                         static_cast<size_t>(t.g) * args.a_group_koff) * kSfBytesPerKStep;
        const int a_x0 = t.g * args.a_group_koff * (kUmmaK / 2);  // A byte column of this group
        int nbox = (t.rows + kABoxRows - 1) / kABoxRows;
        if (kSmallA && nbox > 1) {  // the launch promised at most one box per tile
          raise_device_error(args.err, NVFP4_DEVERR_INTERNAL);
          nbox = 1;
        }
        for (int ks = 0; ks < k_stages; ++ks) {
          const int kv = min(4, k_steps - 4 * ks);
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, args.err,
                                 kPipelineTimeoutNs)) {
            ok = false;
            break;
          }
          const bool b_done = n_issued < early;
          // kQuantA: the A boxes and their scales are resident (quantised in this CTA)
          const uint32_t a_bytes = kQuantA ? 0u : nbox * (kABoxRows * kStageK / 2) + kv * kSfBytesPerKStep;
          mbar_arrive_expect_tx(&full[stage], a_bytes + (b_done ? 0 : kTileBytesB + kv * kSfBytesPerKStep));
          if constexpr (!kQuantA) {
            uint8_t *a_dst = sA + stage * kAB;
            for (int b = 0; b < nbox; ++b)
              tma_load_2d(a_dst + b * (kABoxRows * kStageK / 2), &tmA, a_x0 + ks * (kStageK / 2),
                          t.a_row0 + b * kABoxRows, &full[stage], pol_a);
            bulk_load(sSFA + stage * kSfBytesStage, sfa + static_cast<size_t>(ks) * kSfBytesStage,
                      kv * kSfBytesPerKStep, &full[stage], pol_a);
          }
          if (!b_done) {
            // the tile-major weights: block (tile, stage) is 128 rows of 128 bytes, contiguous
            tma_load_2d(sB + stage * kTileBytesB, mb, 0, (b_row0 / kBlockN * k_stages + ks) * kBlockN, &full[stage],
                        pol_w);
            bulk_load(sSFB + stage * kSfBytesStage, sfb + static_cast<size_t>(ks) * kSfBytesStage,
                      kv * kSfBytesPerKStep, &full[stage], pol_w);
          }
          ++n_issued;
          issued = (issued & ~(0x101u << stage)) | (1u << stage) | (phase << (stage + 8));
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if constexpr (kTok1) {
          // The fused down projection of this tile: its h columns 64 nt .. 64 nt + 63 are K step
          // nt of w2; every w2 row tile of the group contributes 128 rows x 32 bytes.
          if (ok && args.p2_acc != nullptr) {
            const int n_rt = args.p2_N / kBlockN;
            const int kst2 = args.p2_K / kUmmaK, ks2 = (kst2 + 3) / 4;
            const bool sh = t.g == args.shared_group;
            const CUtensorMap *m2 = sh ? &tmC : &tmA;
            const int rt0 = sh ? 0 : t.g * n_rt;
            const int slab = t.nt >> 2, x2 = (t.nt & 3) * 32;
            const uint8_t *sf2 = (sh ? args.p2_sf_shared
                                     : args.p2_sf + static_cast<size_t>(t.g) * args.p2_N * (args.p2_K / 16)) +
                                 static_cast<size_t>(t.nt) * kSfBytesPerKStep;
            for (int p = 0; p * kP2RowTiles < n_rt; ++p) {
              const int nq = min(kP2RowTiles, n_rt - p * kP2RowTiles);
              if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, args.err, kPipelineTimeoutNs)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&full[stage], nq * (kP2TileBytes + kSfBytesPerKStep));
              for (int q = 0; q < nq; ++q) {
                const int rt = p * kP2RowTiles + q;
                tma_load_2d(sB + stage * kTileBytesB + q * kP2TileBytes, m2, x2, ((rt0 + rt) * ks2 + slab) * kBlockN,
                            &full[stage], pol_stream);
                bulk_load(sSFB + stage * kSfBytesStage + q * kSfBytesPerKStep,
                          sf2 + static_cast<size_t>(rt) * kst2 * kSfBytesPerKStep, kSfBytesPerKStep, &full[stage],
                          pol_stream);
              }
              issued = (issued & ~(0x101u << stage)) | (1u << stage) | (phase << (stage + 8));
              if (++stage == S) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA leaves (this wait
        // ignores the abort flag; it is bounded by its own 100 ms limit)
        volatile int never = 0;
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s))
            mbar_wait_bounded(&full[s], (issued >> (s + 8)) & 1u, &never, nullptr, 100000000ull);
      }
    } else if (kTok1 && lane == 1) {
      // The routing kernel has finished once this returns; its schedule must be the one
      // this CTA derived from the ids.
      pdl_wait();
      pdl_trigger();
      bool same = __ldg(args.tile_offsets + args.G) == total_mtiles;
      for (int i = 0; same && i < total_mtiles; ++i) {
        const int4 r = __ldg(args.tile_table + i), e = sched[i];
        same = r.x == e.x && r.y == e.y && r.z == e.z && r.w == e.w;
      }
      if (!same) raise_device_error(args.err, NVFP4_DEVERR_INTERNAL);
    }
  } else if (warp == 1 || (R::kIssuers > 1 && warp >= 6)) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer(s)
      // Issuer iss takes the K stages ks with ks % kIssuers == iss into its own accumulator.
      const int iss = warp == 1 ? 0 : warp - 5;
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      const uint32_t sA0 = smem_u32(sA), sB0 = smem_u32(sB);
      int p2n = 0;  // kTok1: down-projection stages so far (slot buffer p2n & 1)
      for (int idx = first; ok && idx < total_tiles; idx += grid, ++it) {
        const int acc = kAccBufs == 2 ? (it & 1) : 0;
        const uint32_t acc_phase = kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
        if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, abort_flag, args.err,
                               kPipelineTimeoutNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (R::kSwapAB ? iss * kABoxRows : acc * kBlockN);
        for (int ks = 0; ks < k_stages; ++ks) {
          const int kv = min(4, k_steps - 4 * ks);
          if (R::kIssuers > 1 && ks % R::kIssuers != iss) {  // another issuer's stage
            if (++stage == S) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          if (!mbar_wait_bounded(&full[stage], phase, abort_flag, args.err,
                                 kPipelineTimeoutNs)) {
            ok = false;
            break;
          }
          // the stage's scales are in TMEM once the four epilogue warps arrived
          if (!mbar_wait_bounded(&sf_ready[stage], phase, abort_flag, args.err,
                                 kPipelineTimeoutNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_col = tmem_base + R::kAccColsR + stage * kTmemSfCols;
          const uint64_t adesc = smem_desc(sA0 + (kQuantA ? ks : stage) * kAB, 16, 1024, 2);
          const uint64_t bdesc = smem_desc(sB0 + stage * kTileBytesB, 16, 1024, 2);
          for (int j = 0; j < kv; ++j) {
            // +32 bytes of K per step inside the 128-byte swizzle row (descriptor units of 16 B)
            if constexpr (R::kSwapAB)  // weights x tokens: the scale blocks swap places too
              tc_mma_nvf4(d_tmem, bdesc + 2 * j, adesc + 2 * j, kIdescSwap, sf_col + 16 + j * 4, sf_col + j * 4,
                          ks != iss || j != 0);
            else
              tc_mma_nvf4(d_tmem, adesc + 2 * j, bdesc + 2 * j, kIdesc, sf_col + j * 4, sf_col + 16 + j * 4,
                          ks != 0 || j != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        if constexpr (kTok1) {
          if (args.p2_acc != nullptr) {
            const int n_rt = args.p2_N / kBlockN;
            const uint64_t bdesc2 = smem_desc(smem_u32(p2_tile), 16, 256, 6);
            // the down projection takes the accumulator columns as one more use: its slot
            // buffers overlap the w13 accumulator, which the W13 epilogue must have read
            ++it;
            ok = mbar_wait_bounded(&tempty[0], (it & 1) ^ 1, abort_flag, args.err, kPipelineTimeoutNs);
            for (int p = 0; ok && p * kP2RowTiles < n_rt; ++p, ++p2n) {
              const int nq = min(kP2RowTiles, n_rt - p * kP2RowTiles);
              const int b = p2n & 1;
              if (!mbar_wait_bounded(&p2_empty[b], ((p2n >> 1) & 1) ^ 1, abort_flag, args.err, kPipelineTimeoutNs) ||
                  !mbar_wait_bounded(&full[stage], phase, abort_flag, args.err, kPipelineTimeoutNs) ||
                  !mbar_wait_bounded(&sf_ready[stage], phase, abort_flag, args.err, kPipelineTimeoutNs)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t sf_col = tmem_base + R::kAccColsR + stage * kTmemSfCols;
              for (int q = 0; q < nq; ++q)
                tc_mma_nvf4(tmem_base + b * (kP2RowTiles * kP2N) + q * kP2N,
                            smem_desc(sB0 + stage * kTileBytesB + q * kP2TileBytes, 16, 256, 6), bdesc2, kIdescP2,
                            sf_col + 4 * q, sf_col + 16, 0u);
              tc_commit(&empty[stage]);
              tc_commit(&p2_full[b]);
              if (++stage == S) {
                stage = 0;
                phase ^= 1;
              }
            }
            if (!ok) break;
          }
        }
      }
      // every MMA this thread issued has completed before TMEM is released
      volatile int never = 0;
      tc_commit(drain);
      mbar_wait_bounded(drain, 0, &never, nullptr, 100000000ull);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes [32*quarter, 32*quarter + 32)
    const int m = quarter * 32 + lane;
    float gs_scalar = 0.f;
    if constexpr (kTok1) {
      gs_scalar = quantize_token_a(args, sA, sSFA, q_scratch, threadIdx.x - 2 * 32);
    } else if constexpr (kQuantA) {
      // one tile per CTA (the launch guarantees it): its group's K columns
      const int g = first < total_tiles ? entry(first / n_tiles).x : 0;
      gs_scalar = quantize_resident_a(args, g, sA, sSFA, q_scratch, threadIdx.x - 2 * 32);
    } else if constexpr (kEpi != static_cast<int>(Epi::kW2)) {
      gs_scalar = __ldg(args.gs_a);
    }
    // Scale staging.  Each K step's 512-byte swizzled block holds, at 16 r + 4 c, the
    // four UE4M3 scales (64 K) of operand row 32 c + r.  Every 32-lane quarter of TMEM
    // receives the same copy of the block: lane 32 q + r, column (scale address + c)
    // holds the word of row 32 c + r, the arrangement the MMA reads scales from.  This
    // warp writes its own quarter; lane r loads the 16 bytes at 16 r.
    const uint32_t sf_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + R::kAccColsR;
    const int sf_off = lane * 16;
    int sstage = 0;
    uint32_t sphase = 0;
    int it = 0;   // uses of the accumulator columns (a tile, then kTok1's down-projection stages)
    int ht = 0;   // tiles through h_s (small-A W13)
    bool p2_ordered = false;  // kTok1: the routing kernel (which zeroes the fp32 output) has finished
    int p2n = 0;              // kTok1: down-projection stages so far (slot buffer p2n & 1)
    int4 next = first < total_tiles ? entry(first / n_tiles) : make_int4(0, 0, 0, 0);
    for (int idx = first; idx < total_tiles; idx += grid, ++it) {
      const Tile t = make_tile(next, idx, n_tiles);
      if (idx + grid < total_tiles) next = entry((idx + grid) / n_tiles);
      const int acc = kAccBufs == 2 ? (it & 1) : 0;
      const uint32_t acc_phase = kAccBufs == 2 ? ((it >> 1) & 1) : (it & 1);
      // Per-tile epilogue scalars, loaded before this tile's main loop so that their
      // latency is hidden behind it.
      const bool sh = t.g == args.shared_group;
      const float ws2 = sh ? __ldg(args.ws2_shared) : __ldg(args.ws2 + t.g);
      float g_aux = 0.f;  // W13: static scale of h; W2: global scale of the w2 input
      int seg_base = 0;   // W2: first sorted entry of the group
      if constexpr (kEpi == static_cast<int>(Epi::kW13)) g_aux = __ldg(args.gs_out + t.g);
      if constexpr (kEpi == static_cast<int>(Epi::kW2)) {
        g_aux = __ldg(args.gs_a + t.g);
        if (!sh) seg_base = __ldg(args.offsets + t.g);
      }
      const bool row_ok = m < t.rows;
      // MoE small-A tiles are 32 rows high and may start 32 j rows into a scale block
      // (dense and uniform-group tiles start at row 0)
      constexpr bool kRotA = kSmallA && !kTok1 && kEpi != static_cast<int>(Epi::kLinear);
      const int sfa_rot = kRotA ? (t.a_row0 / kABoxRows) & 3 : 0;
      bool ok = true;
      for (int ks = 0; ks < k_stages; ++ks) {
        const int kv = min(4, k_steps - 4 * ks);
        ok = mbar_wait_bounded(&full[sstage], sphase, abort_flag, args.err, kPipelineTimeoutNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const uint8_t *pa = sSFA + (kQuantA ? ks : sstage) * kSfBytesStage + sf_off;
        const uint8_t *pb = sSFB + sstage * kSfBytesStage + sf_off;
        uint32_t ra[16], rb[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // kTok1: A rows 0..7 are the token (its scale word of the K step), the rest zero;
          // kQuantA: the scale word of row `lane` (rows 32.. of the block are not read: N <= 32)
          const uint4 wa = kTok1 ? make_uint4(j < kv && lane < 8 ? reinterpret_cast<const uint32_t *>(sSFA)[4 * ks + j]
                                                                 : 0u, 0u, 0u, 0u)
                           : kQuantA ? make_uint4(j < kv ? reinterpret_cast<const uint32_t *>(sSFA)[(4 * ks + j) * 32 + lane]
                                                         : 0u, 0u, 0u, 0u)
                           : j < kv ? *reinterpret_cast<const uint4 *>(pa + j * kSfBytesPerKStep)
                                    : make_uint4(0u, 0u, 0u, 0u);
          const uint4 wb = j < kv ? *reinterpret_cast<const uint4 *>(pb + j * kSfBytesPerKStep)
                                  : make_uint4(0u, 0u, 0u, 0u);
          ra[4 * j] = wa.x, ra[4 * j + 1] = wa.y, ra[4 * j + 2] = wa.z, ra[4 * j + 3] = wa.w;
          rb[4 * j] = wb.x, rb[4 * j + 1] = wb.y, rb[4 * j + 2] = wb.z, rb[4 * j + 3] = wb.w;
        }
        // Warp-uniform and taken by few tiles: only a group of more than 32 rows (the shared
        // expert above 32 tokens, a popular expert, an expert listed twice by a token) has
        // small-A tiles that do not start a scale block.
        if (kRotA && __builtin_expect(sfa_rot != 0, 0)) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 v = rotate_words(make_uint4(ra[4 * j], ra[4 * j + 1], ra[4 * j + 2], ra[4 * j + 3]), sfa_rot);
            ra[4 * j] = v.x, ra[4 * j + 1] = v.y, ra[4 * j + 2] = v.z, ra[4 * j + 3] = v.w;
          }
        }
        tmem_st16(sf_lane + sstage * kTmemSfCols, ra);
        tmem_st16(sf_lane + sstage * kTmemSfCols + 16, rb);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[sstage]);
        if (++sstage == S) {
          sstage = 0;
          sphase ^= 1;
        }
      }
      if (!ok) break;
      // W2: token and routing weight of this thread's row, while the last MMAs run
      float w2_scale = 0.f;
      int64_t w2_tok = 0;
      if constexpr (kEpi == static_cast<int>(Epi::kW2)) {
        if (row_ok) {
          const int seg_row = t.mt * (kSmallA ? kABoxRows : kBlockM) + m;
          float w = 1.f;
          if (sh) {
            w2_tok = seg_row;
          } else {
            const int f = __ldg(args.sorted_idx + seg_base + seg_row);
            w2_tok = f / args.topk;
            w = __ldg(args.topk_w + f);
          }
          w2_scale = g_aux * ws2 * w;
        }
      }
      ok = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, args.err, kPipelineTimeoutNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * kBlockN);
      // A warp whose 32 accumulator rows are all padding (a group's last m tile) has
      // nothing to read or store; it only releases the accumulator.
      const bool warp_live = R::kSwapAB || quarter * 32 < t.rows;
      // Each warp hands its accumulator lanes back to the MMA as soon as it has read
      // them, so the next tile's MMAs overlap this tile's global stores.
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      };

      constexpr bool kTeamH = kSmallA && kEpi == static_cast<int>(Epi::kW13);
      if constexpr (kTeamH) {
        // The tile's rows sit in lane quarter 0: its warp computes h into h_s and hands
        // the accumulator back; then all four warps re-quantise h, four lanes per block.
        const float gs2 = g_aux;
        const float six_gs2 = __fmul_rn(6.0f, gs2);
        const int I = args.out_ld * 2;
        if (quarter == 0) {
          ok = mbar_wait_bounded(h_empty, (ht & 1) ^ 1, abort_flag, args.err, kPipelineTimeoutNs);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const float alpha = gs_scalar * ws2;
          float *hrow = h_s + m * kHRowFloats;
          if constexpr (kTok1) {
            // Every row of a one-token tile is the token: lane 0's accumulator row (gate columns
            // 0..63, up columns 64..127) goes through shared memory (rows 1.. of h_s) to the 32
            // lanes, two h columns each, into row 0 of h_s.
            float *raw = h_s + kHRowFloats;
#pragma unroll
            for (int c0 = 0; c0 < 8; c0 += 4) {
              uint32_t r[4][16];
#pragma unroll
              for (int q = 0; q < 4; ++q) tmem_ld16(tbase + (c0 + q) * 16, r[q]);
              tmem_ld_wait();
              if (c0 == 4) release();
              if (lane == 0) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    reinterpret_cast<float4 *>(raw + (c0 + q) * 16)[i] =
                        make_float4(__uint_as_float(r[q][4 * i]), __uint_as_float(r[q][4 * i + 1]),
                                    __uint_as_float(r[q][4 * i + 2]), __uint_as_float(r[q][4 * i + 3]));
              }
            }
            __syncwarp();
            const float2 g2 = *reinterpret_cast<const float2 *>(raw + 2 * lane);
            const float2 u2 = *reinterpret_cast<const float2 *>(raw + kBlockN / 2 + 2 * lane);
            const float2 hh = make_float2(silu_mul(g2.x * alpha, u2.x * alpha), silu_mul(g2.y * alpha, u2.y * alpha));
            __syncwarp();
            *reinterpret_cast<float2 *>(h_s + 2 * lane) = hh;
            if (args.h_debug != nullptr)
              for (int r = 0; r < t.rows; ++r)
                *reinterpret_cast<float2 *>(args.h_debug + (t.a_row0 + r) * I + t.nt * 64 + 2 * lane) = hh;
          }
#pragma unroll
          for (int c = 0; c < (kTok1 ? 0 : 4); ++c) {
            uint32_t rg[16], ru[16];
            tmem_ld16(tbase + c * 16, rg);
            tmem_ld16(tbase + kBlockN / 2 + c * 16, ru);
            tmem_ld_wait();
            if (c == 3) release();
            float h[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              h[i] = silu_mul(__uint_as_float(rg[i]) * alpha, __uint_as_float(ru[i]) * alpha);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<float4 *>(hrow + c * 16)[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
            if (args.h_debug != nullptr && row_ok) {
              float4 *hd = reinterpret_cast<float4 *>(args.h_debug + (t.a_row0 + m) * I + t.nt * 64 + c * 16);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                hd[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(h_full);
        } else {
          release();
        }
        ok = mbar_wait_bounded(h_full, ht & 1, abort_flag, args.err, kPipelineTimeoutNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        // Thread e of the 128 takes the 16-bit piece j = e % 16 (elements 4j..4j+3) of row
        // r0 + e / 16: the four lanes of a block share its amax, sixteen lanes make a row's
        // 32 code bytes and its scale word.
        const int e = static_cast<int>(threadIdx.x) - 64;
        const int j = e & 15;
        uint8_t *out = static_cast<uint8_t *>(args.out);
        const int trows = min(t.rows, kABoxRows);  // a tile breaking the small-A promise raised an error
        for (int r0 = 0; r0 < trows; r0 += 8) {
          const int row = r0 + (e >> 4);
          const bool act = row < trows;
          // (kTok1: every row is the token, whose h is row 0)
          const float4 v = act ? *reinterpret_cast<const float4 *>(h_s + (kTok1 ? 0 : row) * kHRowFloats + 4 * j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          uint32_t sfb;
          const uint32_t bits = encode_block16_x4(v, gs2, six_gs2, &sfb);
          const uint32_t hi = __shfl_down_sync(0xffffffffu, bits, 1);
          uint32_t sfw = sfb << (8 * (j >> 2));
          sfw |= __shfl_xor_sync(0xffffffffu, sfw, 4);
          sfw |= __shfl_xor_sync(0xffffffffu, sfw, 8);
          if (act) {
            const int64_t p = t.a_row0 + row;
            if ((j & 1) == 0)
              *reinterpret_cast<uint32_t *>(out + p * args.out_ld + t.nt * 32 + 2 * j) = bits | (hi << 16);
            if (j == 0) *reinterpret_cast<uint32_t *>(args.out_sf + sf_word_offset(p, t.nt, I / 64)) = sfw;
            if constexpr (kTok1) {
              // the same row as the fused down projection's B operand: 32 bytes, 32-byte swizzle
              // (16-byte chunk c of row r at chunk c ^ ((r >> 2) & 1))
              if ((j & 1) == 0)
                *reinterpret_cast<uint32_t *>(p2_tile + row * 32 + ((((j >> 3) ^ (row >> 2)) & 1) << 4) + ((2 * j) & 15)) =
                    bits | (hi << 16);
              if (j == 0) p2_sfw[row] = sfw;
            }
          }
        }
        if constexpr (kTok1) fence_proxy_async_shared();  // the MMAs read p2_tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(h_empty);
        if constexpr (kTok1) {
          // every warp's rows of p2_tile and p2_sfw are written once this tile's h_empty phase completes
          if (args.p2_acc != nullptr) {
            ok = mbar_wait_bounded(h_empty, ht & 1, abort_flag, args.err, kPipelineTimeoutNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
          }
        }
        ++ht;
        if constexpr (kTok1) {
          // The fused down projection of the tile (see the producer): stage the w2 scale blocks
          // (A) and the h rows' scales (B), then add the MMA results of the token's column.
          if (args.p2_acc != nullptr) {
            if (!p2_ordered) {
              pdl_wait();
              p2_ordered = true;
            }
            const int n_rt = args.p2_N / kBlockN;
            float wsum = 1.f;  // the group's routing weight: the shared group takes the token once
            if (!sh) {
              wsum = 0.f;
              for (int f = 0; f < args.topk; ++f)
                if (__ldg(args.tok1_ids + f) == t.g) wsum += __ldg(args.p2_topk_w + f);
            }
            const float alpha2 = gs2 * (sh ? __ldg(args.p2_ws2_shared) : __ldg(args.p2_ws2 + t.g)) * wsum;
            const uint32_t hq_sfw = lane < trows ? p2_sfw[lane] : 0u;
            const uint64_t pol_y = policy_evict_last();
            ++it;  // the down projection's use of the accumulator columns (see the MMA)
            const int P = (n_rt + kP2RowTiles - 1) / kP2RowTiles;
            // stage p's scales: the w2 scale blocks (A of the MMA, four columns each) and the
            // h rows' scale words (B, lanes 0..15 of column 16)
            auto stage_sf = [&](int p) -> bool {
              const int nq = min(kP2RowTiles, n_rt - p * kP2RowTiles);
              bool fine = mbar_wait_bounded(&full[sstage], sphase, abort_flag, args.err, kPipelineTimeoutNs);
              fine = __all_sync(0xffffffffu, fine);
              if (!fine) return false;
              uint32_t ra[16], rb[16];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 wa = q < nq ? *reinterpret_cast<const uint4 *>(sSFB + sstage * kSfBytesStage +
                                                                          q * kSfBytesPerKStep + sf_off)
                                        : make_uint4(0u, 0u, 0u, 0u);
                ra[4 * q] = wa.x, ra[4 * q + 1] = wa.y, ra[4 * q + 2] = wa.z, ra[4 * q + 3] = wa.w;
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) rb[i] = 0u;
              rb[0] = hq_sfw;
              tmem_st16(sf_lane + sstage * kTmemSfCols, ra);
              tmem_st16(sf_lane + sstage * kTmemSfCols + 16, rb);
              tmem_st_wait();
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&sf_ready[sstage]);
              if (++sstage == S) {
                sstage = 0;
                sphase ^= 1;
              }
              return true;
            };
            ok = stage_sf(0) && (P < 2 || stage_sf(1));
            const uint32_t tq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            for (int p = 0; ok && p < P; ++p, ++p2n) {
              const int nq = min(kP2RowTiles, n_rt - p * kP2RowTiles);
              const int b = p2n & 1;
              ok = mbar_wait_bounded(&p2_full[b], (p2n >> 1) & 1, abort_flag, args.err, kPipelineTimeoutNs);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
              tc_fence_after();
              uint32_t v[kP2RowTiles];
#pragma unroll
              for (int q = 0; q < kP2RowTiles; ++q)
                v[q] = q < nq ? tmem_ld1(tq + b * (kP2RowTiles * kP2N) + q * kP2N) : 0u;
              tmem_ld_wait();
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&p2_empty[b]);
              // w2 row 32 quarter + lane of row tile 4 p + q is output column 128 (4 p + q) + 32 quarter + lane
#pragma unroll
              for (int q = 0; q < kP2RowTiles; ++q) {
                if (q < nq) {
                  const float y0 = __uint_as_float(v[q]) * alpha2;
                  const float y1 = __shfl_down_sync(0xffffffffu, y0, 1);
                  const float y2 = __shfl_down_sync(0xffffffffu, y0, 2);
                  const float y3 = __shfl_down_sync(0xffffffffu, y0, 3);
                  if ((lane & 3) == 0)
                    red_add_v4(reinterpret_cast<float4 *>(args.p2_acc + (p * kP2RowTiles + q) * kBlockN + quarter * 32 +
                                                          lane),
                               y0, y1, y2, y3, pol_y);
                }
              }
              if (p + 2 < P) ok = stage_sf(p + 2);
            }
            if (!ok) break;
            // the accumulator columns are free for the next tile's w13
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[0]);
          }
        }
      } else if (!warp_live) {
        release();
      } else if constexpr (kEpi == static_cast<int>(Epi::kLinear) && R::kSwapAB) {
        // accumulator lane m is output feature 128 nt + m, column r token a_row0 + r; the
        // issuers' accumulators (as many as there are K stages, up to kIssuers) add up
        const float alpha = gs_scalar * ws2;
        const int nacc = min(R::kIssuers, k_stages);
        const int64_t ld = args.out_ld;
        __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(args.out) + static_cast<int64_t>(t.a_row0) * ld +
                           static_cast<int64_t>(t.g) * args.out_group_cols + t.nt * kBlockN + m;
        // features past N (a dense linear's last tile when N % 128 != 0) are padding
        const bool col_ok = t.nt * kBlockN + m < args.out_group_cols;
        if (t.rows <= 0) release();
#pragma unroll 1
        for (int c0 = 0; c0 < t.rows; c0 += 16) {
          uint32_t r[R::kIssuers][16];
#pragma unroll
          for (int i = 0; i < R::kIssuers; ++i)
            if (i < nacc) tmem_ld16(tbase + i * kABoxRows + c0, r[i]);
          tmem_ld_wait();
          if (c0 + 16 >= t.rows) release();
          float v[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = __uint_as_float(r[0][q]);
#pragma unroll
          for (int i = 1; i < R::kIssuers; ++i)
            if (i < nacc)
#pragma unroll
              for (int q = 0; q < 16; ++q) v[q] += __uint_as_float(r[i][q]);
          if (col_ok)
#pragma unroll
            for (int q = 0; q < 16; ++q)
              if (c0 + q < t.rows) y[(c0 + q) * ld] = __float2bfloat16_rn(v[q] * alpha);
        }
      } else if constexpr (kEpi == static_cast<int>(Epi::kLinear)) {
        const float alpha = gs_scalar * ws2;
        const bool out32 = (reinterpret_cast<uintptr_t>(args.out) & 31u) == 0;
        const int64_t row = t.a_row0 + m;
        __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(args.out) +
                           row * static_cast<int64_t>(args.out_ld) +
                           static_cast<int64_t>(t.g) * args.out_group_cols + t.nt * kBlockN;
        const int n_chunks = min(kBlockN, args.out_group_cols - t.nt * kBlockN) / 16;  // 16-column chunks left of N
        // four TMEM loads in flight per wait
#pragma unroll 1
        for (int c0 = 0; c0 < kBlockN / 16; c0 += 4) {
          uint32_t r[4][16];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld16(tbase + (c0 + q) * 16, r[q]);
          tmem_ld_wait();
          if (c0 + 4 == kBlockN / 16) release();
          if (row_ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int c = c0 + q;
              if (c >= n_chunks) break;  // a dense linear's last tile may end at N % 128 != 0
              uint32_t packed[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const __nv_bfloat162 v = __floats2bfloat162_rn(
                    __uint_as_float(r[q][2 * i]) * alpha, __uint_as_float(r[q][2 * i + 1]) * alpha);
                packed[i] = *reinterpret_cast<const uint32_t *>(&v);
              }
              // 32 bytes per row and chunk: one 256-bit store when the output is 32-byte
              // aligned (row strides and column offsets are multiples of 32 bytes)
              if (out32) {
                st_global_v8(y + c * 16, packed);
              } else {
                uint4 *dst = reinterpret_cast<uint4 *>(y + c * 16);
                dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
              }
            }
          }
        }
      } else if constexpr (kEpi == static_cast<int>(Epi::kW13)) {
        const float alpha = gs_scalar * ws2;
        const float gs2 = g_aux;
        const float six_gs2 = __fmul_rn(6.0f, gs2);
        const int64_t p = t.a_row0 + m;
        const int I = args.out_ld * 2;
        // h of this thread's row, one 16-column block at a time (encoded at once, so that one
        // block of h is live); the accumulator is handed back once it has been read
        uint32_t codes[8];
        uint32_t sfw = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rg[16], ru[16];
          tmem_ld16(tbase + c * 16, rg);
          tmem_ld16(tbase + kBlockN / 2 + c * 16, ru);
          tmem_ld_wait();
          if (c == 3) release();
          float h[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            h[i] = silu_mul(__uint_as_float(rg[i]) * alpha, __uint_as_float(ru[i]) * alpha);
          if (args.h_debug != nullptr && row_ok) {
            float4 *hd = reinterpret_cast<float4 *>(args.h_debug + p * I + t.nt * 64 + c * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i) hd[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
          }
          uint32_t cw[2];
          const uint32_t sfb = encode_block16(h, gs2, six_gs2, cw);
          codes[2 * c] = cw[0];
          codes[2 * c + 1] = cw[1];
          sfw |= sfb << (8 * c);
        }
        if (row_ok) {
          // 32 code bytes of this row and tile; the workspace is 256-byte aligned and
          // rows are I/2 (a multiple of 32) bytes apart
          st_global_v8(static_cast<uint8_t *>(args.out) + p * args.out_ld + t.nt * 32, codes);
          *reinterpret_cast<uint32_t *>(args.out_sf + sf_word_offset(p, t.nt, I / 64)) = sfw;
        }
      } else {  // kW2
        const float scale = w2_scale;
        const int64_t tok = w2_tok;
        // the accumulator rows stay in L2 between the k + 1 contributions to a token while
        // the weights stream past with evict_first
        const uint64_t pol_y = policy_evict_last();
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(args.out) +
                                                 tok * args.out_ld + t.nt * kBlockN);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t r[4][16];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld16(tbase + h * 64 + q * 16, r[q]);
          tmem_ld_wait();
          if (h == 1) release();
          if (row_ok) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                red_add_v4(dst + h * 16 + q * 4 + i, __uint_as_float(r[q][4 * i]) * scale,
                           __uint_as_float(r[q][4 * i + 1]) * scale, __uint_as_float(r[q][4 * i + 2]) * scale,
                           __uint_as_float(r[q][4 * i + 3]) * scale, pol_y);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, R::kTmemColsR);

}

// Bounded-wait probe: one thread waits on a barrier that never completes.
__global__ void wait_timeout_probe_kernel(uint64_t timeout_ns, uint32_t *err) {
  __shared__ uint64_t bar;
  pdl_wait();
  pdl_trigger();
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool done = mbar_wait_bounded(&bar, 0, &abort_flag, err, timeout_ns);
    if (done) raise_device_error(err, 0x80000000u);  // impossible: nothing arrives
  }
}

template <int kEpi, bool kSmallA, bool kQuantA = false>
cudaError_t launch_gemm_t(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tbs,
                          const GemmArgs &args, int grid, bool one_per_sm, cudaStream_t s,
                          const CUtensorMap *tc = nullptr) {
  using R = Ring<kSmallA, kQuantA, kQuantA && kEpi == static_cast<int>(Epi::kW13)>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(nvfp4_gemm_kernel<kEpi, kSmallA, kQuantA>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(R::kSmemSolo));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  // A grid no larger than the SM count asks for enough shared memory to keep one CTA per
  // SM, so its tiles spread over as many SMs as there are tiles.
  return launch_pdl(nvfp4_gemm_kernel<kEpi, kSmallA, kQuantA>, dim3(grid), dim3(R::kThreads),
                    one_per_sm ? R::kSmemSolo : R::kSmem, s, ta, tb, tbs, tc ? *tc : tb, args);
}

template <int kEpi>
cudaError_t launch_gemm_e(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tbs,
                          const GemmArgs &args, int grid, bool one_per_sm, bool small_a, cudaStream_t s) {
  return small_a ? launch_gemm_t<kEpi, true>(ta, tb, tbs, args, grid, one_per_sm, s)
                 : launch_gemm_t<kEpi, false>(ta, tb, tbs, args, grid, one_per_sm, s);
}

}  // namespace

cudaError_t launch_gemm(Epi epi, const CUtensorMap &ta, const CUtensorMap &tb,
                        const CUtensorMap &tbs, const GemmArgs &args, int grid, bool one_per_sm,
                        bool small_a, cudaStream_t s) {
  switch (epi) {
    case Epi::kLinear:
      return launch_gemm_e<static_cast<int>(Epi::kLinear)>(ta, tb, tbs, args, grid, one_per_sm, small_a, s);
    case Epi::kW13:
      return launch_gemm_e<static_cast<int>(Epi::kW13)>(ta, tb, tbs, args, grid, one_per_sm, small_a, s);
    case Epi::kW2:
      return launch_gemm_e<static_cast<int>(Epi::kW2)>(ta, tb, tbs, args, grid, one_per_sm, small_a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_quant_a(const CUtensorMap &tb, const GemmArgs &args, int grid, cudaStream_t s) {
  return launch_gemm_t<static_cast<int>(Epi::kLinear), true, true>(tb, tb, tb, args, grid, true, s);
}

cudaError_t launch_gemm_tok1(const CUtensorMap &tb, const CUtensorMap &tbs, const CUtensorMap &t2,
                             const CUtensorMap &t2s, const GemmArgs &args, int grid, cudaStream_t s) {
  return launch_gemm_t<static_cast<int>(Epi::kW13), true, true>(t2, tb, tbs, args, grid, false, s, &t2s);
}

cudaError_t launch_wait_timeout_probe(uint32_t timeout_us, uint32_t *err, cudaStream_t s) {
  wait_timeout_probe_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(timeout_us) * 1000ull, err);
  return cudaGetLastError();
}

}  // namespace nvfp4
