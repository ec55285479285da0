// Router gate: the NVFP4 gate weight dequantised to bf16, round-tripped through FP8-E4M3 with
// one per-tensor scale s = amax / 448 (prepare, once), then per call logits = x @ wg^T on the
// tensor cores (tcgen05.mma kind::f16: bf16 operands staged by TMA, fp32 accumulators in
// TMEM; 128-token x 128-expert tiles split over K so that a decode or chunk-sized batch still
// spreads over the SMs), a softmax over the experts and the top-k with weights renormalised
// over the k chosen.  The K splits write fp32 partial logits; the softmax kernel sums them in
// a fixed order, so the logits do not depend on the order in which the splits finish.
#include "common.cuh"

namespace nvfp4 {

namespace {

constexpr int kPrepThreads = 256;

// bf16 value of one dequantised NVFP4 weight: bf16(fl32(fl32(e2m1 * e4m3) * ws2))
__device__ __forceinline__ float nvfp4_weight_bf16(uint32_t code, float scale, float ws2) {
  const uint32_t mag = code & 7u;
  // E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}: subnormal 0.5 * m below code 2, else 2^(e-1) * (1 + m/2)
  const float e2m1 = mag < 2 ? 0.5f * static_cast<float>(mag)
                             : static_cast<float>(1u << ((mag >> 1) - 1)) * ((mag & 1u) ? 1.5f : 1.0f);
  const float v = __fmul_rn(__fmul_rn(e2m1, scale), ws2);
  return __bfloat162float(__float2bfloat16_rn((code & 8u) ? -v : v));
}

// Sixteen weights of one scale block: codes (8 bytes) and the block's E4M3 scale.
__device__ __forceinline__ void load_block(const uint8_t *w, const uint8_t *sf, int64_t blk, float ws2,
                                           float (&v)[16]) {
  const uint2 c = __ldg(reinterpret_cast<const uint2 *>(w) + blk);
  const float scale = ue4m3_to_f32(__ldg(sf + blk));
  const uint32_t cw[2] = {c.x, c.y};
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = nvfp4_weight_bf16((cw[i >> 3] >> ((i & 7) * 4)) & 15u, scale, ws2);
}

__global__ void __launch_bounds__(kPrepThreads) router_amax_kernel(const uint8_t *__restrict__ w,
                                                                  const uint8_t *__restrict__ sf,
                                                                  const float *__restrict__ ws2p, int64_t nblocks,
                                                                  uint32_t *__restrict__ partials) {
  __shared__ uint32_t red[32];
  pdl_wait();
  pdl_trigger();
  const float ws2 = __ldg(ws2p);
  uint32_t m = 0;
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks;
       b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float v[16];
    load_block(w, sf, b, ws2, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) m = max(m, (__float_as_uint(v[i]) >> 16) & 0x7FFFu);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) m = max(m, red[i]);
    partials[blockIdx.x] = m;
  }
}

__global__ void __launch_bounds__(kPrepThreads) router_qdq_kernel(const uint8_t *__restrict__ w,
                                                                 const uint8_t *__restrict__ sf,
                                                                 const float *__restrict__ ws2p, int64_t nblocks,
                                                                 const uint32_t *__restrict__ partials, int nparts,
                                                                 uint16_t *__restrict__ wg) {
  __shared__ uint32_t red[32];
  pdl_wait();
  pdl_trigger();
  uint32_t m = 0;
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) m = max(m, partials[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  const float s = __fdiv_rn(__uint_as_float(red[0] << 16), 448.0f);
  const float r = __frcp_rn(s);
  const float ws2 = __ldg(ws2p);
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks;
       b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float v[16];
    load_block(w, sf, b, ws2, v);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float d[2] = {0.f, 0.f};
      if (s != 0.f) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t q = static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fmul_rn(v[i + h], r), __NV_SATFINITE, __NV_E4M3));
          const float mag = __fmul_rn(ue4m3_to_f32(q & 0x7Fu), s);
          d[h] = (q & 0x80u) ? -mag : mag;
        }
      }
      const __nv_bfloat162 p = __floats2bfloat162_rn(d[0], d[1]);
      o[i >> 1] = *reinterpret_cast<const uint32_t *>(&p);
    }
    uint4 *dst = reinterpret_cast<uint4 *>(wg + b * 16);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// ---------------------------------------------------------------- logits on the tensor cores

constexpr int kRtTile = 128;            // tokens (MMA M) and experts (MMA N) per tile
constexpr int kRtStageK = 64;           // bf16 elements of K per stage: 128 bytes per row
constexpr int kRtStages = 4;
constexpr int kRtBox = kRtTile * kRtStageK * 2;  // 16 KiB per operand and stage
constexpr int kRtThreads = 192;         // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr size_t kRtSmem = 1024 + 2 * kRtStages * kRtBox + 128;
// bf16 x bf16 -> fp32, K-major A and B, M = 128, N = 128
constexpr uint32_t kRtIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t(kRtTile) >> 3) << 17) |
                              ((uint32_t(kRtTile) >> 4) << 24);

// D(tmem, fp32) (+)= A(smem, bf16) * B(smem, bf16)^T, M = 128, N = 128, K = 16.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One CTA per (token tile, expert tile, K split): partial[split][t][e] = sum over the split's
// K range of x[t][k] * wg[e][k] (fp32 from exact bf16 products), for t < T and e < E.  A
// split with an empty K range writes zeros.
__global__ void __launch_bounds__(kRtThreads, 1)
    router_logits_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                            int T, int E, int H, int splits, int stages_per_split, float *__restrict__ partial,
                            uint32_t *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = sA + kRtStages * kRtBox;
  uint64_t *full = reinterpret_cast<uint64_t *>(sB + kRtStages * kRtBox);
  uint64_t *empty = full + kRtStages;
  uint64_t *done = empty + kRtStages;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (E + kRtTile - 1) / kRtTile;
  const int split = static_cast<int>(blockIdx.x) % splits;
  const int nt = (static_cast<int>(blockIdx.x) / splits) % n_tiles;
  const int mt = static_cast<int>(blockIdx.x) / (splits * n_tiles);
  const int k_total = H / kRtStageK;
  const int k0 = min(k_total, split * stages_per_split), k1 = min(k_total, k0 + stages_per_split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kRtTile);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0 && k1 > k0) {
      // ------------------------------------------------------------ TMA producer
      const uint64_t pol_x = policy_evict_last();   // the token rows are re-read by every expert tile
      const uint64_t pol_w = policy_evict_first();  // each gate row is read once per call
      uint32_t issued = 0;
      bool ok = true;
      for (int k = k0; k < k1; ++k) {
        const int i = k - k0, s = i % kRtStages;
        const uint32_t ph = (i / kRtStages) & 1u;
        if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, err, kPipelineTimeoutNs)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], 2 * kRtBox);
        tma_load_2d(sA + s * kRtBox, &tmX, k * kRtStageK * 2, mt * kRtTile, &full[s], pol_x);
        tma_load_2d(sB + s * kRtBox, &tmW, k * kRtStageK * 2, nt * kRtTile, &full[s], pol_w);
        issued = (issued & ~(0x101u << s)) | (1u << s) | (ph << (s + 8));
      }
      if (!ok) {  // let the copies in flight land before the CTA leaves
        volatile int never = 0;
        for (int s = 0; s < kRtStages; ++s)
          if (issued & (1u << s)) mbar_wait_bounded(&full[s], (issued >> (s + 8)) & 1u, &never, nullptr, 100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && k1 > k0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t sA0 = smem_u32(sA), sB0 = smem_u32(sB);
      for (int k = k0; k < k1; ++k) {
        const int i = k - k0, s = i % kRtStages;
        if (!mbar_wait_bounded(&full[s], (i / kRtStages) & 1u, abort_flag, err, kPipelineTimeoutNs)) break;
        tc_fence_after();
        const uint64_t adesc = smem_desc(sA0 + s * kRtBox, 16, 1024, 2);
        const uint64_t bdesc = smem_desc(sB0 + s * kRtBox, 16, 1024, 2);
#pragma unroll
        for (int j = 0; j < kRtStageK / 16; ++j)  // K = 16 per MMA: +32 bytes in the 128-byte row
          tc_mma_bf16(tmem_base, adesc + 2 * j, bdesc + 2 * j, kRtIdesc, (i | j) != 0);
        tc_commit(&empty[s]);
      }
      tc_commit(done);  // fires once every MMA issued above has completed
    }
  } else {
    // -------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int t = mt * kRtTile + quarter * 32 + lane;
    bool ok = true;
    if (k1 > k0) {
      ok = mbar_wait_bounded(done, 0, abort_flag, err, kPipelineTimeoutNs);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    float *dst = partial + (static_cast<int64_t>(split) * T + t) * E + nt * kRtTile;
    const int e_live = min(kRtTile, E - nt * kRtTile);
#pragma unroll 1
    for (int c = 0; c < kRtTile / 16; ++c) {
      uint32_t r[16];
      if (k1 > k0 && ok) {
        tmem_ld16(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + c * 16, r);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) r[q] = 0u;
      }
      if (t < T && c * 16 < e_live) {  // E % 16 == 0 is not required: the tail is written one by one
        // 16-byte stores need every row start 16-byte aligned: E % 4 == 0 (the buffer is 256-aligned)
        if (c * 16 + 16 <= e_live && (E & 3) == 0) {
          float4 *d4 = reinterpret_cast<float4 *>(dst + c * 16);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d4[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
                                __uint_as_float(r[4 * q + 3]));
        } else {
          const int n = min(16, e_live - c * 16);
          for (int q = 0; q < n; ++q) dst[c * 16 + q] = __uint_as_float(r[q]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kRtTile);
}

// One CTA per token.  Its threads sum the K splits' partial logits of their experts (each
// expert's partials in split order, so the logits are the same from call to call) into shared
// memory; warp 0 then takes the softmax over E (<= 1024) logits and the top-k by repeated warp
// arg-max (larger probability first, lower expert id on ties), weights renormalised over the
// k chosen.  logits (optional) receives the summed logits.
constexpr int kTopkThreads = 512;
template <int kPer>  // experts per lane: E <= 32 * kPer
__global__ void __launch_bounds__(kTopkThreads) router_topk_kernel(const float *__restrict__ partial, int splits,
                                                                   int64_t T, int64_t E, int topk,
                                                                   int32_t *__restrict__ ids,
                                                                   float *__restrict__ weights,
                                                                   float *__restrict__ logits) {
  __shared__ float s_logit[kMaxExperts];
  pdl_wait();
  pdl_trigger();
  const int64_t t = blockIdx.x;
  const int64_t sstride = T * E;
  for (int64_t e = threadIdx.x; e < E; e += blockDim.x) {
    // every split's partial in flight at once (one round trip), then summed in split order
    const float *p = partial + t * E + e;
    float part[kRouterMaxSplits];
#pragma unroll
    for (int sp = 0; sp < kRouterMaxSplits; ++sp) part[sp] = sp < splits ? __ldg(p + sp * sstride) : 0.f;
    float v = 0.f;
#pragma unroll
    for (int sp = 0; sp < kRouterMaxSplits; ++sp)
      if (sp < splits) v = __fadd_rn(v, part[sp]);
    s_logit[e] = v;
    if (logits != nullptr) logits[t * E + e] = v;
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  float p[kPer];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int64_t e = lane + 32 * i;
    p[i] = e < E ? s_logit[e] : -INFINITY;
    mx = fmaxf(mx, p[i]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    p[i] = (lane + 32 * i < E) ? expf(__fsub_rn(p[i], mx)) : 0.f;
    sum = __fadd_rn(sum, p[i]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, o));
#pragma unroll
  for (int i = 0; i < kPer; ++i) p[i] = __fdiv_rn(p[i], sum);
  float chosen = 0.f, wsum = 0.f;
  int my_id = -1;
  for (int j = 0; j < topk; ++j) {
    float bv = -1.f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      if (e < E && p[i] >= 0.f && (p[i] > bv || (p[i] == bv && e < bi))) {
        bv = p[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    wsum = __fadd_rn(wsum, bv);
    if (lane == j) {
      my_id = bi;
      chosen = bv;
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i == bi) p[i] = -1.f;  // taken
  }
  if (lane < topk) {
    ids[t * topk + lane] = my_id;
    weights[t * topk + lane] = __fdiv_rn(chosen, wsum);
  }
}

}  // namespace

int router_partial_count(int64_t nblocks) {
  const int64_t n = (nblocks + kPrepThreads * 16 - 1) / (kPrepThreads * 16);
  return static_cast<int>(n < 1 ? 1 : (n > kMaxPartials ? kMaxPartials : n));
}

cudaError_t launch_router_prepare(const uint8_t *w, const uint8_t *sf, const float *ws2, int64_t E, int64_t H,
                                  uint32_t *partials, void *wg, cudaStream_t s) {
  const int64_t nblocks = E * H / 16;
  const int nparts = router_partial_count(nblocks);
  cudaError_t e = launch_pdl(router_amax_kernel, dim3(nparts), dim3(kPrepThreads), 0, s, w, sf, ws2, nblocks,
                             partials);
  if (e != cudaSuccess) return e;
  return launch_pdl(router_qdq_kernel, dim3(nparts), dim3(kPrepThreads), 0, s, w, sf, ws2, nblocks,
                    static_cast<const uint32_t *>(partials), nparts, static_cast<uint16_t *>(wg));
}

int router_splits(int64_t T, int64_t E, int64_t H) {
  const int64_t tiles = ((T + kRtTile - 1) / kRtTile) * ((E + kRtTile - 1) / kRtTile);
  const int64_t k_total = H / kRtStageK;
  int64_t splits = tiles > 0 ? kRouterTargetCtas / tiles : 1;
  splits = splits < 1 ? 1 : (splits > kRouterMaxSplits ? kRouterMaxSplits : splits);
  if (splits > k_total) splits = k_total > 0 ? k_total : 1;
  const int64_t per = (k_total + splits - 1) / splits;  // no split is left without K stages
  return static_cast<int>(per > 0 ? (k_total + per - 1) / per : 1);
}

cudaError_t launch_router(const CUtensorMap &tm_x, const CUtensorMap &tm_w, int64_t T, int64_t H, int64_t E, int topk,
                          int32_t *ids, float *weights, float *logits, float *partial, uint32_t *err, cudaStream_t s) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(router_logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kRtSmem));
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int splits = router_splits(T, E, H);
  const int64_t k_total = H / kRtStageK;
  const int per = static_cast<int>((k_total + splits - 1) / splits);
  const int64_t ctas = ((T + kRtTile - 1) / kRtTile) * ((E + kRtTile - 1) / kRtTile) * splits;
  cudaError_t e = launch_pdl(router_logits_tc_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kRtThreads), kRtSmem, s,
                             tm_x, tm_w, static_cast<int>(T), static_cast<int>(E), static_cast<int>(H), splits, per,
                             partial, err);
  if (e != cudaSuccess) return e;
  auto kernel = E <= 128 ? router_topk_kernel<4>
                         : (E <= 256 ? router_topk_kernel<8> : (E <= 512 ? router_topk_kernel<16> : router_topk_kernel<32>));
  static_assert(32 * 32 >= kMaxExperts, "experts per lane");
  return launch_pdl(kernel, dim3(static_cast<unsigned>(T)), dim3(kTopkThreads), 0, s,
                    static_cast<const float *>(partial), splits, T, E, topk, ids, weights, logits);
}

}  // namespace nvfp4
