// Router gate: the NVFP4 gate weight dequantised to bf16, round-tripped through FP8-E4M3 with
// one per-tensor scale s = amax / 448 (prepare, once), then per call logits = x @ wg^T in fp32
// on the CUDA cores (a small contraction next to the expert GEMMs: 384 x 7168 per token), a
// softmax over the experts and the top-k with weights renormalised over the k chosen.
#include "common.cuh"

namespace nvfp4 {

namespace {

constexpr int kPrepThreads = 256;
constexpr int kGateExperts = 8;   // experts per block (one warp each)
constexpr int kGateTokens = 32;   // tokens per block

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

// logits[t][e] = sum_h x[t][h] * wg[e][h]; warp w of a block owns expert e, lanes stride the
// row in 8-element chunks (fp32 products and sums), then a butterfly reduction.
__global__ void __launch_bounds__(kGateExperts * 32) router_logits_kernel(const uint16_t *__restrict__ x,
                                                                          const uint16_t *__restrict__ wg, int64_t T,
                                                                          int64_t E, int64_t H,
                                                                          float *__restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * kGateExperts + warp;
  if (e >= E) return;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * kGateTokens;
  const int64_t t1 = min(T, t0 + kGateTokens);
  const uint4 *wrow = reinterpret_cast<const uint4 *>(wg + e * H);
  const int64_t chunks = H / 8;
  for (int64_t t = t0; t < t1; ++t) {
    const uint4 *xrow = reinterpret_cast<const uint4 *>(x + t * H);
    float acc = 0.f;
    for (int64_t c = lane; c < chunks; c += 32) {
      const uint4 a = __ldg(xrow + c), b = __ldg(wrow + c);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc = __fadd_rn(acc, __fmul_rn(__uint_as_float(aw[i] << 16), __uint_as_float(bw[i] << 16)));
        acc = __fadd_rn(acc, __fmul_rn(__uint_as_float(aw[i] & 0xFFFF0000u), __uint_as_float(bw[i] & 0xFFFF0000u)));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    if (lane == 0) logits[t * E + e] = acc;
  }
}

// One warp per token: softmax over E (<= 1024) logits, then top-k by repeated warp arg-max
// (larger probability first, lower expert id on ties), weights renormalised over the k chosen.
__global__ void router_topk_kernel(const float *__restrict__ logits, int64_t T, int64_t E, int topk,
                                   int32_t *__restrict__ ids, float *__restrict__ weights) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  constexpr int kPer = kMaxExperts / 32;
  float p[kPer];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int64_t e = lane + 32 * i;
    p[i] = e < E ? logits[t * E + e] : -INFINITY;
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

cudaError_t launch_router(const void *x, int64_t T, int64_t H, const void *wg, int64_t E, int topk, int32_t *ids,
                          float *weights, float *logits, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((E + kGateExperts - 1) / kGateExperts),
                  static_cast<unsigned>((T + kGateTokens - 1) / kGateTokens));
  cudaError_t e = launch_pdl(router_logits_kernel, grid, dim3(kGateExperts * 32), 0, s,
                             static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(wg), T, E, H, logits);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (T + 7) / 8;
  return launch_pdl(router_topk_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    static_cast<const float *>(logits), T, E, topk, ids, weights);
}

}  // namespace nvfp4
