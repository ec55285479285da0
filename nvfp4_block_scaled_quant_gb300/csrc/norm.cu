// RMSNorm feeding the NVFP4 activation quantiser.
//
// Per row r:  inv_r = 1 / sqrt(fl32(sum_k x^2) / K + eps)   (IEEE sqrt and division)
//             y[r,k] = bf16( fl32( fl32(x[r,k] * inv_r) * gamma[k] ) )
// The per-row statistics kernel computes inv_r (fp32 sum in a fixed order: each thread over
// its strided 8-element chunks, then a butterfly warp reduction and a warp-0 reduction of
// the warp sums), the block maxima of |y| for the dynamic global scale, and optionally
// writes y.  The fused quantiser recomputes y from x, inv_r and gamma with the same
// operations, so the fused path (stats -> normalise+quantise) and the unfused path
// (stats writing y -> quantise y) produce identical codes, scales and gs.
#include "common.cuh"

namespace nvfp4 {

namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float normed(float x, float inv, float g) {
  return bf16_round(__fmul_rn(__fmul_rn(x, inv), g));
}

// Chunks of 8 elements a thread keeps in registers between the two passes over a row: rows of
// up to kNormCache * 256 * 8 elements are read once; longer rows are read again (from L2).
constexpr int kNormCache = 4;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_stats_kernel(
    const uint16_t *__restrict__ x, int64_t M, int64_t K, int64_t ldx, const uint16_t *__restrict__ gamma,
    float eps, float *__restrict__ inv_rms, uint32_t *__restrict__ partials, uint16_t *__restrict__ y) {
  __shared__ float red[32];
  __shared__ float s_inv;
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int64_t chunks = K / 8;
  const bool cached = chunks <= static_cast<int64_t>(kNormCache) * blockDim.x;
  uint32_t m = 0;
  for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
    const uint4 *row = reinterpret_cast<const uint4 *>(x + r * ldx);
    uint4 keep[kNormCache];
    if (cached) {  // every chunk of the row is loaded before any is used
#pragma unroll
      for (int u = 0; u < kNormCache; ++u) {
        const int64_t c = threadIdx.x + u * static_cast<int64_t>(blockDim.x);
        keep[u] = c < chunks ? __ldg(row + c) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float acc = 0.f;
    auto add_squares = [&](const uint4 v) {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xFFFF0000u);
        acc = __fadd_rn(acc, __fmul_rn(a, a));
        acc = __fadd_rn(acc, __fmul_rn(b, b));
      }
    };
    // each thread sums its chunks c = tid, tid + 256, ... in increasing order (both paths)
    if (cached) {
#pragma unroll
      for (int u = 0; u < kNormCache; ++u)
        if (threadIdx.x + u * static_cast<int64_t>(blockDim.x) < chunks) add_squares(keep[u]);
    } else {
      for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) add_squares(__ldg(row + c));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (warp == 0) {
      float s = lane < nwarps ? red[lane] : 0.f;
#pragma unroll
      for (int o = 16; o; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
      if (lane == 0) {
        const float mean = __fdiv_rn(s, static_cast<float>(K));
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
        s_inv = inv;
        if (inv_rms) inv_rms[r] = inv;
      }
    }
    __syncthreads();
    const float inv = s_inv;
    const uint4 *grow = reinterpret_cast<const uint4 *>(gamma);
    auto normalise = [&](int64_t c, const uint4 v) {
      const uint4 gv = __ldg(grow + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = normed(__uint_as_float(w[i] << 16), inv, __uint_as_float(gw[i] << 16));
        const float hi = normed(__uint_as_float(w[i] & 0xFFFF0000u), inv, __uint_as_float(gw[i] & 0xFFFF0000u));
        const uint32_t bl = __float_as_uint(lo) >> 16, bh = __float_as_uint(hi) >> 16;
        m = max(m, max(bl & 0x7FFFu, bh & 0x7FFFu));
        o[i] = bl | (bh << 16);
      }
      if (y) reinterpret_cast<uint4 *>(y + r * K)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    };
    if (cached) {
#pragma unroll
      for (int u = 0; u < kNormCache; ++u) {
        const int64_t c = threadIdx.x + u * static_cast<int64_t>(blockDim.x);
        if (c < chunks) normalise(c, keep[u]);
      }
    } else {
      for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) normalise(c, __ldg(row + c));
    }
    __syncthreads();  // red / s_inv are reused by the next row
  }
  if (partials) {
    __shared__ uint32_t mred[32];
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) mred[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < nwarps; ++i) m = max(m, mred[i]);
      partials[blockIdx.x] = m;
    }
  }
}

// 16-element blocks of the normalised rows, walked by a fixed grid as the plain quantiser
// (kNormUnroll blocks' loads in flight per thread, gs derived once per CTA); same layouts.
constexpr int kNormUnroll = 2;
template <typename Idx>  // int32_t when every block index and byte offset of the launch fits
__global__ void __launch_bounds__(kNormThreads, kStreamCtasPerSm) rmsnorm_quantize_kernel(
    const uint16_t *__restrict__ x, int64_t M_, int64_t K_, int64_t ldx_, const uint16_t *__restrict__ gamma,
    const float *__restrict__ inv_rms, const uint32_t *__restrict__ partials, int nparts,
    const float *__restrict__ gs_static, float *__restrict__ gs_out, uint8_t *__restrict__ q,
    uint8_t *__restrict__ sf, int sf_layout, int64_t rows_total) {
  __shared__ uint32_t scratch[32];
  pdl_wait();
  pdl_trigger();
  const Idx M = static_cast<Idx>(M_), K = static_cast<Idx>(K_), ldx = static_cast<Idx>(ldx_);
  const Idx kb = K / 16;
  const Idx total = static_cast<Idx>(rows_total) * kb;
  const Idx stride = static_cast<Idx>(gridDim.x) * static_cast<Idx>(blockDim.x);
  const int lane = threadIdx.x & 31;
  const Idx wbase0 = static_cast<Idx>(blockIdx.x) * static_cast<Idx>(blockDim.x) + static_cast<Idx>(threadIdx.x & ~31);
  // (row, block) of each of this thread's kNormUnroll blocks, advanced without division
  const Idx step = kNormUnroll * stride;
  const Idx step_r = step / kb, step_c = step - step_r * kb;
  RowColT<Idx> pos[kNormUnroll];
#pragma unroll
  for (int u = 0; u < kNormUnroll; ++u) pos[u].init(wbase0 + u * stride + lane, kb);
  uint4 a[kNormUnroll], b[kNormUnroll];
  float inv[kNormUnroll];
  auto load = [&](Idx wb) {
#pragma unroll
    for (int u = 0; u < kNormUnroll; ++u) {
      const Idx g = wb + u * stride + lane;
      a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
      inv[u] = 0.f;
      if (g < total && pos[u].r < M) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + pos[u].r * ldx + pos[u].c * 16);
        a[u] = __ldg(src);
        b[u] = __ldg(src + 1);
        inv[u] = __ldg(inv_rms + pos[u].r);
      }
    }
  };
  load(wbase0);
  float gs;
  if (partials) {
    gs = gs_from_partials(partials, nparts, scratch);
    if (blockIdx.x == 0 && threadIdx.x == 0) *gs_out = gs;
  } else {
    gs = *gs_static;
  }
  const float six_gs = __fmul_rn(6.0f, gs);
  for (Idx wb = wbase0; wb < total; wb += step) {  // uniform over the warp
    if (wb != wbase0) load(wb);
#pragma unroll
    for (int u = 0; u < kNormUnroll; ++u) {
      const Idx g = wb + u * stride + lane;
      const bool valid = g < total;
      const Idx r = pos[u].r, c = pos[u].c;
      pos[u].advance(step_r, step_c, kb);
      const bool live = valid && r < M;
      uint32_t sfb = 0;
      if (live) {
        const uint4 *gsrc = reinterpret_cast<const uint4 *>(gamma + c * 16);
        const uint4 ga = __ldg(gsrc), gb2 = __ldg(gsrc + 1);
        const uint32_t w[8] = {a[u].x, a[u].y, a[u].z, a[u].w, b[u].x, b[u].y, b[u].z, b[u].w};
        const uint32_t gw[8] = {ga.x, ga.y, ga.z, ga.w, gb2.x, gb2.y, gb2.z, gb2.w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[2 * i] = normed(__uint_as_float(w[i] << 16), inv[u], __uint_as_float(gw[i] << 16));
          v[2 * i + 1] = normed(__uint_as_float(w[i] & 0xFFFF0000u), inv[u], __uint_as_float(gw[i] & 0xFFFF0000u));
        }
        uint32_t codes[2];
        sfb = encode_block16(v, gs, six_gs, codes);
        *reinterpret_cast<uint2 *>(q + r * (K / 2) + c * 8) = make_uint2(codes[0], codes[1]);
      }
      if (sf_layout == NVFP4_SF_LINEAR) {
        if (live) sf[r * kb + c] = static_cast<uint8_t>(sfb);
      } else {
        uint32_t word = sfb << ((lane & 3) * 8);
        word |= __shfl_xor_sync(0xffffffffu, word, 1);
        word |= __shfl_xor_sync(0xffffffffu, word, 2);
        if (valid && (lane & 3) == 0) {
          if constexpr (sizeof(Idx) == 4)
            *reinterpret_cast<uint32_t *>(sf + sf_word_offset32(static_cast<uint32_t>(r), static_cast<uint32_t>(c >> 2),
                                                                static_cast<uint32_t>(kb >> 2))) = word;
          else
            *reinterpret_cast<uint32_t *>(sf + sf_word_offset(r, c >> 2, kb >> 2)) = word;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_rmsnorm_stats(const void *x, int64_t M, int64_t K, int64_t ldx, const void *gamma, float eps,
                                 float *inv_rms, uint32_t *partials, int nparts, void *y, cudaStream_t s) {
  return launch_pdl(rmsnorm_stats_kernel, dim3(nparts), dim3(kNormThreads), 0, s, static_cast<const uint16_t *>(x),
                    M, K, ldx, static_cast<const uint16_t *>(gamma), eps, inv_rms, partials,
                    static_cast<uint16_t *>(y));
}

cudaError_t launch_rmsnorm_quantize(const void *x, int64_t M, int64_t K, int64_t ldx, const void *gamma,
                                    const float *inv_rms, const uint32_t *partials, int nparts,
                                    const float *gs_static, float *gs_out, uint8_t *q, uint8_t *sf, int sf_layout,
                                    cudaStream_t s) {
  const int64_t rows_total = sf_layout == NVFP4_SF_LINEAR ? M : ((M + 127) / 128) * 128;
  const int64_t items = rows_total * (K / 16);
  int64_t blocks = items > 0 ? (items + kNormThreads - 1) / kNormThreads : 1;
  if (blocks > stream_grid_cap()) blocks = stream_grid_cap();
  // 32-bit indexing when every block index (plus a grid step) and every byte offset fits
  const int64_t lim = int64_t(1) << 31;
  const bool small = rows_total * (K / 16) + 2 * kNormUnroll * blocks * kNormThreads < lim &&
                     (M > 0 ? (M - 1) * ldx + K : 0) * 2 < lim && rows_total * K < lim;
  auto kernel = small ? rmsnorm_quantize_kernel<int32_t> : rmsnorm_quantize_kernel<int64_t>;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(blocks)), dim3(kNormThreads), 0, s,
                    static_cast<const uint16_t *>(x), M, K, ldx, static_cast<const uint16_t *>(gamma), inv_rms,
                    partials, nparts, gs_static, gs_out, q, sf, sf_layout, rows_total);
}

}  // namespace nvfp4
