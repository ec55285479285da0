// Activation quantisation (amax reduction + NVFP4 block encoding) and the one-time
// weight prepare step (scale swizzle, gate/up row interleave).
//
// Both are HBM-bound streams: 16-byte vector loads along K, one thread per
// 16-element scale block, the four scale bytes of one 64-element group gathered
// with warp shuffles into one 32-bit store of the tensor-core layout.
#include "common.cuh"

namespace nvfp4 {

namespace {

constexpr int kAmaxThreads = 256;
constexpr int kQuantThreads = 256;

__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t w) {
  // |bf16| compares like an unsigned integer once the sign bit is cleared
  return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}

__device__ __forceinline__ uint32_t block_reduce_max(uint32_t v, uint32_t *scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < static_cast<int>(blockDim.x >> 5) ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) scratch[0] = v;
  }
  __syncthreads();
  return scratch[0];
}

// Block partial maxima of |x| (as bf16 bit patterns).  Block b reduces rows
// b, b + gridDim.x, ...
__global__ void __launch_bounds__(kAmaxThreads) amax_partials_kernel(const uint16_t *__restrict__ x,
                                                                     int64_t M, int64_t K,
                                                                     int64_t ldx,
                                                                     uint32_t *__restrict__ partials) {
  __shared__ uint32_t scratch[32];
  pdl_wait();
  pdl_trigger();
  const int64_t chunks = K / 8;
  uint32_t m = 0;
  for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
    const uint4 *row = reinterpret_cast<const uint4 *>(x + r * ldx);
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) {
      const uint4 v = __ldg(row + c);
      m = max(m, max(max(max_abs_bf16x2(v.x), max_abs_bf16x2(v.y)),
                     max(max_abs_bf16x2(v.z), max_abs_bf16x2(v.w))));
    }
  }
  m = block_reduce_max(m, scratch);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// Encode one 16-element block (two 16-byte halves a, b of bf16 pairs) and store its codes;
// returns the E4M3 scale byte.
__device__ __forceinline__ uint32_t encode_and_store(uint4 a, uint4 b, float gs, float six_gs, uint8_t *qdst) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t codes[2];
  const uint32_t sfb = encode_block16_bf16(w, gs, six_gs, codes);
  *reinterpret_cast<uint2 *>(qdst) = make_uint2(codes[0], codes[1]);
  return sfb;
}

// Store the scale byte of block (r, c): one byte (row-major layout) or, in the swizzled
// layout, one 32-bit word per four consecutive blocks of a row, gathered from lanes 4i..4i+3
// (all 32 lanes must call this together).
template <typename Idx>
__device__ __forceinline__ void store_scale(uint8_t *sf, int sf_layout, bool valid, bool live, Idx r, Idx c, Idx kb,
                                            uint32_t sfb) {
  if (sf_layout == NVFP4_SF_LINEAR) {
    if (live) sf[r * kb + c] = static_cast<uint8_t>(sfb);
  } else {
    const int lane = threadIdx.x & 31;
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

// 16-element blocks of a (M, K) bf16 tensor, consecutive threads on consecutive blocks of a
// row (so lanes 4i..4i+3 share one swizzled scale word; K % 64 == 0).  A fixed grid walks all
// blocks with kQuantUnroll blocks' loads in flight per thread, and each CTA derives gs once.
// The swizzled output also covers the padding rows up to a multiple of 128 (scale 0, no codes).
constexpr int kQuantUnroll = 2;
template <typename Idx>  // int32_t when every block index and byte offset of the launch fits
__global__ void __launch_bounds__(kQuantThreads, kStreamCtasPerSm) quantize_kernel(
    const uint16_t *__restrict__ x, int64_t M_, int64_t K_, int64_t ldx_,
    const uint32_t *__restrict__ partials, int nparts, const float *__restrict__ gs_static,
    float *__restrict__ gs_out, uint8_t *__restrict__ q, uint8_t *__restrict__ sf,
    int sf_layout, int64_t rows_total) {
  __shared__ uint32_t scratch[32];
  pdl_wait();
  pdl_trigger();
  const Idx M = static_cast<Idx>(M_), K = static_cast<Idx>(K_), ldx = static_cast<Idx>(ldx_);
  const Idx kb = K / 16;
  const Idx total = static_cast<Idx>(rows_total) * kb;
  const Idx stride = static_cast<Idx>(gridDim.x) * static_cast<Idx>(blockDim.x);
  const int lane = threadIdx.x & 31;
  const Idx wbase0 = static_cast<Idx>(blockIdx.x) * static_cast<Idx>(blockDim.x) + static_cast<Idx>(threadIdx.x & ~31);
  // (row, block) of each of this thread's kQuantUnroll blocks, advanced without division
  const Idx step = kQuantUnroll * stride;
  const Idx step_r = step / kb, step_c = step - step_r * kb;
  RowColT<Idx> pos[kQuantUnroll];
#pragma unroll
  for (int u = 0; u < kQuantUnroll; ++u) pos[u].init(wbase0 + u * stride + lane, kb);
  // the first blocks' loads are issued before the gs reduction, which their latency overlaps
  uint4 a[kQuantUnroll], b[kQuantUnroll];
  auto load = [&](Idx wb) {
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const Idx g = wb + u * stride + lane;
      a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
      if (g < total && pos[u].r < M) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + pos[u].r * ldx + pos[u].c * 16);
        a[u] = __ldg(src);
        b[u] = __ldg(src + 1);
      }
    }
  };
  load(wbase0);
  float gs = 0.f;
  if (nparts == 0) {
    // Small input (at most kInlineAmaxElems elements): every block reduces the whole of x
    // itself, one launch fewer.  Block 0 writes gs (0 when M == 0).
    uint32_t m = 0;
    const Idx chunks = K / 8;
    RowColT<Idx> ix;
    ix.init(static_cast<Idx>(threadIdx.x), chunks);
    const Idx sr = static_cast<Idx>(blockDim.x) / chunks, sc = static_cast<Idx>(blockDim.x) - sr * chunks;
    for (Idx i = threadIdx.x; i < M * chunks; i += blockDim.x, ix.advance(sr, sc, chunks)) {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + ix.r * ldx) + ix.c);
      m = max(m, max(max(max_abs_bf16x2(v.x), max_abs_bf16x2(v.y)), max(max_abs_bf16x2(v.z), max_abs_bf16x2(v.w))));
    }
    m = block_reduce_max(m, scratch);
    gs = __fdiv_rn(__uint_as_float(m << 16), 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *gs_out = gs;
  } else if (partials) {
    gs = gs_from_partials(partials, nparts, scratch);
    if (blockIdx.x == 0 && threadIdx.x == 0) *gs_out = gs;
  } else {
    gs = *gs_static;
  }
  const float six_gs = __fmul_rn(6.0f, gs);
  for (Idx wb = wbase0; wb < total; wb += step) {  // uniform over the warp
    if (wb != wbase0) load(wb);
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const Idx g = wb + u * stride + lane;
      const bool valid = g < total;
      const Idx r = pos[u].r, c = pos[u].c;
      const bool live = valid && r < M;
      uint32_t sfb = 0;
      if (live) sfb = encode_and_store(a[u], b[u], gs, six_gs, q + r * (K / 2) + c * 8);
      store_scale(sf, sf_layout, valid, live, r, c, kb, sfb);
      pos[u].advance(step_r, step_c, kb);
    }
  }
}

// Prepared weight layout.  Codes are tile-major: for each group, 128-row tile and 128-byte
// column slab of K (256 FP4 elements), the tile's 128 rows x 128 bytes sit in one contiguous
// 16 KiB block (row r of the tile at 128 r), rows permuted for the w13 interleave and slabs
// past K/2 bytes filled with zero codes; a GEMM stage then reads one contiguous block.
// Scales: one 32-bit word (4 scales) per thread, written in the swizzled layout.
__device__ __forceinline__ int64_t interleave_src_row(int64_t n, int64_t N, int flags) {
  if (!(flags & NVFP4_PREP_W13_INTERLEAVE)) return n;
  const int64_t tile = n >> 7, j = n & 127;
  return j < 64 ? tile * 64 + j : N / 2 + tile * 64 + (j - 64);
}

__global__ void prepare_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ sf,
                               int64_t G, int64_t N, int64_t K, int flags,
                               uint8_t *__restrict__ w_out, uint8_t *__restrict__ sf_out) {
  // No early trigger: the launch after this one may read the prepared weights before its
  // own wait (the GEMMs stream their first weight stages early), so it starts only once
  // this grid has completed.
  pdl_wait();
  const int64_t row_bytes = K / 2;                // a multiple of 32 (K % 64 == 0)
  const int64_t slabs = (row_bytes + 127) / 128;  // 128-byte column slabs per row
  const int64_t tiles = (N + 127) / 128;          // (one group with N % 128 != 0: rows from N on are zero)
  const int64_t code_items = G * tiles * slabs * 1024;  // 16-byte chunks of the tile-major blocks
  const int64_t words_per_group = tiles * 128 * K / 64;  // 4 scales per word
  const int64_t total = code_items + G * words_per_group;
  const int64_t kb = K / 16, kc4 = K / 64;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < code_items) {
      const int64_t blk = i >> 10, within = i & 1023;  // block (group, tile, slab); 16-byte chunk
      const int64_t r = within >> 3, c16 = within & 7;
      const int64_t tile = blk / slabs, s = blk - tile * slabs;
      const int64_t g = tile / tiles, nt = tile - g * tiles;
      const int64_t n = nt * 128 + r;
      const int64_t src = g * N + interleave_src_row(n, N, flags);
      const int64_t byte = s * 128 + c16 * 16;
      const uint4 v = byte < row_bytes && n < N ? __ldg(reinterpret_cast<const uint4 *>(w + src * row_bytes + byte))
                                                : make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4 *>(w_out)[i] = v;
    } else {
      const int64_t j = i - code_items;
      const int64_t g = j / words_per_group, wi = j - g * words_per_group;
      const int64_t blk = wi >> 7, within = wi & 127;
      const int64_t rb = blk / kc4, cb = blk - rb * kc4;
      const int64_t r = rb * 128 + (within & 3) * 32 + (within >> 2);
      const int64_t src = g * N + interleave_src_row(r, N, flags);
      const uint32_t word = r < N ? __ldg(reinterpret_cast<const uint32_t *>(sf + src * kb + cb * 4)) : 0u;
      reinterpret_cast<uint32_t *>(sf_out + g * (tiles * 128 * kb))[wi] = word;
    }
  }
}

}  // namespace

int amax_partial_count(int64_t M, int64_t K) {
  (void)K;
  if (M <= 0) return 1;
  return static_cast<int>(M < kMaxPartials ? M : kMaxPartials);
}

cudaError_t launch_amax_partials(const void *x, int64_t M, int64_t K, int64_t ldx,
                                 uint32_t *partials, int nparts, cudaStream_t s) {
  return launch_pdl(amax_partials_kernel, dim3(nparts), dim3(kAmaxThreads), 0, s,
                    static_cast<const uint16_t *>(x), M, K, ldx, partials);
}

int stream_grid_cap() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1024;
  if (cached[dev] == 0) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = (sms > 0 ? sms : 128) * kStreamCtasPerSm;
  }
  return cached[dev];
}

cudaError_t launch_quantize(const void *x, int64_t M, int64_t K, int64_t ldx,
                            const uint32_t *partials, int nparts, const float *gs_static,
                            float *gs_out, uint8_t *q, uint8_t *sf, int sf_layout,
                            cudaStream_t s) {
  const int64_t rows_total = sf_layout == NVFP4_SF_LINEAR ? M : ((M + 127) / 128) * 128;
  const int64_t items = rows_total * (K / 16);
  int64_t blocks = items > 0 ? (items + kQuantThreads - 1) / kQuantThreads : 1;
  if (blocks > stream_grid_cap()) blocks = stream_grid_cap();
  // 32-bit indexing when every block index (plus a grid step) and every byte offset of x, the
  // codes and the scales stays below 2^31
  const int64_t lim = int64_t(1) << 31;
  const bool small = rows_total * (K / 16) + 2 * kQuantUnroll * blocks * kQuantThreads < lim &&
                     (M > 0 ? (M - 1) * ldx + K : 0) * 2 < lim && rows_total * K < lim;
  return small ? launch_pdl(quantize_kernel<int32_t>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantThreads), 0, s,
                            static_cast<const uint16_t *>(x), M, K, ldx, partials, nparts, gs_static, gs_out, q, sf,
                            sf_layout, rows_total)
               : launch_pdl(quantize_kernel<int64_t>, dim3(static_cast<unsigned>(blocks)), dim3(kQuantThreads), 0, s,
                            static_cast<const uint16_t *>(x), M, K, ldx, partials, nparts, gs_static, gs_out, q, sf,
                            sf_layout, rows_total);
}

cudaError_t launch_act_quant(const void *x, int64_t M, int64_t K, int64_t ldx, bool dynamic, uint32_t *partials,
                             const float *gs_static, float *gs_out, uint8_t *q, uint8_t *sf, int sf_layout,
                             cudaStream_t s) {
  if (!dynamic) return launch_quantize(x, M, K, ldx, nullptr, 1, gs_static, gs_out, q, sf, sf_layout, s);
  if (M * K <= kInlineAmaxElems)  // nparts = 0: the quantise blocks reduce x themselves
    return launch_quantize(x, M, K, ldx, nullptr, 0, gs_static, gs_out, q, sf, sf_layout, s);
  const int nparts = amax_partial_count(M, K);
  const cudaError_t e = launch_amax_partials(x, M, K, ldx, partials, nparts, s);
  if (e != cudaSuccess) return e;
  return launch_quantize(x, M, K, ldx, partials, nparts, gs_static, gs_out, q, sf, sf_layout, s);
}

cudaError_t launch_prepare(const uint8_t *w, const uint8_t *sf, int64_t G, int64_t N, int64_t K,
                           int flags, uint8_t *w_out, uint8_t *sf_out, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return launch_pdl(prepare_kernel, dim3(sms * 8), dim3(256), 0, s, w, sf, G, N, K, flags, w_out, sf_out);
}

}  // namespace nvfp4
