// MoE routing (histogram, scans, stable permutation), the dispatch step that
// quantises each token once and writes its codes into the row of every expert
// segment it is routed to, and the final fp32 -> bf16 conversion.
#include "common.cuh"

namespace nvfp4 {

namespace {

constexpr int kRouteThreads = 512;
constexpr int kDispatchThreads = 256;
constexpr int kDestRegs = 8;  // destination rows held in registers (top-k up to 8)
constexpr int kRankWarps = kRouteThreads / 32;
constexpr int kRankPerWarp = 512;                      // entries per warp and chunk
constexpr int kRankChunk = kRankWarps * kRankPerWarp;  // entries ranked per pass
constexpr int kSmallRank = 256;                        // up to this many entries one warp ranks
constexpr int kHistUnroll = 8;                         // id loads in flight per histogram step

// dynamic shared memory of the routing block (counts, cursors, deltas, scan scratch,
// per-warp counts)
size_t route_smem_bytes(int E) {
  return sizeof(int) * (static_cast<size_t>(E) * (6 + kRankWarps) + 1 + 96 + 6);
}

// Block-wide exclusive scans over n counts (n <= 4 * blockDim): the counts, the counts
// rounded up to 128 rows, and the tiles of 2^tile_shift rows they take.  Writes
// out_x[0..n] (n+1 entries, the last one the total; n >= 1); out_pad and out_tiles may
// be null.
__device__ void block_scan3(const int *in_count, int n, int tile_shift, int *out_off, int *out_pad,
                            int *out_tiles, int *tmp /* 3 * 32 ints */) {
  const int tile_round = (1 << tile_shift) - 1;
  const int per = (n + blockDim.x - 1) / blockDim.x;  // <= 4
  const int lo = threadIdx.x * per;
  int s0 = 0, s1 = 0, s2 = 0;
  for (int i = 0; i < per; ++i) {
    const int idx = lo + i;
    if (idx < n) {
      const int c = in_count[idx];
      s0 += c;
      s1 += (c + 127) & ~127;
      s2 += (c + tile_round) >> tile_shift;
    }
  }
  // inclusive warp scan of the thread sums
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int i0 = s0, i1 = s1, i2 = s2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, i0, o), b = __shfl_up_sync(0xffffffffu, i1, o),
              c = __shfl_up_sync(0xffffffffu, i2, o);
    if (lane >= o) {
      i0 += a;
      i1 += b;
      i2 += c;
    }
  }
  if (lane == 31) {
    tmp[warp] = i0;
    tmp[32 + warp] = i1;
    tmp[64 + warp] = i2;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int a = lane < nw ? tmp[lane] : 0, b = lane < nw ? tmp[32 + lane] : 0,
        c = lane < nw ? tmp[64 + lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, a, o), y = __shfl_up_sync(0xffffffffu, b, o),
                z = __shfl_up_sync(0xffffffffu, c, o);
      if (lane >= o) {
        a += x;
        b += y;
        c += z;
      }
    }
    if (lane < nw) {  // exclusive prefix of the warp totals
      tmp[lane] = a - tmp[lane];
      tmp[32 + lane] = b - tmp[32 + lane];
      tmp[64 + lane] = c - tmp[64 + lane];
    }
  }
  __syncthreads();
  int e0 = tmp[warp] + i0 - s0, e1 = tmp[32 + warp] + i1 - s1, e2 = tmp[64 + warp] + i2 - s2;
  for (int i = 0; i < per; ++i) {
    const int idx = lo + i;
    if (idx < n) {
      out_off[idx] = e0;
      if (out_pad) out_pad[idx] = e1;
      if (out_tiles) out_tiles[idx] = e2;
      const int c = in_count[idx];
      e0 += c;
      e1 += (c + 127) & ~127;
      e2 += (c + tile_round) >> tile_shift;
    }
    if (idx == n - 1) {
      out_off[n] = e0;
      if (out_pad) out_pad[n] = e1;
      if (out_tiles) out_tiles[n] = e2;
    }
  }
}

// Block 0 routes; blocks 1.. compute amax partials of x (when partials != nullptr)
// and zero the fp32 accumulator y_acc (T*H floats).
//
// Routing keeps flat order within each expert (a stable counting sort of the
// T*k entries).  Up to kSmallRank entries one warp walks them 32 at a time.
// Beyond that the entries go in chunks of kRankChunk: warp w owns the
// contiguous slice [w*kRankPerWarp, (w+1)*kRankPerWarp) of the chunk, counts
// its entries per expert, a scan over the warps (per expert, in warp order)
// turns the counts into starting positions, and a second walk hands out
// consecutive positions to equal experts in flat order.
__device__ void route_block(const int32_t *__restrict__ ids, int T, int topk, int E, int has_shared,
                            RouteBufs rb, uint32_t *err) {
  {
    extern __shared__ int route_smem[];
    int *s_cnt = route_smem;        // G = E (+1 shared) counts
    int *s_cursor = s_cnt + E + 1;  // next free sorted position per expert
    int *s_delta = s_cursor + E;    // padded row - sorted position, per expert
    int *s_tmp = s_delta + E;       // scan scratch (96)
    int *s_off = s_tmp + 96;        // G + 1 exclusive scans: rows, padded rows, tiles
    int *s_pad = s_off + E + 2;
    int *s_tiles = s_pad + E + 2;
    int *s_wcnt = s_tiles + E + 2;  // kRankWarps x E per-warp counts, then positions
    const int G = E + (has_shared ? 1 : 0);
    const int Tk = T * topk;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int g = threadIdx.x; g < G; g += blockDim.x) s_cnt[g] = 0;
    __syncthreads();
    // histogram: one shared-memory atomic per entry (cheaper than grouping equal ids with
    // a warp match first); each warp has kHistUnroll loads in flight before it uses the first
    for (int f0 = warp * 32; f0 < Tk; f0 += blockDim.x * kHistUnroll) {
      int ev[kHistUnroll];
#pragma unroll
      for (int u = 0; u < kHistUnroll; ++u) {
        const int f = f0 + u * blockDim.x + lane;
        ev[u] = f < Tk ? __ldg(ids + f) : -1;
      }
#pragma unroll
      for (int u = 0; u < kHistUnroll; ++u) {
        const int f = f0 + u * blockDim.x + lane;
        int e = ev[u];
        if (f < Tk && (e < 0 || e >= E)) {
          raise_device_error(err, NVFP4_DEVERR_BAD_EXPERT_ID);
          e = -1;
        }
        if (e >= 0) atomicAdd(&s_cnt[e], 1);
      }
    }
    if (has_shared && threadIdx.x == 0) s_cnt[E] = T;
    __syncthreads();
    block_scan3(s_cnt, G, rb.tile_shift, s_off, s_pad, s_tiles, s_tmp);
    __syncthreads();
    for (int g = threadIdx.x; g <= G; g += blockDim.x) {
      if (g < G) rb.counts[g] = s_cnt[g];
      rb.offsets[g] = s_off[g];
      if (rb.pad_offsets) rb.pad_offsets[g] = s_pad[g];
      if (rb.tile_offsets) rb.tile_offsets[g] = s_tiles[g];
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      s_cursor[e] = s_off[e];
      s_delta[e] = s_pad[e] - s_off[e];
    }
    // the GEMMs' tile schedule: one entry per tile of 2^tile_shift rows of each group's
    // segment in the permuted buffers; kTileMulti marks the tiles of a group that spans
    // several (they read the same weights)
    if (rb.tile_table) {
      const int tr = 1 << rb.tile_shift;
      for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const int c = s_cnt[g], t0 = s_tiles[g], p0 = s_pad[g];
        const int multi = c > tr ? kTileMulti : 0;
        for (int mt = 0; mt * tr < c; ++mt)
          rb.tile_table[t0 + mt] = make_int4(g, mt | multi, min(tr, c - mt * tr), p0 + mt * tr);
      }
    }
    __syncthreads();
    // Hand out positions to the 32 entries starting at f0 (warp-uniform), taking
    // each expert's next position from slot[e] and advancing it.
    auto place32 = [&](int f0, int e, int *slot) {
      const int f = f0 + lane;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int leader = __ffs(peers) - 1;
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int start = 0;
      if (lane == leader && e >= 0) {
        start = slot[e];
        slot[e] = start + __popc(peers);
      }
      start = __shfl_sync(0xffffffffu, start, leader);
      if (f < Tk) {
        if (e >= 0) {
          const int pos = start + rank;
          rb.sorted_idx[pos] = f;
          rb.inv_idx[f] = pos;
          if (rb.dest_rows) rb.dest_rows[f] = s_delta[e] + pos;
        } else {
          rb.inv_idx[f] = -1;
          if (rb.dest_rows) rb.dest_rows[f] = -1;
        }
      }
      __syncwarp();
    };
    auto load_id = [&](int f) {
      int e = f < Tk ? __ldg(ids + f) : -1;
      return (e < 0 || e >= E) ? -1 : e;
    };
    if (Tk <= kSmallRank) {
      if (warp == 0)
        for (int f0 = 0; f0 < Tk; f0 += 32) place32(f0, load_id(f0 + lane), s_cursor);
      return;
    }
    for (int base = 0; base < Tk; base += kRankChunk) {
      for (int i = threadIdx.x; i < kRankWarps * E; i += blockDim.x) s_wcnt[i] = 0;
      __syncthreads();
      int *my_cnt = s_wcnt + warp * E;
      const int w0 = base + warp * kRankPerWarp;
      int my_e[kRankPerWarp / 32];
#pragma unroll
      for (int j = 0; j < kRankPerWarp / 32; ++j) {
        const int e = load_id(w0 + 32 * j + lane);
        my_e[j] = e;
        if (e >= 0) atomicAdd(&my_cnt[e], 1);  // counts only: the order of the atomics is free
      }
      __syncthreads();
      for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = s_cursor[e];
        for (int w = 0; w < kRankWarps; ++w) {
          const int c = s_wcnt[w * E + e];
          s_wcnt[w * E + e] = run;
          run += c;
        }
        s_cursor[e] = run;
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kRankPerWarp / 32; ++j) place32(w0 + 32 * j, my_e[j], my_cnt);
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kRouteThreads) route_amax_kernel(
    const int32_t *__restrict__ ids, int T, int topk, int E, int has_shared, RouteBufs rb,
    const uint16_t *__restrict__ x, int64_t H, uint32_t *__restrict__ partials, int nparts,
    float *__restrict__ y_acc, uint32_t *err) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0) {
    route_block(ids, T, topk, E, has_shared, rb, err);
    return;
  }
  // amax partials + zeroing
  const int b = blockIdx.x - 1, nb = gridDim.x - 1;
  if (partials && b < nparts) {
    // partial b covers rows b, b + nparts, ... so every row lands in exactly one partial
    __shared__ uint32_t scratch[32];
    uint32_t m = 0;
    const int64_t chunks = H / 8;
    for (int64_t r = b; r < T; r += nparts) {
      const uint4 *row = reinterpret_cast<const uint4 *>(x + r * H);
      for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x) {
        const uint4 v = __ldg(row + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) m = max(m, scratch[i]);
      partials[b] = m;
    }
  }
  const int64_t n4 = static_cast<int64_t>(T) * H / 4;
  float4 *y4 = reinterpret_cast<float4 *>(y_acc);
  for (int64_t i = static_cast<int64_t>(b) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(nb) * blockDim.x)
    y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// One thread's share of the dispatch: the 16-element block c of token t, and the
// token's destination rows (routed entries, -1 when dropped).
struct DispatchIn {
  uint4 a, b;
  int dest[kDestRegs];
};

__device__ __forceinline__ void dispatch_load(const uint16_t *__restrict__ x, bool valid, int64_t t, int64_t c,
                                              int64_t H, int topk, const RouteBufs &rb, DispatchIn &in) {
  in.a = make_uint4(0u, 0u, 0u, 0u);
  in.b = in.a;
  if (valid) {
    const uint4 *src = reinterpret_cast<const uint4 *>(x + t * H + c * 16);
    in.a = __ldg(src);
    in.b = __ldg(src + 1);
  }
  const int *dest_src = rb.dest_rows + t * topk;
#pragma unroll
  for (int j = 0; j < kDestRegs; ++j)
    in.dest[j] = (valid && j < topk && topk <= kDestRegs) ? __ldg(dest_src + j) : -1;
}

// Encode the block with gs and write its codes and scale word into every destination
// row (the routed rows, then the shared segment).  Every lane of the warp calls this:
// the four scale bytes of a 64-element group are gathered with shuffles.
__device__ __forceinline__ void dispatch_store(const DispatchIn &in, bool valid, int64_t t, int64_t c, int64_t H,
                                               int topk, int E, int has_shared, const RouteBufs &rb, float gs,
                                               uint8_t *__restrict__ xq, uint8_t *__restrict__ xsf) {
  const int64_t kb = H / 16;
  const float six_gs = __fmul_rn(6.0f, gs);
  uint32_t codes[2] = {0u, 0u}, sfb = 0;
  if (valid) {
    const uint32_t w[8] = {in.a.x, in.a.y, in.a.z, in.a.w, in.b.x, in.b.y, in.b.z, in.b.w};
    sfb = encode_block16_bf16(w, gs, six_gs, codes);
  }
  const int lane = threadIdx.x & 31;
  uint32_t word = sfb << ((lane & 3) * 8);
  word |= __shfl_xor_sync(0xffffffffu, word, 1);
  word |= __shfl_xor_sync(0xffffffffu, word, 2);
  if (!valid) return;
  const uint2 cv = make_uint2(codes[0], codes[1]);
  const bool sf_writer = (lane & 3) == 0;
  auto put = [&](int64_t p) {
    *reinterpret_cast<uint2 *>(xq + p * (H / 2) + c * 8) = cv;
    if (sf_writer) *reinterpret_cast<uint32_t *>(xsf + sf_word_offset(p, c >> 2, kb >> 2)) = word;
  };
  if (topk <= kDestRegs) {
#pragma unroll
    for (int j = 0; j < kDestRegs; ++j)
      if (in.dest[j] >= 0) put(in.dest[j]);
  } else {
    const int *dest_src = rb.dest_rows + t * topk;
    for (int j = 0; j < topk; ++j) {
      const int p = __ldg(dest_src + j);
      if (p >= 0) put(p);
    }
  }
  if (has_shared) put(static_cast<int64_t>(__ldg(rb.pad_offsets + E)) + t);
}

// One thread per 16-element block of x (T, H).  Every token is quantised once
// and its codes and scales are written to its row in each routed expert's
// segment (and the shared expert's segment).
__global__ void __launch_bounds__(kDispatchThreads, 1) dispatch_quant_kernel(
    const uint16_t *__restrict__ x, int T, int64_t H, int topk, int E, int has_shared,
    const int32_t *__restrict__ ids, RouteBufs rb, const uint32_t *__restrict__ partials,
    int nparts, const float *__restrict__ gs_static, float *__restrict__ gs_out,
    uint8_t *__restrict__ xq, uint8_t *__restrict__ xsf) {
  __shared__ uint32_t scratch[32];
  pdl_wait();
  pdl_trigger();
  const int64_t kb = H / 16;
  const int64_t gb = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool valid = gb < static_cast<int64_t>(T) * kb;
  // (32-bit division while the index fits)
  const int64_t t = !valid ? 0 : (gb <= 0x7FFFFFFF ? static_cast<int64_t>(static_cast<uint32_t>(gb) / static_cast<uint32_t>(kb)) : gb / kb);
  const int64_t c = valid ? gb - t * kb : 0;
  // The block's 16 elements and the token's destination rows are loaded first, so
  // their latency overlaps the gs reduction.
  DispatchIn in;
  dispatch_load(x, valid, t, c, H, topk, rb, in);
  float gs;
  if (partials) {
    gs = gs_from_partials(partials, nparts, scratch);
    if (blockIdx.x == 0 && threadIdx.x == 0) *gs_out = gs;
  } else {
    gs = *gs_static;
  }
  dispatch_store(in, valid, t, c, H, topk, E, has_shared, rb, gs, xq, xsf);
}

__global__ void finalize_kernel(const float4 *__restrict__ acc, int64_t n4, uint2 *__restrict__ y) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = acc[i];
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    y[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo),
                      *reinterpret_cast<const uint32_t *>(&hi));
  }
}

}  // namespace

cudaError_t launch_route_amax(const int32_t *ids, int T, int topk, int E, int has_shared,
                              RouteBufs rb, const void *x, int64_t H, uint32_t *partials,
                              int nparts, float *y_acc, uint32_t *err, cudaStream_t s) {
  // enough helper blocks to zero y_acc quickly and to give every partial a block
  const int64_t n4 = static_cast<int64_t>(T) * H / 4;
  int helpers = static_cast<int>((n4 + kRouteThreads * 8 - 1) / (kRouteThreads * 8));
  if (partials && helpers < nparts) helpers = nparts;
  if (helpers < 1) helpers = 1;
  if (helpers > 1024) helpers = 1024;
  const size_t smem = route_smem_bytes(E);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(route_amax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(route_smem_bytes(kMaxExperts)));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(route_amax_kernel, dim3(1 + helpers), dim3(kRouteThreads), smem, s, ids, T, topk, E,
                    has_shared, rb, static_cast<const uint16_t *>(x), H, partials, nparts, y_acc, err);
}

cudaError_t launch_dispatch_quant(const void *x, int T, int64_t H, int topk, int E,
                                  int has_shared, const int32_t *ids, RouteBufs rb,
                                  const uint32_t *partials, int nparts, const float *gs_static,
                                  float *gs_out, uint8_t *xq, uint8_t *xsf, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(T) * (H / 16);
  const int64_t blocks = items > 0 ? (items + kDispatchThreads - 1) / kDispatchThreads : 1;
  return launch_pdl(dispatch_quant_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kDispatchThreads), 0, s,
                    static_cast<const uint16_t *>(x), T, H, topk, E, has_shared, ids, rb, partials, nparts,
                    gs_static, gs_out, xq, xsf);
}

cudaError_t launch_finalize(const float *y_acc, int64_t n, void *y, cudaStream_t s) {
  const int64_t n4 = n / 4;
  int64_t blocks = (n4 + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(finalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    reinterpret_cast<const float4 *>(y_acc), n4, static_cast<uint2 *>(y));
}

}  // namespace nvfp4
