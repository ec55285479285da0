// Device primitives for sm_103a: mbarriers, TMA, tcgen05 (TMEM, UMMA), bounded waits,
// and the NVFP4 block encoder shared by the activation quantiser and the fused
// GEMM epilogue.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace nvfp4 {

// ---------------------------------------------------------------- small helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void raise_device_error(uint32_t *err, uint32_t flag) {
  if (err) atomicOr(err, flag);
}

// Programmatic dependent launch: wait for the previous grid on the stream to complete
// (and its writes to be visible); allow the next grid to start launching.  Every kernel
// of the library triggers only after its own wait returned, so when a library kernel
// starts, every grid two or more launches back on the stream has completed.  The weight
// preparation kernel does not trigger at all: the launch after it starts once it has
// completed, so weights are final for any library kernel that reads them early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Raise the expected transaction bytes of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up when
// *abort becomes non-zero (another role gave up) or after timeout_ns; on a
// timeout it raises NVFP4_DEVERR_PIPELINE_TIMEOUT and sets *abort.  Returns
// true when the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort, uint32_t *err,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        *abort = 1;
        raise_device_error(err, NVFP4_DEVERR_PIPELINE_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- TMA / bulk copies

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                          uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gmem_src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 prefetch of one box of a tensor map (innermost coordinate 16-byte aligned) and of a
// contiguous range (16-byte aligned, a multiple of 16 bytes); neither waits for the data.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap *map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t *smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), fixed version bits 46..47 = 1, swizzle mode
// in bits 61..63 (0 none, 2 = 128-byte swizzle, 6 = 32-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes, uint32_t swizzle_mode) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
  return d;
}

// D(tmem, fp32) (+)= A(smem) * B(smem)^T, FP4 E2M1 operands with one UE4M3 scale
// per 16 K-elements taken from TMEM; M = 128, N and K = 64 fixed by idesc.
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i receives lane (base lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 1 column: thread i receives lane (base lane + i).
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  return r;
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread i writes lane (base lane + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32"
      " [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One 32-byte global store (256-bit vector); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// y[0..3] += (a, b, c, d): a 16-byte fp32 vector reduction in L2 that returns nothing,
// with an L2 cache policy.  Written out so the scatter-add stays a reduction whatever
// else the kernel contains (a value-returning atomic costs the w2 scatter about 2.4x at
// 4096 tokens).
__device__ __forceinline__ void red_add_v4(float4 *p, float a, float b, float c, float d, uint64_t policy) {
  asm volatile("red.relaxed.gpu.global.add.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(a),
               "f"(b), "f"(c), "f"(d), "l"(policy)
               : "memory");
}

// ---------------------------------------------------------------- CTA pairs (clusters of 2)

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of the object at the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  return a;
}

// Arrive on an mbarrier given by its shared::cluster address, without release semantics.
// For signals about tensor-memory accesses the ordering comes from tcgen05.wait::st / ::ld
// and tcgen05.fence::before_thread_sync; a release at cluster scope also waits for the
// SM's outstanding memory traffic (0.6-0.9 us per arrival while the TMA ring is busy).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait_bounded for a barrier that the peer CTA arrives on: acquire at cluster scope.
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                          uint32_t *err, uint64_t timeout_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        *abort = 1;
        raise_device_error(err, NVFP4_DEVERR_PIPELINE_TIMEOUT);
        return false;
      }
    }
  }
}

// Every thread of both CTAs of the pair must reach this (no thread may skip it).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Tensor memory of a CTA pair: one warp of each CTA of the pair takes part in the
// allocation, the relinquish and the deallocation, with the same column count.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrive on the barrier at the same offset in every CTA of `cta_mask` once the pair's
// tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// D (+)= A * B^T over the CTA pair: M = 256 (128 rows of A and of D in each CTA), N split
// between the two CTAs' shared memory (B rows), one UE4M3 scale per 16 K taken from each
// CTA's tensor memory.  Issued by one thread of the even CTA.
__device__ __forceinline__ void tc_mma_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// ---------------------------------------------------------------- NVFP4 block encoder

// Unsigned E4M3 byte -> fp32 (exact): bias 7, subnormal m * 2^-9 at exponent 0.
__device__ __forceinline__ float ue4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;
}

__device__ __forceinline__ uint32_t f32_to_ue4m3(float s) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3));
}

// Two fp32 values -> one byte of E2M1 codes, v0 in the low nibble, each code
// rounded to nearest-even on |v| with saturation at 6 and the sign bit of v
// kept (so a negative value that rounds to zero gives code 0x8).  The hardware
// conversion keeps the sign of a value that rounds to zero; the bit-exact
// quantiser tests hold it to that (-0.0, -0.1, negative midpoints).
__device__ __forceinline__ uint32_t e2m1x2_signed(float v0, float v1) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp4x2(make_float2(v0, v1), __NV_E2M1, cudaRoundNearest));
}

// Encode one 16-element block whose largest magnitude is amax, with global multiplier gs
// (six_gs = fl32(6 * gs)).  Returns the E4M3 scale byte; codes[0..1] receive the 8 code
// bytes (element 0 in the low nibble of byte 0).
__device__ __forceinline__ uint32_t encode_block16_amax(const float (&v)[16], float amax, float gs, float six_gs,
                                                        uint32_t (&codes)[2]) {
  const float s = (six_gs == 0.f) ? 0.f : __fdiv_rn(amax, six_gs);
  const uint32_t sf = f32_to_ue4m3(s);
  const float d = __fmul_rn(ue4m3_to_f32(sf), gs);
  const float r = __frcp_rn(d);
  if (d == 0.f || isinf(r)) {
    codes[0] = codes[1] = 0u;
    return sf;
  }
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const uint32_t byte = e2m1x2_signed(__fmul_rn(v[i], r), __fmul_rn(v[i + 1], r));
    w[i >> 3] |= byte << ((i & 7) * 4);
  }
  codes[0] = w[0];
  codes[1] = w[1];
  return sf;
}

// Encode one 16-element block with global multiplier gs (six_gs = fl32(6 * gs)).
// Returns the E4M3 scale byte; codes[0..1] receive the 8 code bytes (element 0
// in the low nibble of byte 0).
__device__ __forceinline__ uint32_t encode_block16(const float (&v)[16], float gs, float six_gs,
                                                   uint32_t (&codes)[2]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  return encode_block16_amax(v, amax, gs, six_gs, codes);
}

// The largest magnitude of 16 bf16 values packed two per word, as fp32: |bf16| orders like
// its unsigned bits once the sign is cleared, so two halves are compared per instruction.
__device__ __forceinline__ float amax_bf16x16(const uint32_t (&w)[8]) {
  uint32_t m = w[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int i = 1; i < 8; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
  return __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
}

// bf16 block (two 16-byte halves of bf16 pairs, element 0 in the low half of the first word)
// -> codes and scale byte, as encode_block16 on the unpacked values.
__device__ __forceinline__ uint32_t encode_block16_bf16(const uint32_t (&w)[8], float gs, float six_gs,
                                                        uint32_t (&codes)[2]) {
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  return encode_block16_amax(v, amax_bf16x16(w), gs, six_gs, codes);
}

// The same encoding with one 16-element block spread over four consecutive lanes
// (lanes 4b..4b+3 of the warp; every lane of the warp calls it): each lane holds
// four of the block's elements in v, in order.  The block amax is exchanged with
// shuffles and every lane derives the scale the same way encode_block16 does.
// Returns this lane's two code bytes (its first element in the low nibble of the
// low byte); *sf receives the block's E4M3 scale byte.
__device__ __forceinline__ uint32_t encode_block16_x4(float4 v, float gs, float six_gs, uint32_t *sf) {
  float amax = fmaxf(fmaxf(fmaxf(fmaxf(0.f, fabsf(v.x)), fabsf(v.y)), fabsf(v.z)), fabsf(v.w));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const float s = (six_gs == 0.f) ? 0.f : __fdiv_rn(amax, six_gs);
  *sf = f32_to_ue4m3(s);
  const float d = __fmul_rn(ue4m3_to_f32(*sf), gs);
  const float r = __frcp_rn(d);
  if (d == 0.f || isinf(r)) return 0u;
  return e2m1x2_signed(__fmul_rn(v.x, r), __fmul_rn(v.y, r)) |
         (e2m1x2_signed(__fmul_rn(v.z, r), __fmul_rn(v.w, r)) << 8);
}

// Row and column of a flat block index g = r * kb + c, advanced by a fixed step with no
// division in the loop (the step's own quotient and remainder are computed once).  Idx is
// int32_t where every index and offset of the launch fits, which halves the integer work.
template <typename Idx>
struct RowColT {
  Idx r, c;
  __device__ __forceinline__ void init(Idx g, Idx kb) {
    r = g / kb;
    c = g - r * kb;
  }
  __device__ __forceinline__ void advance(Idx step_r, Idx step_c, Idx kb) {
    c += step_c;
    r += step_r;
    if (c >= kb) {
      c -= kb;
      ++r;
    }
  }
};
using RowCol = RowColT<int64_t>;

// Byte offset of the 32-bit word holding scales (row r, columns 4c'..4c'+3) in
// the swizzled layout, for a buffer whose rows carry K elements (kc4 = K / 64
// four-column groups per row).
__device__ __forceinline__ size_t sf_word_offset(int64_t r, int64_t col4, int64_t kc4) {
  return (static_cast<size_t>(r >> 7) * kc4 + col4) * 512u + static_cast<size_t>(r & 31) * 16u +
         static_cast<size_t>((r & 127) >> 5) * 4u;
}
// The same in 32-bit arithmetic, for buffers below 2^31 bytes.
__device__ __forceinline__ uint32_t sf_word_offset32(uint32_t r, uint32_t col4, uint32_t kc4) {
  return ((r >> 7) * kc4 + col4) * 512u + (r & 31u) * 16u + ((r & 127u) >> 5) * 4u;
}

// Global scale from the block partials: gs = fl32(amax / 2688).
__device__ __forceinline__ float gs_from_partials(const uint32_t *partials, int nparts,
                                                  uint32_t *scratch) {
  uint32_t m = 0;
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) m = max(m, partials[i]);
  // reduce across the block
#pragma unroll
  for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < static_cast<int>(blockDim.x >> 5) ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) scratch[0] = m;
  }
  __syncthreads();
  const float amax = __uint_as_float(scratch[0] << 16);
  return __fdiv_rn(amax, 2688.0f);
}

}  // namespace nvfp4
