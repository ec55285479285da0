// Host side of the C ABI: argument validation, workspace layout, TMA tensor-map
// encoding and the launch sequences of each entry point.  Nothing here
// allocates device memory or synchronises the host (except
// nvfp4_get_device_error).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace nvfp4 {
namespace {

// ---------------------------------------------------------------- error reporting

thread_local char g_last_error[512] = "";

nvfp4_status fail(nvfp4_status st, const char *fn, const char *fmt, ...) {
  int n = std::snprintf(g_last_error, sizeof(g_last_error), "%s: ", fn);
  if (n < 0) n = 0;
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_last_error + n, sizeof(g_last_error) - static_cast<size_t>(n), fmt, ap);
  va_end(ap);
  return st;
}

nvfp4_status cuda_fail(const char *fn, cudaError_t e, const char *what) {
  return fail(NVFP4_ERR_CUDA, fn, "%s: %s", what, cudaGetErrorString(e));
}

#define NV_REQUIRE(cond, status, ...) \
  do {                                \
    if (!(cond)) return fail(status, __func__, __VA_ARGS__); \
  } while (0)

#define NV_CUDA(expr, what)                          \
  do {                                               \
    cudaError_t e_ = (expr);                         \
    if (e_ != cudaSuccess) return cuda_fail(__func__, e_, what); \
  } while (0)

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// ---------------------------------------------------------------- per-device state

__device__ uint32_t g_device_flags;

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sms = 0;
  uint32_t *flags = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

nvfp4_status device_info(const char *fn, DeviceInfo **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(fn, e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_UNSUPPORTED_DEVICE, fn, "device %d", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(fn, e, "cudaDeviceGetAttribute");
    d.supported = major == 10 && minor == 3;
    if (d.supported) {
      void *p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_flags)) != cudaSuccess)
        return cuda_fail(fn, e, "cudaGetSymbolAddress(device flags)");
      d.flags = static_cast<uint32_t *>(p);
    }
    d.ready = true;
    if (!d.supported)
      return fail(NVFP4_ERR_UNSUPPORTED_DEVICE, fn, "device %d is sm_%d%d; this library is built for sm_103a",
                  dev, major, minor);
  }
  if (!d.supported) return fail(NVFP4_ERR_UNSUPPORTED_DEVICE, fn, "device %d is not sm_103", dev);
  *out = &d;
  return NVFP4_OK;
}

// ---------------------------------------------------------------- TMA descriptors

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

nvfp4_status get_encoder(const char *fn, EncodeTiledFn *out) {
  static EncodeTiledFn encode = nullptr;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) encode = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!encode) return fail(NVFP4_ERR_CUDA, fn, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *out = encode;
  return NVFP4_OK;
}

// 2-D byte tensor (rows x row_bytes, row stride ld_bytes) read in boxes of
// 128 bytes x box_rows with the 128-byte swizzle.
nvfp4_status make_map(const char *fn, CUtensorMap *m, const void *base, int64_t row_bytes,
                      int64_t rows, int64_t ld_bytes, int box_rows, int box_bytes = 128,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn encode;
  nvfp4_status st = get_encoder(fn, &encode);
  if (st != NVFP4_OK) return st;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(NVFP4_ERR_CUDA, fn, "cuTensorMapEncodeTiled failed (%d) for %lld x %lld bytes", static_cast<int>(r),
                static_cast<long long>(rows), static_cast<long long>(row_bytes));
  return NVFP4_OK;
}

// Prepared (tile-major) weights of rows x K: blocks of 128 rows x 128 bytes, read through a
// map of 128-byte rows with 128-row boxes.
nvfp4_status make_weight_map(const char *fn, CUtensorMap *m, const void *w, int64_t rows, int64_t K) {
  const int64_t slabs = (K / 2 + 127) / 128;
  return make_map(fn, m, w, 128, rows * slabs, 128, 128);
}

// The same weights read one 64-element K step at a time: boxes of 128 rows x 32 bytes at
// x = 32 (k % 4) of slab k / 4, 32-byte swizzle (the one-token kernel's w2 slices).
nvfp4_status make_weight_slice_map(const char *fn, CUtensorMap *m, const void *w, int64_t rows, int64_t K) {
  const int64_t slabs = (K / 2 + 127) / 128;
  return make_map(fn, m, w, 128, rows * slabs, 128, 128, 32, CU_TENSOR_MAP_SWIZZLE_32B);
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

size_t sf_bytes(int64_t rows, int64_t K) {
  return static_cast<size_t>(round_up(rows, 128)) * static_cast<size_t>(round_up(K / 16, 4));
}

// ---------------------------------------------------------------- dense linear workspace

struct LinearWs {
  size_t xq, xsf, partials, total;
};
LinearWs linear_ws(int64_t M, int64_t K) {
  LinearWs w;
  size_t off = 0;
  w.xq = off;
  off = align256(off + static_cast<size_t>(M) * static_cast<size_t>(K / 2));
  w.xsf = off;
  off = align256(off + sf_bytes(M, K));
  w.partials = off;
  off = align256(off + kMaxPartials * sizeof(uint32_t));
  w.total = off;
  return w;
}

// ---------------------------------------------------------------- MoE workspace

nvfp4_moe_ws_layout moe_layout(int64_t T, int64_t H, int64_t I, int64_t E, int topk, int has_shared) {
  nvfp4_moe_ws_layout L;
  std::memset(&L, 0, sizeof(L));
  const int64_t G = E + (has_shared ? 1 : 0);
  const int64_t Tk = T * topk;
  const int64_t routed_rows = round_up(Tk + 127 * (E < Tk ? E : Tk), 128);
  L.rows_capacity = routed_rows + (has_shared ? round_up(T, 128) : 0);
  const size_t rc = static_cast<size_t>(L.rows_capacity);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  L.counts = take(static_cast<size_t>(G) * 4);
  L.offsets = take(static_cast<size_t>(G + 1) * 4);
  L.pad_offsets = take(static_cast<size_t>(G + 1) * 4);
  L.tile_offsets = take(static_cast<size_t>(G + 1) * 4);
  L.sorted_idx = take(static_cast<size_t>(Tk > 0 ? Tk : 1) * 4);
  L.inv_idx = take(static_cast<size_t>(Tk > 0 ? Tk : 1) * 4);
  L.dest_rows = take(static_cast<size_t>(Tk > 0 ? Tk : 1) * 4);
  // one entry per tile; with kABoxRows-row tiles a group of c rows takes ceil(c / 32)
  // <= 4 ceil(c / 128) entries, and the 128-row padded segments sum to at most rc
  L.tile_table = take(rc / kABoxRows * 16 + 16);
  L.amax_partials = take(kMaxPartials * 4);
  L.xq = take(rc * static_cast<size_t>(H / 2));
  L.xsf = take(sf_bytes(L.rows_capacity, H));
  L.hq = take(rc * static_cast<size_t>(I / 2));
  L.hsf = take(sf_bytes(L.rows_capacity, I));
  L.y_acc = take(static_cast<size_t>(T) * static_cast<size_t>(H) * 4);
  L.total = off;
  return L;
}

nvfp4_status check_moe_shape(const char *fn, int64_t T, int64_t H, int64_t I, int64_t E, int topk) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || topk <= 0)
    return fail(NVFP4_ERR_INVALID_ARG, fn, "sizes must be positive (T >= 0): T=%lld H=%lld I=%lld E=%lld topk=%d",
                (long long)T, (long long)H, (long long)I, (long long)E, topk);
  if (H % 128) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, fn, "H=%lld must be a multiple of 128", (long long)H);
  if (I % 64) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, fn, "I=%lld must be a multiple of 64", (long long)I);
  if (E > kMaxExperts) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, fn, "E=%lld above %d", (long long)E, kMaxExperts);
  if (topk > kMaxTopk) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, fn, "topk=%d above %d", topk, kMaxTopk);
  if (T * topk >= (int64_t(1) << 30) || H > (int64_t(1) << 20) || I > (int64_t(1) << 20))
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, fn, "sizes too large");
  return NVFP4_OK;
}

nvfp4_status check_ws(const char *fn, const void *ws, size_t ws_bytes, size_t need) {
  if (ws_bytes < need)
    return fail(NVFP4_ERR_WORKSPACE, fn, "workspace of %zu bytes, %zu needed", ws_bytes, need);
  if (need && !ws) return fail(NVFP4_ERR_INVALID_ARG, fn, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(NVFP4_ERR_MISALIGNED, fn, "workspace must be 256-byte aligned");
  return NVFP4_OK;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

RouteBufs route_bufs(void *ws, const nvfp4_moe_ws_layout &L) {
  RouteBufs rb;
  rb.counts = at<int>(ws, L.counts);
  rb.offsets = at<int>(ws, L.offsets);
  rb.pad_offsets = at<int>(ws, L.pad_offsets);
  rb.tile_offsets = at<int>(ws, L.tile_offsets);
  rb.sorted_idx = at<int>(ws, L.sorted_idx);
  rb.inv_idx = at<int>(ws, L.inv_idx);
  rb.dest_rows = at<int>(ws, L.dest_rows);
  rb.tile_table = at<int4>(ws, L.tile_table);
  rb.tile_shift = 7;  // kBlockM-row tiles unless the caller sets moe_tile_shift(T)
  return rb;
}

// ---------------------------------------------------------------- stage bodies (validated inputs)

nvfp4_status moe_dispatch_impl(const char *fn, DeviceInfo *d, const void *x, int64_t T, int64_t H, int64_t I,
                               int64_t E, int topk, const int32_t *ids, int has_shared, int a1_gs_mode,
                               float *a1_gs, void *ws, cudaStream_t s) {
  const nvfp4_moe_ws_layout L = moe_layout(T, H, I, E, topk, has_shared);
  RouteBufs rb = route_bufs(ws, L);
  rb.tile_shift = moe_tile_shift(T);  // the GEMM launches on this workspace use the same T
  const bool dyn = a1_gs_mode == NVFP4_GS_DYNAMIC;
  const int nparts = amax_partial_count(T, H);
  uint32_t *partials = dyn ? at<uint32_t>(ws, L.amax_partials) : nullptr;
  NV_CUDA(launch_route_amax(ids, static_cast<int>(T), topk, static_cast<int>(E), has_shared, rb, x, H, partials,
                            nparts, at<float>(ws, L.y_acc), d->flags, s),
          "route kernel launch");
  NV_CUDA(launch_dispatch_quant(x, static_cast<int>(T), H, topk, static_cast<int>(E), has_shared, ids, rb, partials,
                                nparts, a1_gs, a1_gs, at<uint8_t>(ws, L.xq), at<uint8_t>(ws, L.xsf), s),
          "dispatch kernel launch");
  (void)fn;
  return NVFP4_OK;
}

// One-token w13 (nvfp4_moe_forward at T = 1): the w13 CTAs quantise x themselves and take
// their schedule from the top-k ids, so no dispatch launch runs and the weights stream while
// the routing kernel is still working.
struct Tok1 {
  const void *x;
  const int32_t *ids;
  bool dynamic;
  float *a1_gs;
  // the down projection, fused into the same launch (split K over I): w2 codes, scales and
  // weight scales, the shared expert's, the routing weights
  const uint8_t *w2, *w2_sf, *sh_w2, *sh_w2_sf;
  const float *w2_ws2, *sh_ws2, *topk_w;
};

bool tok1_applies(int64_t T, int64_t H, int topk) { return T == 1 && topk <= kTok1MaxTopk && H <= kTok1MaxK; }

// Weight stages of a GEMM's first tile prefetched into L2 beyond its ring before the
// previous launch of the chain completes (w13, w2).
constexpr int kEarlyL2W13 = 0;
constexpr int kEarlyL2W2 = 4;

nvfp4_status moe_gemm_impl(const char *fn, DeviceInfo *d, Epi epi, int64_t T, int64_t H, int64_t I, int64_t E,
                           int topk, const uint8_t *w, const uint8_t *w_sf, const float *w_ws2,
                           const uint8_t *sh_w, const uint8_t *sh_sf, const float *sh_ws2, const float *gs_a,
                           const float *gs_out, const float *topk_w, float *h_debug, void *ws, cudaStream_t s,
                           const Tok1 *tok1 = nullptr) {
  const int has_shared = sh_w != nullptr;
  const nvfp4_moe_ws_layout L = moe_layout(T, H, I, E, topk, has_shared);
  if (T == 0) return NVFP4_OK;
  const bool w13 = epi == Epi::kW13;
  const int64_t N = w13 ? 2 * I : H, K = w13 ? H : I;
  CUtensorMap ta, tb, tbs;
  nvfp4_status st = make_map(fn, &ta, at<uint8_t>(ws, w13 ? L.xq : L.hq), K / 2, L.rows_capacity, K / 2, kABoxRows);
  if (st != NVFP4_OK) return st;
  if ((st = make_weight_map(fn, &tb, w, E * N, K)) != NVFP4_OK) return st;
  if (has_shared) {
    if ((st = make_weight_map(fn, &tbs, sh_w, N, K)) != NVFP4_OK) return st;
  } else {
    tbs = tb;
  }
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.G = static_cast<int>(E) + has_shared;
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.counts = at<int>(ws, L.counts);
  a.offsets = at<int>(ws, L.offsets);
  a.pad_offsets = at<int>(ws, L.pad_offsets);
  a.tile_offsets = at<int>(ws, L.tile_offsets);
  a.tile_table = at<const int4>(ws, L.tile_table);
  a.shared_group = has_shared ? static_cast<int>(E) : -1;
  a.a_sf = at<uint8_t>(ws, w13 ? L.xsf : L.hsf);
  a.a_kc_total = static_cast<int>(K / 64);
  a.b_sf = w_sf;
  a.b_sf_shared = sh_sf;
  a.gs_a = gs_a;
  a.ws2 = w_ws2;
  a.ws2_shared = sh_ws2 ? sh_ws2 + (w13 ? 0 : 1) : nullptr;
  a.gs_out = gs_out;
  a.err = d->flags;
  a.early_b = 1;  // dispatch (or w13) precedes this launch; routing and weights are older
  a.early_l2 = w13 ? kEarlyL2W13 : kEarlyL2W2;
  if (w13) {
    a.out = at<uint8_t>(ws, L.hq);
    a.out_sf = at<uint8_t>(ws, L.hsf);
    a.h_debug = h_debug;
    a.out_ld = static_cast<int>(I / 2);
  } else {
    a.out = at<float>(ws, L.y_acc);
    a.out_ld = static_cast<int>(H);
    a.sorted_idx = at<int>(ws, L.sorted_idx);
    a.topk_w = topk_w;
    a.topk = topk;
  }
  if (tok1 != nullptr) {
    a.qa_x = tok1->x;
    a.qa_ld = H;
    a.qa_gs_static = tok1->dynamic ? nullptr : tok1->a1_gs;
    a.qa_gs_out = tok1->dynamic ? tok1->a1_gs : nullptr;
    a.tok1_ids = tok1->ids;
    a.tok1_E = static_cast<int>(E);
    a.topk = topk;
    a.early_b = 0;  // nothing is read before the wait but the ids and the weights
    CUtensorMap t2, t2s;
    if ((st = make_weight_slice_map(fn, &t2, tok1->w2, E * H, I)) != NVFP4_OK) return st;
    if (has_shared) {
      if ((st = make_weight_slice_map(fn, &t2s, tok1->sh_w2, H, I)) != NVFP4_OK) return st;
    } else {
      t2s = t2;
    }
    a.p2_N = static_cast<int>(H);
    a.p2_K = static_cast<int>(I);
    a.p2_acc = at<float>(ws, L.y_acc);
    a.p2_sf = tok1->w2_sf;
    a.p2_sf_shared = tok1->sh_w2_sf;
    a.p2_ws2 = tok1->w2_ws2;
    a.p2_ws2_shared = tok1->sh_ws2 ? tok1->sh_ws2 + 1 : nullptr;
    a.p2_topk_w = tok1->topk_w;
    NV_CUDA(launch_gemm_tok1(tb, tbs, t2, t2s, a, d->sms * kCtasPerSm, s), "one-token MoE launch");
    return NVFP4_OK;
  }
  // The routing cut the groups into tiles of moe_tile_rows(T) rows: 32-row tiles fit one
  // A box each, so the ring with 4 small stages applies.
  const bool small_a = moe_tile_rows(T) == kABoxRows;
  NV_CUDA(launch_gemm(epi, ta, tb, tbs, a, d->sms * kCtasPerSm, false, small_a, s), "grouped GEMM launch");
  return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

int nvfp4_abi_version(void) { return NVFP4_ABI_VERSION; }

const char *nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NVFP4_ERR_MISALIGNED: return "misaligned pointer or stride";
    case NVFP4_ERR_WORKSPACE: return "workspace too small";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_DEVICE_FAULT: return "device-side fault flag";
    case NVFP4_ERR_TIMEOUT: return "device-side wait timed out";
    case NVFP4_ERR_UNSUPPORTED_DEVICE: return "unsupported device";
  }
  return "unknown status";
}

const char *nvfp4_last_error_string(void) { return g_last_error; }

nvfp4_status nvfp4_get_device_error(void *stream, int32_t *flags) {
  NV_REQUIRE(flags != nullptr, NVFP4_ERR_INVALID_ARG, "flags is NULL");
  DeviceInfo *d;
  nvfp4_status st = device_info(__func__, &d);
  if (st != NVFP4_OK) return st;
  NV_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "cudaStreamSynchronize");
  uint32_t v = 0;
  NV_CUDA(cudaMemcpy(&v, d->flags, sizeof(v), cudaMemcpyDeviceToHost), "read device flags");
  const uint32_t zero = 0;
  NV_CUDA(cudaMemcpy(d->flags, &zero, sizeof(zero), cudaMemcpyHostToDevice), "clear device flags");
  *flags = static_cast<int32_t>(v);
  if (v & NVFP4_DEVERR_PIPELINE_TIMEOUT) return fail(NVFP4_ERR_TIMEOUT, __func__, "device flags 0x%x", v);
  if (v) return fail(NVFP4_ERR_DEVICE_FAULT, __func__, "device flags 0x%x", v);
  return NVFP4_OK;
}

size_t nvfp4_sf_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return sf_bytes(rows, K);
}

size_t nvfp4_quantize_workspace_bytes(int64_t M, int64_t K) {
  (void)M;
  (void)K;
  return kMaxPartials * sizeof(uint32_t);
}

nvfp4_status nvfp4_quantize_act(const void *x, int64_t M, int64_t K, int64_t ldx, int gs_mode, float *gs,
                                uint8_t *q, uint8_t *sf, int sf_layout, void *ws, size_t ws_bytes,
                                void *stream) {
  NV_REQUIRE(M >= 0 && K > 0, NVFP4_ERR_INVALID_ARG, "M=%lld K=%lld", (long long)M, (long long)K);
  NV_REQUIRE(K % 64 == 0, NVFP4_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 64", (long long)K);
  NV_REQUIRE(gs_mode == NVFP4_GS_DYNAMIC || gs_mode == NVFP4_GS_STATIC, NVFP4_ERR_INVALID_ARG, "gs_mode %d", gs_mode);
  NV_REQUIRE(sf_layout == NVFP4_SF_SWIZZLED || sf_layout == NVFP4_SF_LINEAR, NVFP4_ERR_INVALID_ARG, "sf_layout %d",
             sf_layout);
  NV_REQUIRE(gs != nullptr && ((x != nullptr && q != nullptr && sf != nullptr) || M == 0), NVFP4_ERR_INVALID_ARG,
             "NULL pointer argument");
  NV_REQUIRE(ldx >= K && ldx % 8 == 0, NVFP4_ERR_MISALIGNED, "ldx=%lld must be >= K and a multiple of 8",
             (long long)ldx);
  NV_REQUIRE(aligned(x, 16) && aligned(q, 16) && aligned(sf, 16) && aligned(gs, 4), NVFP4_ERR_MISALIGNED,
             "x, q and sf must be 16-byte aligned");
  NV_REQUIRE(M * (ldx > K ? ldx : K) < (int64_t(1) << 40), NVFP4_ERR_UNSUPPORTED_SHAPE, "tensor too large");
  const bool dyn = gs_mode == NVFP4_GS_DYNAMIC;
  if (dyn) {
    nvfp4_status st = check_ws(__func__, ws, ws_bytes, nvfp4_quantize_workspace_bytes(M, K));
    if (st != NVFP4_OK) return st;
  }
  DeviceInfo *d;
  nvfp4_status st = device_info(__func__, &d);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t *partials = dyn ? static_cast<uint32_t *>(ws) : nullptr;
  NV_CUDA(launch_act_quant(x, M, K, ldx, dyn, partials, gs, gs, q, sf, sf_layout, s), "quantize kernel launch");
  return NVFP4_OK;
}

size_t nvfp4_rmsnorm_quantize_workspace_bytes(int64_t M, int64_t K) {
  (void)K;
  if (M < 0) return 0;
  return align256(kMaxPartials * sizeof(uint32_t)) + align256(static_cast<size_t>(M) * sizeof(float));
}

static nvfp4_status check_norm_args(const char *fn, const void *x, int64_t M, int64_t K, int64_t ldx,
                                    const void *gamma, float eps) {
  if (!(M >= 0 && K > 0)) return fail(NVFP4_ERR_INVALID_ARG, fn, "M=%lld K=%lld", (long long)M, (long long)K);
  if (K % 64) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, fn, "K=%lld must be a multiple of 64", (long long)K);
  if (!gamma || (!x && M > 0)) return fail(NVFP4_ERR_INVALID_ARG, fn, "NULL pointer argument");
  if (!(eps >= 0.f) || !(eps < 1e30f)) return fail(NVFP4_ERR_INVALID_ARG, fn, "eps must be finite and >= 0");
  if (ldx < K || ldx % 8) return fail(NVFP4_ERR_MISALIGNED, fn, "ldx=%lld must be >= K and a multiple of 8",
                                      (long long)ldx);
  if (!aligned(x, 16) || !aligned(gamma, 16)) return fail(NVFP4_ERR_MISALIGNED, fn, "x and gamma must be 16-byte aligned");
  return NVFP4_OK;
}

nvfp4_status nvfp4_rmsnorm(const void *x, int64_t M, int64_t K, int64_t ldx, const void *gamma, float eps, void *y,
                           void *stream) {
  nvfp4_status st = check_norm_args(__func__, x, M, K, ldx, gamma, eps);
  if (st != NVFP4_OK) return st;
  NV_REQUIRE(y || M == 0, NVFP4_ERR_INVALID_ARG, "y is NULL");
  NV_REQUIRE(aligned(y, 16), NVFP4_ERR_MISALIGNED, "y must be 16-byte aligned");
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  if (M == 0) return NVFP4_OK;
  NV_CUDA(launch_rmsnorm_stats(x, M, K, ldx, gamma, eps, nullptr, nullptr, amax_partial_count(M, K), y,
                               static_cast<cudaStream_t>(stream)),
          "rmsnorm kernel launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_rmsnorm_quantize(const void *x, int64_t M, int64_t K, int64_t ldx, const void *gamma, float eps,
                                    int gs_mode, float *gs, uint8_t *q, uint8_t *sf, int sf_layout, void *x_normed,
                                    void *ws, size_t ws_bytes, void *stream) {
  nvfp4_status st = check_norm_args(__func__, x, M, K, ldx, gamma, eps);
  if (st != NVFP4_OK) return st;
  NV_REQUIRE(gs_mode == NVFP4_GS_DYNAMIC || gs_mode == NVFP4_GS_STATIC, NVFP4_ERR_INVALID_ARG, "gs_mode %d", gs_mode);
  NV_REQUIRE(sf_layout == NVFP4_SF_SWIZZLED || sf_layout == NVFP4_SF_LINEAR, NVFP4_ERR_INVALID_ARG, "sf_layout %d",
             sf_layout);
  NV_REQUIRE(gs && ((q && sf) || M == 0), NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(aligned(q, 16) && aligned(sf, 16) && aligned(x_normed, 16) && aligned(gs, 4), NVFP4_ERR_MISALIGNED,
             "q, sf and x_normed must be 16-byte aligned");
  if ((st = check_ws(__func__, ws, ws_bytes, nvfp4_rmsnorm_quantize_workspace_bytes(M, K))) != NVFP4_OK) return st;
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool dyn = gs_mode == NVFP4_GS_DYNAMIC;
  const int nparts = amax_partial_count(M, K);
  uint32_t *partials = dyn ? static_cast<uint32_t *>(ws) : nullptr;
  float *inv_rms = at<float>(ws, align256(kMaxPartials * sizeof(uint32_t)));
  if (M > 0)
    NV_CUDA(launch_rmsnorm_stats(x, M, K, ldx, gamma, eps, inv_rms, partials, nparts, x_normed, s),
            "rmsnorm statistics kernel launch");
  else if (dyn)
    NV_CUDA(launch_amax_partials(x, 0, K, ldx, partials, 1, s), "amax kernel launch");
  NV_CUDA(launch_rmsnorm_quantize(x, M, K, ldx, gamma, inv_rms, partials, M > 0 ? nparts : 1, gs, gs, q, sf, sf_layout,
                                  s),
          "rmsnorm quantize kernel launch");
  return NVFP4_OK;
}

// Output widths: a multiple of 128, or of 16 for one group (the dense linear), whose last
// 128-row weight tile is then padded with zero rows.
static bool weight_rows_ok(int64_t G, int64_t N) { return N % 128 == 0 || (G == 1 && N % 16 == 0); }

size_t nvfp4_prepared_weight_bytes(int64_t G, int64_t N, int64_t K) {
  if (G <= 0 || N <= 0 || K <= 0 || K % 64 || !weight_rows_ok(G, N)) return 0;
  return static_cast<size_t>(G) * static_cast<size_t>(round_up(N, 128)) * static_cast<size_t>((K / 2 + 127) / 128) *
         128u;
}

nvfp4_status nvfp4_prepare_weights(const uint8_t *w, const uint8_t *sf, int64_t G, int64_t N, int64_t K, int flags,
                                   uint8_t *w_out, uint8_t *sf_out, void *stream) {
  NV_REQUIRE(w && sf && w_out && sf_out, NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(G > 0 && N > 0 && K > 0, NVFP4_ERR_INVALID_ARG, "G=%lld N=%lld K=%lld", (long long)G, (long long)N,
             (long long)K);
  NV_REQUIRE(flags == NVFP4_PREP_PLAIN || flags == NVFP4_PREP_W13_INTERLEAVE, NVFP4_ERR_INVALID_ARG, "flags %d",
             flags);
  NV_REQUIRE(K % 64 == 0 && weight_rows_ok(G, N) && (N % 128 == 0 || flags == NVFP4_PREP_PLAIN),
             NVFP4_ERR_UNSUPPORTED_SHAPE,
             "K=%lld must be a multiple of 64 and N=%lld of 128 (of 16 for one group without the w13 interleave)",
             (long long)K, (long long)N);
  NV_REQUIRE(aligned(w, 16) && aligned(sf, 16) && aligned(w_out, 16) && aligned(sf_out, 16), NVFP4_ERR_MISALIGNED,
             "pointers must be 16-byte aligned");
  NV_REQUIRE(w != w_out && sf != sf_out, NVFP4_ERR_INVALID_ARG, "prepare cannot run in place");
  DeviceInfo *d;
  nvfp4_status st = device_info(__func__, &d);
  if (st != NVFP4_OK) return st;
  NV_CUDA(launch_prepare(w, sf, G, N, K, flags, w_out, sf_out, static_cast<cudaStream_t>(stream)),
          "prepare kernel launch");
  return NVFP4_OK;
}

size_t nvfp4_linear_workspace_bytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0) return 0;
  return linear_ws(M, K).total;
}

// Dense GEMM, or G uniform groups where group g multiplies columns [gK, (g+1)K) of the
// quantised activations with its own weight (G, N, K/2) into output columns [gN, (g+1)N).
// Weight stages of a linear's first tile prefetched into L2 beyond the ring at kernel start
// (before the dependency wait: the weights are older than the previous launch).
constexpr int kLinearEarlyL2 = 16;

static nvfp4_status gemm_dense(const char *fn, DeviceInfo *d, const uint8_t *xq, const uint8_t *xsf, const float *gs,
                               int64_t M, int64_t K, int64_t N, const uint8_t *w, const uint8_t *w_sf,
                               const float *ws2, void *y, cudaStream_t s, int early_b = 0, int64_t G = 1) {
  if (M == 0) return NVFP4_OK;
  // many rows and N a multiple of 256: 256 x 256 tiles on CTA pairs
  const int pair_clusters = (G == 1 && N % 256 == 0 && M >= kPairMinM) ? gemm_pair_max_clusters() : 0;
  CUtensorMap ta, tb;
  nvfp4_status st = make_map(fn, &ta, xq, G * K / 2, M, G * K / 2, pair_clusters > 0 ? 128 : kABoxRows);
  if (st != NVFP4_OK) return st;
  if ((st = make_weight_map(fn, &tb, w, G * round_up(N, kBlockN), K)) != NVFP4_OK) return st;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.G = static_cast<int>(G);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.dense_M = static_cast<int>(M);
  a.shared_group = -1;
  a.a_sf = xsf;
  a.a_kc_total = static_cast<int>(G * K / 64);
  a.a_group_koff = G > 1 ? static_cast<int>(K / 64) : 0;
  a.b_sf = w_sf;
  a.gs_a = gs;
  a.ws2 = ws2;
  a.out = y;
  a.out_ld = static_cast<int>(G * N);
  a.out_group_cols = static_cast<int>(N);
  a.err = d->flags;
  a.early_b = early_b;
  a.early_l2 = early_b ? kLinearEarlyL2 : 0;  // the first tile's stages beyond the ring, into L2
  if (pair_clusters > 0) {
    const int64_t pair_tiles = ((M + 255) / 256) * (N / 256);
    const int clusters = static_cast<int>(pair_tiles < pair_clusters ? pair_tiles : pair_clusters);
    NV_CUDA(launch_gemm_pair(ta, tb, a, clusters, s), "pair GEMM launch");
    return NVFP4_OK;
  }
  const int64_t tiles = G * ((M + kBlockM - 1) / kBlockM) * ((N + kBlockN - 1) / kBlockN);
  const int grid = static_cast<int>(tiles < d->sms * kCtasPerSm ? tiles : d->sms * kCtasPerSm);
  // M <= 32: every tile has at most one 32-row A box, so the ring with 4 small stages applies
  NV_CUDA(launch_gemm(Epi::kLinear, ta, tb, tb, a, grid, grid <= d->sms, M <= kABoxRows, s), "GEMM launch");
  return NVFP4_OK;
}

// Dense (G = 1) or fixed-group linear for 1 <= M <= 32 rows in one launch: the GEMM CTAs
// quantise x themselves (same arithmetic as nvfp4_quantize_act) into resident A boxes.
// Every CTA reduces the amax over all G*K columns and quantises its group's K of them.
static nvfp4_status linear_fused(const char *fn, DeviceInfo *d, const void *x, int64_t M, int64_t G, int64_t K,
                                 int64_t N, const uint8_t *w, const uint8_t *w_sf, const float *ws2, bool dyn,
                                 float *gs, void *y, cudaStream_t s) {
  CUtensorMap tb;
  nvfp4_status st = make_weight_map(fn, &tb, w, G * round_up(N, kBlockN), K);
  if (st != NVFP4_OK) return st;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.G = static_cast<int>(G);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.dense_M = static_cast<int>(M);
  a.shared_group = -1;
  a.b_sf = w_sf;
  a.ws2 = ws2;
  a.out = y;
  a.out_ld = static_cast<int>(G * N);
  a.out_group_cols = static_cast<int>(N);
  a.err = d->flags;
  a.early_b = 1;  // the weights are older than the previous launch (prepare_weights does not trigger early)
  a.early_l2 = kLinearEarlyL2;  // the tile's stages beyond the ring: into L2 before the dependency wait
  a.qa_x = x;
  a.qa_ld = G * K;
  a.qa_gs_static = dyn ? nullptr : gs;
  a.qa_gs_out = dyn ? gs : nullptr;
  const int64_t tiles = G * ((N + kBlockN - 1) / kBlockN);
  // a dense linear's CTAs may take several tiles (all of group 0); groups need one tile per CTA
  const int grid = static_cast<int>(tiles < d->sms ? tiles : d->sms);
  NV_CUDA(launch_gemm_quant_a(tb, a, grid, s), "fused linear launch");
  return NVFP4_OK;
}

static bool linear_fusable(const DeviceInfo *d, int64_t M, int64_t G, int64_t K, int64_t N) {
  return M >= 1 && M <= kABoxRows && K <= kQuantMaxK && M * K <= kQuantMaxElems &&
         M * G * K <= 4 * kQuantMaxElems && (G == 1 || G * ((N + kBlockN - 1) / kBlockN) <= d->sms);
}

#define NV_CHECK_GEMM_SHAPE(M, K, N)                                                                          \
  NV_REQUIRE((M) >= 0 && (K) > 0 && (N) > 0, NVFP4_ERR_INVALID_ARG, "M=%lld K=%lld N=%lld", (long long)(M),    \
             (long long)(K), (long long)(N));                                                                  \
  NV_REQUIRE((K) % 64 == 0 && (N) % 16 == 0, NVFP4_ERR_UNSUPPORTED_SHAPE,                                     \
             "K=%lld must be a multiple of 64 and N=%lld of 16", (long long)(K), (long long)(N));               \
  NV_REQUIRE((M) < (int64_t(1) << 30) && (N) < (int64_t(1) << 30) && (K) < (int64_t(1) << 24),              \
             NVFP4_ERR_UNSUPPORTED_SHAPE, "sizes too large")

nvfp4_status nvfp4_gemm(const uint8_t *xq, const uint8_t *xsf, const float *gs, int64_t M, int64_t K, int64_t N,
                        const uint8_t *w, const uint8_t *w_sf, const float *ws2, void *y, void *stream) {
  NV_CHECK_GEMM_SHAPE(M, K, N);
  NV_REQUIRE(gs && w && w_sf && ws2 && ((xq && xsf && y) || M == 0), NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(aligned(xq, 16) && aligned(xsf, 16) && aligned(w, 16) && aligned(w_sf, 16) && aligned(y, 16) &&
                 aligned(gs, 4) && aligned(ws2, 4),
             NVFP4_ERR_MISALIGNED, "pointers must be 16-byte aligned");
  DeviceInfo *d;
  nvfp4_status st = device_info(__func__, &d);
  if (st != NVFP4_OK) return st;
  return gemm_dense(__func__, d, xq, xsf, gs, M, K, N, w, w_sf, ws2, y, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_linear(const void *x, int64_t M, int64_t K, int64_t N, const uint8_t *w, const uint8_t *w_sf,
                          const float *ws2, int gs_mode, float *gs, void *y, void *ws, size_t ws_bytes,
                          void *stream) {
  NV_CHECK_GEMM_SHAPE(M, K, N);
  NV_REQUIRE(gs_mode == NVFP4_GS_DYNAMIC || gs_mode == NVFP4_GS_STATIC, NVFP4_ERR_INVALID_ARG, "gs_mode %d", gs_mode);
  NV_REQUIRE(gs && w && w_sf && ws2 && ((x && y) || M == 0), NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(aligned(x, 16) && aligned(w, 16) && aligned(w_sf, 16) && aligned(y, 16) && aligned(gs, 4) &&
                 aligned(ws2, 4),
             NVFP4_ERR_MISALIGNED, "pointers must be 16-byte aligned");
  const LinearWs L = linear_ws(M, K);
  nvfp4_status st = check_ws(__func__, ws, ws_bytes, L.total);
  if (st != NVFP4_OK) return st;
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool dyn = gs_mode == NVFP4_GS_DYNAMIC;
  if (linear_fusable(d, M, 1, K, N)) return linear_fused(__func__, d, x, M, 1, K, N, w, w_sf, ws2, dyn, gs, y, s);
  uint8_t *xq = at<uint8_t>(ws, L.xq), *xsf = at<uint8_t>(ws, L.xsf);
  uint32_t *partials = dyn ? at<uint32_t>(ws, L.partials) : nullptr;
  NV_CUDA(launch_act_quant(x, M, K, K, dyn, partials, gs, gs, xq, xsf, NVFP4_SF_SWIZZLED, s), "quantize kernel launch");
  // the quantise launch just before this GEMM runs after everything that wrote W
  return gemm_dense(__func__, d, xq, xsf, gs, M, K, N, w, w_sf, ws2, y, s, 1);
}

// ---------------------------------------------------------------- no-allocation dense linear
// Scratch of nvfp4_linear_noalloc: one array per device, alive until the process exits.
}  // extern "C"
namespace nvfp4 {
namespace {
__device__ __align__(256) uint8_t g_linear_noalloc_scratch[NVFP4_LINEAR_NOALLOC_MAX_BYTES];
void *g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, resolved once per device.
nvfp4_status noalloc_scratch(const char *fn, void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(fn, e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_linear_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(fn, e, "cudaGetSymbolAddress(no-allocation scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return NVFP4_OK;
}
}  // namespace
}  // namespace nvfp4
extern "C" {

nvfp4_status nvfp4_linear_noalloc(const void *x, int64_t M, int64_t K, int64_t N, const uint8_t *w,
                                  const uint8_t *w_sf, const float *ws2, int gs_mode, float *gs, void *y,
                                  void *stream) {
  NV_CHECK_GEMM_SHAPE(M, K, N);
  NV_REQUIRE(gs_mode == NVFP4_GS_DYNAMIC || gs_mode == NVFP4_GS_STATIC, NVFP4_ERR_INVALID_ARG, "gs_mode %d", gs_mode);
  NV_REQUIRE(gs && w && w_sf && ws2 && ((x && y) || M == 0), NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(aligned(x, 16) && aligned(w, 16) && aligned(w_sf, 16) && aligned(y, 16) && aligned(gs, 4) &&
                 aligned(ws2, 4),
             NVFP4_ERR_MISALIGNED, "pointers must be 16-byte aligned");
  const LinearWs L = linear_ws(M, K);
  NV_REQUIRE(L.total <= NVFP4_LINEAR_NOALLOC_MAX_BYTES, NVFP4_ERR_WORKSPACE,
             "M=%lld K=%lld needs %zu bytes of scratch, above the %u-byte static array; use nvfp4_linear with a "
             "caller workspace",
             (long long)M, (long long)K, L.total, NVFP4_LINEAR_NOALLOC_MAX_BYTES);
  DeviceInfo *d;
  nvfp4_status st = device_info(__func__, &d);
  if (st != NVFP4_OK) return st;
  void *scratch = nullptr;
  if ((st = noalloc_scratch(__func__, &scratch)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool dyn = gs_mode == NVFP4_GS_DYNAMIC;
  if (linear_fusable(d, M, 1, K, N)) return linear_fused(__func__, d, x, M, 1, K, N, w, w_sf, ws2, dyn, gs, y, s);
  uint8_t *xq = at<uint8_t>(scratch, L.xq), *xsf = at<uint8_t>(scratch, L.xsf);
  uint32_t *partials = dyn ? at<uint32_t>(scratch, L.partials) : nullptr;
  NV_CUDA(launch_act_quant(x, M, K, K, dyn, partials, gs, gs, xq, xsf, NVFP4_SF_SWIZZLED, s), "quantize kernel launch");
  // the quantise launch just before this GEMM runs after everything that wrote W
  return gemm_dense(__func__, d, xq, xsf, gs, M, K, N, w, w_sf, ws2, y, s, 1);
}

size_t nvfp4_grouped_linear_workspace_bytes(int64_t M, int64_t G, int64_t K) {
  if (M < 0 || G <= 0 || K < 0) return 0;
  return linear_ws(M, G * K).total;
}

nvfp4_status nvfp4_grouped_linear(const void *x, int64_t M, int64_t G, int64_t K, int64_t N, const uint8_t *w,
                                  const uint8_t *w_sf, const float *ws2, int gs_mode, float *gs, void *y, void *ws,
                                  size_t ws_bytes, void *stream) {
  NV_REQUIRE(G >= 1 && G <= 4096, NVFP4_ERR_INVALID_ARG, "G=%lld", (long long)G);
  NV_CHECK_GEMM_SHAPE(M, G * K, G * N);
  NV_REQUIRE(K % 64 == 0 && N % 128 == 0, NVFP4_ERR_UNSUPPORTED_SHAPE,
             "K=%lld must be a multiple of 64 and N=%lld of 128", (long long)K, (long long)N);
  NV_REQUIRE(gs_mode == NVFP4_GS_DYNAMIC || gs_mode == NVFP4_GS_STATIC, NVFP4_ERR_INVALID_ARG, "gs_mode %d", gs_mode);
  NV_REQUIRE(gs && w && w_sf && ws2 && ((x && y) || M == 0), NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(aligned(x, 16) && aligned(w, 16) && aligned(w_sf, 16) && aligned(y, 16) && aligned(gs, 4) &&
                 aligned(ws2, 4),
             NVFP4_ERR_MISALIGNED, "pointers must be 16-byte aligned");
  const LinearWs L = linear_ws(M, G * K);
  nvfp4_status st = check_ws(__func__, ws, ws_bytes, L.total);
  if (st != NVFP4_OK) return st;
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool dyn = gs_mode == NVFP4_GS_DYNAMIC;
  if (linear_fusable(d, M, G, K, N)) return linear_fused(__func__, d, x, M, G, K, N, w, w_sf, ws2, dyn, gs, y, s);
  uint8_t *xq = at<uint8_t>(ws, L.xq), *xsf = at<uint8_t>(ws, L.xsf);
  uint32_t *partials = dyn ? at<uint32_t>(ws, L.partials) : nullptr;
  NV_CUDA(launch_act_quant(x, M, G * K, G * K, dyn, partials, gs, gs, xq, xsf, NVFP4_SF_SWIZZLED, s),
          "quantize kernel launch");
  return gemm_dense(__func__, d, xq, xsf, gs, M, K, N, w, w_sf, ws2, y, s, 1, G);
}

size_t nvfp4_router_prepare_workspace_bytes(int64_t E, int64_t H) {
  (void)E;
  (void)H;
  return kMaxPartials * sizeof(uint32_t);
}

nvfp4_status nvfp4_router_prepare(const uint8_t *w, const uint8_t *w_sf, const float *ws2, int64_t E, int64_t H,
                                  void *wg, void *ws, size_t ws_bytes, void *stream) {
  NV_REQUIRE(w && w_sf && ws2 && wg, NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(E > 0 && H > 0, NVFP4_ERR_INVALID_ARG, "E=%lld H=%lld", (long long)E, (long long)H);
  NV_REQUIRE(H % 64 == 0 && E <= kMaxExperts, NVFP4_ERR_UNSUPPORTED_SHAPE, "H %% 64 == 0 and E <= %d", kMaxExperts);
  NV_REQUIRE(aligned(w, 16) && aligned(w_sf, 16) && aligned(wg, 16) && aligned(ws2, 4), NVFP4_ERR_MISALIGNED,
             "pointers must be 16-byte aligned");
  nvfp4_status st = check_ws(__func__, ws, ws_bytes, nvfp4_router_prepare_workspace_bytes(E, H));
  if (st != NVFP4_OK) return st;
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  NV_CUDA(launch_router_prepare(w, w_sf, ws2, E, H, static_cast<uint32_t *>(ws), wg, static_cast<cudaStream_t>(stream)),
          "router prepare launch");
  return NVFP4_OK;
}

size_t nvfp4_router_workspace_bytes(int64_t T, int64_t E) {
  if (T < 0 || E < 0) return 0;
  // the K splits' partial logits; the split count is largest when H is (any H % 64 == 0)
  const int64_t splits = router_splits(T, E, int64_t(1) << 24);
  return align256(static_cast<size_t>(splits) * static_cast<size_t>(T) * static_cast<size_t>(E) * sizeof(float));
}

nvfp4_status nvfp4_router(const void *x, int64_t T, int64_t H, const void *wg, int64_t E, int topk, int32_t *ids,
                          float *weights, float *logits, void *ws, size_t ws_bytes, void *stream) {
  NV_REQUIRE(T >= 0 && H > 0 && E > 0 && topk > 0, NVFP4_ERR_INVALID_ARG, "T=%lld H=%lld E=%lld topk=%d",
             (long long)T, (long long)H, (long long)E, topk);
  NV_REQUIRE(H % 64 == 0 && E <= kMaxExperts && topk <= kMaxTopk && topk <= E, NVFP4_ERR_UNSUPPORTED_SHAPE,
             "H %% 64 == 0, E <= %d, topk <= min(%d, E)", kMaxExperts, kMaxTopk);
  NV_REQUIRE(wg && ((x && ids && weights) || T == 0), NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(aligned(x, 16) && aligned(wg, 16) && aligned(ids, 4) && aligned(weights, 4) && aligned(logits, 4),
             NVFP4_ERR_MISALIGNED, "x and wg must be 16-byte aligned");
  NV_REQUIRE(T < (int64_t(1) << 24) && H < (int64_t(1) << 24), NVFP4_ERR_UNSUPPORTED_SHAPE, "sizes too large");
  nvfp4_status st = check_ws(__func__, ws, ws_bytes, nvfp4_router_workspace_bytes(T, E));
  if (st != NVFP4_OK) return st;
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  if (T == 0) return NVFP4_OK;
  CUtensorMap tx, tw;
  if ((st = make_map(__func__, &tx, x, 2 * H, T, 2 * H, 128)) != NVFP4_OK) return st;
  if ((st = make_map(__func__, &tw, wg, 2 * H, E, 2 * H, 128)) != NVFP4_OK) return st;
  NV_CUDA(launch_router(tx, tw, T, H, E, topk, ids, weights, logits, static_cast<float *>(ws), d->flags,
                        static_cast<cudaStream_t>(stream)),
          "router launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_moe_route(const int32_t *ids, int64_t T, int topk, int64_t E, int32_t *counts, int32_t *offsets,
                             int32_t *sorted_idx, int32_t *inv_idx, void *stream) {
  NV_REQUIRE(T >= 0 && topk > 0 && E > 0, NVFP4_ERR_INVALID_ARG, "T=%lld topk=%d E=%lld", (long long)T, topk,
             (long long)E);
  NV_REQUIRE(E <= kMaxExperts && topk <= kMaxTopk && T * topk < (int64_t(1) << 30), NVFP4_ERR_UNSUPPORTED_SHAPE,
             "E <= %d, topk <= %d", kMaxExperts, kMaxTopk);
  NV_REQUIRE(counts && offsets && ((ids && sorted_idx && inv_idx) || T == 0), NVFP4_ERR_INVALID_ARG,
             "NULL pointer argument");
  NV_REQUIRE(aligned(ids, 4) && aligned(counts, 4) && aligned(offsets, 4) && aligned(sorted_idx, 4) &&
                 aligned(inv_idx, 4),
             NVFP4_ERR_MISALIGNED, "int32 arrays must be 4-byte aligned");
  DeviceInfo *d;
  nvfp4_status st = device_info(__func__, &d);
  if (st != NVFP4_OK) return st;
  RouteBufs rb{counts, offsets, nullptr, nullptr, sorted_idx, inv_idx, nullptr, nullptr, moe_tile_shift(T)};
  NV_CUDA(launch_route_amax(ids, static_cast<int>(T), topk, static_cast<int>(E), 0, rb, nullptr, 0, nullptr, 0,
                            nullptr, d->flags, static_cast<cudaStream_t>(stream)),
          "route kernel launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int topk, int has_shared,
                                        nvfp4_moe_ws_layout *out) {
  NV_REQUIRE(out != nullptr, NVFP4_ERR_INVALID_ARG, "out is NULL");
  nvfp4_status st = check_moe_shape(__func__, T, H, I, E, topk);
  if (st != NVFP4_OK) return st;
  *out = moe_layout(T, H, I, E, topk, has_shared ? 1 : 0);
  return NVFP4_OK;
}

size_t nvfp4_moe_workspace_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int topk, int has_shared) {
  if (check_moe_shape("nvfp4_moe_workspace_bytes", T, H, I, E, topk) != NVFP4_OK) return 0;
  return moe_layout(T, H, I, E, topk, has_shared ? 1 : 0).total;
}

}  // extern "C"

namespace nvfp4 {
namespace {

nvfp4_status check_moe_common(const char *fn, int64_t T, int64_t H, int64_t I, int64_t E, int topk, int has_shared,
                              void *ws, size_t ws_bytes) {
  nvfp4_status st = check_moe_shape(fn, T, H, I, E, topk);
  if (st != NVFP4_OK) return st;
  return check_ws(fn, ws, ws_bytes, moe_layout(T, H, I, E, topk, has_shared).total);
}

nvfp4_status check_weights(const char *fn, const uint8_t *w, const uint8_t *sf, const float *ws2) {
  if (!w || !sf || !ws2) return fail(NVFP4_ERR_INVALID_ARG, fn, "NULL weight pointer");
  if (!aligned(w, 16) || !aligned(sf, 16) || !aligned(ws2, 4))
    return fail(NVFP4_ERR_MISALIGNED, fn, "weights and scales must be 16-byte aligned");
  return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" {

nvfp4_status nvfp4_moe_dispatch(const void *x, int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                                const int32_t *topk_ids, int has_shared, int a1_gs_mode, float *a1_gs, void *ws,
                                size_t ws_bytes, void *stream) {
  has_shared = has_shared ? 1 : 0;
  nvfp4_status st = check_moe_common(__func__, T, H, I, E, topk, has_shared, ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  NV_REQUIRE(a1_gs_mode == NVFP4_GS_DYNAMIC || a1_gs_mode == NVFP4_GS_STATIC, NVFP4_ERR_INVALID_ARG,
             "a1_gs_mode %d", a1_gs_mode);
  NV_REQUIRE(a1_gs && ((x && topk_ids) || T == 0), NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(aligned(x, 16) && aligned(topk_ids, 4) && aligned(a1_gs, 4), NVFP4_ERR_MISALIGNED,
             "x must be 16-byte aligned");
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  return moe_dispatch_impl(__func__, d, x, T, H, I, E, topk, topk_ids, has_shared, a1_gs_mode, a1_gs, ws,
                           static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_moe_w13(int64_t T, int64_t H, int64_t I, int64_t E, int topk, const uint8_t *w13,
                           const uint8_t *w13_sf, const float *w13_ws2, const uint8_t *sh_w13,
                           const uint8_t *sh_w13_sf, const float *sh_ws2, const float *a1_gs, const float *a2_gs,
                           float *h_debug, void *ws, size_t ws_bytes, void *stream) {
  const int has_shared = sh_w13 != nullptr;
  nvfp4_status st = check_moe_common(__func__, T, H, I, E, topk, has_shared, ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  if ((st = check_weights(__func__, w13, w13_sf, w13_ws2)) != NVFP4_OK) return st;
  if (has_shared && (st = check_weights(__func__, sh_w13, sh_w13_sf, sh_ws2)) != NVFP4_OK) return st;
  NV_REQUIRE(a1_gs && a2_gs, NVFP4_ERR_INVALID_ARG, "NULL global scale");
  NV_REQUIRE(aligned(a1_gs, 4) && aligned(a2_gs, 4) && aligned(h_debug, 16), NVFP4_ERR_MISALIGNED,
             "misaligned scale or h_debug");
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  return moe_gemm_impl(__func__, d, Epi::kW13, T, H, I, E, topk, w13, w13_sf, w13_ws2, sh_w13, sh_w13_sf, sh_ws2,
                       a1_gs, a2_gs, nullptr, h_debug, ws, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_moe_w2(int64_t T, int64_t H, int64_t I, int64_t E, int topk, const float *topk_w,
                          const uint8_t *w2, const uint8_t *w2_sf, const float *w2_ws2, const uint8_t *sh_w2,
                          const uint8_t *sh_w2_sf, const float *sh_ws2, const float *a2_gs, void *ws,
                          size_t ws_bytes, void *stream) {
  const int has_shared = sh_w2 != nullptr;
  nvfp4_status st = check_moe_common(__func__, T, H, I, E, topk, has_shared, ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  if ((st = check_weights(__func__, w2, w2_sf, w2_ws2)) != NVFP4_OK) return st;
  if (has_shared && (st = check_weights(__func__, sh_w2, sh_w2_sf, sh_ws2)) != NVFP4_OK) return st;
  NV_REQUIRE(a2_gs && (topk_w || T == 0), NVFP4_ERR_INVALID_ARG, "NULL pointer argument");
  NV_REQUIRE(aligned(a2_gs, 4) && aligned(topk_w, 4), NVFP4_ERR_MISALIGNED, "misaligned fp32 array");
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  return moe_gemm_impl(__func__, d, Epi::kW2, T, H, I, E, topk, w2, w2_sf, w2_ws2, sh_w2, sh_w2_sf, sh_ws2, a2_gs,
                       nullptr, topk_w, nullptr, ws, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_moe_finalize(int64_t T, int64_t H, int64_t I, int64_t E, int topk, int has_shared, void *y,
                                void *ws, size_t ws_bytes, void *stream) {
  has_shared = has_shared ? 1 : 0;
  nvfp4_status st = check_moe_common(__func__, T, H, I, E, topk, has_shared, ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  NV_REQUIRE(y || T == 0, NVFP4_ERR_INVALID_ARG, "y is NULL");
  NV_REQUIRE(aligned(y, 16), NVFP4_ERR_MISALIGNED, "y must be 16-byte aligned");
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  if (T == 0) return NVFP4_OK;
  const nvfp4_moe_ws_layout L = moe_layout(T, H, I, E, topk, has_shared);
  NV_CUDA(launch_finalize(at<float>(ws, L.y_acc), T * H, y, static_cast<cudaStream_t>(stream)),
          "finalize kernel launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_moe_forward(const void *x, int64_t T, int64_t H, int64_t I, int64_t E, int topk,
                               const int32_t *topk_ids, const float *topk_w, const uint8_t *w13, const uint8_t *w13_sf,
                               const float *w13_ws2, const uint8_t *w2, const uint8_t *w2_sf, const float *w2_ws2,
                               const uint8_t *sh_w13, const uint8_t *sh_w13_sf, const uint8_t *sh_w2,
                               const uint8_t *sh_w2_sf, const float *sh_ws2, int a1_gs_mode, float *a1_gs,
                               const float *a2_gs, void *y, void *ws, size_t ws_bytes, void *stream) {
  const int has_shared = sh_w13 != nullptr;
  nvfp4_status st = check_moe_common(__func__, T, H, I, E, topk, has_shared, ws, ws_bytes);
  if (st != NVFP4_OK) return st;
  NV_REQUIRE(a1_gs_mode == NVFP4_GS_DYNAMIC || a1_gs_mode == NVFP4_GS_STATIC, NVFP4_ERR_INVALID_ARG,
             "a1_gs_mode %d", a1_gs_mode);
  NV_REQUIRE(a1_gs && a2_gs && ((x && topk_ids && topk_w && y) || T == 0), NVFP4_ERR_INVALID_ARG,
             "NULL pointer argument");
  NV_REQUIRE(aligned(x, 16) && aligned(y, 16) && aligned(topk_ids, 4) && aligned(topk_w, 4) && aligned(a1_gs, 4) &&
                 aligned(a2_gs, 4),
             NVFP4_ERR_MISALIGNED, "x and y must be 16-byte aligned, fp32/int32 arrays 4-byte aligned");
  if ((st = check_weights(__func__, w13, w13_sf, w13_ws2)) != NVFP4_OK) return st;
  if ((st = check_weights(__func__, w2, w2_sf, w2_ws2)) != NVFP4_OK) return st;
  if (has_shared) {
    if ((st = check_weights(__func__, sh_w13, sh_w13_sf, sh_ws2)) != NVFP4_OK) return st;
    if ((st = check_weights(__func__, sh_w2, sh_w2_sf, sh_ws2)) != NVFP4_OK) return st;
  } else {
    NV_REQUIRE(!sh_w2, NVFP4_ERR_INVALID_ARG, "sh_w2 given without sh_w13");
  }
  DeviceInfo *d;
  if ((st = device_info(__func__, &d)) != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tok1_applies(T, H, topk)) {
    // routing and the zeroing of y_acc only; the w13 CTAs reduce the amax and quantise
    const nvfp4_moe_ws_layout L = moe_layout(T, H, I, E, topk, has_shared);
    RouteBufs rb = route_bufs(ws, L);
    rb.tile_shift = moe_tile_shift(T);
    NV_CUDA(launch_route_amax(topk_ids, 1, topk, static_cast<int>(E), has_shared, rb, nullptr, H, nullptr, 0,
                              at<float>(ws, L.y_acc), d->flags, s),
            "route kernel launch");
    const Tok1 tok1{x,   topk_ids, a1_gs_mode == NVFP4_GS_DYNAMIC, a1_gs, w2, w2_sf, sh_w2, sh_w2_sf,
                    w2_ws2, sh_ws2, topk_w};
    if ((st = moe_gemm_impl(__func__, d, Epi::kW13, T, H, I, E, topk, w13, w13_sf, w13_ws2, sh_w13, sh_w13_sf,
                            sh_ws2, a1_gs, a2_gs, nullptr, nullptr, ws, s, &tok1)) != NVFP4_OK)
      return st;
  } else {
    if ((st = moe_dispatch_impl(__func__, d, x, T, H, I, E, topk, topk_ids, has_shared, a1_gs_mode, a1_gs, ws,
                                s)) != NVFP4_OK)
      return st;
    if ((st = moe_gemm_impl(__func__, d, Epi::kW13, T, H, I, E, topk, w13, w13_sf, w13_ws2, sh_w13, sh_w13_sf,
                            sh_ws2, a1_gs, a2_gs, nullptr, nullptr, ws, s)) != NVFP4_OK)
      return st;
  }
  // (at T = 1 the one-token launch did the down projection too)
  if (!tok1_applies(T, H, topk) &&
      (st = moe_gemm_impl(__func__, d, Epi::kW2, T, H, I, E, topk, w2, w2_sf, w2_ws2, sh_w2, sh_w2_sf, sh_ws2, a2_gs,
                          nullptr, topk_w, nullptr, ws, s)) != NVFP4_OK)
    return st;
  if (T == 0) return NVFP4_OK;
  const nvfp4_moe_ws_layout L = moe_layout(T, H, I, E, topk, has_shared);
  NV_CUDA(launch_finalize(at<float>(ws, L.y_acc), T * H, y, s), "finalize kernel launch");
  return NVFP4_OK;
}

nvfp4_status nvfp4_debug_wait_timeout(uint32_t timeout_us, void *stream) {
  NV_REQUIRE(timeout_us > 0 && timeout_us <= 5000000u, NVFP4_ERR_INVALID_ARG, "timeout_us %u outside (0, 5e6]",
             timeout_us);
  DeviceInfo *d;
  nvfp4_status st = device_info(__func__, &d);
  if (st != NVFP4_OK) return st;
  NV_CUDA(launch_wait_timeout_probe(timeout_us, d->flags, static_cast<cudaStream_t>(stream)), "probe launch");
  return NVFP4_OK;
}

}  // extern "C"
