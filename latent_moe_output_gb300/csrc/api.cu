// C ABI of the latent-MoE tail library (declared in include/latent_tail.h):
// host-side argument validation, one-time per-device set-up, TMA tensor-map
// encoding and the token-count dispatch between the decode and prefill
// kernels (the single-GPU counterpart of `_select_tail_tier` in PR #50383,
// which picks the tail implementation from num_tokens alone).
#include "latent_tail.h"
#include "launch.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

namespace {

__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;

struct DeviceSlot {
  bool initialized = false;
  lt_status status = LT_OK;
  lt::DeviceInfo info{};
};

DeviceSlot g_devices[kMaxDevices];
std::mutex g_mutex;

typedef CUresult (*PointerGetAttributeFn)(void*, CUpointer_attribute, CUdeviceptr);
PointerGetAttributeFn g_ptr_attr = nullptr;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

lt_status init_device(int dev, DeviceSlot& slot) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return LT_ERR_CUDA;
  if (major != 10 || minor != 3) return LT_ERR_UNSUPPORTED;  // kernels are built for sm_103a
  lt::DeviceInfo& d = slot.info;
  d.device = dev;
  if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess)
    return LT_ERR_CUDA;
  void* err_ptr = nullptr;
  if (cudaGetSymbolAddress(&err_ptr, g_error_word) != cudaSuccess) return LT_ERR_CUDA;
  d.err_word = static_cast<uint32_t*>(err_ptr);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return LT_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if (g_ptr_attr == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return LT_ERR_CUDA;
    g_ptr_attr = reinterpret_cast<PointerGetAttributeFn>(fn);
  }
  if (lt::setup_norm(d) != cudaSuccess || lt::setup_decode(d) != cudaSuccess ||
      lt::setup_prefill(d) != cudaSuccess || lt::setup_gemv(d) != cudaSuccess)
    return LT_ERR_CUDA;
  return LT_OK;
}

// Per-device state of the current device; set up on first use.
lt_status current_device(const lt::DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceSlot& slot = g_devices[dev];
  if (!slot.initialized) {
    slot.status = init_device(dev, slot);
    slot.initialized = true;
  }
  *out = &slot.info;
  return slot.status;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  uintptr_t lo, hi;
};
Span span(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Span{a, a + bytes};
}
bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi; }

// out may be exactly one of the P shared partials (in-place beta-add): every
// kernel reads all partials of an output element before writing it, and no
// other CTA reads that element.
bool aliases_a_partial(const void* out, const void* shared, int P, int T, int H) {
  const uintptr_t o = reinterpret_cast<uintptr_t>(out);
  const uintptr_t s = reinterpret_cast<uintptr_t>(shared);
  const uintptr_t plane = static_cast<uintptr_t>(T) * H * 2;
  return o >= s && (o - s) % plane == 0 && (o - s) / plane < static_cast<uintptr_t>(P);
}

// Device address through which the current device reaches the page-locked
// host range [p, p + bytes), or nullptr when the range is not entirely inside
// one page-locked host allocation or registration mapped for this device.
// Queries only; never touches the memory.
void* mapped_host_range(const void* p, size_t bytes) {
  if (p == nullptr || bytes == 0 || g_ptr_attr == nullptr) return nullptr;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the (non-sticky) error the failed query recorded
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr) return nullptr;
  CUdeviceptr start = 0;
  size_t size = 0;
  const CUdeviceptr q = static_cast<CUdeviceptr>(reinterpret_cast<uintptr_t>(p));
  if (g_ptr_attr(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, q) != CUDA_SUCCESS ||
      g_ptr_attr(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, q) != CUDA_SUCCESS)
    return nullptr;
  if (q < start || q - start > size || bytes > size - (q - start)) return nullptr;
  return a.devicePointer;
}

lt_status check_shape(int P, int T, int L, int H) {
  if (P < 1 || P > 64 || T < 0 || T > (1 << 24) || L < 8 || L > 16384 || H < 8 ||
      H > (1 << 20))
    return LT_ERR_INVALID_ARG;
  if (L % 8 != 0 || H % 8 != 0) return LT_ERR_ALIGNMENT;
  return LT_OK;
}

lt_status check_range(int H, int c0, int c1) {
  if (c0 < 0 || c1 > H || c0 >= c1) return LT_ERR_INVALID_ARG;
  if (c0 % 8 != 0 || c1 % 8 != 0) return LT_ERR_ALIGNMENT;
  return LT_OK;
}

lt_status check_ptrs(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p == nullptr) return LT_ERR_INVALID_ARG;
  for (const void* p : ptrs)
    if (!aligned16(p)) return LT_ERR_ALIGNMENT;
  return LT_OK;
}

size_t latent_bytes(int T, int L) { return static_cast<size_t>(T) * L * 2; }

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

lt_status launch_status(cudaError_t e) { return e == cudaSuccess ? LT_OK : LT_ERR_CUDA; }

// Whether a call of T tokens at latent width L runs the decode kernel (else the
// prefill kernel).
bool decode_path(int T, int L) { return lt::decode_supported(T, L); }

lt_status run_project(const lt::ProjectArgs& a, const lt::DeviceInfo& dev, cudaStream_t s) {
  if (decode_path(a.T, a.L)) return launch_status(lt::launch_decode(a, dev, s));
  return launch_status(lt::launch_prefill(a, dev, s));
}

lt_status forward_impl(const uint16_t* routed, const uint16_t* shared, const float* g,
                       const uint16_t* W, uint16_t* out, int P, int T, int L, int H, float eps,
                       int c0, int c1, void* ws, size_t ws_bytes, lt_stream stream,
                       bool early_trigger = true, bool routed_in_device_memory = true,
                       bool shared_on_host = false) {
  lt_status st = check_shape(P, T, L, H);
  if (st != LT_OK) return st;
  if ((st = check_range(H, c0, c1)) != LT_OK) return st;
  if (g != nullptr && (!std::isfinite(eps) || !(eps > 0.f))) return LT_ERR_INVALID_ARG;
  if (T == 0) return LT_OK;
  if ((st = check_ptrs({routed, shared, W, out})) != LT_OK) return st;
  if (g != nullptr && !aligned16(g)) return LT_ERR_ALIGNMENT;
  const size_t need = latent_tail_workspace_size(P, T, L, H);
  if (ws == nullptr || ws_bytes < need) return LT_ERR_WORKSPACE;
  if (!aligned16(ws)) return LT_ERR_ALIGNMENT;
  const Span so = span(out, static_cast<size_t>(T) * H * 2);
  const Span sw = span(ws, need);
  const Span ss = span(shared, static_cast<size_t>(P) * T * H * 2);
  const Span inputs[] = {span(routed, static_cast<size_t>(P) * T * L * 2),
                         span(g, g ? static_cast<size_t>(L) * 4 : 0),
                         span(W, static_cast<size_t>(H) * L * 2)};
  for (const Span& in : inputs)
    if (overlaps(so, in) || overlaps(sw, in)) return LT_ERR_INVALID_ARG;
  if (overlaps(sw, ss) || overlaps(so, sw)) return LT_ERR_INVALID_ARG;
  if (overlaps(so, ss) && !aliases_a_partial(out, shared, P, T, H)) return LT_ERR_INVALID_ARG;

  const lt::DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != LT_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (routed_in_device_memory && T <= lt::kGemvMaxTokens &&
      lt::gemv_supported(T, L, c0, c1, *dev)) {  // the whole tail in one launch
    const lt::GemvArgs ga{routed, g, nullptr, shared, W, out, P, T, L, H, c0, c1, eps,
                          shared_on_host};
    return launch_status(lt::launch_gemv(ga, *dev, s));
  }
  uint16_t* y = static_cast<uint16_t*>(ws);
  lt::NormArgs na{routed, g, y, P, T, L, eps, nullptr, 0, false};
  if (decode_path(T, L)) {
    // The decode kernel streams W in whole 128-row tiles covering [c0, c1).
    const int r0 = c0 / lt::kDecodeTileRows * lt::kDecodeTileRows;
    const int r1 = std::min(H, (c1 + lt::kDecodeTileRows - 1) / lt::kDecodeTileRows *
                                   lt::kDecodeTileRows);
    const size_t w_bytes = static_cast<size_t>(r1 - r0) * L * 2;
    if (w_bytes <= lt::kMaxWPrefetchBytes) {
      na.l2_prefetch = W + static_cast<size_t>(r0) * L;
      na.l2_prefetch_bytes = w_bytes;
    }
    // (not for page-locked host partials: the bulk L2 prefetch is only used on
    // device memory)
    na.prefetch_routed = routed_in_device_memory;
  }
  if ((st = launch_status(lt::launch_norm(na, true, *dev, s))) != LT_OK) return st;
  const lt::ProjectArgs pa{y, shared, W, out, P, T, L, H, c0, c1, true, early_trigger, true};
  return run_project(pa, *dev, s);
}

}  // namespace

namespace lt {

bool make_map_bf16_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows) {
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estrides[2] = {1, 1};
  const CUresult r =
      g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estrides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace lt

extern "C" {

LT_API size_t latent_tail_workspace_size(int P, int T, int L, int H) {
  if (T <= 0 || check_shape(P, T, L, H) != LT_OK) return 0;
  return round256(latent_bytes(T, L));
}

LT_API lt_status latent_tail_forward(const uint16_t* routed, const uint16_t* shared,
                                     const float* norm_weight, const uint16_t* W, uint16_t* out,
                                     int P, int T, int L, int H, float eps, void* workspace,
                                     size_t workspace_bytes, lt_stream stream) {
  return forward_impl(routed, shared, norm_weight, W, out, P, T, L, H, eps, 0, H, workspace,
                      workspace_bytes, stream);
}

LT_API lt_status latent_tail_forward_cols(const uint16_t* routed, const uint16_t* shared,
                                          const float* norm_weight, const uint16_t* W,
                                          uint16_t* out, int P, int T, int L, int H, float eps,
                                          int col_start, int col_end, void* workspace,
                                          size_t workspace_bytes, lt_stream stream) {
  return forward_impl(routed, shared, norm_weight, W, out, P, T, L, H, eps, col_start, col_end,
                      workspace, workspace_bytes, stream);
}

LT_API size_t latent_tail_host_workspace_size(int P, int T, int L, int H) {
  if (T <= 0 || check_shape(P, T, L, H) != LT_OK) return 0;
  size_t b = round256(latent_bytes(T, L));
  if (T <= lt::kGemvMaxTokens)  // staging for the routed partials (one-launch kernel)
    b += round256(static_cast<size_t>(P) * T * L * 2);
  if (!decode_path(T, L))  // prefill kernel: staging for the partials and the result
    b += round256(static_cast<size_t>(P) * T * L * 2) + round256(static_cast<size_t>(P) * T * H * 2) +
         round256(static_cast<size_t>(T) * H * 2);
  return b;
}

LT_API lt_status latent_tail_forward_host(const uint16_t* routed_host, const uint16_t* shared_host,
                                          const float* norm_weight, const uint16_t* W,
                                          uint16_t* out_host, int P, int T, int L, int H,
                                          float eps, void* workspace, size_t workspace_bytes,
                                          lt_stream stream) {
  lt_status st = check_shape(P, T, L, H);
  if (st != LT_OK) return st;
  if (norm_weight != nullptr && (!std::isfinite(eps) || !(eps > 0.f))) return LT_ERR_INVALID_ARG;
  if (T == 0) return LT_OK;
  if ((st = check_ptrs({routed_host, shared_host, W, out_host})) != LT_OK) return st;
  const size_t need = latent_tail_host_workspace_size(P, T, L, H);
  if (workspace == nullptr || workspace_bytes < need) return LT_ERR_WORKSPACE;
  if (!aligned16(workspace)) return LT_ERR_ALIGNMENT;
  if (norm_weight != nullptr && !aligned16(norm_weight)) return LT_ERR_ALIGNMENT;
  const Span sw = span(workspace, need);
  if (overlaps(sw, span(W, static_cast<size_t>(H) * L * 2)) ||
      overlaps(sw, span(norm_weight, norm_weight ? static_cast<size_t>(L) * 4 : 0)))
    return LT_ERR_INVALID_ARG;
  const size_t r_bytes = static_cast<size_t>(P) * T * L * 2;
  const size_t s_bytes = static_cast<size_t>(P) * T * H * 2;
  const size_t o_bytes = static_cast<size_t>(T) * H * 2;
  const Span so = span(out_host, o_bytes);
  if (overlaps(so, span(routed_host, r_bytes))) return LT_ERR_INVALID_ARG;
  if (overlaps(so, span(shared_host, s_bytes)) && !aliases_a_partial(out_host, shared_host, P, T, H))
    return LT_ERR_INVALID_ARG;
  const lt::DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != LT_OK) return st;
  void* rd = mapped_host_range(routed_host, r_bytes);
  void* sd = mapped_host_range(shared_host, s_bytes);
  void* od = mapped_host_range(out_host, o_bytes);
  if (rd == nullptr || sd == nullptr || od == nullptr) return LT_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t y_bytes = round256(latent_bytes(T, L));
  if (T <= lt::kGemvMaxTokens && lt::gemv_supported(T, L, 0, H, *dev)) {
    // The one-launch kernel reads the routed partials once per CTA: a copy
    // kernel brings them (P*T*L*2 bytes) into the workspace first; shared and
    // out stay on the host link, read and written once. Same kernel, same bits
    // as the device call.
    uint16_t* r_st = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + y_bytes);
    if (lt::launch_stage(rd, r_st, r_bytes, *dev, s) != cudaSuccess) return LT_ERR_CUDA;
    return forward_impl(r_st, static_cast<const uint16_t*>(sd), norm_weight, W,
                        static_cast<uint16_t*>(od), P, T, L, H, eps, 0, H, workspace, y_bytes,
                        stream, /*early_trigger=*/true, /*routed_in_device_memory=*/true,
                        /*shared_on_host=*/true);
  }
  if (decode_path(T, L)) {
    // The kernels read the partials and write the result across the host link.
    // Here the host link, not the W stream, bounds a call, and releasing the
    // next call only after the MMAs measured faster than the early release.
    return forward_impl(static_cast<const uint16_t*>(rd), static_cast<const uint16_t*>(sd),
                        norm_weight, W, static_cast<uint16_t*>(od), P, T, L, H, eps, 0, H,
                        workspace, y_bytes, stream, /*early_trigger=*/false,
                        /*routed_in_device_memory=*/false);
  }
  // Larger calls: stage through device memory with one copy per tensor.
  uint8_t* w8 = static_cast<uint8_t*>(workspace);
  uint16_t* r_st = reinterpret_cast<uint16_t*>(w8 + y_bytes);
  uint16_t* s_st = reinterpret_cast<uint16_t*>(w8 + y_bytes + round256(r_bytes));
  uint16_t* o_st =
      reinterpret_cast<uint16_t*>(w8 + y_bytes + round256(r_bytes) + round256(s_bytes));
  if (cudaMemcpyAsync(r_st, routed_host, r_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(s_st, shared_host, s_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return LT_ERR_CUDA;
  if ((st = forward_impl(r_st, s_st, norm_weight, W, o_st, P, T, L, H, eps, 0, H, workspace,
                         y_bytes, stream)) != LT_OK)
    return st;
  return launch_status(cudaMemcpyAsync(out_host, o_st, o_bytes, cudaMemcpyDeviceToHost, s));
}

LT_API lt_status latent_tail_norm(const uint16_t* routed, const float* norm_weight,
                                  uint16_t* latent, int P, int T, int L, float eps,
                                  lt_stream stream) {
  lt_status st = check_shape(P, T, L, 8);
  if (st != LT_OK) return st;
  if (norm_weight != nullptr && (!std::isfinite(eps) || !(eps > 0.f))) return LT_ERR_INVALID_ARG;
  if (T == 0) return LT_OK;
  if ((st = check_ptrs({routed, latent})) != LT_OK) return st;
  if (norm_weight != nullptr && !aligned16(norm_weight)) return LT_ERR_ALIGNMENT;
  const Span sy = span(latent, latent_bytes(T, L));
  if (overlaps(sy, span(routed, static_cast<size_t>(P) * T * L * 2)) ||
      overlaps(sy, span(norm_weight, norm_weight ? static_cast<size_t>(L) * 4 : 0)))
    return LT_ERR_INVALID_ARG;
  const lt::DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != LT_OK) return st;
  const lt::NormArgs na{routed, norm_weight, latent, P, T, L, eps, nullptr, 0, false};
  return launch_status(lt::launch_norm(na, false, *dev, reinterpret_cast<cudaStream_t>(stream)));
}

LT_API lt_status latent_tail_project_cols(const uint16_t* latent, const uint16_t* shared,
                                          const uint16_t* W, uint16_t* out, int P, int T, int L,
                                          int H, int col_start, int col_end, lt_stream stream) {
  lt_status st = check_shape(P, T, L, H);
  if (st != LT_OK) return st;
  if ((st = check_range(H, col_start, col_end)) != LT_OK) return st;
  if (T == 0) return LT_OK;
  if ((st = check_ptrs({latent, shared, W, out})) != LT_OK) return st;
  const Span so = span(out, static_cast<size_t>(T) * H * 2);
  if (overlaps(so, span(latent, latent_bytes(T, L))) ||
      overlaps(so, span(W, static_cast<size_t>(H) * L * 2)))
    return LT_ERR_INVALID_ARG;
  if (overlaps(so, span(shared, static_cast<size_t>(P) * T * H * 2)) &&
      !aliases_a_partial(out, shared, P, T, H))
    return LT_ERR_INVALID_ARG;
  const lt::DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != LT_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T <= lt::kGemvMaxTokens && lt::gemv_supported(T, L, col_start, col_end, *dev)) {
    const lt::GemvArgs ga{nullptr, nullptr, latent, shared, W, out, P, T, L, H,
                          col_start, col_end, 0.f, false};
    return launch_status(lt::launch_gemv(ga, *dev, s));
  }
  // The decode kernel is launched as a programmatic dependent with every read
  // after its dependency wait: back-to-back calls overlap one launch's start-up
  // (barrier set-up, TMEM allocation) with the previous launch's tail.
  const bool dep = decode_path(T, L);
  const lt::ProjectArgs pa{latent, shared, W, out, P,   T,   L,    H,
                           col_start, col_end, dep, dep, false};
  return run_project(pa, *dev, s);
}

LT_API lt_status latent_tail_check(lt_stream stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LT_ERR_CUDA;
  const lt::DeviceInfo* dev = nullptr;
  lt_status st = current_device(&dev);
  if (st != LT_OK) return st;
  uint32_t word = 0;
  if (cudaMemcpy(&word, dev->err_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return LT_ERR_CUDA;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(dev->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return LT_ERR_CUDA;
    if (word & lt::kErrWaitTimeout) return LT_ERR_TIMEOUT;
  }
  return LT_OK;
}

LT_API lt_status latent_tail_selftest_wait_timeout(unsigned int limit_us, lt_stream stream) {
  if (limit_us < 1 || limit_us > 1000000) return LT_ERR_INVALID_ARG;
  const lt::DeviceInfo* dev = nullptr;
  lt_status st = current_device(&dev);
  if (st != LT_OK) return st;
  return launch_status(lt::launch_wait_probe(static_cast<uint64_t>(limit_us) * 1000u, *dev,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

LT_API const char* latent_tail_status_string(lt_status status) {
  switch (status) {
    case LT_OK: return "LT_OK: success";
    case LT_ERR_INVALID_ARG: return "LT_ERR_INVALID_ARG: invalid argument";
    case LT_ERR_ALIGNMENT: return "LT_ERR_ALIGNMENT: pointer or size not aligned";
    case LT_ERR_UNSUPPORTED: return "LT_ERR_UNSUPPORTED: device is not sm_103";
    case LT_ERR_WORKSPACE: return "LT_ERR_WORKSPACE: workspace missing or too small";
    case LT_ERR_CUDA: return "LT_ERR_CUDA: CUDA call or kernel launch failed";
    case LT_ERR_TIMEOUT: return "LT_ERR_TIMEOUT: a bounded device wait expired";
  }
  return "unknown lt_status";
}

}  // extern "C"
