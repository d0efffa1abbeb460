// latent_tail_forward_noalloc: the whole tail without a caller-provided
// workspace, for callers that have no way to allocate device memory.
//
// Who needs it: code that receives only its input and output buffers from a
// host runtime that owns all device memory (a plugin or custom-op interface
// with no allocator hook), and code that runs where allocating is not
// allowed or not wanted at call time. Such a caller cannot obtain the
// workspace latent_tail_forward asks for.
//
// How: the path's only scratch, the normalized latent y[T, L], lives in the
// file-scope device array below. Every GPU that loads this library holds it, 8 MiB, until the
// process exits. Host code must not pass the
// array's name to a kernel (on the host it names a host-side shadow, not
// device memory); its device address is looked up once per device with
// cudaGetSymbolAddress and cached.
#include "latent_tail.h"

#include <cuda_runtime.h>

#include <mutex>

static constexpr size_t kStaticScratchBytes = LT_NOALLOC_MAX_SCRATCH_BYTES;

// The scratch itself: one per device, shared by every call on that device.
static __device__ __align__(256) unsigned char g_static_latent[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the static scratch on the current device. The lookup runs
// on the first call per device, with that device current. A device this
// library has no code for (anything but compute capability 10.3) is reported
// as unsupported before the lookup, which would fail there; a failed lookup
// clears the error it leaves in the runtime so later, unrelated error checks
// do not see it.
lt_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return LT_ERR_CUDA;
    if (major != 10 || minor != 3) return LT_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_latent) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LT_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LT_OK;
}

}  // namespace

extern "C" LT_API lt_status latent_tail_forward_noalloc(const uint16_t* routed,
                                                        const uint16_t* shared,
                                                        const float* norm_weight,
                                                        const uint16_t* W, uint16_t* out, int P,
                                                        int T, int L, int H, float eps,
                                                        lt_stream stream) {
  const size_t need = latent_tail_workspace_size(P, T, L, H);
  if (need > kStaticScratchBytes) return LT_ERR_WORKSPACE;  // too large for the array
  if (T <= 0 || need == 0)  // nothing to stage: let the regular entry point validate / no-op
    return latent_tail_forward(routed, shared, norm_weight, W, out, P, T, L, H, eps, nullptr, 0,
                               stream);
  void* scratch = nullptr;
  const lt_status st = scratch_on_current_device(&scratch);
  if (st != LT_OK) return st;
  return latent_tail_forward(routed, shared, norm_weight, W, out, P, T, L, H, eps, scratch,
                             kStaticScratchBytes, stream);
}
