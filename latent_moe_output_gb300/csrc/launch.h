// Library-internal host interface between the C-ABI layer (api.cu) and the
// kernel translation units. Not installed, not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lt {

// Device error word bits (set with atomicOr by kernels, read by latent_tail_check).
constexpr uint32_t kErrWaitTimeout = 1u;

// Largest token count the decode (split-K, swap-AB) kernel serves; above it,
// or when its buffers do not fit (decode_supported), the persistent
// tensor-core kernel runs. Set where the two kernels cross over at L = 2048,
// H = 7168, P = 8 (forward call, GB300): 21.4 against 23.7 us at T = 224,
// 25.8 against 24.4 us at T = 256.
constexpr int kDecodeMaxTokens = 224;

// Up to this many tokens a call runs the CUDA-core kernel that does the whole
// tail in one launch (gemv.cu), when one SM's slice of W fits in its shared
// memory and L <= 4096.
constexpr int kGemvMaxTokens = 2;

// Encodes a 2-D bf16 row-major [rows, cols] tensor map with a (64 x box_rows)
// box and 128-byte swizzle, without L2 sector promotion: every box reads
// 128-byte row pieces whose neighbours are read much later, if at all (see the
// prefill kernel's shared-partial map). Returns false if the driver rejects it.
bool make_map_bf16_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows);

struct DeviceInfo {
  int device;
  int num_sms;
  int max_smem_optin;
  uint32_t* err_word;  // device address of the error word
};

struct NormArgs {
  const uint16_t* routed;  // [P,T,L]
  const float* g;          // [L]
  uint16_t* y;             // [T,L]
  int P, T, L;
  float eps;
  // Optional L2 prefetch, issued before the dependency wait, of the W rows the
  // projection kernel streams next (l2_prefetch_bytes a multiple of 16).
  const void* l2_prefetch;
  size_t l2_prefetch_bytes;
  // Also prefetch all of `routed` into L2 before the wait, ahead of W, so that
  // its reads after the wait do not queue behind the W traffic.
  bool prefetch_routed;
};

// Prefetches larger than these are skipped: they would not stay in L2.
constexpr size_t kMaxRoutedPrefetchBytes = size_t(16) << 20;
constexpr size_t kMaxWPrefetchBytes = size_t(64) << 20;

// W rows per decode tile: the decode kernel reads W in whole tiles of this
// many rows, starting at absolute multiples of it.
constexpr int kDecodeTileRows = 128;

struct ProjectArgs {
  const uint16_t* y;       // [T,L]
  const uint16_t* shared;  // [P,T,H]
  const uint16_t* W;       // [H,L]
  uint16_t* out;           // [T,H]
  int P, T, L, H;
  int col_start, col_end;
  bool pdl;                // launched as a programmatic dependent: may start before the
                           // preceding kernel on the stream has finished
  // Decode kernel: let the next kernel on the stream launch as soon as each CTA
  // has issued its last W copy (else once its MMAs are done). Earlier lets the
  // next call's norm kernel prefetch its W into L2 during this call's tail.
  bool early_trigger;
  // Everything but y was complete when this kernel was released: the preceding
  // kernel is the norm kernel of the same call, which waited for all earlier work
  // before releasing it, so W and the shared partials may be read before the
  // dependency wait. Otherwise (pdl without it) every input is read after the wait.
  bool inputs_ready;
};

// The whole tail on CUDA cores for T <= kGemvMaxTokens. With latent == nullptr
// the kernel reduces `routed` and normalizes it itself; otherwise it reads the
// latent [T, L] (latent_tail_project_cols) and ignores routed, g and eps.
struct GemvArgs {
  const uint16_t* routed;  // [P,T,L]
  const float* g;          // [L] or null (no norm)
  const uint16_t* latent;  // [T,L] or null
  const uint16_t* shared;  // [P,T,H]
  const uint16_t* W;       // [H,L]
  uint16_t* out;           // [T,H]
  int P, T, L, H;
  int col_start, col_end;
  float eps;
  bool shared_on_host;     // shared is mapped page-locked host memory: not prefetched
};

cudaError_t launch_norm(const NormArgs& a, bool trigger_dependents, const DeviceInfo& dev,
                        cudaStream_t stream);
cudaError_t launch_gemv(const GemvArgs& a, const DeviceInfo& dev, cudaStream_t stream);
// Copies `bytes` (a multiple of 16, both pointers 16-byte aligned) from mapped
// page-locked host memory to device memory in a kernel launched as a
// programmatic dependent (no copy-engine round trip on the stream).
cudaError_t launch_stage(const void* src, void* dst, size_t bytes, const DeviceInfo& dev,
                         cudaStream_t stream);
// Whether launch_gemv serves this shape on this device (T and the W slice fit).
bool gemv_supported(int T, int L, int col_start, int col_end, const DeviceInfo& dev);
// Whether launch_decode serves T tokens of latent width L (T <= kDecodeMaxTokens
// and its buffers fit in shared memory; always true for T <= 128).
bool decode_supported(int T, int L);
cudaError_t launch_decode(const ProjectArgs& a, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_prefill(const ProjectArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// One CTA waiting on a barrier nothing arrives at, bounded by limit_ns.
cudaError_t launch_wait_probe(uint64_t limit_ns, const DeviceInfo& dev, cudaStream_t stream);

// One-time per-device function attributes (dynamic shared memory limits).
cudaError_t setup_norm(const DeviceInfo& dev);
cudaError_t setup_decode(const DeviceInfo& dev);
cudaError_t setup_prefill(const DeviceInfo& dev);
cudaError_t setup_gemv(const DeviceInfo& dev);

}  // namespace lt
