// Steps 1-2 of the latent-MoE tail: sum the P routed partials of each token in
// FP32 and apply RMSNorm with weight g, writing the bf16 latent y[T,L]. With no
// weight (g == nullptr, the pages' `transform.norm is None` branch) the latent
// is the partial sum itself.
//
// Follows `allreduce_norm_latent_out` in PR #50383's `_shard_up_proj_tail`
// (all-reduce first, then the norm) and F.rms_norm as the PR #51253 test
// calls it: y = x * rsqrt(mean(x^2) + eps) * g, mean over L.
//
// One CTA per token row: 256 threads each own 8-element (16-byte) chunks of
// the row, load all P partials of a chunk before accumulating (p ascending),
// keep x in registers (L <= 2048: one chunk per thread) or else in shared
// memory, reduce the sum of squares with warp shuffles and
// then write y = (x * r) * g rounded to bf16. Memory-bound: P*L*2 bytes in,
// L*2 bytes out per token, every load a 16-byte vector.
//
// Calls that the decode kernel serves also pass the W rows the projection
// kernel is about to stream: the grid then has at least one CTA per SM, and
// every CTA issues bulk L2 prefetches of its share of those rows before the
// dependency wait, so the HBM reads of W start while the preceding work is
// still finishing. CTAs beyond the T token rows only prefetch (and wait, so the
// grid's completion still implies the preceding work's).
#include "launch.h"
#include "ptx.cuh"

#include <algorithm>

namespace lt {
namespace {

constexpr int kNormThreads = 256;
constexpr int kMaxL = 16384;
constexpr size_t kPrefetchPiece = 16384;
constexpr size_t kRoutedPiece = 4096;  // small, so every SM issues one early

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void add8(float (&a)[8], const uint4& v) {
  a[0] += bf16_lo(v.x);
  a[1] += bf16_hi(v.x);
  a[2] += bf16_lo(v.y);
  a[3] += bf16_hi(v.y);
  a[4] += bf16_lo(v.z);
  a[5] += bf16_hi(v.z);
  a[6] += bf16_lo(v.w);
  a[7] += bf16_hi(v.w);
}

// kRegs: L <= 8 * kNormThreads, so each thread owns at most one 8-element chunk
// and keeps it in registers between the reduction and the write (no shared
// memory for x, fewer registers than staging it through shared memory).
template <bool kRegs>
__global__ void __launch_bounds__(kNormThreads)
    norm_kernel(const uint16_t* __restrict__ routed, const float* __restrict__ g,
                uint16_t* __restrict__ y, int P, int T, int L, float eps, int trigger,
                const uint8_t* __restrict__ pf, size_t pf_bytes, size_t pf_routed_bytes) {
  extern __shared__ float4 xs4[];  // !kRegs: the token's x[L] in FP32
  __shared__ float red[kNormThreads / 32];
  // Optional: pull `routed` and then the projection's W rows into L2 before
  // waiting, spread over the CTAs of the grid first (piece i goes to CTA
  // i % grid). `routed` goes first on every SM so that its lines arrive before
  // the W stream; if the preceding work is still writing it, the lines are
  // simply updated in L2 and read after the wait below.
  if (pf_routed_bytes != 0) {
    const uint8_t* r8 = reinterpret_cast<const uint8_t*>(routed);
    const size_t pieces = (pf_routed_bytes + kRoutedPiece - 1) / kRoutedPiece;
    for (size_t i = blockIdx.x + static_cast<size_t>(gridDim.x) * threadIdx.x; i < pieces;
         i += static_cast<size_t>(gridDim.x) * kNormThreads) {
      const size_t off = i * kRoutedPiece;
      const size_t n = pf_routed_bytes - off < kRoutedPiece ? pf_routed_bytes - off : kRoutedPiece;
      l2_prefetch_bulk(r8 + off, static_cast<uint32_t>(n));
    }
    __syncthreads();
  }
  if (pf_bytes != 0) {
    const size_t pieces = (pf_bytes + kPrefetchPiece - 1) / kPrefetchPiece;
    for (size_t i = blockIdx.x + static_cast<size_t>(gridDim.x) * threadIdx.x; i < pieces;
         i += static_cast<size_t>(gridDim.x) * kNormThreads) {
      const size_t off = i * kPrefetchPiece;
      const size_t n = pf_bytes - off < kPrefetchPiece ? pf_bytes - off : kPrefetchPiece;
      l2_prefetch_bulk(pf + off, static_cast<uint32_t>(n));
    }
  }
  // Launched as a programmatic dependent of whatever precedes it on the stream:
  // wait for that work (it may produce `routed` or still read the latent buffer)
  // before touching memory, then let the projection kernel start its prologue.
  pdl_wait();
  if (trigger) pdl_launch_dependents();
  if (static_cast<int>(blockIdx.x) >= T) return;  // CTAs that only prefetched

  const int t = blockIdx.x;
  const int nchunk = L >> 3;
  const size_t row_stride = static_cast<size_t>(T) * L;
  const uint16_t* base = routed + static_cast<size_t>(t) * L;

  float ss = 0.f;
  // kRegs: the weights of this thread's single chunk are requested now, with
  // its partials, instead of after the reduction (one round trip less on the
  // path to y).
  const float4* g4 = reinterpret_cast<const float4*>(g);
  float4 g0_reg = make_float4(0.f, 0.f, 0.f, 0.f), g1_reg = g0_reg;
  if (kRegs && g != nullptr && static_cast<int>(threadIdx.x) < nchunk) {
    g0_reg = __ldg(g4 + 2 * threadIdx.x);
    g1_reg = __ldg(g4 + 2 * threadIdx.x + 1);
  }
  float keep[8];  // kRegs: this thread's chunk of x
#pragma unroll
  for (int j = 0; j < 8; ++j) keep[j] = 0.f;
  for (int c = threadIdx.x; c < nchunk; c += kNormThreads) {
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const uint16_t* src = base + static_cast<size_t>(c) * 8;
    int p = 0;
    for (; p + 8 <= P; p += 8) {
      uint4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = ld_stream_v4(src + (p + k) * row_stride);
#pragma unroll
      for (int k = 0; k < 8; ++k) add8(a, v[k]);
    }
    for (; p < P; ++p) add8(a, ld_stream_v4(src + p * row_stride));
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += a[j] * a[j];
    if constexpr (kRegs) {
#pragma unroll
      for (int j = 0; j < 8; ++j) keep[j] = a[j];
    } else {
      xs4[2 * c] = make_float4(a[0], a[1], a[2], a[3]);
      xs4[2 * c + 1] = make_float4(a[4], a[5], a[6], a[7]);
    }
  }

  ss = warp_sum(ss);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  // The eight warp sums, added in the order of a halving shuffle tree over them.
  static_assert(kNormThreads == 256, "eight warp sums");
  const float total = ((red[0] + red[4]) + (red[2] + red[6])) + ((red[1] + red[5]) + (red[3] + red[7]));
  const float r = 1.0f / sqrtf(total / static_cast<float>(L) + eps);

  uint4* dst = reinterpret_cast<uint4*>(y + static_cast<size_t>(t) * L);
  for (int c = threadIdx.x; c < nchunk; c += kNormThreads) {
    float4 x0, x1;
    if constexpr (kRegs) {
      x0 = make_float4(keep[0], keep[1], keep[2], keep[3]);
      x1 = make_float4(keep[4], keep[5], keep[6], keep[7]);
    } else {
      x0 = xs4[2 * c];
      x1 = xs4[2 * c + 1];
    }
    uint4 o;
    if (g == nullptr) {  // no norm: round the partial sum itself
      o.x = pack_bf16x2(x0.x, x0.y);
      o.y = pack_bf16x2(x0.z, x0.w);
      o.z = pack_bf16x2(x1.x, x1.y);
      o.w = pack_bf16x2(x1.z, x1.w);
    } else {
      const float4 g0 = kRegs ? g0_reg : __ldg(g4 + 2 * c);
      const float4 g1 = kRegs ? g1_reg : __ldg(g4 + 2 * c + 1);
      o.x = pack_bf16x2(x0.x * r * g0.x, x0.y * r * g0.y);
      o.y = pack_bf16x2(x0.z * r * g0.z, x0.w * r * g0.w);
      o.z = pack_bf16x2(x1.x * r * g1.x, x1.y * r * g1.y);
      o.w = pack_bf16x2(x1.z * r * g1.z, x1.w * r * g1.w);
    }
    dst[c] = o;
  }
}

}  // namespace

cudaError_t setup_norm(const DeviceInfo&) {
  return cudaFuncSetAttribute(norm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kMaxL * static_cast<int>(sizeof(float)));
}

cudaError_t launch_norm(const NormArgs& a, bool trigger_dependents, const DeviceInfo& dev,
                        cudaStream_t stream) {
  if (a.l2_prefetch_bytes % 16 != 0 || reinterpret_cast<uintptr_t>(a.l2_prefetch) % 16 != 0)
    return cudaErrorInvalidValue;
  const size_t routed_bytes = static_cast<size_t>(a.P) * a.T * a.L * 2;  // a multiple of 16
  const size_t pf_routed =
      a.prefetch_routed && routed_bytes <= kMaxRoutedPrefetchBytes ? routed_bytes : 0;
  cudaLaunchConfig_t cfg{};
  // With a prefetch, at least one CTA per SM so that every SM's copy engine
  // issues a share of it.
  const int grid =
      a.l2_prefetch_bytes != 0 || pf_routed != 0 ? std::max(a.T, dev.num_sms) : a.T;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kNormThreads, 1, 1);
  const bool regs = a.L <= 8 * kNormThreads;  // one 8-element chunk per thread at most
  cfg.dynamicSmemBytes = regs ? 0 : static_cast<size_t>(a.L) * sizeof(float);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int trig = trigger_dependents ? 1 : 0;
  const uint8_t* pf = static_cast<const uint8_t*>(a.l2_prefetch);
  return regs ? cudaLaunchKernelEx(&cfg, norm_kernel<true>, a.routed, a.g, a.y, a.P, a.T, a.L,
                                   a.eps, trig, pf, a.l2_prefetch_bytes, pf_routed)
              : cudaLaunchKernelEx(&cfg, norm_kernel<false>, a.routed, a.g, a.y, a.P, a.T, a.L,
                                   a.eps, trig, pf, a.l2_prefetch_bytes, pf_routed);
}

}  // namespace lt
