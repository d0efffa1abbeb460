// The whole latent-MoE tail for one or two tokens on CUDA cores, in one
// launch:
//   x[t,l]   = sum_p routed[p,t,l]                        (FP32, p ascending)
//   y[t,l]   = x[t,l] * rsqrt(mean_l x[t,l]^2 + eps) * g[l]  (FP32, not rounded)
//   out[t,h] = bf16_rn( sum_l y[t,l] * W[h,l] + sum_p shared[p,t,h] ),  h in [c0,c1)
// that is `allreduce_norm_latent_out` followed by the narrowed beta-add
// `hidden_shard.addmm_(latent, up_proj_shard.t())` of PR #50383's
// `_shard_up_proj_tail`, with the shared partials of the final all-reduce summed
// in the epilogue.
//
// With T <= 2 the product is a matrix-vector product. A tensor-core MMA
// occupies an SM's tensor core for the same ~78 ns whatever its N, so here the
// dot products run as FP32 FMAs and the kernel is shaped around streaming W
// once:
//   * one CTA per slice of rpc consecutive W rows (output columns, rpc a
//     multiple of 8), about one per SM. Before its dependency wait the CTA asks
//     L2 for its share of the small inputs and then for its W slice (a prefetch
//     only warms L2, which any write of the preceding kernel updates);
//   * after the wait every thread issues the first loads of its routed pieces
//     and of its shared-partial columns, and only then does one thread copy
//     the W slice (rpc * L * 2 contiguous bytes; H = 7168, L = 2048: 48 rows,
//     192 KB) into shared memory with one-dimensional bulk copies, one per 8
//     rows, each with its own mbarrier: whatever the SM requests after the
//     slice comes back behind it;
//   * while the slice streams in, every thread builds its own 8-element pieces
//     (i, i + 256, ...) of the T normalized latent rows in FP32, in registers
//     (each CTA reduces all P routed partials itself: P*T*L*2 bytes, 32 KB per
//     CTA at T = 1, P = 8, L = 2048); the sum of squares goes through one block
//     reduction. Then the sums of the P shared partials of the CTA's columns,
//     8 columns per thread;
//   * as each 8-row chunk lands, every thread forms the 8 x T partial dot
//     products of its latent pieces with the chunk (each W byte is read from
//     shared memory once), a halving shuffle tree leaves each warp's total of
//     accumulator (t, row) on one lane, and the warp stores it;
//   * at the end the 8 warp totals of every output are summed in warp order,
//     the shared sum is added, and the T x rpc results are stored as bf16.
// Each CTA's share of the routed reads grows with T and competes with its W
// slice for the SM's intake; at T >= 3 the two-kernel path (norm kernel, then
// the tensor-core decode kernel) is faster.
// Every CTA computes the latent in the same order, chunks start at absolute
// multiples of 8 columns, and each output element is formed in the same order
// whatever the column range, so column ranges tiling [0, H) reproduce the full
// call bit for bit.
// kFromLatent: y [T, L] (bf16, written by earlier work) is read instead of being
// computed (latent_tail_project_cols).
#include "launch.h"
#include "ptx.cuh"

#include <algorithm>

namespace lt {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerChunk = 8;
constexpr int kMaxChunks = 16;          // mbarriers, one per 8 W rows
constexpr int kMaxPieces = 2;           // 8-element latent pieces per thread: L <= 4096
constexpr int kSmemLimit = 225 * 1024;  // + static smem <= opt-in maximum
constexpr int kStageThreads = 256;

struct GemvParams {
  const uint16_t* routed;  // [P, T, L] (computed latent)
  const float* g;          // [L] or null (no norm)
  const uint16_t* latent;  // [T, L] (kFromLatent)
  const uint16_t* shared;  // [P, T, H]
  const uint16_t* W;       // [H, L]
  uint16_t* out;           // [T, H]
  int P, H, L;
  int col_start, col_end;
  int rpc;                  // W rows per CTA, a multiple of 8
  float eps;
  bool prefetch_shared;     // false when `shared` is page-locked host memory
  uint32_t ssum_offset;     // byte offset of ssum [T][rpc] FP32 in shared memory
  uint32_t part_offset;     // byte offset of the warp totals [chunk][warp][8 * T]
  uint32_t* err;
};

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

__device__ __forceinline__ void widen8(float (&a)[8], const uint4& v) {
  a[0] = bf16_lo(v.x);
  a[1] = bf16_hi(v.x);
  a[2] = bf16_lo(v.y);
  a[3] = bf16_hi(v.y);
  a[4] = bf16_lo(v.z);
  a[5] = bf16_hi(v.z);
  a[6] = bf16_lo(v.w);
  a[7] = bf16_hi(v.w);
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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sums N per-lane accumulators (N a power of two, 8 <= N <= 32) over the warp.
// Returns, on lane i, the total of accumulator i % N. Lane bits at or above N
// are folded by a plain butterfly; below it each step keeps the half of the
// live accumulators that lane bit o selects and adds the partner's other half.
template <int N>
__device__ __forceinline__ float reduce_lanes(float (&v)[N], int lane) {
#pragma unroll
  for (int o = 16; o >= N; o >>= 1)
#pragma unroll
    for (int j = 0; j < N; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], o);
#pragma unroll
  for (int n = N; n > 1; n >>= 1) {
    const int o = n >> 1;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float send = up ? v[j] : v[j + n / 2];
      const float keep = up ? v[j + n / 2] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// Shared memory from the 128-byte-aligned base: [0, rpc * L * 2) the W slice
// (row r at r * L * 2), then ssum [kT][rpc] FP32 at ssum_offset and the warp
// totals [chunk][warp][8 * kT] FP32 at part_offset.
template <bool kFromLatent, int kT>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const GemvParams p) {
  static_assert(kT == 1 || kT == 2, "one or two tokens");
  constexpr int kAcc = kRowsPerChunk * kT;  // 8 or 16 accumulators per thread
  constexpr int kPB = 8;                    // partials loaded per batch
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar[kMaxChunks];
  __shared__ float red[kWarps][kT];
  __shared__ float rnorm[kT];
  __shared__ int abort_flag;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int row0 = p.col_start + static_cast<int>(blockIdx.x) * p.rpc;
  const int nrows = min(p.rpc, p.col_end - row0);  // a multiple of 8
  const int nchunks = nrows / kRowsPerChunk;
  const uint32_t chunk_bytes = static_cast<uint32_t>(kRowsPerChunk * p.L * 2);
  const uint16_t* wsrc = p.W + static_cast<size_t>(row0) * p.L;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 127u) & ~127u) - raw_u32);
  float* ssum = reinterpret_cast<float*>(smem + p.ssum_offset);
  float* part = reinterpret_cast<float*>(smem + p.part_offset);
  volatile int* abort_v = &abort_flag;

  if (tid == 0) {
    for (int c = 0; c < nchunks; ++c) mbar_init(smem_u32(&bar[c]), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  // Ask L2 for the small inputs first, so that their reads below do not queue
  // behind the W stream in HBM: this CTA's 1/grid share of the latent source
  // (routed or latent, read by every CTA) and its own shared-partial columns.
  // Prefetches only warm L2, which any write of the preceding kernel updates.
  if (p.prefetch_shared && tid < p.P * kT) {
    const uint16_t* src = p.shared + static_cast<size_t>(tid) * p.H + row0;  // row (p, t)
    l2_prefetch_bulk(src, static_cast<uint32_t>(nrows) * 2);
  }
  if (tid == kThreads - 1) {
    const uint8_t* src = reinterpret_cast<const uint8_t*>(kFromLatent ? p.latent : p.routed);
    const size_t total = static_cast<size_t>(kFromLatent ? 1 : p.P) * kT * p.L * 2;
    const size_t piece = ((total + gridDim.x - 1) / gridDim.x + 15) / 16 * 16;
    const size_t off = static_cast<size_t>(blockIdx.x) * piece;
    if (off < total) l2_prefetch_bulk(src + off, static_cast<uint32_t>(min(piece, total - off)));
  }
  __syncthreads();
  if (tid == 0)
    for (int c = 0; c < nchunks; ++c)
      l2_prefetch_bulk(wsrc + static_cast<size_t>(c) * kRowsPerChunk * p.L, chunk_bytes);
  // Every input (W included) may be written by the work before this kernel on
  // the stream: nothing is read into the SM before the dependency wait.
  pdl_wait();

  // The first loads of the small inputs are issued before the W copies, so that
  // their data does not queue behind the W slice on its way into the SM:
  // partials 0 .. kPB-1 of this thread's first latent piece (or that piece of
  // the latent) and of its first shared-sum item.
  const int npieces = p.L / 8;
  const int n8 = nrows / 8;
  const size_t rplane = static_cast<size_t>(kT) * p.L;
  const size_t splane = static_cast<size_t>(kT) * p.H;
  uint4 rv[kT][kPB];
  uint4 sv[kPB];
  if (tid < npieces) {
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      if (kFromLatent) {
        rv[t][0] = ld_l2_v4(p.latent + static_cast<size_t>(t) * p.L + tid * 8);
      } else {
#pragma unroll
        for (int q = 0; q < kPB; ++q)
          if (q < p.P)
            rv[t][q] = ld_l2_v4(p.routed + tid * 8 + q * rplane + static_cast<size_t>(t) * p.L);
      }
    }
  }
  if (tid < kT * n8) {
    const int t = tid / n8;
    const uint16_t* src = p.shared + static_cast<size_t>(t) * p.H + row0 + (tid - t * n8) * 8;
#pragma unroll
    for (int q = 0; q < kPB; ++q)
      if (q < p.P) sv[q] = ld_l2_v4(src + q * splane);
  }
  __syncthreads();  // every thread's first loads are in flight
  if (tid == 0) {
    pdl_launch_dependents();  // the next kernel may set up while this one runs
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t b = smem_u32(&bar[c]);
      mbar_arrive_expect_tx(b, chunk_bytes);
      bulk_load(smem_u32(smem) + static_cast<uint32_t>(c) * chunk_bytes,
                wsrc + static_cast<size_t>(c) * kRowsPerChunk * p.L, chunk_bytes, b);
    }
  }

  // (a) This thread's latent pieces k = tid + 256 * i (elements 8k .. 8k + 7) of
  //     the kT tokens in FP32, kept in registers: x summed over the P partials
  //     (p ascending), then, with a norm weight, x * r * g with r from the FP32
  //     sum of x^2.
  float y[kMaxPieces][kT][8];
  float ss[kT];
#pragma unroll
  for (int t = 0; t < kT; ++t) ss[t] = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxPieces; ++i) {
    const int k = tid + kThreads * i;
#pragma unroll
    for (int t = 0; t < kT; ++t)
#pragma unroll
      for (int e = 0; e < 8; ++e) y[i][t][e] = 0.f;
    if (k >= npieces) continue;
    if (kFromLatent) {
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        if (i != 0) rv[t][0] = ld_l2_v4(p.latent + static_cast<size_t>(t) * p.L + k * 8);
        widen8(y[i][t], rv[t][0]);
      }
    } else {
      const uint16_t* src = p.routed + k * 8;
      for (int pp = 0; pp < p.P; pp += kPB) {
        if (i != 0 || pp != 0) {
#pragma unroll
          for (int q = 0; q < kPB; ++q)
#pragma unroll
            for (int t = 0; t < kT; ++t)
              if (pp + q < p.P)
                rv[t][q] = ld_l2_v4(src + (pp + q) * rplane + static_cast<size_t>(t) * p.L);
        }
#pragma unroll
        for (int q = 0; q < kPB; ++q)
#pragma unroll
          for (int t = 0; t < kT; ++t)
            if (pp + q < p.P) add8(y[i][t], rv[t][q]);
      }
#pragma unroll
      for (int t = 0; t < kT; ++t)
#pragma unroll
        for (int e = 0; e < 8; ++e) ss[t] += y[i][t][e] * y[i][t][e];
    }
  }
  if (!kFromLatent && p.g != nullptr) {
#pragma unroll
    for (int t = 0; t < kT; ++t) {
      const float v = warp_sum(ss[t]);
      if (lane == 0) red[warp][t] = v;
    }
    __syncthreads();
    if (tid < kT) {
      float s = 0.f;
      for (int w = 0; w < kWarps; ++w) s += red[w][tid];
      rnorm[tid] = 1.0f / sqrtf(s / static_cast<float>(p.L) + p.eps);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kMaxPieces; ++i) {
      const int k = tid + kThreads * i;
      if (k >= npieces) continue;
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.g) + 2 * k);
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.g) + 2 * k + 1);
      const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int t = 0; t < kT; ++t) {
        const float r = rnorm[t];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[i][t][e] = y[i][t][e] * r * gv[e];
      }
    }
  }

  // (b) Sums of the P shared partials of this CTA's columns (p ascending), 8
  //     columns per thread.
  for (int it = tid; it < kT * n8; it += kThreads) {
    const int t = it / n8;
    const int q8 = it - t * n8;
    const uint16_t* src = p.shared + static_cast<size_t>(t) * p.H + row0 + q8 * 8;
    float s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) s[e] = 0.f;
    for (int pp = 0; pp < p.P; pp += kPB) {
      if (it != tid || pp != 0) {
#pragma unroll
        for (int q = 0; q < kPB; ++q)
          if (pp + q < p.P) sv[q] = ld_l2_v4(src + (pp + q) * splane);
      }
#pragma unroll
      for (int q = 0; q < kPB; ++q)
        if (pp + q < p.P) add8(s, sv[q]);
    }
    float4* dst = reinterpret_cast<float4*>(ssum + t * p.rpc + q8 * 8);
    dst[0] = make_float4(s[0], s[1], s[2], s[3]);
    dst[1] = make_float4(s[4], s[5], s[6], s[7]);
  }

  // (c) Each chunk as it lands: this thread's 8 x kT partial dot products, then
  //     the warp's totals, stored per (chunk, warp).
  for (int c = 0; c < nchunks; ++c) {
    const bool ok = mbar_wait(smem_u32(&bar[c]), 0, p.err, abort_v);
    if (!__all_sync(0xffffffffu, ok)) break;
    const uint8_t* wc = smem + static_cast<size_t>(c) * chunk_bytes;
    float acc[kAcc];
#pragma unroll
    for (int j = 0; j < kAcc; ++j) acc[j] = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPieces; ++i) {
      const int k = tid + kThreads * i;
      if (k >= npieces) continue;
#pragma unroll
      for (int rr = 0; rr < kRowsPerChunk; ++rr) {
        float w[8];
        widen8(w, *reinterpret_cast<const uint4*>(wc + static_cast<size_t>(rr) * p.L * 2 + k * 16));
#pragma unroll
        for (int t = 0; t < kT; ++t) {
          float s = acc[t * kRowsPerChunk + rr];
#pragma unroll
          for (int e = 0; e < 8; ++e) s = fmaf(w[e], y[i][t][e], s);
          acc[t * kRowsPerChunk + rr] = s;
        }
      }
    }
    const float v = reduce_lanes<kAcc>(acc, lane);
    if (lane < kAcc) part[(c * kWarps + warp) * kAcc + lane] = v;
  }
  __syncthreads();

  if (*abort_v) {  // let copies still in flight land before the CTA exits
    if (tid == 0)
      for (int c = 0; c < nchunks; ++c) wait_drain(smem_u32(&bar[c]), 0);
    return;
  }
  // (d) out[t, row0 + r] = bf16(sum over warps, in order, + shared sum).
  for (int i = tid; i < kT * nrows; i += kThreads) {
    const int t = i / nrows;
    const int r = i - t * nrows;
    const float* pc = part + (r / kRowsPerChunk) * kWarps * kAcc + t * kRowsPerChunk +
                      (r % kRowsPerChunk);
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += pc[w * kAcc];
    __nv_bfloat16 b = __float2bfloat16_rn(s + ssum[t * p.rpc + r]);
    p.out[static_cast<size_t>(t) * p.H + row0 + r] = *reinterpret_cast<uint16_t*>(&b);
  }
}

// Copies `n` 16-byte words (page-locked host memory mapped into the device's
// address space -> device memory) for the host-buffer entry point, as a
// programmatic dependent: it waits for the preceding work on the stream, which
// may still read dst, and lets the next kernel set up at once.
__global__ void __launch_bounds__(kStageThreads) stage_kernel(const uint4* src, uint4* dst,
                                                              size_t n) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t stride = static_cast<size_t>(gridDim.x) * kStageThreads;
  for (size_t i = static_cast<size_t>(blockIdx.x) * kStageThreads + threadIdx.x; i < n;
       i += stride)
    dst[i] = src[i];
}

struct GemvPlan {
  int rpc, grid;
  size_t smem;
  uint32_t ssum_offset, part_offset;
};

bool plan_gemv(int T, int L, int width, int num_sms, GemvPlan& g) {
  if (T < 1 || T > kGemvMaxTokens || num_sms < 1 || width < 8 || width % 8 != 0 || L % 8 != 0 ||
      L > kMaxPieces * kThreads * 8)
    return false;
  const int per_sm = (width + num_sms - 1) / num_sms;
  g.rpc = (per_sm + kRowsPerChunk - 1) / kRowsPerChunk * kRowsPerChunk;
  if (g.rpc > kMaxChunks * kRowsPerChunk) return false;
  const size_t w_bytes = static_cast<size_t>(g.rpc) * L * 2;     // a multiple of 128
  const size_t ssum_bytes = static_cast<size_t>(T) * g.rpc * 4;  // a multiple of 32
  const size_t part_bytes =
      static_cast<size_t>(g.rpc / kRowsPerChunk) * kWarps * kRowsPerChunk * T * 4;
  g.ssum_offset = static_cast<uint32_t>(w_bytes);
  g.part_offset = static_cast<uint32_t>(w_bytes + ssum_bytes);
  g.smem = 128 + w_bytes + ssum_bytes + part_bytes;
  if (g.smem > static_cast<size_t>(kSmemLimit)) return false;
  g.grid = (width + g.rpc - 1) / g.rpc;
  return true;
}

template <bool kFromLatent, int kT>
cudaError_t launch(const GemvParams& p, const GemvPlan& g, cudaStream_t stream) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(g.grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<kFromLatent, kT>, p);
}

template <bool kFromLatent>
cudaError_t launch_t(int T, const GemvParams& p, const GemvPlan& g, cudaStream_t stream) {
  static_assert(kGemvMaxTokens == 2, "one instantiation per token count");
  return T == 1 ? launch<kFromLatent, 1>(p, g, stream) : launch<kFromLatent, 2>(p, g, stream);
}

template <bool kFromLatent>
cudaError_t set_limits() {
  cudaError_t e = cudaFuncSetAttribute(gemv_kernel<kFromLatent, 1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_kernel<kFromLatent, 2>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
}

}  // namespace

cudaError_t setup_gemv(const DeviceInfo&) {
  const cudaError_t e = set_limits<false>();
  return e != cudaSuccess ? e : set_limits<true>();
}

bool gemv_supported(int T, int L, int col_start, int col_end, const DeviceInfo& dev) {
  GemvPlan g;
  return plan_gemv(T, L, col_end - col_start, dev.num_sms, g);
}

cudaError_t launch_gemv(const GemvArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  GemvPlan g;
  if (!plan_gemv(a.T, a.L, a.col_end - a.col_start, dev.num_sms, g))
    return cudaErrorInvalidConfiguration;
  GemvParams p{};
  p.routed = a.routed;
  p.g = a.g;
  p.latent = a.latent;
  p.shared = a.shared;
  p.W = a.W;
  p.out = a.out;
  p.P = a.P;
  p.H = a.H;
  p.L = a.L;
  p.col_start = a.col_start;
  p.col_end = a.col_end;
  p.rpc = g.rpc;
  p.eps = a.eps;
  p.prefetch_shared = !a.shared_on_host;
  p.ssum_offset = g.ssum_offset;
  p.part_offset = g.part_offset;
  p.err = dev.err_word;
  return a.latent != nullptr ? launch_t<true>(a.T, p, g, stream)
                             : launch_t<false>(a.T, p, g, stream);
}

cudaError_t launch_stage(const void* src, void* dst, size_t bytes, const DeviceInfo& dev,
                         cudaStream_t stream) {
  if (bytes % 16 != 0 || reinterpret_cast<uintptr_t>(src) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(dst) % 16 != 0)
    return cudaErrorInvalidValue;
  const size_t n = bytes / 16;
  if (n == 0) return cudaSuccess;
  const size_t blocks = (n + kStageThreads - 1) / kStageThreads;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(std::min<size_t>(blocks, dev.num_sms)), 1, 1);
  cfg.blockDim = dim3(kStageThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stage_kernel, static_cast<const uint4*>(src),
                            static_cast<uint4*>(dst), n);
}

}  // namespace lt
