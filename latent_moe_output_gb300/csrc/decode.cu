// Steps 3-5 of the latent-MoE tail for decode-sized token counts (T <= 128):
//   out[t,h] = bf16_rn( sum_l y[t,l] * W[h,l] + sum_p shared[p,t,h] ),  h in [c0,c1)
// The narrowed beta-add GEMM of PR #50383's `_shard_up_proj_tail`
// (`hidden_shard.addmm_(latent, up_proj_shard.t())`) with the shared-partial
// sum of the final all-reduce folded into the epilogue.
//
// At these sizes the call is bound by streaming W (H*L*2 bytes) from HBM once,
// so the kernel is shaped around that stream:
//   * swap-AB tensor-core product: the MMA's M=128 rows are W rows (output
//     columns h), its N are the T tokens padded to a multiple of 16, K = L;
//     the FP32 accumulator D[h][t] lives in TMEM;
//   * one CTA per (128-row tile, K slice). The KS slices of a tile form one
//     thread-block cluster; the KS partial accumulators are summed through
//     distributed shared memory in a fixed order (q = 0..KS-1), so results do
//     not depend on the requested column range;
//   * W and y K-blocks (64 wide, 128-byte rows) arrive by TMA into a stage
//     ring; one thread issues TMA, one issues tcgen05.mma; under programmatic
//     dependent launch the W loads of the first stages are issued before
//     waiting for the norm kernel that produces y;
//   * epilogue: each CTA finishes 128/KS rows for all tokens, adding the P
//     shared partials (p ascending) in FP32 and storing bf16.
#include "launch.h"
#include "ptx.cuh"

#include <algorithm>

namespace lt {
namespace {

constexpr int kBlockM = 128;                           // W rows per tile
constexpr int kBlockK = 64;                            // K per stage (128-byte rows)
constexpr int kThreads = 128;
constexpr int kMaxStages = 8;
constexpr uint32_t kWStageBytes = kBlockM * kBlockK * 2;  // 16 KB
constexpr int kSmemBudget = 72 * 1024;                  // keeps 3 CTAs per SM

struct DecodeParams {
  const uint16_t* shared;
  uint16_t* out;
  int P, T, L, H;
  int col_start, col_end;
  int tile0;       // absolute index of the first 128-row tile
  int ks;          // K slices per tile == cluster size
  int kb_per_cta;  // K-blocks per slice
  int total_kb;    // ceil(L / 64)
  int npad;        // MMA N: tokens rounded up to a multiple of 16
  int stages;
  int tmem_cols;
  int pdl;
  uint32_t* err;
};

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap w_map,
                  const __grid_constant__ CUtensorMap y_map, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages];
  __shared__ uint64_t empty_bar[kMaxStages];
  __shared__ uint64_t acc_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int h0 = (p.tile0 + static_cast<int>(blockIdx.y)) * kBlockM;
  const int kb_begin = static_cast<int>(rank) * p.kb_per_cta;
  const int nkb = max(0, min(p.total_kb, kb_begin + p.kb_per_cta) - kb_begin);
  const uint32_t stage_bytes = kWStageBytes + static_cast<uint32_t>(p.npad) * 128u;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  float* part = reinterpret_cast<float*>(smem_raw + (sbase - raw_u32));  // [npad][128]

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&acc_bar), 1);
    abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_map(&w_map);
    tma_prefetch_map(&y_map);
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), static_cast<uint32_t>(p.tmem_cols));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_v = &abort_flag;

  if (warp == 0) {
    if (lane == 0 && nkb > 0) {
      // ---------------- TMA producer ----------------
      const int pre = min(p.stages, nkb);
      for (int i = 0; i < pre; ++i) {
        const uint32_t st = sbase + static_cast<uint32_t>(i) * stage_bytes;
        const uint32_t fb = smem_u32(&full_bar[i]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        tma_load_2d(st, &w_map, fb, (kb_begin + i) * kBlockK, h0);
      }
      if (p.pdl) pdl_wait();  // y is written by the preceding norm kernel
      for (int i = 0; i < pre; ++i) {
        const uint32_t st = sbase + static_cast<uint32_t>(i) * stage_bytes;
        tma_load_2d(st + kWStageBytes, &y_map, smem_u32(&full_bar[i]), (kb_begin + i) * kBlockK,
                    0);
      }
      int issued = pre;
      for (int i = pre; i < nkb; ++i) {
        const int s = i % p.stages;
        const uint32_t round = static_cast<uint32_t>(i / p.stages);
        if (!mbar_wait(smem_u32(&empty_bar[s]), (round & 1u) ^ 1u, p.err, abort_v)) break;
        const uint32_t st = sbase + static_cast<uint32_t>(s) * stage_bytes;
        const uint32_t fb = smem_u32(&full_bar[s]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        tma_load_2d(st, &w_map, fb, (kb_begin + i) * kBlockK, h0);
        tma_load_2d(st + kWStageBytes, &y_map, fb, (kb_begin + i) * kBlockK, 0);
        issued = i + 1;
      }
      if (*abort_v) {  // let copies already in flight land before the CTA exits
        for (int i = max(0, issued - p.stages); i < issued; ++i)
          wait_drain(smem_u32(&full_bar[i % p.stages]), static_cast<uint32_t>(i / p.stages) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && nkb > 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = umma_idesc_bf16(kBlockM, p.npad);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % p.stages;
        const uint32_t round = static_cast<uint32_t>(i / p.stages);
        if (!mbar_wait(smem_u32(&full_bar[s]), round & 1u, p.err, abort_v)) break;
        tc_fence_after();
        const uint32_t a = sbase + static_cast<uint32_t>(s) * stage_bytes;
        const uint32_t b = a + kWStageBytes;
#pragma unroll
        for (int k = 0; k < kBlockK / 16; ++k)
          umma_bf16(tmem, umma_desc_sw128(a + 32u * k), umma_desc_sw128(b + 32u * k), idesc,
                    (i | k) != 0 ? 1u : 0u);
        umma_commit(smem_u32(&empty_bar[s]));
      }
      umma_commit(smem_u32(&acc_bar));  // fires once every issued MMA has completed
    }
    __syncwarp();
  }

  // ---------------- epilogue part 1: TMEM -> shared-memory partial ----------------
  const bool have_acc = nkb > 0;
  bool ok = true;
  if (have_acc) {
    ok = mbar_wait(smem_u32(&acc_bar), 0, p.err, abort_v);
    tc_fence_after();
  }
  ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below needs a converged warp
  {
    const int row = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    for (int c = 0; c < p.npad; c += 16) {
      float v[16];
      __syncwarp();  // tcgen05.ld needs the whole warp converged
      if (have_acc && ok) {
        tmem_ld16(tmem + lane_base + static_cast<uint32_t>(c), v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c + j < p.T) part[(c + j) * kBlockM + row] = v[j];
    }
  }
  __syncwarp();
  cluster_sync();  // every slice's partial is now visible to the cluster

  // ---------------- epilogue part 2: split-K sum + shared partials ----------------
  {
    const int rpc = kBlockM / p.ks;  // rows finished by this CTA
    const int r0 = static_cast<int>(rank) * rpc;
    const int my_row = threadIdx.x % rpc;
    const int ngroups = kThreads / rpc;
    const int tg = threadIdx.x / rpc;
    const int h = h0 + r0 + my_row;
    const bool col_ok = h >= p.col_start && h < p.col_end;
    const uint32_t part_u32 = smem_u32(part);
    uint32_t peer[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) peer[q] = q < p.ks ? map_to_rank(part_u32, q) : 0u;
    const size_t plane = static_cast<size_t>(p.T) * p.H;
    for (int t = tg; t < p.T; t += ngroups) {
      const uint32_t off = static_cast<uint32_t>((t * kBlockM + r0 + my_row) * 4);
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < p.ks) acc += ld_dsmem_f32(peer[q] + off);
      if (col_ok) {
        const unsigned short* src =
            reinterpret_cast<const unsigned short*>(p.shared) + static_cast<size_t>(t) * p.H + h;
        float s = 0.f;
        for (int pp = 0; pp < p.P; ++pp)
          s += __uint_as_float(static_cast<uint32_t>(__ldg(src + pp * plane)) << 16);
        const __nv_bfloat16 o = __float2bfloat16_rn(acc + s);
        p.out[static_cast<size_t>(t) * p.H + h] = *reinterpret_cast<const uint16_t*>(&o);
      }
    }
  }
  __syncwarp();
  cluster_sync();  // peers have finished reading this CTA's partial

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (*abort_v && have_acc && lane == 0) wait_drain(smem_u32(&acc_bar), 0);
    __syncwarp();
    tmem_dealloc(tmem, static_cast<uint32_t>(p.tmem_cols));
  }
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

int next_pow2_at_least(int v, int lo) {
  int r = lo;
  while (r < v) r <<= 1;
  return r;
}

#ifdef LT_TUNING
#include <cstdlib>
int env_int(const char* name, int dflt) {
  const char* s = std::getenv(name);
  return s ? std::atoi(s) : dflt;
}
#endif

}  // namespace

cudaError_t setup_decode(const DeviceInfo&) {
  return cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              1024 + 64 * 1024 + kSmemBudget);
}

cudaError_t launch_decode(const ProjectArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  DecodeParams p{};
  p.shared = a.shared;
  p.out = a.out;
  p.P = a.P;
  p.T = a.T;
  p.L = a.L;
  p.H = a.H;
  p.col_start = a.col_start;
  p.col_end = a.col_end;
  p.total_kb = ceil_div(a.L, kBlockK);
  p.npad = ceil_div(std::max(a.T, 1), 16) * 16;
  // K split: a fixed function of L (never of the column range), so that every
  // output element is summed in the same order whatever range is requested.
  int ks = std::max(1, std::min(8, p.total_kb / 4));
  while (ks & (ks - 1)) ks &= ks - 1;  // power of two: 128 rows split evenly
#ifdef LT_TUNING
  ks = env_int("LT_DECODE_KS", ks);
#endif
  p.ks = ks;
  p.kb_per_cta = ceil_div(p.total_kb, ks);
  const uint32_t stage_bytes = kWStageBytes + static_cast<uint32_t>(p.npad) * 128u;
  int stages = std::min(p.kb_per_cta, std::max(1, kSmemBudget / static_cast<int>(stage_bytes)));
  stages = std::min(stages, kMaxStages);
#ifdef LT_TUNING
  stages = std::min(std::max(1, env_int("LT_DECODE_STAGES", stages)), kMaxStages);
#endif
  p.stages = stages;
  p.tmem_cols = next_pow2_at_least(p.npad, 32);
  p.pdl = a.pdl ? 1 : 0;
  p.err = dev.err_word;
  const int tile_first = a.col_start / kBlockM;
  const int tile_last = (a.col_end - 1) / kBlockM;
  p.tile0 = tile_first;
  const int ntiles = tile_last - tile_first + 1;
  const size_t part_bytes = static_cast<size_t>(p.npad) * kBlockM * sizeof(float);
  const size_t smem = 1024 + std::max(static_cast<size_t>(stages) * stage_bytes, part_bytes);

  CUtensorMap w_map, y_map;
  if (!make_map_bf16_sw128(&w_map, a.W, a.H, a.L, kBlockM)) return cudaErrorInvalidValue;
  if (!make_map_bf16_sw128(&y_map, a.y, a.T, a.L, static_cast<uint32_t>(p.npad)))
    return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(ks), static_cast<unsigned>(ntiles), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  attrs[n].id = cudaLaunchAttributeClusterDimension;
  attrs[n].val.clusterDim.x = static_cast<unsigned>(ks);
  attrs[n].val.clusterDim.y = 1;
  attrs[n].val.clusterDim.z = 1;
  ++n;
  if (a.pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = static_cast<unsigned>(n);
  return cudaLaunchKernelEx(&cfg, decode_kernel, w_map, y_map, p);
}

}  // namespace lt
