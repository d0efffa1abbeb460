// Steps 3-5 of the latent-MoE tail for prefill-sized token counts (T > 128):
//   out[t,h] = bf16_rn( sum_l y[t,l] * W[h,l] + sum_p shared[p,t,h] ),  h in [c0,c1)
// The narrowed beta-add GEMM of PR #50383's `_shard_up_proj_tail`
// (`hidden_shard.addmm_(latent, up_proj_shard.t())`), with the shared-partial
// sum of the final all-reduce done in the GEMM epilogue.
//
// Persistent, warp-specialized tcgen05 kernel, one CTA per SM:
//   warp 0      TMA producer: y tile [128 tokens x 64] and W tile [256 rows x 64]
//               per K-block into a 4-stage ring (128-byte swizzle);
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//               (M = 128 tokens, N = 256 output columns, K = 16 per instruction);
//   warps 2..5  epilogue: TMEM -> registers (32 columns at a time), add the P
//               shared partials with 16-byte loads, round to bf16, 16-byte stores.
// Two TMEM accumulators (2 x 256 columns) let the epilogue of one tile run
// while the MMAs of the next tile accumulate. Output tiles sit at absolute
// multiples of 256 columns, so a column-range call computes each element
// exactly as the full call does.
#include "launch.h"
#include "ptx.cuh"

#include <algorithm>

namespace lt {
namespace {

constexpr int kTileT = 128;  // tokens per tile (MMA M)
constexpr int kTileH = 256;  // output columns per tile (MMA N)
constexpr int kBlockK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kAStage = kTileT * kBlockK * 2;  // 16 KB of y
constexpr uint32_t kBStage = kTileH * kBlockK * 2;  // 32 KB of W
constexpr uint32_t kStageBytes = kAStage + kBStage;
constexpr uint32_t kTmemCols = 2 * kTileH;
constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes;

struct PrefillParams {
  const uint16_t* shared;
  uint16_t* out;
  int P, T, L, H;
  int col_start, col_end;
  int htile0;       // absolute index of the first 256-column tile
  int n_htiles;
  int n_ttiles;
  int total_kb;
  int pdl;
  uint32_t* err;
};

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

struct TileCoord {
  int t0, h0;
};

__device__ __forceinline__ TileCoord tile_coord(const PrefillParams& p, int tile) {
  TileCoord c;
  c.t0 = (tile / p.n_htiles) * kTileT;
  c.h0 = (p.htile0 + tile % p.n_htiles) * kTileH;
  return c;
}

// Adds 8 bf16 values of one shared partial to s[0..7].
__device__ __forceinline__ void add8(float* s, const uint4& v) {
  s[0] += bf16_lo(v.x);
  s[1] += bf16_hi(v.x);
  s[2] += bf16_lo(v.y);
  s[3] += bf16_hi(v.y);
  s[4] += bf16_lo(v.z);
  s[5] += bf16_hi(v.z);
  s[6] += bf16_lo(v.w);
  s[7] += bf16_hi(v.w);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap y_map,
                   const __grid_constant__ CUtensorMap w_map, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages];
  __shared__ uint64_t empty_bar[kStages];
  __shared__ uint64_t accf_bar[2];
  __shared__ uint64_t acce_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int num_tiles = p.n_ttiles * p.n_htiles;
  const int my_tiles =
      static_cast<int>(blockIdx.x) < num_tiles
          ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
          : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&accf_bar[a]), 1);
      mbar_init(smem_u32(&acce_bar[a]), 4 * 32);
    }
    abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_map(&y_map);
    tma_prefetch_map(&w_map);
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_v = &abort_flag;

  if (warp == 0) {
    if (lane == 0 && my_tiles > 0) {
      // ---------------- TMA producer ----------------
      const int total = my_tiles * p.total_kb;
      const int pre = min(kStages, total);
      auto coord_of = [&](int it, TileCoord& c, int& kb) {
        const int local = it / p.total_kb;
        kb = it - local * p.total_kb;
        c = tile_coord(p, static_cast<int>(blockIdx.x) + local * static_cast<int>(gridDim.x));
      };
      for (int it = 0; it < pre; ++it) {  // W does not depend on the norm kernel
        TileCoord c;
        int kb;
        coord_of(it, c, kb);
        const uint32_t st = sbase + static_cast<uint32_t>(it) * kStageBytes;
        const uint32_t fb = smem_u32(&full_bar[it]);
        mbar_arrive_expect_tx(fb, kStageBytes);
        tma_load_2d(st + kAStage, &w_map, fb, kb * kBlockK, c.h0);
      }
      if (p.pdl) pdl_wait();
      for (int it = 0; it < pre; ++it) {
        TileCoord c;
        int kb;
        coord_of(it, c, kb);
        const uint32_t st = sbase + static_cast<uint32_t>(it) * kStageBytes;
        tma_load_2d(st, &y_map, smem_u32(&full_bar[it]), kb * kBlockK, c.t0);
      }
      int issued = pre;
      for (int it = pre; it < total; ++it) {
        const int s = it % kStages;
        const uint32_t round = static_cast<uint32_t>(it / kStages);
        if (!mbar_wait(smem_u32(&empty_bar[s]), (round & 1u) ^ 1u, p.err, abort_v)) break;
        TileCoord c;
        int kb;
        coord_of(it, c, kb);
        const uint32_t st = sbase + static_cast<uint32_t>(s) * kStageBytes;
        const uint32_t fb = smem_u32(&full_bar[s]);
        mbar_arrive_expect_tx(fb, kStageBytes);
        tma_load_2d(st, &y_map, fb, kb * kBlockK, c.t0);
        tma_load_2d(st + kAStage, &w_map, fb, kb * kBlockK, c.h0);
        issued = it + 1;
      }
      if (*abort_v) {
        for (int it = max(0, issued - kStages); it < issued; ++it)
          wait_drain(smem_u32(&full_bar[it % kStages]), static_cast<uint32_t>(it / kStages) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && my_tiles > 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = umma_idesc_bf16(kTileT, kTileH);
      int it = 0;
      bool alive = true;
      for (int i = 0; i < my_tiles && alive; ++i) {
        const int acc = i & 1;
        const uint32_t use = static_cast<uint32_t>(i >> 1);
        if (!mbar_wait(smem_u32(&acce_bar[acc]), (use & 1u) ^ 1u, p.err, abort_v)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(acc * kTileH);
        for (int kb = 0; kb < p.total_kb; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t round = static_cast<uint32_t>(it / kStages);
          if (!mbar_wait(smem_u32(&full_bar[s]), round & 1u, p.err, abort_v)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = sbase + static_cast<uint32_t>(s) * kStageBytes;
          const uint32_t b = a + kAStage;
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k)
            umma_bf16(d, umma_desc_sw128(a + 32u * k), umma_desc_sw128(b + 32u * k), idesc,
                      (kb | k) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&empty_bar[s]));
        }
        umma_commit(smem_u32(&accf_bar[acc]));
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const size_t plane = static_cast<size_t>(p.T) * p.H;
    for (int i = 0; i < my_tiles; ++i) {
      const int acc = i & 1;
      const uint32_t use = static_cast<uint32_t>(i >> 1);
      bool ok = mbar_wait(smem_u32(&accf_bar[acc]), use & 1u, p.err, abort_v);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const TileCoord c =
          tile_coord(p, static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x));
      const int t = c.t0 + q * 32 + lane;
      const bool row_ok = t < p.T;
      const uint32_t dcol = tmem + lane_base + static_cast<uint32_t>(acc * kTileH);
#pragma unroll 1
      for (int ch = 0; ch < kTileH / 32; ++ch) {
        const int hb = c.h0 + ch * 32;
        float v[32];
        __syncwarp();  // tcgen05.ld needs the whole warp converged
        tmem_ld32(dcol + static_cast<uint32_t>(ch * 32), v);
        if (ch == kTileH / 32 - 1) {  // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          mbar_arrive(smem_u32(&acce_bar[acc]));
        }
        if (!row_ok || hb >= p.col_end || hb + 32 <= p.col_start) continue;
        bool gv[4];  // 8-column groups inside [col_start, col_end) (col_end <= H)
#pragma unroll
        for (int g = 0; g < 4; ++g) gv[g] = hb + g * 8 >= p.col_start && hb + g * 8 < p.col_end;
        float s[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) s[j] = 0.f;
        const uint16_t* src = p.shared + static_cast<size_t>(t) * p.H + hb;
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        int pp = 0;
        for (; pp + 4 <= p.P; pp += 4) {
          uint4 w[4][4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int g = 0; g < 4; ++g)
              w[k][g] = gv[g] ? ld_stream_v4(src + (pp + k) * plane + g * 8) : zero;
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int g = 0; g < 4; ++g) add8(&s[g * 8], w[k][g]);
        }
        for (; pp < p.P; ++pp) {
#pragma unroll
          for (int g = 0; g < 4; ++g)
            add8(&s[g * 8], gv[g] ? ld_stream_v4(src + pp * plane + g * 8) : zero);
        }
        uint16_t* dst = p.out + static_cast<size_t>(t) * p.H + hb;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          if (!gv[g]) continue;
          uint4 o;
          o.x = pack_bf16x2(v[g * 8 + 0] + s[g * 8 + 0], v[g * 8 + 1] + s[g * 8 + 1]);
          o.y = pack_bf16x2(v[g * 8 + 2] + s[g * 8 + 2], v[g * 8 + 3] + s[g * 8 + 3]);
          o.z = pack_bf16x2(v[g * 8 + 4] + s[g * 8 + 4], v[g * 8 + 5] + s[g * 8 + 5]);
          o.w = pack_bf16x2(v[g * 8 + 6] + s[g * 8 + 6], v[g * 8 + 7] + s[g * 8 + 7]);
          *reinterpret_cast<uint4*>(dst + g * 8) = o;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (*abort_v && lane == 0) {  // no MMA may still write TMEM when it is freed
      const int last = my_tiles - 1;
      for (int i = max(0, last - 1); i <= last; ++i)
        wait_drain(smem_u32(&accf_bar[i & 1]), static_cast<uint32_t>(i >> 1) & 1u);
    }
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

cudaError_t setup_prefill(const DeviceInfo&) {
  return cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmemBytes));
}

cudaError_t launch_prefill(const ProjectArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  PrefillParams p{};
  p.shared = a.shared;
  p.out = a.out;
  p.P = a.P;
  p.T = a.T;
  p.L = a.L;
  p.H = a.H;
  p.col_start = a.col_start;
  p.col_end = a.col_end;
  p.htile0 = a.col_start / kTileH;
  p.n_htiles = (a.col_end - 1) / kTileH - p.htile0 + 1;
  p.n_ttiles = ceil_div(a.T, kTileT);
  p.total_kb = ceil_div(a.L, kBlockK);
  p.pdl = a.pdl ? 1 : 0;
  p.err = dev.err_word;
  const long long tiles = static_cast<long long>(p.n_htiles) * p.n_ttiles;
  const int grid = static_cast<int>(std::min<long long>(dev.num_sms, tiles));

  CUtensorMap y_map, w_map;
  if (!make_map_bf16_sw128(&y_map, a.y, a.T, a.L, kTileT)) return cudaErrorInvalidValue;
  if (!make_map_bf16_sw128(&w_map, a.W, a.H, a.L, kTileH)) return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[1];
  int n = 0;
  if (a.pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = static_cast<unsigned>(n);
  return cudaLaunchKernelEx(&cfg, prefill_kernel, y_map, w_map, p);
}

}  // namespace lt
