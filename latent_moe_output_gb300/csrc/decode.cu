// Steps 3-5 of the latent-MoE tail for decode-sized token counts (T <= 224):
//   out[t,h] = bf16_rn( sum_l y[t,l] * W[h,l] + sum_p shared[p,t,h] ),  h in [c0,c1)
// The narrowed beta-add GEMM of PR #50383's `_shard_up_proj_tail`
// (`hidden_shard.addmm_(latent, up_proj_shard.t())`) with the shared-partial
// sum of the final all-reduce folded into the epilogue.
//
// At these sizes the call is bound by streaming W (H*L*2 bytes) from HBM once,
// so the kernel is shaped around that stream:
//   * swap-AB tensor-core product: the MMA's M = 128 rows are W rows (output
//     columns h), its N are the T tokens padded to a multiple of 16, K = L;
//     the FP32 accumulator D[h][t] lives in TMEM;
//   * one CTA per (128-row tile, K slice); the KS slices of a tile form one
//     thread-block cluster. KS = 8 for up to 16 tokens (four CTAs per SM),
//     KS = 4 (two CTAs per SM) up to 96 tokens while its buffers fit in half
//     an SM, else 2;
//   * W boxes (128 x 64, 128-byte swizzle) are requested before the rest of the
//     set-up, and under programmatic dependent launch before waiting for the
//     norm kernel that writes y (which has already prefetched W into L2); one
//     thread issues TMA, one issues tcgen05.mma;
//   * with early release, each CTA lets the next kernel on the stream launch
//     once it has issued its last W copy, so the next call's norm kernel
//     prefetches its W while this call finishes;
//   * while W streams in, the epilogue warps sum the P shared partials of the
//     rows this CTA finishes (p ascending, FP32) into shared memory;
//   * after the MMAs and a cluster barrier (every stage ring of the cluster is
//     then free), every CTA pushes each accumulator row into the ring of the
//     cluster CTA that finishes that row (DSMEM stores, token-major so that a
//     warp's stores are contiguous), a second cluster barrier, then each CTA
//     adds the KS partials in fixed slice order plus the shared sum and stores
//     bf16. The summation order never depends on the requested column range.
#include "launch.h"
#include "ptx.cuh"

#include <algorithm>

namespace lt {
namespace {

constexpr int kBlockM = kDecodeTileRows;                  // W rows per tile
constexpr int kBlockK = 64;                               // K per stage (128-byte rows)
constexpr int kThreads = 192;                             // TMA, MMA, 4 epilogue warps
constexpr int kEpiThreads = 128;
constexpr int kMaxStages = 16;
constexpr uint32_t kWStageBytes = kBlockM * kBlockK * 2;  // 16 KB
constexpr int kSmemLimit = 220 * 1024;                   // + static smem <= opt-in max
constexpr int kSmemBudget = 210 * 1024;                   // one CTA per SM
constexpr int kHalfSmBudget = 110 * 1024;                 // two CTAs per SM
// Four K slices (two CTAs per SM) only up to this many padded tokens: at 97-112
// tokens two slices on one CTA per SM were faster (GB300, P = 8, L = 2048,
// H = 7168, forward call 15.6-15.9 against 16.7-17.2 us at T = 104 and 112),
// at 96 and below four (14.0 against 14.8 us at T = 96, 13.1 against 15.0 at 80).
constexpr int kFourSliceMaxNpad = 96;
// Eight K slices (448 CTAs at H = 7168, clusters of 8, four CTAs per SM) for up to
// 16 tokens: every SM then streams about the same share of W (against 256 KB on 72
// SMs and 128 KB on the other 80 with four slices). Measured 1-3 % faster per call
// at T = 3...16 (GB300, P = 8, L = 2048, H = 7168: T = 16 10.46-10.48 against
// 10.58-10.63 us, T = 3 9.58 against 9.83-9.88 us).
constexpr int kEightSliceMaxNpad = 16;
constexpr int kQuarterSmBudget = 55 * 1024;  // four CTAs per SM

constexpr int kTwoPerSm = 0;
constexpr int kOnePerSmMode = 1;
constexpr int kFourPerSm = 2;

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
  uint32_t ssum_offset;  // byte offsets (from the 1024-aligned base) of the shared-partial
  uint32_t slot_offset;  // sums and of the received K-slice partials (0: in the ring)
  int pdl;
  int inputs_ready;         // W and shared complete at launch (only y is awaited)
  int trigger_after_issue;  // allow dependents once the last W copy is issued
  uint32_t* err;
};

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
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

// Shared-memory layout from the 1024-aligned base:
//   [0, region)        stage ring: W box [128 x 64] then y box [npad x 64], 128B swizzle
//   [ssum_offset, ..)  ssum[t][r]: sum_p shared[p, t, h0 + r0 + r] for this CTA's rows
//   [slot_offset, ..)  slot[src][t][r]: the K-slice partial of row r0 + r pushed by CTA
//                      src; above 32 tokens slot_offset is 0: the partials then reuse
//                      the ring once every CTA of the cluster has finished its MMAs,
//                      which leaves room for more stages (region = the larger of the two)
// kMode: how many CTAs the launch puts on an SM. kTwoPerSm (KS = 4), kOnePerSm
// (KS <= 2; see (a) below) or kFourPerSm (KS = 8, register use capped so that
// four CTAs fit in the register file).
template <int kMode>
__global__ void __launch_bounds__(kThreads, kMode == kFourPerSm ? 4 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap w_map,
                  const __grid_constant__ CUtensorMap y_map, const DecodeParams p) {
  constexpr bool kOnePerSm = kMode == kOnePerSmMode;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages];
  __shared__ uint64_t empty_bar[kMaxStages];
  __shared__ uint64_t acc_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // K slice of this CTA; equal to its rank in the cluster (grid x == cluster x).
  const uint32_t rank = blockIdx.x;
  const int h0 = (p.tile0 + static_cast<int>(blockIdx.y)) * kBlockM;
  const int kb_begin = static_cast<int>(rank) * p.kb_per_cta;
  const int nkb = max(0, min(p.total_kb, kb_begin + p.kb_per_cta) - kb_begin);
  const uint32_t stage_bytes = kWStageBytes + static_cast<uint32_t>(p.npad) * 128u;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_u32);
  float* ssum = reinterpret_cast<float*>(sgen + p.ssum_offset);
  float* slot = reinterpret_cast<float*>(sgen + p.slot_offset);
  const int rpc = kBlockM / p.ks;  // output rows this CTA finishes
  const int r0 = static_cast<int>(rank) * rpc;
  const int groups = rpc / 8;      // 8-row (16-byte) groups per token
  volatile int* abort_v = &abort_flag;
  const int pre = min(p.stages, nkb);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&acc_bar), 1);
    abort_flag = 0;
    mbar_fence_init();
    // When W does not depend on the preceding kernel, request the first stages
    // now, before the rest of the set-up, so the HBM stream starts at once.
    if (!p.pdl || p.inputs_ready)
      for (int i = 0; i < pre; ++i) {
        const uint32_t fb = smem_u32(&full_bar[i]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        tma_load_2d(sbase + static_cast<uint32_t>(i) * stage_bytes, &w_map, fb,
                    (kb_begin + i) * kBlockK, h0);
      }
  }
  if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), static_cast<uint32_t>(p.tmem_cols));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const bool have_acc = nkb > 0;
  bool acc_ok = true;  // epilogue warps: the accumulator is complete and readable

  if (warp == 0) {
    if (lane == 0 && nkb > 0) {
      // ---------------- TMA producer ----------------
      if (p.pdl) pdl_wait();  // y is written by the preceding kernel
      for (int i = 0; i < pre; ++i) {
        const uint32_t st = sbase + static_cast<uint32_t>(i) * stage_bytes;
        const uint32_t fb = smem_u32(&full_bar[i]);
        if (p.pdl && !p.inputs_ready) {  // W after the wait too
          mbar_arrive_expect_tx(fb, stage_bytes);
          tma_load_2d(st, &w_map, fb, (kb_begin + i) * kBlockK, h0);
        }
        tma_load_2d(st + kWStageBytes, &y_map, fb, (kb_begin + i) * kBlockK, 0);
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
      if (p.trigger_after_issue) pdl_launch_dependents();
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
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    // (a) While W streams in: sum the P shared partials of this CTA's rows,
    //     p ascending in FP32, into shared memory. After a norm kernel of the same
    //     call they are read without waiting: the work that wrote them finished
    //     before that kernel released this one. Read from L2, never through a
    //     possibly stale L1.
    if (p.pdl && !p.inputs_ready) pdl_wait();
    const int et = threadIdx.x - 64;
    const size_t plane = static_cast<size_t>(p.T) * p.H;
    const int items = p.T * groups;
    if constexpr (kOnePerSm) {
      // With one CTA per SM this sum can outlast the MMAs, so a thread takes two
      // 8-column pieces at a time (16 loads in flight). With two CTAs per SM the
      // extra loads and registers cost more than they saved (the loop below).
      constexpr int per = 2;
      for (int i0 = et; i0 < items; i0 += per * kEpiThreads) {
        const uint16_t* src[2];
        bool live[2], load[2];
        float a[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = i0 + u * kEpiThreads;
          const int t = i / groups;
          const int h = h0 + r0 + (i - t * groups) * 8;
          live[u] = i < items;
          load[u] = live[u] && h >= p.col_start && h < p.col_end;
          src[u] = p.shared + static_cast<size_t>(t) * p.H + h;
#pragma unroll
          for (int j = 0; j < 8; ++j) a[u][j] = 0.f;
        }
        int pp = 0;
        for (; pp + 8 <= p.P; pp += 8) {
          uint4 v[2][8];
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (load[u])
#pragma unroll
              for (int k = 0; k < 8; ++k) v[u][k] = ld_l2_v4(src[u] + (pp + k) * plane);
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (load[u])
#pragma unroll
              for (int k = 0; k < 8; ++k) add8(a[u], v[u][k]);
        }
        for (; pp < p.P; ++pp)
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (load[u]) add8(a[u], ld_l2_v4(src[u] + pp * plane));
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (!live[u]) continue;
          const int i = i0 + u * kEpiThreads;
          const int t = i / groups;
          float4* dst = reinterpret_cast<float4*>(ssum + t * rpc + (i - t * groups) * 8);
          dst[0] = make_float4(a[u][0], a[u][1], a[u][2], a[u][3]);
          dst[1] = make_float4(a[u][4], a[u][5], a[u][6], a[u][7]);
        }
      }
    } else {
      for (int i = et; i < items; i += kEpiThreads) {
        const int t = i / groups;
        const int g = i - t * groups;
        const int h = h0 + r0 + g * 8;
        float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (h >= p.col_start && h < p.col_end) {
          const uint16_t* src = p.shared + static_cast<size_t>(t) * p.H + h;
          int pp = 0;
          for (; pp + 8 <= p.P; pp += 8) {
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = ld_l2_v4(src + (pp + k) * plane);
#pragma unroll
            for (int k = 0; k < 8; ++k) add8(a, v[k]);
          }
          for (; pp < p.P; ++pp) add8(a, ld_l2_v4(src + pp * plane));
        }
        float4* dst = reinterpret_cast<float4*>(ssum + t * rpc + g * 8);
        dst[0] = make_float4(a[0], a[1], a[2], a[3]);
        dst[1] = make_float4(a[4], a[5], a[6], a[7]);
      }
    }
    // (b) Wait for this CTA's MMAs (its ring is then no longer read).
    if (have_acc) {
      acc_ok = mbar_wait(smem_u32(&acc_bar), 0, p.err, abort_v);
      tc_fence_after();
    }
    acc_ok = __all_sync(0xffffffffu, acc_ok);  // tcgen05.ld below needs a converged warp
    if (lane == 0 && warp == 2 && !p.trigger_after_issue)
      pdl_launch_dependents();  // the next call may start its prologue
  }
  if (p.slot_offset == 0) {  // the same for every CTA of the launch
    __syncwarp();
    tc_fence_before();
    cluster_sync();  // every CTA of the cluster is past its MMAs: its ring may take the partials
    tc_fence_after();
  }

  // (c) Accumulator rows -> the shared memory of the CTA that finishes them
  //     (distributed shared memory stores into its slot[rank]). The lanes of a
  //     warp hold consecutive rows, which slot keeps adjacent for each token, so
  //     every store of the warp fills one contiguous 128-byte line.
  if (warp >= 2) {
    const int q = warp & 3;            // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int owner = row / rpc;
    const uint32_t dst_row = smem_u32(slot) +
        static_cast<uint32_t>((static_cast<int>(rank) * p.npad * rpc + (row - owner * rpc)) * 4);
    const uint32_t dsm = map_to_rank(dst_row, static_cast<uint32_t>(owner));
    const uint32_t token_stride = static_cast<uint32_t>(rpc) * 4u;
    for (int c = 0; c < p.npad; c += 16) {
      float v[16];
      __syncwarp();
      if (have_acc && acc_ok) {
        tmem_ld16(tmem + lane_base + static_cast<uint32_t>(c), v);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j)
        st_dsmem_f32(dsm + static_cast<uint32_t>(c + j) * token_stride, v[j]);
    }
  }
  __syncwarp();
  cluster_sync();  // all K-slice partials of this CTA's rows have arrived

  // (d) Finish this CTA's rows: K-slice partials summed in fixed order
  //     (slice 0..KS-1), plus the shared-partial sum, rounded to bf16. A thread
  //     keeps a run of consecutive rows (8 with one CTA per SM, where it saved
  //     ~0.5 us at T = 128; 4 otherwise) and takes every tstep-th token, four
  //     tokens' loads at a time; the lanes of a warp read consecutive pieces of
  //     slot and ssum. The run length divides rpc and the 192 threads.
  {
    constexpr int kRun = kOnePerSm ? 8 : 4;
    const int runs = rpc / kRun;
    const int g = static_cast<int>(threadIdx.x) % runs;
    const int tstep = kThreads / runs;
    const int h = h0 + r0 + g * kRun;
    if (h >= p.col_start && h < p.col_end) {  // ranges are multiples of 8
      for (int t0 = static_cast<int>(threadIdx.x) / runs; t0 < p.T; t0 += 4 * tstep) {
        float v[4][kRun];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = t0 + u * tstep;
          if (t >= p.T) break;
          float acc[kRun];
#pragma unroll
          for (int j = 0; j < kRun; ++j) acc[j] = 0.f;
          for (int src = 0; src < p.ks; ++src) {
            const float4* sp =
                reinterpret_cast<const float4*>(slot + (src * p.npad + t) * rpc + g * kRun);
#pragma unroll
            for (int j4 = 0; j4 < kRun / 4; ++j4) {
              const float4 a = sp[j4];
              acc[4 * j4] += a.x;
              acc[4 * j4 + 1] += a.y;
              acc[4 * j4 + 2] += a.z;
              acc[4 * j4 + 3] += a.w;
            }
          }
          const float4* ss4 = reinterpret_cast<const float4*>(ssum + t * rpc + g * kRun);
#pragma unroll
          for (int j4 = 0; j4 < kRun / 4; ++j4) {
            const float4 s = ss4[j4];
            v[u][4 * j4] = acc[4 * j4] + s.x;
            v[u][4 * j4 + 1] = acc[4 * j4 + 1] + s.y;
            v[u][4 * j4 + 2] = acc[4 * j4 + 2] + s.z;
            v[u][4 * j4 + 3] = acc[4 * j4 + 3] + s.w;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int t = t0 + u * tstep;
          if (t >= p.T) break;
          uint16_t* dst = p.out + static_cast<size_t>(t) * p.H + h;
          if constexpr (kRun == 8) {
            uint4 o;
            o.x = pack_bf16x2(v[u][0], v[u][1]);
            o.y = pack_bf16x2(v[u][2], v[u][3]);
            o.z = pack_bf16x2(v[u][4], v[u][5]);
            o.w = pack_bf16x2(v[u][6], v[u][7]);
            *reinterpret_cast<uint4*>(dst) = o;
          } else {
            st_global_v2(dst, pack_bf16x2(v[u][0], v[u][1]), pack_bf16x2(v[u][2], v[u][3]));
          }
        }
      }
    }
  }

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

struct DecodePlan {
  int total_kb, npad, ks, stages;
  uint32_t ssum_offset, slot_offset;
  size_t smem;
};

// K split, stage count and shared-memory layout: a fixed function of (T, L),
// never of the column range, so every output element is summed in the same
// order whatever range is requested. Eight slices (448 CTAs at H = 7168, four
// per SM) for up to 16 tokens when their buffers fit in a quarter of an SM's
// shared memory, four (224 CTAs, two per SM) for up to 96 tokens when they fit
// in half, else two (112 CTAs, one per SM), else one. Returns false when even
// that does not fit.
bool plan_decode(int T, int L, DecodePlan& g) {
  if (T < 1 || T > kDecodeMaxTokens || L < 1) return false;
  g.total_kb = ceil_div(L, kBlockK);
  g.npad = ceil_div(T, 16) * 16;
  const uint32_t stage_bytes = kWStageBytes + static_cast<uint32_t>(g.npad) * 128u;
  // The received K-slice partials take 128 rows x npad FP32 whatever the split.
  // Above 32 tokens they reuse the ring (one more cluster barrier, more stages:
  // the region is then the larger of the two), else they have their own bytes.
  const bool in_ring = g.npad > 32;
  const size_t sl = (static_cast<size_t>(kBlockM) * g.npad * 4 + 1023) & ~size_t(1023);
  auto ss_bytes = [&](int cand) {
    return (static_cast<size_t>(g.npad) * (kBlockM / cand) * 4 + 1023) & ~size_t(1023);
  };
  auto region_for = [&](long st) {
    const size_t ring = static_cast<size_t>(st) * stage_bytes;
    return in_ring ? std::max(ring, sl) : ring;
  };
  auto smem_for = [&](int cand, long st) {
    return 1024 + region_for(st) + ss_bytes(cand) + (in_ring ? 0 : sl);
  };
  const long fixed_extra = in_ring ? 0 : static_cast<long>(sl);
  int ks = 1;
  int stages = 1;
  for (int cand : {8, 4, 2}) {
    if (g.total_kb < 4 * cand) continue;  // at least 4 K-blocks per slice
    if ((cand - 1) * ceil_div(g.total_kb, cand) >= g.total_kb) continue;  // no empty slice
    if (cand == 8 && g.npad > kEightSliceMaxNpad) continue;
    if (cand == 4 && g.npad > kFourSliceMaxNpad) continue;
    const long budget =
        cand == 8 ? kQuarterSmBudget : cand == 4 ? kHalfSmBudget : kSmemBudget;
    long st = (budget - 1024 - static_cast<long>(ss_bytes(cand)) - fixed_extra) /
              static_cast<long>(stage_bytes);
    st = std::min<long>({st, ceil_div(g.total_kb, cand), kMaxStages});
    if (st < (cand == 4 ? 3 : 2) || smem_for(cand, st) > static_cast<size_t>(budget)) continue;
    ks = cand;
    stages = static_cast<int>(st);
    break;
  }
  if (ks == 1) {
    const long st = (kSmemBudget - 1024 - static_cast<long>(ss_bytes(1)) - fixed_extra) /
                    static_cast<long>(stage_bytes);
    stages = static_cast<int>(std::max<long>(1, std::min<long>({st, g.total_kb, kMaxStages})));
  }
  const size_t region = region_for(stages);
  g.ks = ks;
  g.stages = stages;
  g.ssum_offset = static_cast<uint32_t>(region);
  g.slot_offset = in_ring ? 0u : static_cast<uint32_t>(region + ss_bytes(ks));
  g.smem = smem_for(ks, stages);
  return g.smem <= static_cast<size_t>(kSmemLimit);
}

}  // namespace

cudaError_t setup_decode(const DeviceInfo&) {
  for (const void* f : {reinterpret_cast<const void*>(decode_kernel<kTwoPerSm>),
                        reinterpret_cast<const void*>(decode_kernel<kOnePerSmMode>),
                        reinterpret_cast<const void*>(decode_kernel<kFourPerSm>)}) {
    const cudaError_t e =
        cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

bool decode_supported(int T, int L) {
  DecodePlan g;
  return plan_decode(T, L, g);
}

cudaError_t launch_decode(const ProjectArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  DecodePlan g;
  if (!plan_decode(a.T, a.L, g)) return cudaErrorInvalidConfiguration;
  DecodeParams p{};
  p.shared = a.shared;
  p.out = a.out;
  p.P = a.P;
  p.T = a.T;
  p.L = a.L;
  p.H = a.H;
  p.col_start = a.col_start;
  p.col_end = a.col_end;
  p.total_kb = g.total_kb;
  p.npad = g.npad;
  p.ks = g.ks;
  p.kb_per_cta = ceil_div(g.total_kb, g.ks);
  p.stages = g.stages;
  p.ssum_offset = g.ssum_offset;
  p.slot_offset = g.slot_offset;
  const int ks = g.ks;
  p.tmem_cols = next_pow2_at_least(p.npad, 32);
  p.pdl = a.pdl ? 1 : 0;
  p.inputs_ready = a.inputs_ready ? 1 : 0;
  p.trigger_after_issue = a.early_trigger ? 1 : 0;
  p.err = dev.err_word;
  const int tile_first = a.col_start / kBlockM;
  const int tile_last = (a.col_end - 1) / kBlockM;
  p.tile0 = tile_first;
  const int ntiles = tile_last - tile_first + 1;
  const size_t smem = g.smem;

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
  if (ks == 8) return cudaLaunchKernelEx(&cfg, decode_kernel<kFourPerSm>, w_map, y_map, p);
  return ks <= 2 ? cudaLaunchKernelEx(&cfg, decode_kernel<kOnePerSmMode>, w_map, y_map, p)
                 : cudaLaunchKernelEx(&cfg, decode_kernel<kTwoPerSm>, w_map, y_map, p);
}

}  // namespace lt
