// Steps 3-5 of the latent-MoE tail for prefill-sized token counts (T > 224, and
// T > 128 when the decode kernel's buffers do not fit):
//   out[t,h] = bf16_rn( sum_l y[t,l] * W[h,l] + sum_p shared[p,t,h] ),  h in [c0,c1)
// The narrowed beta-add GEMM of PR #50383's `_shard_up_proj_tail`
// (`hidden_shard.addmm_(latent, up_proj_shard.t())`), with the shared-partial
// sum of the final all-reduce done in the GEMM epilogue.
//
// At these sizes the dominant traffic is the P shared partials (P*T*H*2 bytes,
// 69-74% of all bytes), so the kernel is built around two concurrent streams:
// the tensor-core mainloop, fed from L2 (y and W are re-read per tile), and
// the HBM stream of shared partials, fed by TMA independently of the MMAs.
//
// What one SM can take in per unit time (bytes in flight over the L2 / HBM
// round trip) bounds the kernel, so the bytes a CTA must ingest per tile
// matter. Pairs of CTAs (a 2-CTA cluster) therefore share one tensor-core
// product (tcgen05 cta_group::2, M = 256 tokens, N = tile width): each CTA loads
// its own 128 tokens of y and half of the W tile, which halves the operand bytes
// per CTA. The tile width is 256 columns; 128 for T <= 256 so that the few
// tiles of a short call still occupy twice the CTA pairs; 192 where it fills
// the pairs' waves better (at H = 7168, T in (256, 1024] and (1280, 1536]);
// and 512 with a single shared partial from 4096 tokens on, when the wide
// tiles need at most half the waves (a template parameter, chosen from T, P,
// H and the SM count, never from the column range).
//
// Persistent, warp-specialized kernel, one CTA per SM, 7 warps per CTA:
//   warp 0      operand producer: y [128 tokens x 64] and W [width/2 rows x 64]
//               per K-block into this CTA's stage ring (128B swizzle, L2
//               evict-last: every operand tile is read by many CTAs);
//   warp 1      TMEM allocation for the pair; in the even CTA the single-thread
//               MMA issuer (both CTAs' TMA copies of a stage complete on the even
//               CTA's barrier; its commits arrive on the stage and accumulator
//               barriers of both CTAs);
//   warp 6      shared-partial producer: for every tile, 64-column chunk and
//               partial p, one TMA box [128 tokens x 64 columns] into a slot
//               ring (L2 evict-first: read once);
//   warps 2..5  epilogue, one token row per thread: sum the P partial boxes of
//               a chunk in FP32 (p ascending), add the accumulator columns from
//               this CTA's TMEM (two accumulators, so the next tile's MMAs run
//               during this tile's epilogue; one with 512-column tiles), round
//               to bf16 and store 16-byte vectors. When every pair owns a
//               single tile (and the tiles are not 512 wide) there is no next
//               tile to overlap: the epilogue then parks each chunk's FP32 sums
//               in the idle second accumulator's TMEM columns while the MMAs
//               run, and adds them to the accumulator afterwards (same bits).
// Output tiles sit at absolute multiples of the tile width, so a column-range
// call computes each element exactly as the full call does.
#include "launch.h"
#include "ptx.cuh"

#include <algorithm>

namespace lt {
namespace {

constexpr int kTileT = 128;   // tokens per CTA (half of the pair's MMA M = 256)
constexpr int kTileH = 256;   // output columns per tile (MMA N)
constexpr int kNarrowTileH = 128;  // T <= 256: twice the tiles, so twice the pairs busy
// 192-column tiles: at H = 7168 a 256-token group has 38 of them, so two
// groups fill the 76 CTA pairs of a GB300 exactly (against 56 of 76 with 256
// columns), and four groups run in two full waves (against 112 tiles for 76
// pairs). A 192-column tile took ~0.9 of the time of a 256-column one in full
// waves (P = 8), so the launch takes it when (waves with 192) x 9 <= (waves
// with 256) x 10: at H = 7168, T in (256, 1024] and (1280, 1536].
constexpr int kMidTileH = 192;
// 512-column tiles for a single shared partial (P = 1, where the tensor cores
// bind): two N = 256 instructions per K-step into one 512-column accumulator.
// Each CTA then takes in 48 KB per K-block for 128 x 512 outputs instead of
// 32 KB for 128 x 256, at the price of the second accumulator: the epilogue
// no longer overlaps the next tile's MMAs. Taken when the wide tiles need at
// most half the waves of the 256-column ones (P = 1, H = 7168, projection us,
// same box, 256 / 512 columns: T = 4096 90.4-90.6 / 87.4, T = 8192 173.9-176.3 /
// 168.5-170.6; at T = 2048, 3 waves against 2 with the second one half empty,
// 49.3 / 58.5). Below 4096 tokens they were not measured to win and are not used.
constexpr int kWideTileH = 512;
constexpr int kWideMinTokens = 4096;
constexpr int kBlockK = 64;
constexpr int kMaxStages = 6;
constexpr int kChunk = 64;    // output columns per shared-partial box
constexpr int kMaxSlots = 8;  // shared-partial ring depth limit
constexpr int kThreads = 224;
constexpr uint32_t kAStage = kTileT * kBlockK * 2;  // 16 KB of y
// Stage = y [128 x 64] then this CTA's half of the W tile [tile_h/2 x 64].
constexpr uint32_t stage_bytes_for(int tile_h) {
  return kAStage + static_cast<uint32_t>(tile_h / 2) * kBlockK * 2;
}
constexpr uint32_t kSlotBytes = kTileT * kChunk * 2;  // 16 KB
constexpr uint32_t kTmemCols = 2 * kTileH;
constexpr size_t kSmemLimit = 226 * 1024;  // + static shared memory <= opt-in maximum

// Shared memory splits between the operand ring (feeds the MMAs from L2) and
// the shared-partial ring (feeds the epilogue from HBM); both hide latency, so
// the split follows the share of the shared-partial bytes, i.e. P (measured,
// projection us, same box): P = 8, T = 8192: 4 + 6 216.7, 4 + 5 221.5, 3 + 7
// 239.2, 3 + 8 239.9; P = 16, T = 16384: 3 + 8 669, 3 + 7 676, 4 + 6 682,
// 4 + 5 701.
constexpr int kStagesFewPartials = 4;  // 2 <= P <= 8
constexpr int kSlotsFewPartials = 6;
constexpr int kStagesManyPartials = 3;  // P > 8
constexpr int kSlotsManyPartials = 8;
// With a single shared partial the epilogue needs far fewer bytes in flight and
// the tensor cores bind, so the operand ring gets them: P = 1, T = 8192 ran at
// 172.1 us with 6 + 2 against 175.5 us with 4 + 5.
constexpr int kSinglePartialStages = 6;
constexpr int kSinglePartialSlots = 2;
// 128-column tiles (T <= 256): 24 KB stages, six of them beside five slots.
constexpr int kNarrowStages = 6;
constexpr int kNarrowSlots = 5;
// 192-column tiles: 28 KB stages. P = 8 (forward call, us, same box; 4 + 7,
// 5 + 5, 3 + 8, 4 + 6): T = 320 26.40, 25.90, 28.87, 26.33; T = 640 47.23,
// 45.38, 50.62, 46.78; T = 1024 51.50, 49.98, 55.09, 51.05. P > 8: 3 + 8.
constexpr int kMidStagesFewPartials = 5;
constexpr int kMidSlotsFewPartials = 5;
constexpr int kMidStagesManyPartials = 3;
constexpr int kMidSlotsManyPartials = 8;
// 512-column tiles: 48 KB stages, four of them beside the two slots of P = 1.
constexpr int kWideStages = 4;
constexpr int kWideSlots = 2;

size_t smem_bytes(int stages, int slots, int tile_h) {
  return 1024 + static_cast<size_t>(stages) * stage_bytes_for(tile_h) +
         static_cast<size_t>(slots) * kSlotBytes;
}

struct PrefillParams {
  uint16_t* out;
  int P, T, L, H;
  int col_start, col_end;
  int tile_h;       // output columns per tile: kTileH, kMidTileH or kNarrowTileH
  int htile0;       // absolute index of the first tile_h-column tile
  int n_htiles;
  int n_tpairs;     // 256-token groups (one per CTA pair and tile)
  int total_kb;
  int stages;       // operand ring depth
  int slots;        // shared-partial ring depth
  int pdl;
  // Every pair owns at most one tile: the epilogue parks each chunk's shared sums
  // in the idle second accumulator's TMEM columns while the mainloop runs.
  int stage_sums;
  uint32_t* err;
};

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}

struct TileCoord {
  int t0, h0;  // this CTA's first token and the tile's first output column
};

// Pair tile `tile` -> coordinates for the CTA of rank `rank` in the pair.
template <int kTileW>
__device__ __forceinline__ TileCoord tile_coord(const PrefillParams& p, int tile, int rank) {
  TileCoord c;
  c.t0 = (tile / p.n_htiles) * (2 * kTileT) + rank * kTileT;
  c.h0 = (p.htile0 + tile % p.n_htiles) * kTileW;
  return c;
}

// First output column (relative to the tile's) of the 64 accumulator columns
// [64 ch, 64 ch + 64). Each CTA of the pair holds tile_w / 2 consecutive W rows,
// and an instruction takes the first half of its N columns from the even CTA's
// rows and the second half from the odd CTA's. With 512-column tiles two N = 256
// instructions per K-step take rows 0-127 and then 128-255 of each CTA, so the
// accumulator's 128-column blocks hold tile columns 0, 256, 128 and 384.
template <int kTileW>
__device__ __forceinline__ int chunk_offset(int ch) {
  if constexpr (kTileW > 256) {
    const int blk = ch >> 1;
    return ((blk & 1) << 8) | ((blk >> 1) << 7) | ((ch & 1) << 6);
  } else {
    return ch * kChunk;
  }
}

// A 64-column chunk is processed only if it meets [col_start, col_end).
__device__ __forceinline__ bool chunk_active(const PrefillParams& p, int hc) {
  return hc < p.col_end && hc + kChunk > p.col_start;
}

// Adds the 8 bf16 values of a 16-byte word to s[0..7].
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

// kTileW: output columns per tile (MMA N), a compile-time constant so that the
// issue loops keep their address arithmetic constant.
template <int kTileW>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap y_map,
                   const __grid_constant__ CUtensorMap w_map,
                   const __grid_constant__ CUtensorMap s_map, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages];   // even CTA: both CTAs' stage s landed
  __shared__ uint64_t empty_bar[kMaxStages];  // stage consumed by the pair MMAs
  __shared__ uint64_t accf_bar[2];            // accumulator ready (both CTAs)
  __shared__ uint64_t acce_bar[2];            // even CTA: accumulator drained by both
  __shared__ uint64_t sfull_bar[kMaxSlots];
  __shared__ uint64_t sempty_bar[kMaxSlots];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());  // 0 issues the pair MMAs
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  const int n_pairs = static_cast<int>(gridDim.x) >> 1;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  const int n_stages = p.stages;
  constexpr int tile_h = kTileW;
  constexpr bool kWide = kTileW > 256;   // two instructions per K-step, one accumulator
  constexpr int kAccs = kWide ? 1 : 2;   // accumulators (each tile_h TMEM columns)
  constexpr int kInstrN = kWide ? 256 : kTileW;
  // Parking shared sums needs the idle second accumulator.
  const bool stage_sums = !kWide && p.stage_sums != 0;
  constexpr int half_h = tile_h / 2;        // W rows loaded by each CTA of the pair
  constexpr int n_chunks = tile_h / kChunk;
  constexpr uint32_t stage_bytes = stage_bytes_for(tile_h);
  const int n_slots = p.slots;
  const uint32_t slot_base = sbase + static_cast<uint32_t>(n_stages) * stage_bytes;
  const uint8_t* slot_gen = smem_raw + (slot_base - raw_u32);
  const int num_tiles = p.n_tpairs * p.n_htiles;
  const int my_tiles = pair < num_tiles ? (num_tiles - 1 - pair) / n_pairs + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < n_stages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&accf_bar[a]), 1);
      mbar_init(smem_u32(&acce_bar[a]), 2 * 4);  // one arrival per epilogue warp of the pair
    }
    for (int s = 0; s < n_slots; ++s) {
      mbar_init(smem_u32(&sfull_bar[s]), 1);
      mbar_init(smem_u32(&sempty_bar[s]), 4);  // one arrival per epilogue warp
    }
    abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_map(&y_map);
    tma_prefetch_map(&w_map);
    tma_prefetch_map(&s_map);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(&tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_v = &abort_flag;

  if (warp == 0) {
    if (lane == 0 && my_tiles > 0) {
      // ---------------- operand producer (this CTA's halves) ----------------
      // Both CTAs' loads of stage s complete on the even CTA's full_bar[s]; the
      // even CTA expects the bytes of both.
      const uint64_t keep = policy_evict_last();
      const int total = my_tiles * p.total_kb;
      const int pre = min(n_stages, total);
      auto coord_of = [&](int it, TileCoord& c, int& kb) {
        const int local = it / p.total_kb;
        kb = it - local * p.total_kb;
        c = tile_coord<kTileW>(p, pair + local * n_pairs, rank);
      };
      auto full_of = [&](int s) { return map_to_rank(smem_u32(&full_bar[s]), 0); };
      for (int it = 0; it < pre; ++it) {  // W does not depend on the norm kernel
        TileCoord c;
        int kb;
        coord_of(it, c, kb);
        const uint32_t st = sbase + static_cast<uint32_t>(it) * stage_bytes;
        if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full_bar[it]), 2 * stage_bytes);
        tma_load_2d_pair_hint(st + kAStage, &w_map, full_of(it), kb * kBlockK,
                              c.h0 + rank * half_h, keep);
      }
      if (p.pdl) pdl_wait();
      for (int it = 0; it < pre; ++it) {
        TileCoord c;
        int kb;
        coord_of(it, c, kb);
        const uint32_t st = sbase + static_cast<uint32_t>(it) * stage_bytes;
        tma_load_2d_pair_hint(st, &y_map, full_of(it), kb * kBlockK, c.t0, keep);
      }
      int issued = pre;
      for (int it = pre; it < total; ++it) {
        const int s = it % n_stages;
        const uint32_t round = static_cast<uint32_t>(it / n_stages);
        if (!mbar_wait_cluster(smem_u32(&empty_bar[s]), (round & 1u) ^ 1u, p.err, abort_v)) break;
        TileCoord c;
        int kb;
        coord_of(it, c, kb);
        const uint32_t st = sbase + static_cast<uint32_t>(s) * stage_bytes;
        if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full_bar[s]), 2 * stage_bytes);
        tma_load_2d_pair_hint(st, &y_map, full_of(s), kb * kBlockK, c.t0, keep);
        tma_load_2d_pair_hint(st + kAStage, &w_map, full_of(s), kb * kBlockK, c.h0 + rank * half_h,
                              keep);
        issued = it + 1;
      }
      if (*abort_v && rank == 0) {  // the even CTA's barriers count both CTAs' copies
        for (int it = max(0, issued - n_stages); it < issued; ++it)
          wait_drain(smem_u32(&full_bar[it % n_stages]), static_cast<uint32_t>(it / n_stages) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && my_tiles > 0) {
      if (rank == 0) {
        // ---------------- pair MMA issuer ----------------
        const uint32_t idesc = umma_idesc_bf16(2 * kTileT, kInstrN);
        int it = 0;
        bool alive = true;
        for (int i = 0; i < my_tiles && alive; ++i) {
          const int acc = i % kAccs;
          const uint32_t use = static_cast<uint32_t>(i / kAccs);
          if (!mbar_wait_cluster(smem_u32(&acce_bar[acc]), (use & 1u) ^ 1u, p.err, abort_v)) break;
          tc_fence_after();
          const uint32_t d = tmem + static_cast<uint32_t>(acc * tile_h);
          for (int kb = 0; kb < p.total_kb; ++kb, ++it) {
            const int s = it % n_stages;
            const uint32_t round = static_cast<uint32_t>(it / n_stages);
            if (!mbar_wait_cluster(smem_u32(&full_bar[s]), round & 1u, p.err, abort_v)) {
              alive = false;
              break;
            }
            tc_fence_after();
            const uint32_t a = sbase + static_cast<uint32_t>(s) * stage_bytes;
            const uint32_t b = a + kAStage;
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k) {
              umma_bf16_pair(d, umma_desc_sw128(a + 32u * k), umma_desc_sw128(b + 32u * k), idesc,
                             (kb | k) != 0 ? 1u : 0u);
              if constexpr (kWide)  // W rows 128..255 of each CTA -> columns 256..511
                umma_bf16_pair(d + 256u, umma_desc_sw128(a + 32u * k),
                               umma_desc_sw128(b + 128u * 128u + 32u * k), idesc,
                               (kb | k) != 0 ? 1u : 0u);
            }
            umma_commit_pair(smem_u32(&empty_bar[s]), 0x3);
          }
          umma_commit_pair(smem_u32(&accf_bar[acc]), 0x3);
        }
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    if (lane == 0 && my_tiles > 0) {
      // ---------------- shared-partial producer ----------------
      const uint64_t once = policy_evict_first();
      int k = 0;
      bool alive = true;
      for (int i = 0; i < my_tiles && alive; ++i) {
        const TileCoord c = tile_coord<kTileW>(p, pair + i * n_pairs, rank);
        if (c.t0 >= p.T) continue;  // no rows of this CTA in the tile
        for (int ch = 0; ch < n_chunks && alive; ++ch) {
          const int hc = c.h0 + chunk_offset<kTileW>(ch);
          if (!chunk_active(p, hc)) continue;
          for (int pp = 0; pp < p.P; ++pp, ++k) {
            const int s = k % n_slots;
            const uint32_t round = static_cast<uint32_t>(k / n_slots);
            if (!mbar_wait(smem_u32(&sempty_bar[s]), (round & 1u) ^ 1u, p.err, abort_v)) {
              alive = false;
              break;
            }
            const uint32_t fb = smem_u32(&sfull_bar[s]);
            mbar_arrive_expect_tx(fb, kSlotBytes);
            tma_load_2d_hint(slot_base + static_cast<uint32_t>(s) * kSlotBytes, &s_map, fb, hc,
                             pp * p.T + c.t0, once);
          }
        }
      }
      if (*abort_v) {
        for (int kk = max(0, k - n_slots); kk < k; ++kk)
          wait_drain(smem_u32(&sfull_bar[kk % n_slots]), static_cast<uint32_t>(kk / n_slots) & 1u);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;       // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;  // token row within this CTA's half of the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    // Accumulator `a` fully read by this warp: hand it back to the MMA issuer.
    auto release_acc = [&](int a) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t bar = smem_u32(&acce_bar[a]);
        if (rank == 0)
          mbar_arrive(bar);
        else
          mbar_arrive_remote(map_to_rank(bar, 0));
      }
    };
    // out[t, hc .. hc+63] = bf16(acc + shared sum), only inside [col_start, col_end).
    auto emit = [&](int t, int hc, const float* v0, const float* v1, const float* sums) {
      uint16_t* dst = p.out + static_cast<size_t>(t) * p.H + hc;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const int hh = hc + g * 8;
        if (hh < p.col_start || hh >= p.col_end) continue;
        const float* a = g < 4 ? &v0[g * 8] : &v1[(g - 4) * 8];
        const float* b = &sums[g * 8];
        uint4 o;
        o.x = pack_bf16x2(a[0] + b[0], a[1] + b[1]);
        o.y = pack_bf16x2(a[2] + b[2], a[3] + b[3]);
        o.z = pack_bf16x2(a[4] + b[4], a[5] + b[5]);
        o.w = pack_bf16x2(a[6] + b[6], a[7] + b[7]);
        st_stream_v4(dst + g * 8, o);
      }
    };
    int k = 0;
    bool alive = true;
    for (int i = 0; i < my_tiles && alive; ++i) {
      const int acc = i % kAccs;
      const uint32_t use = static_cast<uint32_t>(i / kAccs);
      const TileCoord c = tile_coord<kTileW>(p, pair + i * n_pairs, rank);
      const int t = c.t0 + r;
      const bool row_ok = t < p.T;
      const bool has_rows = c.t0 < p.T;
      const uint32_t dcol = tmem + lane_base + static_cast<uint32_t>(acc * tile_h);
      bool acc_ready = false;
#pragma unroll 1
      for (int ch = 0; ch < n_chunks; ++ch) {
        const int hc = c.h0 + chunk_offset<kTileW>(ch);
        const bool active = has_rows && chunk_active(p, hc);
        float s[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) s[j] = 0.f;
        if (active) {
          // sum the P partial boxes of this chunk, p ascending
          for (int pp = 0; pp < p.P; ++pp, ++k) {
            const int sl = k % n_slots;
            const uint32_t round = static_cast<uint32_t>(k / n_slots);
            bool ok = mbar_wait(smem_u32(&sfull_bar[sl]), round & 1u, p.err, abort_v);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
              alive = false;
              break;
            }
            const uint8_t* row_ptr = slot_gen + sl * kSlotBytes + r * 128;
#pragma unroll
            for (int g = 0; g < 8; ++g) {  // 16-byte chunk g of the row sits at g ^ (r % 8)
              const uint4 v = *reinterpret_cast<const uint4*>(row_ptr + ((g ^ (r & 7)) << 4));
              add8(&s[g * 8], v);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sempty_bar[sl]));
          }
          if (!alive) break;
        }
        if (stage_sums) {
          // Single tile per pair: the second accumulator's columns are idle, so
          // park this chunk's FP32 sums there and go on to the next chunk's
          // partials without waiting for the MMAs; the sums are added below.
          __syncwarp();  // tcgen05.st needs the whole warp converged
          const uint32_t scol = tmem + lane_base + static_cast<uint32_t>(tile_h + ch * kChunk);
          tmem_st32(scol, &s[0]);
          tmem_st32(scol + 32u, &s[32]);
          continue;
        }
        if (!acc_ready) {
          bool ok = mbar_wait_cluster(smem_u32(&accf_bar[acc]), use & 1u, p.err, abort_v);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) {
            alive = false;
            break;
          }
          tc_fence_after();
          acc_ready = true;
        }
        float v0[32], v1[32];
        __syncwarp();  // tcgen05.ld needs the whole warp converged
        tmem_ld32(dcol + static_cast<uint32_t>(ch * kChunk), v0);
        tmem_ld32(dcol + static_cast<uint32_t>(ch * kChunk + 32), v1);
        if (ch == n_chunks - 1) release_acc(acc);
        if (!active || !row_ok) continue;
        emit(t, hc, v0, v1, s);
      }
      if (stage_sums && alive) {
        // The parked sums plus the accumulator, chunk by chunk.
        tmem_wait_st();
        bool ok = mbar_wait_cluster(smem_u32(&accf_bar[acc]), use & 1u, p.err, abort_v);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < n_chunks; ++ch) {
          const int hc = c.h0 + chunk_offset<kTileW>(ch);
          const bool active = has_rows && chunk_active(p, hc);
          float v0[32], v1[32], sums[kChunk];
          __syncwarp();
          tmem_ld32(dcol + static_cast<uint32_t>(ch * kChunk), v0);
          tmem_ld32(dcol + static_cast<uint32_t>(ch * kChunk + 32), v1);
          const uint32_t scol = tmem + lane_base + static_cast<uint32_t>(tile_h + ch * kChunk);
          tmem_ld32(scol, *reinterpret_cast<float(*)[32]>(&sums[0]));
          tmem_ld32(scol + 32u, *reinterpret_cast<float(*)[32]>(&sums[32]));
          if (ch == n_chunks - 1) release_acc(acc);
          if (!active || !row_ok) continue;
          emit(t, hc, v0, v1, sums);
        }
      }
    }
  }

  // Neither CTA may leave while the pair's MMAs could still read its shared
  // memory or write its TMEM, or while its peer could still signal it.
  tc_fence_before();
  __syncthreads();
  if (warp == 1 && rank == 0 && *abort_v && lane == 0) {
    const int last = my_tiles - 1;
    for (int i = max(0, last - (kAccs - 1)); i <= last; ++i)
      wait_drain(smem_u32(&accf_bar[i % kAccs]), static_cast<uint32_t>(i / kAccs) & 1u);
  }
  __syncwarp();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

cudaError_t setup_prefill(const DeviceInfo&) {
  for (const void* f : {reinterpret_cast<const void*>(prefill_kernel<kTileH>),
                        reinterpret_cast<const void*>(prefill_kernel<kMidTileH>),
                        reinterpret_cast<const void*>(prefill_kernel<kNarrowTileH>),
                        reinterpret_cast<const void*>(prefill_kernel<kWideTileH>)}) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kSmemLimit));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_prefill(const ProjectArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  PrefillParams p{};
  p.out = a.out;
  p.P = a.P;
  p.T = a.T;
  p.L = a.L;
  p.H = a.H;
  p.col_start = a.col_start;
  p.col_end = a.col_end;
  // A fixed function of T (never of the column range), so that every output
  // element is computed the same way whatever range a call asks for.
  // (Of T, H and the device: a column range never changes it.)
  if (a.T <= 2 * kTileT) {
    p.tile_h = kNarrowTileH;
  } else {
    const int groups = ceil_div(a.T, 2 * kTileT);
    const int pairs = std::max(1, dev.num_sms / 2);
    auto waves = [&](int w) { return ceil_div(groups * ceil_div(a.H, w), pairs); };
    if (a.P == 1 && a.T >= kWideMinTokens && 2 * waves(kWideTileH) <= waves(kTileH))
      p.tile_h = kWideTileH;
    else
      p.tile_h = 9 * waves(kMidTileH) <= 10 * waves(kTileH) ? kMidTileH : kTileH;
  }
  p.htile0 = a.col_start / p.tile_h;
  p.n_htiles = (a.col_end - 1) / p.tile_h - p.htile0 + 1;
  p.n_tpairs = ceil_div(a.T, 2 * kTileT);
  p.total_kb = ceil_div(a.L, kBlockK);
  if (p.tile_h == kWideTileH) {
    p.stages = kWideStages;
    p.slots = kWideSlots;
  } else if (a.P == 1) {  // one box per chunk: the operand ring gets the bytes (measured)
    p.stages = kSinglePartialStages;
    p.slots = kSinglePartialSlots;
  } else if (p.tile_h == kNarrowTileH) {
    p.stages = kNarrowStages;
    p.slots = kNarrowSlots;
  } else if (p.tile_h == kMidTileH) {
    p.stages = a.P <= 8 ? kMidStagesFewPartials : kMidStagesManyPartials;
    p.slots = a.P <= 8 ? kMidSlotsFewPartials : kMidSlotsManyPartials;
  } else if (a.P <= 8) {
    p.stages = kStagesFewPartials;
    p.slots = kSlotsFewPartials;
  } else {
    p.stages = kStagesManyPartials;
    p.slots = kSlotsManyPartials;
  }
  // the barrier arrays hold kMaxStages / kMaxSlots entries
  if (p.stages < 1 || p.stages > kMaxStages || p.slots < 1 || p.slots > kMaxSlots)
    return cudaErrorInvalidConfiguration;
  const size_t smem = smem_bytes(p.stages, p.slots, p.tile_h);
  if (smem > kSmemLimit) return cudaErrorInvalidConfiguration;
  p.pdl = a.pdl ? 1 : 0;
  p.err = dev.err_word;
  const long long tiles = static_cast<long long>(p.n_htiles) * p.n_tpairs;
  // one tile per pair at most (and a second accumulator to park the sums in)
  p.stage_sums = tiles <= dev.num_sms / 2 && p.tile_h != kWideTileH ? 1 : 0;
  const int grid = 2 * static_cast<int>(std::min<long long>(dev.num_sms / 2, tiles));

  // The shared partials as one 2-D tensor [P*T rows, H columns]: the box for
  // (partial p, tokens t0..t0+127) starts at row p*T + t0. Rows past T inside
  // a partial belong to the next partial and are never stored; rows past P*T
  // and columns past H read as zero. No tensor map asks for 256-byte L2
  // promotion: here the other 128 bytes of each sector belong to the next
  // column chunk, read only after all P partials of this one, by which time the
  // read-once stream has evicted them. Promotion on this map cost 22% of the
  // stress projection (901 against 704 us) and 12% of the prefill one.
  CUtensorMap y_map, w_map, s_map;
  if (!make_map_bf16_sw128(&y_map, a.y, a.T, a.L, kTileT)) return cudaErrorInvalidValue;
  if (!make_map_bf16_sw128(&w_map, a.W, a.H, a.L, static_cast<uint32_t>(p.tile_h / 2)))
    return cudaErrorInvalidValue;
  if (!make_map_bf16_sw128(&s_map, a.shared, static_cast<uint64_t>(a.P) * a.T, a.H, kTileT))
    return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  attrs[n].id = cudaLaunchAttributeClusterDimension;  // CTA pairs
  attrs[n].val.clusterDim.x = 2;
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
  if (p.tile_h == kNarrowTileH)
    return cudaLaunchKernelEx(&cfg, prefill_kernel<kNarrowTileH>, y_map, w_map, s_map, p);
  if (p.tile_h == kMidTileH)
    return cudaLaunchKernelEx(&cfg, prefill_kernel<kMidTileH>, y_map, w_map, s_map, p);
  if (p.tile_h == kWideTileH)
    return cudaLaunchKernelEx(&cfg, prefill_kernel<kWideTileH>, y_map, w_map, s_map, p);
  return cudaLaunchKernelEx(&cfg, prefill_kernel<kTileH>, y_map, w_map, s_map, p);
}

}  // namespace lt
