// Latent-MoE output tail: plain CPU oracle.
//
// TEST INFRASTRUCTURE ONLY. This file is the correctness reference for the
// CUDA library. Only the tests, the smoke check and the benchmark's CPU
// baseline may load it; the library itself never calls it, and the two share
// no code, header, table or helper.
//
// What it computes (one definition, written out plainly):
//
//   x[t,l]   = sum_p routed[p,t,l]                         (routed partial sum)
//   y[t,l]   = x[t,l] * rsqrt(mean_l x[t,l]^2 + eps) * g[l] (RMSNorm with weight)
//   out[t,h] = sum_l y[t,l] * W[h,l] + sum_p shared[p,t,h]  (up-projection plus
//                                                           summed shared partials)
//   for h in the half-open column range [col_start, col_end).
//
// Sources ("Kimi-K3 latent MoE" vLLM PR digests):
//   * PR #51253 report, section "关键源码片段" (test source), the
//     `_check_matches_replicated` expectation: F.linear(F.rms_norm(all-reduced
//     routed, (LATENT_SIZE,), norm.weight, EPS), up_proj.weight) plus the
//     all-reduced shared output. The all-reduce over tensor-parallel ranks is the
//     sum over the P stacked partials here.
//   * same test, `_check_writes_only_its_own_shard`: a rank owning columns
//     [start,end) adds latent . W[start:end]^T into exactly those columns.
//   * PR #50383 report, source of `_shard_up_proj_tail`: reduce then norm
//     (`allreduce_norm_latent_out`), narrow W rows and shared columns to the
//     shard, then the beta-add `hidden_shard.addmm_(latent, up_proj_shard.t())`.
//   * RMSNorm as PyTorch's F.rms_norm defines it: x * rsqrt(mean(x^2) + eps) *
//     weight, eps inside the square root, mean over the latent dimension.
//   * the same source's branch for `transform.norm is None`: the latent is the
//     all-reduced routed output itself. Here: g == NULL selects it (y = x, eps
//     unused).
//
// Precision: the loop body is instantiated for float (the FP32 oracle the
// parity tests use, matching the FP32 reference convention of PR #50593's
// contract test) and for double (used by the oracle's own pins to bound the
// FP32 rounding). Inputs are bf16 bit patterns widened exactly. There is no
// intermediate rounding, no blocking and no reordering: partial sums run with p
// ascending, squares and dot products with l ascending.
//
// Build: g++ -O2 -ffp-contract=off -shared -fPIC (no fast-math, no FMA
// contraction, so x86 and Arm hosts give the same bits).
//
// LT_ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake so
// the CPU tests can show that their pins catch it. Production builds of the
// oracle never define it.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifndef LT_ORACLE_MUTANT
#define LT_ORACLE_MUTANT 0
#endif

namespace {

float widen_bf16(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// Argument checks shared by both instantiations. Returns 0 when the call is
// well formed, a negative code otherwise.
int check_args(const void* routed, const void* shared, const float* g,
               const void* W, long P, long T, long L, long H, long c0, long c1,
               const void* out) {
  if (P < 1 || T < 0 || L < 1 || H < 1) return -1;
  if (c0 < 0 || c1 > H || c0 >= c1) return -2;
  if (T > 0 && (!routed || !shared || !W || !out)) return -3;
  return 0;
}

// Steps 1 and 2 for one token: partial sum, then RMSNorm with weight.
template <typename Acc>
void normalized_latent(const uint16_t* routed, const float* g, long P, long T,
                       long L, long t, Acc eps, Acc* x, Acc* y) {
  for (long l = 0; l < L; ++l) {
    Acc s = 0;
#if LT_ORACLE_MUTANT == 5
    // mistake: partials read as if laid out [T,P,L]
    for (long p = 0; p < P; ++p) s += widen_bf16(routed[((t * P) + p) * L + l]);
#else
    for (long p = 0; p < P; ++p) s += widen_bf16(routed[((p * T) + t) * L + l]);
#endif
    x[l] = s;
  }
  if (g == nullptr) {  // no norm: the latent is the partial sum itself
#if LT_ORACLE_MUTANT == 10
    // mistake: the no-norm branch still normalizes (with unit weight)
    Acc ss0 = 0;
    for (long l = 0; l < L; ++l) ss0 += x[l] * x[l];
    const Acc r0 = static_cast<Acc>(1) / std::sqrt(ss0 / static_cast<Acc>(L) + eps);
    for (long l = 0; l < L; ++l) y[l] = x[l] * r0;
#else
    for (long l = 0; l < L; ++l) y[l] = x[l];
#endif
    return;
  }
  Acc ss = 0;
#if LT_ORACLE_MUTANT == 9
  // mistake: squares of the partials summed instead of the square of the sum
  for (long l = 0; l < L; ++l)
    for (long p = 0; p < P; ++p) {
      Acc v = widen_bf16(routed[((p * T) + t) * L + l]);
      ss += v * v;
    }
#else
  for (long l = 0; l < L; ++l) ss += x[l] * x[l];
#endif
#if LT_ORACLE_MUTANT == 2
  Acc ms = ss;  // mistake: sum of squares, not the mean
#else
  Acc ms = ss / static_cast<Acc>(L);
#endif
#if LT_ORACLE_MUTANT == 1
  Acc r = static_cast<Acc>(1) / (std::sqrt(ms) + eps);  // mistake: eps outside
#else
  Acc r = static_cast<Acc>(1) / std::sqrt(ms + eps);
#endif
  for (long l = 0; l < L; ++l) {
#if LT_ORACLE_MUTANT == 6
    y[l] = x[l] * r;  // mistake: norm weight dropped
#else
    y[l] = x[l] * r * static_cast<Acc>(g[l]);
#endif
  }
}

template <typename Acc>
int forward(const uint16_t* routed, const uint16_t* shared, const float* g,
            const uint16_t* W, long P, long T, long L, long H, double eps,
            long c0, long c1, Acc* out) {
  int rc = check_args(routed, shared, g, W, P, T, L, H, c0, c1, out);
  if (rc) return rc;
  const long width = c1 - c0;
  const Acc e = static_cast<Acc>(eps);
  std::vector<Acc> x(L), y(L);
  for (long t = 0; t < T; ++t) {
    normalized_latent<Acc>(routed, g, P, T, L, t, e, x.data(), y.data());
    for (long h = c0; h < c1; ++h) {
      Acc acc = 0;
#if LT_ORACLE_MUTANT == 3
      // mistake: W read transposed, as if it were [L,H]
      for (long l = 0; l < L; ++l) acc += y[l] * widen_bf16(W[l * H + h]);
#elif LT_ORACLE_MUTANT == 8
      // mistake: W row taken relative to the column range start
      for (long l = 0; l < L; ++l) acc += y[l] * widen_bf16(W[(h - c0) * L + l]);
#else
      for (long l = 0; l < L; ++l) acc += y[l] * widen_bf16(W[h * L + l]);
#endif
      Acc s = 0;
#if LT_ORACLE_MUTANT == 4
      for (long p = 1; p < P; ++p)  // mistake: first shared partial dropped
        s += widen_bf16(shared[((p * T) + t) * H + h]);
#elif LT_ORACLE_MUTANT == 7
      for (long p = 0; p < P; ++p)  // mistake: shared read as [T,P,H]
        s += widen_bf16(shared[((t * P) + p) * H + h]);
#else
      for (long p = 0; p < P; ++p)
        s += widen_bf16(shared[((p * T) + t) * H + h]);
#endif
      out[t * width + (h - c0)] = acc + s;
    }
  }
  return 0;
}

template <typename Acc>
int latent(const uint16_t* routed, const float* g, long P, long T, long L,
           double eps, Acc* y_out) {
  if (P < 1 || T < 0 || L < 1) return -1;
  if (T > 0 && (!routed || !y_out)) return -3;
  std::vector<Acc> x(L);
  for (long t = 0; t < T; ++t)
    normalized_latent<Acc>(routed, g, P, T, L, t, static_cast<Acc>(eps), x.data(),
                           y_out + t * L);
  return 0;
}

}  // namespace

extern "C" {

// out[T, col_end-col_start] (row-major, FP32) for routed [P,T,L], shared
// [P,T,H], W [H,L] given as bf16 bit patterns and g [L] in FP32 (g == NULL:
// no norm).
int lt_oracle_forward_f32(const uint16_t* routed, const uint16_t* shared,
                          const float* g, const uint16_t* W, long P, long T,
                          long L, long H, double eps, long col_start,
                          long col_end, float* out) {
  return forward<float>(routed, shared, g, W, P, T, L, H, eps, col_start,
                        col_end, out);
}

// The same computation in double.
int lt_oracle_forward_f64(const uint16_t* routed, const uint16_t* shared,
                          const float* g, const uint16_t* W, long P, long T,
                          long L, long H, double eps, long col_start,
                          long col_end, double* out) {
  return forward<double>(routed, shared, g, W, P, T, L, H, eps, col_start,
                         col_end, out);
}

// The normalized latent y[T,L] alone (steps 1 and 2), FP32.
int lt_oracle_latent_f32(const uint16_t* routed, const float* g, long P, long T,
                         long L, double eps, float* y) {
  return latent<float>(routed, g, P, T, L, eps, y);
}

// The normalized latent y[T,L] alone, double.
int lt_oracle_latent_f64(const uint16_t* routed, const float* g, long P, long T,
                         long L, double eps, double* y) {
  return latent<double>(routed, g, P, T, L, eps, y);
}

int lt_oracle_mutant_id(void) { return LT_ORACLE_MUTANT; }

}  // extern "C"
