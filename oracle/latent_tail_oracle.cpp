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
// The oracle's own tests plant mistakes in a temporary copy of this file (a
// text patch per mistake) to show that its pins catch each one; this file
// itself holds only the definition.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

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
    for (long p = 0; p < P; ++p) s += widen_bf16(routed[((p * T) + t) * L + l]);
    x[l] = s;
  }
  if (g == nullptr) {  // no norm: the latent is the partial sum itself
    for (long l = 0; l < L; ++l) y[l] = x[l];
    return;
  }
  Acc ss = 0;
  for (long l = 0; l < L; ++l) ss += x[l] * x[l];
  const Acc ms = ss / static_cast<Acc>(L);
  const Acc r = static_cast<Acc>(1) / std::sqrt(ms + eps);
  for (long l = 0; l < L; ++l) y[l] = x[l] * r * static_cast<Acc>(g[l]);
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
      for (long l = 0; l < L; ++l) acc += y[l] * widen_bf16(W[h * L + l]);
      Acc s = 0;
      for (long p = 0; p < P; ++p)
        s += widen_bf16(shared[((p * T) + t) * H + h]);
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

}  // extern "C"
