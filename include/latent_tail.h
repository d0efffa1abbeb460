/*
 * latent_tail.h - C ABI of the GB300 (sm_103a) latent-MoE output tail.
 *
 * The operation (Kimi-K3 latent MoE, as the vLLM PR #50383 and #51253 digests
 * describe it):
 *
 *   x[t,l]   = sum_{p<P} routed[p,t,l]                      routed partial sum
 *   y[t,l]   = x[t,l] * rsqrt(mean_l x[t,l]^2 + eps) * g[l]  RMSNorm with weight
 *   out[t,h] = sum_l y[t,l] * W[h,l] + sum_{p<P} shared[p,t,h]
 *
 * Sources, by page and section:
 *   - PR #51253 report, test source section: `_check_matches_replicated`
 *     (expected = F.linear(F.rms_norm(all-reduced routed, (L,), g, EPS), W)
 *     plus the all-reduced shared output) and `_check_writes_only_its_own_shard`
 *     (a rank owning columns [start,end) adds latent . W[start:end]^T into only
 *     those columns; the rest stays bit-identical).
 *   - PR #50383 report, source of `_shard_up_proj_tail`: all-reduce then norm
 *     (`allreduce_norm_latent_out`), `weight.narrow(0, start, size)` and
 *     `shared_output.narrow(-1, start, size)`, then the beta-add epilogue
 *     `hidden_shard.addmm_(latent, up_proj_shard.t())`.
 *   On one GPU the P tensor-parallel partials are stacked tensors that the
 *   kernels reduce; the column-parallel shard is the [col_start, col_end) option.
 *
 * Conventions for every entry point:
 *   - bf16 tensors are passed as `uint16_t*` holding bfloat16 bit patterns.
 *   - All arrays are DEVICE memory on the current CUDA device (except the
 *     host buffers of latent_tail_forward_host), contiguous and row-major,
 *     allocated and owned by the caller. Every pointer must be
 *     16-byte aligned. The library never allocates, frees or keeps a pointer
 *     after the call returns.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream). No call synchronizes the host, except
 *     latent_tail_check.
 *   - Arguments are validated on the host before anything is enqueued. On a
 *     non-OK status nothing was launched and no memory was touched.
 *   - T == 0 is a no-op that returns LT_OK.
 *   - Shape limits: 1 <= P <= 64; 8 <= L <= 16384 and L % 8 == 0;
 *     8 <= H <= 1048576 and H % 8 == 0; 0 <= T <= 2^24. Violations give
 *     LT_ERR_INVALID_ARG (range) or LT_ERR_ALIGNMENT (multiple of 8).
 *   - Device-side waits are bounded: a wait that expires sets a device error
 *     word and the kernel returns early; latent_tail_check reports it as
 *     LT_ERR_TIMEOUT.
 */
#ifndef LATENT_TAIL_H
#define LATENT_TAIL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define LT_API __attribute__((visibility("default")))
#else
#define LT_API
#endif

typedef enum lt_status {
  LT_OK = 0,
  LT_ERR_INVALID_ARG = 1, /* null pointer, bad shape/range, overlap, bad eps */
  LT_ERR_ALIGNMENT = 2,   /* pointer not 16-byte aligned, or L/H/range not % 8 */
  LT_ERR_UNSUPPORTED = 3, /* current device is not compute capability 10.3 */
  LT_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
  LT_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  LT_ERR_TIMEOUT = 6      /* a bounded device-side wait expired */
} lt_status;

/* Same object as cudaStream_t. */
typedef struct CUstream_st* lt_stream;

/*
 * Bytes of device workspace latent_tail_forward / _forward_cols need for T
 * tokens of latent width L: the normalized latent y [T, L] in bf16, rounded up
 * to 256 bytes. P and H do not change it. Returns 0 for T <= 0 or invalid
 * shapes. Host-only, never touches the GPU.
 */
LT_API size_t latent_tail_workspace_size(int P, int T, int L, int H);

/*
 * Whole tail for all H output columns (equivalent to latent_tail_forward_cols
 * with col_start = 0, col_end = H).
 *   routed      [P, T, L] bf16  routed-expert latent partials
 *   shared      [P, T, H] bf16  shared-expert output partials
 *   norm_weight [L]       fp32  RMSNorm weight g, or NULL for the pages'
 *                               `transform.norm is None` branch: no RMSNorm, the
 *                               latent is the partial sum itself (eps unused)
 *   W           [H, L]    bf16  up-projection weight (row h = output column h)
 *   out         [T, H]    bf16  result, round-to-nearest-even; must not overlap
 *                               routed, W, g or the workspace. It may be exactly
 *                               one of the shared partials (out == shared + p*T*H):
 *                               the pages' in-place `addmm_` into the shared
 *                               output; any other overlap with shared is rejected
 *   eps                         RMSNorm epsilon, finite and > 0 (when norm_weight
 *                               is not NULL)
 *   workspace, workspace_bytes  at least latent_tail_workspace_size(P,T,L,H)
 *                               bytes of device scratch; its contents on entry
 *                               are ignored and on return are unspecified
 * For T <= 2 (when L <= 4096 and one SM's share of W fits in its shared
 * memory, e.g. L = 2048 at H = 7168) one CUDA-core kernel does the whole tail;
 * the normalized latent then stays in FP32, unrounded, and the workspace is
 * not used. Otherwise two kernels run: reduce + RMSNorm into the workspace
 * (bf16), then the up-projection with the shared-partial epilogue (decode
 * kernel for T <= 224 when its buffers fit in shared memory, which they always
 * do for T <= 128 and do at L = 2048; persistent tensor-core kernel otherwise),
 * chained by programmatic dependent launch. When the decode kernel runs (and
 * T > 2) the first kernel also prefetches routed and the W rows
 * into L2 before it waits for the preceding work on the stream (an L2
 * prefetch is only a hint: if that work is still writing routed, the lines are
 * updated in L2 and every read happens after the wait). Calls issued back to
 * back on one stream may share one workspace. Capturable in a CUDA graph.
 */
LT_API lt_status latent_tail_forward(const uint16_t* routed, const uint16_t* shared,
                                     const float* norm_weight, const uint16_t* W,
                                     uint16_t* out, int P, int T, int L, int H,
                                     float eps, void* workspace, size_t workspace_bytes,
                                     lt_stream stream);

/*
 * Column-parallel form: writes only out[t, h] for col_start <= h < col_end.
 * Every other byte of out (still the full [T, H] buffer) is left untouched.
 * 0 <= col_start < col_end <= H, both multiples of 8. Each written element is
 * computed exactly as latent_tail_forward computes it, so a set of calls whose
 * ranges tile [0, H) reproduces the full call bit for bit.
 */
LT_API lt_status latent_tail_forward_cols(const uint16_t* routed, const uint16_t* shared,
                                          const float* norm_weight, const uint16_t* W,
                                          uint16_t* out, int P, int T, int L, int H,
                                          float eps, int col_start, int col_end,
                                          void* workspace, size_t workspace_bytes,
                                          lt_stream stream);

/*
 * Steps 1-2 alone (the pages' `allreduce_norm_latent_out`): latent[t,l] =
 * bf16_rn(x[t,l] * rsqrt(mean_l x^2 + eps) * g[l]) with x = sum_p routed[p,t,l]
 * accumulated in FP32; with norm_weight == NULL, latent = bf16_rn(x).
 *   routed [P, T, L] bf16, norm_weight [L] fp32, latent [T, L] bf16 (output,
 *   must not overlap the inputs).
 */
LT_API lt_status latent_tail_norm(const uint16_t* routed, const float* norm_weight,
                                  uint16_t* latent, int P, int T, int L, float eps,
                                  lt_stream stream);

/*
 * Steps 3-5 alone (the pages' narrowed `addmm_` beta-add plus the shared-partial
 * sum): out[t,h] = bf16_rn(sum_l latent[t,l] * W[h,l] + sum_p shared[p,t,h]) for
 * col_start <= h < col_end; other columns untouched.
 *   latent [T, L] bf16, shared [P, T, H] bf16, W [H, L] bf16, out [T, H] bf16
 *   (out may be exactly one of the shared partials, as in latent_tail_forward).
 * Range rules as in latent_tail_forward_cols; results are bit-identical to the
 * projection step of latent_tail_forward given the same latent. With P = 1 this
 * is the per-rank compute after the reference's all-reduce.
 * When the decode kernel serves the call (see latent_tail_forward) it is
 * launched as a programmatic dependent of the work
 * before it on the stream: it may start (set up its barriers and tensor memory)
 * before that work has finished, but it reads no input and writes no output
 * until that work is complete, so back-to-back calls overlap only set-up.
 */
LT_API lt_status latent_tail_project_cols(const uint16_t* latent, const uint16_t* shared,
                                          const uint16_t* W, uint16_t* out, int P, int T,
                                          int L, int H, int col_start, int col_end,
                                          lt_stream stream);

/*
 * Synchronizes `stream`, then reports (and clears) the current device's error
 * word: LT_ERR_TIMEOUT if a bounded device wait expired since the last check,
 * LT_ERR_CUDA if the stream reported an error, LT_OK otherwise.
 */
LT_API lt_status latent_tail_check(lt_stream stream);

/*
 * Diagnostic for the bounded device waits: enqueues one CTA that waits on a
 * barrier nothing ever completes, through the same bounded wait the kernels
 * use, with a limit of limit_us microseconds (1 .. 1000000). The wait expires,
 * the device error word records a timeout and the kernel returns; the next
 * latent_tail_check on the stream reports LT_ERR_TIMEOUT and clears it. No
 * fault, trap or hang is involved and the context stays usable.
 */
LT_API lt_status latent_tail_selftest_wait_timeout(unsigned int limit_us, lt_stream stream);

/*
 * Allocation-free form of latent_tail_forward (the pages have no counterpart;
 * this exists for callers, not for the method). Some callers cannot allocate
 * device memory: a custom op or plugin that a host runtime hands only its
 * input and output buffers, with no allocator to call, or code that must not
 * allocate while it runs. They cannot supply the workspace that
 * latent_tail_forward needs, so this entry point keeps that scratch (the
 * normalized latent, T * L * 2 bytes) in a fixed device array inside the
 * library instead:
 *   - the array holds LT_NOALLOC_MAX_SCRATCH_BYTES (8 MiB) on every GPU that
 *     loads the library, until the process exits; calls whose
 *     latent_tail_workspace_size(P, T, L, H) exceeds it return LT_ERR_WORKSPACE
 *     and launch nothing (at L = 2048 that allows T <= 2048);
 *   - nothing is allocated or freed by the call (no cudaMalloc / cudaFree);
 *   - the first call on a device looks up the array's device address on that
 *     device; make that first call before capturing a stream into a graph;
 *   - all calls on a device share the one array and it keeps the previous
 *     call's contents (every call rewrites all of the latent it reads, so
 *     nothing needs to start at zero).
 *     Calls whose GPU work overlaps in time
 *     (different streams without ordering, or different host threads) race on
 *     the array and give wrong results: order them on one stream.
 * Arguments, output and errors are as for latent_tail_forward, minus the
 * workspace.
 */
#define LT_NOALLOC_MAX_SCRATCH_BYTES ((size_t)8 << 20)
LT_API lt_status latent_tail_forward_noalloc(const uint16_t* routed, const uint16_t* shared,
                                             const float* norm_weight, const uint16_t* W,
                                             uint16_t* out, int P, int T, int L, int H,
                                             float eps, lt_stream stream);

/*
 * Bytes of device workspace latent_tail_forward_host needs: the normalized
 * latent as for latent_tail_workspace_size, plus device staging for routed when
 * T <= 2, and for routed, shared and out when the call runs the persistent
 * tensor-core kernel (above 224 tokens, or above 128 when the decode kernel's
 * buffers do not fit; see latent_tail_forward), each rounded up to 256 bytes.
 * Returns 0 for T <= 0 or invalid shapes. Host-only, never touches the GPU.
 */
LT_API size_t latent_tail_host_workspace_size(int P, int T, int L, int H);

/*
 * End-to-end form of latent_tail_forward for inputs that arrive in, and a
 * result that leaves to, host memory (serving glue that holds the partials on
 * the CPU side; the pages' tail always runs on device tensors, so this is a
 * library convenience, not a step of the method).
 *   routed_host [P, T, L], shared_host [P, T, H], out_host [T, H]: bf16 in
 *     PAGE-LOCKED host memory mapped for the current device (cudaHostAlloc /
 *     cudaMallocHost, or cudaHostRegister with cudaHostRegisterMapped), each
 *     lying inside one such allocation, 16-byte aligned. Anything else
 *     (pageable memory, device memory, a range running past its allocation)
 *     gives LT_ERR_INVALID_ARG before any work is enqueued.
 *   norm_weight, W: device memory, as in latent_tail_forward.
 *   out_host: same overlap rules as out in latent_tail_forward (it may be
 *     exactly one of the shared partials).
 *   workspace: latent_tail_host_workspace_size(P, T, L, H) bytes of device
 *     memory, not overlapping W or norm_weight.
 * When the one-launch kernel serves the shape (T <= 2, as for
 * latent_tail_forward), a copy kernel first brings the routed partials into
 * the workspace; the kernel then reads shared and writes out through the host
 * link. Otherwise, when the decode kernel serves the call, the kernels read the
 * partials and write the result through the host link directly: no staging
 * copy, the host bytes cross the link once.
 * For the persistent kernel the partials are copied into the workspace (one cudaMemcpyAsync per
 * tensor), the device path runs, and the result is copied back. Like every
 * call it is asynchronous: out_host holds the result once `stream` has been
 * synchronized, and the host buffers must not be modified before then.
 * Results are bit-identical to latent_tail_forward on the same values.
 */
LT_API lt_status latent_tail_forward_host(const uint16_t* routed_host,
                                          const uint16_t* shared_host,
                                          const float* norm_weight, const uint16_t* W,
                                          uint16_t* out_host, int P, int T, int L, int H,
                                          float eps, void* workspace, size_t workspace_bytes,
                                          lt_stream stream);

/* Static, human-readable name of a status code. Never NULL. */
LT_API const char* latent_tail_status_string(lt_status status);

#ifdef __cplusplus
}
#endif

#endif /* LATENT_TAIL_H */
