/*
 * muon.h -- C ABI of the GB300 (sm_103a) Muon optimizer-step library.
 *
 * The operation: the per-matrix Muon step over whole weight matrices held on
 * one rank -- "How PyTorch Scaled a Near-1T MoE on Europe's Public
 * Supercomputer", section "Three optimizations that changed the economics",
 * FlexShard bullet: Muon is applied to almost all weight matrices, its
 * Newton-Schulz update works on full matrices, and whole experts are placed
 * on one rank so that the orthogonalisation needs no communication.  Muon
 * keeps a single optimizer state per matrix (the momentum) -- "Domyn is
 * training a 1T-parameter MoE on Europe's Jupiter supercomputer, and
 * published the recipe", section "What moved the number".
 *
 * The pages state no formula.  This library computes, per m x n matrix
 * (r = min(m, n), k = max(m, n); "oriented" = transposed when m > n):
 *
 *   M   <- fma(mu, M, G)                      fp32 momentum, one rounding
 *   U    = fma(mu, M, G)  (Nesterov)          fp32, one rounding (or U = M)
 *   X0   = bf16(U^(oriented) * sigma),  sigma = fp32(1 / (|U|_F + eps))
 *   repeat `steps` times, (a, b, c) = (3.4445, -4.7750, 2.0315) by default:
 *     A  = bf16(X X^T)                        r x r, fp32 accumulation
 *     B  = bf16(b A + c A A)                  r x r, fp32 accumulation
 *     X  = bf16(a X + B X)                    r x k, fp32 accumulation
 *   O    = X (un-oriented)
 *   W   <- round_W( fma(-s, O, dcy * W) ),  dcy = 1 - lr*wd,
 *                                           s   = lr * 0.2 * sqrt(max(m, n))
 *          (dcy and s are computed in double on the host, rounded once to fp32)
 *
 * Conventions shared by every call:
 *  - Matrices are dense, row-major, contiguous, on the current CUDA device;
 *    every device pointer must be 16-byte aligned.  Host arrays (the pointer
 *    arrays, rows, cols, coeffs, opts) are read during the call only.
 *  - The caller owns every matrix.  W, G and M of one matrix must not alias
 *    each other, and no two matrices may overlap.
 *  - Calls are asynchronous on `stream` (0 = legacy default stream) and do
 *    not synchronise the host, except for the first allocation of the
 *    library-owned workspace (below).  Device-side failures (a bounded wait
 *    that ran out inside a kernel) are reported by muon_device_status().
 *  - Validation happens before any work is enqueued: on a non-OK return
 *    nothing was enqueued and no argument was modified.  count == 0 is a
 *    no-op returning MUON_OK.
 *  - Workspace: the library keeps one device workspace per device, grown with
 *    stream-ordered allocation on the caller's stream (never on a side
 *    stream) and reused by later calls; calls on different streams are
 *    ordered through an event.  If the workspace for a whole batch cannot be
 *    allocated, the matrices run in consecutive groups with smaller workspaces
 *    (same results); MUON_ERR_OOM only if no grouping finds memory.
 *    muon_step_ex() can take a caller-provided workspace instead.
 *    muon_release_workspace() frees it.
 *  - Thread safety: calls may come from several host threads; the library
 *    serialises them internally.
 *  - CUDA graphs: muon_step, muon_step_ex and muon_ns5_batched may be captured
 *    on a stream once a call with the same shapes has run outside the capture
 *    (so that the workspace exists); a capture that would need a larger
 *    workspace fails with MUON_ERR_UNSUPPORTED.  Captured work is not ordered
 *    against the library's uncaptured calls on other streams.
 *  - Device lifetime: the library keeps per-device state for the life of the
 *    process (the workspace, its streams and events, kernel attributes, the
 *    device address of muon_ns5_batched_static's scratch array).  It does not
 *    survive cudaDeviceReset() or the teardown of the device's primary
 *    context: after either, make no further call of this library in the
 *    process.
 */
#ifndef MUON_GB300_H
#define MUON_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MUON_API __attribute__((visibility("default")))
#else
#define MUON_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MUON_OK = 0,
    MUON_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment, aliasing, dtype */
    MUON_ERR_UNSUPPORTED = 2,   /* no sm_100-family device, or a shape above the limits */
    MUON_ERR_CUDA = 3,          /* a CUDA runtime call failed (see muon_last_error) */
    MUON_ERR_OOM = 4,           /* workspace allocation failed or caller workspace too small */
    MUON_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out (muon_device_status) */
    MUON_ERR_CORRUPT = 6        /* a debug guard region of the workspace was overwritten
                                   (MUON_DEBUG_GUARD=1; muon_device_status) */
} muon_status;

typedef enum { MUON_BF16 = 0, MUON_F32 = 1 } muon_dtype;

/* Largest supported dimension (rows or cols) of one matrix. */
#define MUON_MAX_DIM 32768

/*
 * In-place Newton-Schulz orthogonalisation (with Frobenius normalisation and
 * automatic orientation) of `count` bf16 matrices -- the "orthogonalisation on
 * full matrices" of the FlexShard bullet above, without the momentum or the
 * weight update.
 *   ptrs[i]  device pointer to matrix i, bf16, rows[i] x cols[i], row-major;
 *            overwritten with O (bf16).
 *   rows, cols  host arrays of `count` dims, each in [1, MUON_MAX_DIM].
 *   steps    number of iterations, 0..64 (0 = normalise only).
 *   coeffs   host float[3] {a, b, c}, or NULL for {3.4445, -4.7750, 2.0315}.
 * Returns a muon_status.
 */
MUON_API int muon_ns5_batched(void* const* ptrs, const int* rows, const int* cols, int count,
                     int steps, const float* coeffs, cudaStream_t stream);

/*
 * muon_ns5_batched with a coefficient schedule.  The pages give no Newton-
 * Schulz coefficients at all; this generalises the fixed triple:
 *   coeffs_per_step = 0: coeffs is NULL or one {a, b, c} used at every step
 *   coeffs_per_step = 1: coeffs holds `steps` triples {a_t, b_t, c_t}, the
 *                        t-th used at iteration t (NULL = defaults)
 * Other arguments and behaviour as muon_ns5_batched.
 */
MUON_API int muon_ns_batched_ex(void* const* ptrs, const int* rows, const int* cols, int count,
                                int steps, const float* coeffs, int coeffs_per_step,
                                cudaStream_t stream);

/* Size of the device scratch array behind muon_ns5_batched_static (64 MiB). */
#define MUON_STATIC_SCRATCH_BYTES (64u << 20)

/*
 * muon_ns5_batched for callers that cannot allocate device memory.  The pages
 * have no counterpart of this call; it exists for callers that must not call
 * cudaMalloc -- code running while a framework's caching allocator owns the
 * device budget (a stray allocation outside it can push the job out of
 * memory), latency-critical paths that cannot take cudaMalloc's implicit
 * synchronisation, and hosts that give the library a fixed memory budget.
 *
 * Same arguments, same kernels and same results as muon_ns5_batched, but the
 * scratch (norm partials, per-matrix scales, padded iterates) lives in one
 * file-scope device array of MUON_STATIC_SCRATCH_BYTES that every GPU loading
 * the library holds until the process exits.  No call allocates or frees
 * device memory.
 *  - Limit: batches whose scratch (muon_workspace_bytes(rows, cols, count))
 *    exceeds MUON_STATIC_SCRATCH_BYTES are rejected with MUON_ERR_UNSUPPORTED
 *    and a message giving both sizes; nothing is enqueued.  For example one
 *    1024 x 4096 matrix fits, one 2048 x 6144 matrix does not.
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress) with that device current; make that first
 *    call before any stream capture on the device.
 *  - Sharing: every call uses the same array and it keeps the previous call's
 *    contents; every scratch element is written before it is read, so nothing
 *    needs clearing.  Calls whose work overlaps on the GPU (other streams,
 *    other host threads) race on the array: order them on one stream or with
 *    events.
 */
MUON_API int muon_ns5_batched_static(void* const* ptrs, const int* rows, const int* cols, int count,
                                     int steps, const float* coeffs, cudaStream_t stream);

/*
 * One full Muon step on `count` matrices with bf16 weights, bf16 gradients and
 * fp32 momentum, Nesterov, 5 steps, default coefficients, eps = 1e-7.
 *   W[i]  device pointer, bf16 rows[i] x cols[i], updated in place.
 *   G[i]  device pointer, bf16, read only.
 *   M[i]  device pointer, fp32, updated in place (bit-exact fp32 arithmetic).
 *   lr, mu, wd  learning rate, momentum, decoupled weight decay (finite).
 */
MUON_API int muon_step(void* const* W, const void* const* G, float* const* M,
              const int* rows, const int* cols, int count,
              float lr, float mu, float wd, cudaStream_t stream);

typedef struct {
    int w_dtype;              /* muon_dtype of every W (default MUON_BF16) */
    int g_dtype;              /* muon_dtype of every G (default MUON_BF16) */
    int steps;                /* Newton-Schulz iterations, 0..64 (default 5) */
    const float* coeffs;      /* host float[3] or NULL (default) */
    float eps;                /* normalisation epsilon, >= 0 (default 1e-7) */
    int nesterov;             /* 1 = Nesterov look-ahead (default), 0 = U = M */
    void* workspace;          /* optional caller workspace (device, 256-byte aligned) */
    size_t workspace_bytes;   /* its size.  Smaller than muon_workspace_bytes(...) for the
                                 whole batch: the matrices run in consecutive groups that
                                 fit, one after the other on the stream (same results);
                                 MUON_ERR_OOM only if one matrix alone does not fit */
    void* const* o_out;       /* optional host array of `count` device pointers (bf16,
                                 rows[i] x cols[i], 16-byte aligned, not overlapping any
                                 other buffer) that receive the orthogonalised update O;
                                 NULL (default) = not written */
    int coeffs_per_step;      /* 0 (default): coeffs is one (a, b, c) triple used at
                                 every iteration; 1: coeffs holds `steps` triples, one
                                 per iteration (a coefficient schedule) */
    int g_count;              /* gradients per matrix, 1..64 (default 1): G[i] points to
                                 g_count contiguous rows[i] x cols[i] matrices (for
                                 example one per micro-batch or per sender) that are
                                 summed in fp32, in order, g = G_0 + G_1 + ..., inside
                                 the momentum pass -- bf16 gradients sent separately
                                 and summed in fp32 locally ("Training a trillion-
                                 parameter AI on the GPUs powering Europe's fastest
                                 supercomputer") without an fp32 accumulation buffer */
    int ns_fp8_gram;          /* 0 (default) or 1: the FP8 variant of Newton-Schulz for
                                 the matrices on the tensor-core path -- an answer to the
                                 open question of FP8 for expert matrix math ("Domyn is
                                 training a 1T-parameter MoE on Europe's Jupiter
                                 supercomputer, and published the recipe", section
                                 "What moved the number").  Each iteration's Gram
                                 product A = X X^T takes E4M3 operands: X scaled by
                                 2^8 (exact; the iterates' elements stay below 1.21,
                                 so 448 is never reached for the default coefficients),
                                 rounded to nearest even, summed in fp32, unscaled by
                                 2^-16, then rounded to bf16.  The E4M3 copy needs one
                                 more byte of workspace per element of every
                                 tensor-core iterate (a caller workspace sized by
                                 muon_workspace_bytes runs the batch in groups).  The
                                 polynomial and the
                                 update stay bf16 (E4M3 operands there move O by 10-50 %:
                                 X' = a X + B X cancels to about 0.7 X).  O then lies
                                 within about 8e-2 relative Frobenius error of the bf16
                                 result.  Matrices small enough for the shared-memory
                                 path (about 128 x 256 and below) stay bf16 there. */
} muon_step_opts;

/* Fill `opts` with the defaults listed above. */
MUON_API void muon_step_opts_init(muon_step_opts* opts);

/* muon_step with explicit options (opts may be NULL for the defaults). */
MUON_API int muon_step_ex(void* const* W, const void* const* G, float* const* M,
                 const int* rows, const int* cols, int count,
                 float lr, float mu, float wd, const muon_step_opts* opts,
                 cudaStream_t stream);

/*
 * muon_step_ex on optimizer state kept in host memory -- "Domyn is training a
 * 1T-parameter MoE on Europe's Jupiter supercomputer...", section "What moved
 * the number": optimizer state offloaded to Grace memory over NVLink-C2C.
 *   W[i], G[i], M[i]  HOST pointers to pinned (page-locked: cudaMallocHost or
 *                     cudaHostRegister) memory, same layouts and dtypes as
 *                     muon_step_ex; W and M are updated in place.
 *   opts              as muon_step_ex, but workspace and o_out must be NULL.
 * The matrices are streamed through the current device in chunks of about
 * 1 GiB of state (the first and the last at most 256 MB) with three staging sets, overlapping the copy in of the next
 * chunk and the copy out of the previous one with the step on the current one
 * (two library-owned copy streams, ordered with events).  The call is
 * asynchronous on `stream`: the host buffers may be read or reused only after
 * `stream` has completed the step.  Staging memory (three chunks) is allocated
 * stream-ordered on `stream` and kept for later calls.  All arguments are
 * validated before anything is enqueued; unpinned host memory is rejected
 * with MUON_ERR_INVALID_ARG.  A failure after the copies have started (a
 * staging or workspace allocation, an enqueue) returns the error with
 * `stream` still ordered after every copy already enqueued, so the host
 * buffers are safe to touch once `stream` completes; the matrices of the
 * chunks before the failing one may already be updated (W and M written
 * back), those from it on are not.
 */
MUON_API int muon_step_host(void* const* W, const void* const* G, float* const* M,
                            const int* rows, const int* cols, int count,
                            float lr, float mu, float wd, const muon_step_opts* opts,
                            cudaStream_t stream);

/*
 * AdamW for the parameters Muon does not cover -- "Domyn is training a
 * 1T-parameter MoE...", table "The model and the machine": Muon for about
 * 99.5% of parameters, AdamW for the rest (vectors, norms, embeddings).
 *   P[i]  device pointer to a flat parameter of numel[i] elements (p_dtype),
 *         updated in place;
 *   G[i]  its gradient (g_dtype), read only;
 *   M[i], V[i]  fp32 first and second moments, updated in place;
 *   numel[i] >= 0 (0 = skipped); every non-empty buffer 16-byte aligned, no
 *   overlaps (MUON_ERR_INVALID_ARG otherwise).
 *   lr, eps, wd finite, eps >= 0; beta1, beta2 in [0, 1); step >= 1 is the
 *   1-based step number used for bias correction.
 * Per element, each operation rounded once in fp32:
 *   m' = fma(beta1, m, (1-beta1)*g);  v' = fma(beta2, v, (1-beta2)*(g*g));
 *   p' = round_P(fma(-lr/(1-beta1^t), m' / (sqrt(v') / sqrt(1-beta2^t) + eps),
 *                    (1-lr*wd)*p))
 * where the scalars are computed in double and rounded to fp32 once
 * (1/sqrt(1-beta2^t) is applied as a multiplication).  Asynchronous on
 * `stream`; no workspace.
 */
MUON_API int muon_adamw_step(void* const* P, const void* const* G, float* const* M, float* const* V,
                             const long long* numel, int count, int p_dtype, int g_dtype,
                             float lr, float beta1, float beta2, float eps, float wd, int step,
                             cudaStream_t stream);

/* Device workspace (bytes) that one call on these shapes needs; 0 on bad args. */
MUON_API size_t muon_workspace_bytes(const int* rows, const int* cols, int count);

/* Static description of a status code. */
MUON_API const char* muon_status_string(int status);

/* Detail of the calling thread's last non-OK return ("" if none). */
MUON_API const char* muon_last_error(void);

/* Synchronise the current device's work on `stream`, then read and clear the
 * device-side status word (MUON_OK; MUON_ERR_TIMEOUT after a kernel's bounded
 * wait ran out; MUON_ERR_CORRUPT when MUON_DEBUG_GUARD=1 is set and a guard
 * region around a workspace region was overwritten).  Returns MUON_ERR_CUDA if
 * the stream reported an error. */
MUON_API int muon_device_status(cudaStream_t stream, int* device_status);

/* Free the library-owned workspace of the current device (synchronises it). */
MUON_API void muon_release_workspace(void);

/*
 * Kernel timing (for benchmarks).  While enabled, every kernel launch the
 * library makes is bracketed by a pair of CUDA events recorded on the
 * launching stream; muon_profile_read() synchronises those events and returns
 * per-kernel totals.  Disabled by default; enabling adds two event records per
 * launch.  Names: norm_pass, norm_finalize, pack, ns_gemm_gram, ns_gemm_poly,
 * ns_gemm_update, ns_gemm_final (the last update with the weight update or
 * the store of O in its epilogue), ns_small, unpack, adamw.
 */
typedef struct {
    char name[40];            /* kernel name */
    int launches;             /* launches since the last reset */
    double total_ms;          /* summed event-measured durations */
    double flops;             /* nominal algorithmic FLOPs of those launches */
    double bytes;             /* algorithmic HBM bytes of those launches */
} muon_kernel_stat;

MUON_API int muon_profile_enable(int on);                   /* 1 = on, 0 = off; resets totals */
MUON_API int muon_profile_read(muon_kernel_stat* out, int max_entries, int* n_entries);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H */
