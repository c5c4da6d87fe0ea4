/*
 * libgma — Gaussian Mixture Attention (GMA) forward hot path for one GB300
 * (sm_103a).  C ABI over caller-owned memory and a CUDA stream.
 *
 * The method is the one described by the explainer page "Gaussian Mixture
 * Attention: Linear-Time Sequence Mixing via Probabilistic Latent Routing"
 * (technical summary, sections "핵심 메커니즘" and "변형 및 학습"):
 *
 *   routing      gamma_{i,k} = p(z = k | x_i) under a K-component GMM with
 *                means mu_k, diagonal variances sigma_k^2 = softplus(var_raw_k)
 *                and priors pi = softmax(logit_pi); Q_X and K_X rows share the
 *                same components (one GMM per head).
 *   write        Vt = Gamma_K^T V  (K x d_v),  Z = Gamma_K^T 1  (K)
 *   read         O  = Gamma_Q Vt / (Gamma_Q Z + eps)   (eps added once per row)
 *   causal       Vt, Z are inclusive prefix sums over positions j <= i; the
 *                library evaluates them in the chunkwise-parallel form of the
 *                linear-attention page ("선형 어텐션 원리 정리", section
 *                "쉽게 이해하기": dense products inside a chunk, a carried state
 *                between chunks), which is exact, not an approximation.
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *     and contiguous, 16-byte aligned (else GMA_ERR_ALIGNMENT).  The library
 *     never allocates, frees or retains them.
 *   - Work is enqueued on `stream` (0 = legacy default stream) and is
 *     asynchronous: the call returns before the GPU finishes.  Launch
 *     failures are reported as GMA_ERR_CUDA; faults inside a kernel surface
 *     at the caller's next synchronisation.
 *   - Arguments are validated on the host before anything is launched; on
 *     any error nothing is enqueued.  Unsupported sizes return
 *     GMA_ERR_UNSUPPORTED; nothing falls back to another implementation.
 *   - `ws` is caller-owned device scratch of at least
 *     gma_workspace_size(shape, op) bytes (GMA_ERR_WORKSPACE otherwise).  Its
 *     contents on entry are ignored and on return are unspecified.  Calls
 *     that run concurrently must use different workspaces.
 *   - Bounded waits.  The tensor-core kernels wait on mbarriers (for TMA
 *     copies and tensor-core products) with a limit of about 2 s of SM
 *     cycles.  If a wait expires, the kernel stops issuing work, waits (again
 *     bounded) for what it has already issued, and returns, leaving the
 *     call's outputs undefined (NaN where the waiting threads owned the rows);
 *     it also sets the device's timeout flag.  The next
 *     compute call on that device that sees the flag returns GMA_ERR_TIMEOUT
 *     (launching nothing) and clears it; gma_sync_status(stream) waits for
 *     the stream and reports it deterministically.  An expired wait means the
 *     asynchronous units did not make progress: treat the CUDA context as
 *     unusable.
 *   - Calls are reentrant.  The library's only global state is created once
 *     and never changes results: the two copy streams per device of
 *     gma_forward_causal_host (created by its first call), the scratch array
 *     of gma_decode_step_noalloc, the timeout flags (one word per device in
 *     page-locked host memory, allocated by the first call that launches a
 *     tensor-core kernel: make that call before any stream capture), and the
 *     thread-local last CUDA error.
 *
 * Supported sizes: d_route in {16, 32, 64, 128}; d_v in {16, 32, 64, 128};
 * 1 <= K <= 512; B, H, N >= 1 with B*H*N*max(d_route, d_v, K) < 2^40;
 * causal chunk as described in gma_shape; B*H <= 65535.  N = 0 is
 * accepted, the sequence pointers may then be NULL, and the call does nothing
 * (a causal call copies state_in to state_out, or zeroes it).
 */
#ifndef GMA_H
#define GMA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gma_stream_t; /* binary-compatible with cudaStream_t */

typedef enum {
    GMA_OK = 0,
    GMA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum value */
    GMA_ERR_UNSUPPORTED = 2, /* valid but not implemented: d_route, d_v, K or chunk */
    GMA_ERR_ALIGNMENT = 3,   /* a tensor pointer is not 16-byte aligned */
    GMA_ERR_WORKSPACE = 4,   /* ws is null or smaller than gma_workspace_size() */
    GMA_ERR_CUDA = 5,        /* a CUDA launch or runtime call failed */
    GMA_ERR_TIMEOUT = 6      /* a bounded wait inside a kernel expired (see gma_sync_status) */
} gma_status;

typedef enum { GMA_F32 = 0, GMA_BF16 = 1 } gma_dtype;

typedef enum {
    GMA_OP_RESPONSIBILITIES = 0,
    GMA_OP_BIDIR = 1,
    GMA_OP_CAUSAL = 2,
    GMA_OP_DECODE = 3,
    GMA_OP_CAUSAL_HOST = 4,  /* gma_forward_causal_host: staging + the causal workspace */
    GMA_OP_USAGE = 5,        /* gma_responsibility_stats */
    GMA_OP_BACKWARD = 6      /* gma_backward (causal or bidirectional) */
} gma_op;

typedef struct {
    int B, H, N;        /* batch, heads, tokens per sequence (ignored by decode) */
    int d_route;        /* width of the Q_X / K_X routing rows */
    int d_v;            /* width of the value rows and of the output */
    int K;              /* number of Gaussian components per head */
    int chunk;          /* causal chunk length C in {16, 32, 64, 128}; 0 selects
                           128 where the tensor-core path applies (K <= 128 or
                           K in {256, 384, 512}, and d_v = 64, or d_v = 128 with
                           bf16 products), else 64; 128 is accepted only there */
    float eps;          /* read-phase stabiliser, added to Gamma_Q Z (>= 0) */
    gma_dtype x_dtype;  /* storage type of Q_X and K_X */
    gma_dtype v_dtype;  /* storage type of V */
    gma_dtype gemm_dtype; /* GMA_F32: chunk products carry fp32 operands (the
                             1e-4 path); GMA_BF16: Gamma, V and P are rounded to
                             bf16 as product operands, accumulation stays fp32 */
} gma_shape;

/* Per-head GMM parameters, fp32 device pointers (one GMM per head, shared by
 * Q_X and K_X and by every batch element):
 *   mu       [H, K, d_route]  component means
 *   var_raw  [H, K, d_route]  raw variances; sigma^2 = softplus(var_raw)
 *   logit_pi [H, K]           mixture logits;  pi = softmax over K          */
typedef struct {
    const float *mu;
    const float *var_raw;
    const float *logit_pi;
} gma_params;

/* Bytes of device scratch that `op` needs for `shape` (0 on invalid input). */
size_t gma_workspace_size(const gma_shape *shape, gma_op op);

/* Routing step alone (the "probabilistic latent routing" of "핵심 메커니즘"):
 *   x      [B, H, N, d_route]  routing rows (x_dtype)
 *   gamma  [B, H, N, K]        fp32 output, each row a probability vector.   */
gma_status gma_responsibilities(const gma_shape *shape, gma_params params, const void *x,
                                float *gamma, void *ws, size_t ws_bytes, gma_stream_t stream);

/* Responsibility diagnostics (the interpretability reading of "결과 및 성능":
 * components in use, usage entropy, hard assignments), as a reduction over
 * the responsibilities of the routing rows x [B, H, N, d_route] (x_dtype),
 * which the call computes in its workspace.  Per head h, over the B*N rows
 * of that head:
 *   usage    [H, K] fp32    soft usage, sum_i gamma_ik
 *   counts   [H, K] int64   hard assignments: rows whose argmax is k (the
 *                           lowest k among equal values)
 *   entropy  [H, 2] fp32    entropy of usage[h] / sum(usage[h]) and of
 *                           counts[h] / (B N), each divided by log K (0 when
 *                           K = 1); a value of 1 means uniform use
 *   assign   nullable [B, H, N] int32: the argmax of every row
 * The number of components in use is the count of k with counts[h][k] > 0.
 * Sums run in a fixed order: repeated calls give identical results.
 * Workspace: gma_workspace_size(shape, GMA_OP_USAGE).                        */
gma_status gma_responsibility_stats(const gma_shape *shape, gma_params params, const void *x,
                                    float *usage, long long *counts, float *entropy, int *assign,
                                    void *ws, size_t ws_bytes, gma_stream_t stream);

/* Bidirectional forward (write phase then read phase of "핵심 메커니즘"):
 *   qx, kx [B, H, N, d_route] (x_dtype);  v [B, H, N, d_v] (v_dtype)
 *   out    [B, H, N, d_v] fp32:  O = Gamma_Q Vt / (Gamma_Q Z + eps).        */
gma_status gma_forward_bidir(const gma_shape *shape, gma_params params, const void *qx,
                             const void *kx, const void *v, float *out, void *ws,
                             size_t ws_bytes, gma_stream_t stream);

/* Cross-attention (named as an extension in "의의 및 주장"): the queries of one
 * sequence read the latent memory written by the keys and values of another.
 * shape->N is the number of query rows; n_kv >= 0 the number of key/value
 * rows (every other field is shared).  Same arithmetic as the bidirectional
 * form, which it equals when the two sequences are the same.
 *   qx  [B, H, N, d_route] (x_dtype)      kx [B, H, n_kv, d_route] (x_dtype)
 *   v   [B, H, n_kv, d_v]  (v_dtype)      out [B, H, N, d_v] fp32
 * With n_kv = 0 the memory is empty and out = 0 / (0 + eps).  kx and v may be
 * NULL when n_kv = 0; every pointer may be NULL when N = 0 (nothing is done).
 * Workspace: gma_cross_workspace_size(shape, n_kv) bytes (0 on invalid input). */
size_t gma_cross_workspace_size(const gma_shape *shape, int n_kv);
gma_status gma_forward_cross(const gma_shape *shape, int n_kv, gma_params params, const void *qx,
                             const void *kx, const void *v, float *out, void *ws, size_t ws_bytes,
                             gma_stream_t stream);

/* Causal forward (prefix-sum variant of "변형 및 학습"): O_i reads the memory
 * written by positions j <= i.
 *   qx, kx, v, out  as gma_forward_bidir
 *   state_in   nullable [B, H, K*d_v + K] fp32: memory left by earlier tokens
 *              (Vt as K rows of d_v, then Z); NULL means empty.
 *   state_out  nullable [B, H, K*d_v + K] fp32: memory after the N tokens
 *              (state_in included).  May alias state_in.                     */
gma_status gma_forward_causal(const gma_shape *shape, gma_params params, const void *qx,
                              const void *kx, const void *v, const float *state_in,
                              float *state_out, float *out, void *ws, size_t ws_bytes,
                              gma_stream_t stream);

/* Causal forward on HOST buffers: the library copies the inputs in and the
 * output out itself, in groups of (batch, head) slices, so that the copies of
 * one group overlap the computation of another (slices are independent in
 * the method).  Same arithmetic and results as gma_forward_causal.
 *   qx, kx, v   host [B, H, N, ...] as gma_forward_causal (page-locked memory
 *               gives asynchronous copies; pageable memory works, slower)
 *   out         host [B, H, N, d_v] fp32
 *   state_in, state_out   device, as gma_forward_causal
 *   ws          device scratch of gma_workspace_size(shape, GMA_OP_CAUSAL_HOST)
 *               bytes: device copies of the inputs and the output, then the
 *               causal workspace.
 * The call enqueues its work after everything already on `stream` and returns;
 * the output is on the host once `stream` has completed.  The copies run on
 * two internal streams joined to `stream` by events.                       */
gma_status gma_forward_causal_host(const gma_shape *shape, gma_params params, const void *qx,
                                   const void *kx, const void *v, const float *state_in,
                                   float *state_out, float *out, void *ws, size_t ws_bytes,
                                   gma_stream_t stream);

/* Gradients of the causal (causal = 1) or bidirectional (causal = 0) forward,
 * for end-to-end training ("변형 및 학습": the GMM parameters are learned by
 * backpropagation through the softplus and softmax reparameterisations).
 * Given dout = dL/dO [B, H, N, d_v] (fp32), the call recomputes the forward
 * (responsibilities, memory) and writes, all fp32:
 *   dqx, dkx  [B, H, N, d_route]   (gradients of the stored Q_X, K_X values)
 *   dv        [B, H, N, d_v]
 *   dmu, dvar_raw [H, K, d_route], dlogit_pi [H, K]: summed over the batch
 *             and over both routings (one GMM per head), overwritten.
 * The arithmetic is fp32 on CUDA cores (shape->gemm_dtype and shape->chunk
 * are ignored: chunks of 64 rows); every reduction runs in a fixed order, so
 * repeated calls give identical results.  The causal form starts from an
 * empty memory (no state_in).  Workspace: gma_workspace_size(shape,
 * GMA_OP_BACKWARD).  N = 0 gives zero parameter gradients.                  */
gma_status gma_backward(const gma_shape *shape, int causal, gma_params params, const void *qx,
                        const void *kx, const void *v, const float *dout, float *dqx, float *dkx,
                        float *dv, float *dmu, float *dvar_raw, float *dlogit_pi, void *ws,
                        size_t ws_bytes, gma_stream_t stream);

/* One recurrent decode step (the causal form advanced by one token; constant
 * memory per head as in "선형 어텐션 원리 정리"): the token is written into the
 * memory first, then its query reads it.
 *   qx, kx [B, H, d_route] (x_dtype); v [B, H, d_v] (v_dtype)
 *   state  [B, H, K*d_v + K] fp32, updated in place
 *   out    [B, H, d_v] fp32.  shape->N is ignored.                          */
gma_status gma_decode_step(const gma_shape *shape, gma_params params, const void *qx,
                           const void *kx, const void *v, float *state, float *out, void *ws,
                           size_t ws_bytes, gma_stream_t stream);

/* Profiling variant of gma_forward_causal, for benchmarks.  It runs exactly
 * the same launches on `stream`, and records events[i] just before launch i
 * and events[n_stages] after the last one, so that the caller can time every
 * kernel of the step with cudaEventElapsedTime.
 *   prof->events     in:  GMA_PROFILE_MAX_STAGES + 1 cudaEvent_t handles
 *                         (created by the caller, timing enabled)
 *   prof->n_stages   out: number of launches of this call
 *   prof->stage_name out: static, NUL-terminated kernel names (not owned)   */
#define GMA_PROFILE_MAX_STAGES 8
typedef struct {
    void *events[GMA_PROFILE_MAX_STAGES + 1];
    int n_stages;
    const char *stage_name[GMA_PROFILE_MAX_STAGES];
} gma_profile;

gma_status gma_forward_causal_profiled(const gma_shape *shape, gma_params params, const void *qx,
                                       const void *kx, const void *v, const float *state_in,
                                       float *state_out, float *out, void *ws, size_t ws_bytes,
                                       gma_stream_t stream, gma_profile *prof);

/* Profiling variants of gma_forward_bidir and gma_decode_step, with the same
 * event protocol as gma_forward_causal_profiled.                             */
gma_status gma_forward_bidir_profiled(const gma_shape *shape, gma_params params, const void *qx,
                                      const void *kx, const void *v, float *out, void *ws,
                                      size_t ws_bytes, gma_stream_t stream, gma_profile *prof);
gma_status gma_decode_step_profiled(const gma_shape *shape, gma_params params, const void *qx,
                                    const void *kx, const void *v, float *state, float *out,
                                    void *ws, size_t ws_bytes, gma_stream_t stream,
                                    gma_profile *prof);

/* Decode step for callers that cannot allocate device memory.
 *
 * No counterpart in the paper: this is a deployment convenience.  Some hosts
 * cannot call cudaMalloc at the point where they run a decode step: plugins
 * whose host application owns every device allocation, code held to a fixed
 * memory budget, or loops that must not take the allocator's latency or
 * failure modes.  This entry point computes exactly what gma_decode_step
 * computes, with the same arguments minus the workspace, and allocates
 * nothing: its scratch (the per-head parameters prepared for the step) lives
 * in a file-scope device array of GMA_NOALLOC_SCRATCH_BYTES bytes that every
 * GPU which loads the library holds until the process exits.
 *   - The scratch of the calling thread's current device is used.  The
 *     first call on a device looks up the array's device address (once per
 *     device); make that first call before any stream capture.
 *   - Shapes whose scratch would exceed GMA_NOALLOC_SCRATCH_BYTES, i.e.
 *     256-byte-rounded H*K*d_route*8 plus 256-byte-rounded H*K*4, are
 *     rejected with GMA_ERR_WORKSPACE and nothing is launched.
 *   - Every call shares the one array.  Calls whose work overlaps on the GPU
 *     (for example on two streams without ordering between them) race on it
 *     and give undefined results; order them.  Each call rewrites the whole
 *     part of the array it reads, so no clearing is needed between calls.
 * All other arguments, layouts and errors are those of gma_decode_step.     */
#define GMA_NOALLOC_SCRATCH_BYTES (8u << 20)

gma_status gma_decode_step_noalloc(const gma_shape *shape, gma_params params, const void *qx,
                                   const void *kx, const void *v, float *state, float *out,
                                   gma_stream_t stream);

/* Waits for `stream` to complete, then reports a bounded wait that expired in
 * one of the library's kernels on the calling thread's current device since
 * the last report: GMA_ERR_TIMEOUT (and the flag is cleared), GMA_ERR_CUDA if
 * the synchronisation failed (gma_last_cuda_error names the error), else
 * GMA_OK.  This is the status-reporting half of the bounded waits described
 * under "Bounded waits" above (no counterpart on the pages: a property of
 * this implementation's asynchronous kernels).                              */
gma_status gma_sync_status(gma_stream_t stream);

/* Test hook of the timeout path, with no counterpart on the pages: enqueues
 * one kernel whose only work is a wait, bounded by limit_cycles SM cycles,
 * on an mbarrier that nothing ever arrives on (no copy or product is issued
 * against it, so nothing is in flight when it gives up).  The wait expires
 * and is reported like those of the compute kernels: the next compute call
 * or gma_sync_status returns GMA_ERR_TIMEOUT.  limit_cycles in [1, 4e9]
 * (GMA_ERR_INVALID_ARG otherwise); about 2e6 is one millisecond at 2 GHz.  */
gma_status gma_test_wait_timeout(long long limit_cycles, gma_stream_t stream);

/* Static description of a status code (never NULL). */
const char *gma_status_string(gma_status status);

/* Name of the CUDA error behind the last GMA_ERR_CUDA returned on the calling
 * thread ("cudaSuccess" if there was none).  Static string.                 */
const char *gma_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GMA_H */
