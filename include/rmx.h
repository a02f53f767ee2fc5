/*
 * rmx.h -- C ABI of the fused RankMixer block (forward + backward) for GB300.
 *
 * The operation is the RankMixer block of the page "Subgraph-fusion-based
 * Mega-kernel Generation", section "Exact computation":
 *
 *   out1   = norm1(token_mixer(norm0(x)) + x)          outer LNs: eps 1e-3
 *   Z[b,t] = out1[b,t] @ w1[t] + b1[t];  (U, G) = split(Z) into halves
 *   hidden = LN_x(U) * silu(LN_gate(G))                 inner LNs: eps 1e-5
 *   out2[b,t] = hidden[b,t] @ wout[t] + bout[t]
 *   y      = norm2(out1 + out2)
 *
 * token_mixer: reshape [B,T,D] to [B,T,T,D/T], swap the two T axes, reshape
 * back.  The backward returns the gradient of sum(dy * y) with respect to x
 * and to every parameter (section "Workload and interfaces": the runner
 * differentiates the complete block with a same-shape upstream gradient).
 *
 * Conventions shared by every entry point:
 *  - All tensors are dense, row-major, in the storage dtype of the config
 *    (float32, bfloat16 or float16) unless stated otherwise.  Arithmetic,
 *    statistics and accumulation are float32 on the device.
 *  - Device pointers are allocated and owned by the caller.  The library never
 *    allocates device memory and never synchronises a stream, except
 *    rmx_check() and the *_sync helpers that say so.
 *  - Every device pointer must be 16-byte aligned.
 *  - Calls enqueue work on `stream` (NULL = the legacy default stream) and
 *    return once it is enqueued.  Errors found on the host (arguments, sizes,
 *    alignment) are returned before anything is enqueued.  A device-side wait
 *    that gave up (RMX_ERR_TIMEOUT) is reported by rmx_check().
 *  - Gradients are overwritten, never accumulated (the page's timed loop
 *    sets gradients to None before every step).
 *  - No C++ exception crosses this boundary.
 */
#ifndef RMX_H
#define RMX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle; identical to cudaStream_t / CUstream. */
typedef struct CUstream_st* rmx_stream;

typedef enum {
  RMX_OK = 0,
  RMX_ERR_INVALID_ARG = 1,   /* bad shape, null pointer, bad dtype           */
  RMX_ERR_UNSUPPORTED = 2,   /* valid block, but outside what the kernels do */
  RMX_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned             */
  RMX_ERR_WORKSPACE = 4,     /* a caller buffer is smaller than required     */
  RMX_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed            */
  RMX_ERR_TIMEOUT = 6        /* a bounded device-side wait gave up           */
} rmx_status;

/* Storage type of every tensor, and the contract of the four per-token
 * contractions:
 *   RMX_F32       float32, contractions in IEEE float32 on the CUDA cores
 *                 (strict: no TF32);
 *   RMX_BF16, RMX_F16  16-bit storage, contractions on the tensor cores with
 *                 float32 accumulation;
 *   RMX_F32_TF32  float32 storage, contractions on the tensor cores with the
 *                 operands read as TF32 (10-bit mantissa; the hardware drops
 *                 the low 13 bits of each float32 operand) and float32
 *                 accumulation -- the page's "--dtype float32 --tf32" option
 *                 (section "Run the benchmark").  Everything outside the
 *                 contractions is float32 as under RMX_F32. */
typedef enum { RMX_F32 = 0, RMX_BF16 = 1, RMX_F16 = 2, RMX_F32_TF32 = 3 } rmx_dtype;

/* Block shape.  x, y, dy, dx are [B,T,D]; H is the FFN width (H = k*D on the
 * page, k in {2,3}).  Requires B >= 0, T >= 1, D >= 1, H >= 1, D % T == 0.
 * B == 0 is an empty batch: the forward does nothing and the backward writes
 * zero gradients. */
typedef struct {
  int B, T, D, H;
  int dtype; /* rmx_dtype */
} rmx_config;

/* Parameters (device pointers, storage dtype), section "Workload and
 * interfaces": w1 [T,D,2H], b1 [T,2H], wout [T,H,D], bout [T,D]; the three
 * outer NezhaLayerNorms' gamma/beta [D]; the inner LayerNorms' weight/bias
 * [H] (lnx_* = norm_x applied to U, lng_* = norm_gate applied to G). */
typedef struct {
  const void *w1, *b1, *wout, *bout;
  const void *gamma0, *beta0, *gamma1, *beta1, *gamma2, *beta2;
  const void *lnx_w, *lnx_b, *lng_w, *lng_b;
} rmx_params;

/* Parameter gradients, same shapes and dtype as rmx_params (device). */
typedef struct {
  void *w1, *b1, *wout, *bout;
  void *gamma0, *beta0, *gamma1, *beta1, *gamma2, *beta2;
  void *lnx_w, *lnx_b, *lng_w, *lng_b;
} rmx_grads;

/* Bytes of the `saved` buffer that rmx_forward fills and rmx_backward reads:
 * out1 [B,T,D], Z [B,T,2H], hidden [B,T,H], s2 = out1 + out2 [B,T,D] in the
 * storage dtype, then ten float32 row statistics (mean and 1/sqrt(var+eps) of
 * norm0, norm1, norm2, LN_x, LN_gate) of length B*T, then forward-only
 * scratch (per-tile partial statistics of Z), then norm1's input
 * s1 = token_mix(norm0(x)) + x [B,T,D] in the storage dtype.  Each segment
 * starts on a 256-byte boundary.
 * Rows whose length is not a multiple of 8 elements (D or H) are processed
 * as zero-padded copies of pitch roundup(D, 8) and roundup(H, 8): the
 * tensors above then have those pitches, and `saved` also holds the padded
 * copies of x, y and every parameter (the backward reuses them).  Under
 * RMX_F32_TF32 it also holds transposed copies of w1 and wout.
 * Returns 0 for an invalid config. */
size_t rmx_saved_bytes(const rmx_config* cfg);

/* Bytes of backward scratch (device, caller-owned, contents undefined between
 * calls); for padded rows it includes the padded copies of dy, dx and every
 * gradient, under RMX_F32_TF32 transposed copies of hidden, ds2, out1 and dZ.
 * Returns 0 for an invalid config. */
size_t rmx_workspace_bytes(const rmx_config* cfg);

/* Forward pass.  x [B,T,D] (device) -> y [B,T,D] (device), filling `saved`
 * (device, >= rmx_saved_bytes) for the backward.  x and y may not alias. */
rmx_status rmx_forward(const rmx_config* cfg, const void* x, const rmx_params* params,
                       void* saved, size_t saved_bytes, void* y, rmx_stream stream);

/* Backward pass for upstream gradient dy [B,T,D] (device).  x must be the
 * same input buffer, unchanged, that was passed to the matching rmx_forward
 * (the backward reads it instead of keeping a copy, as autograd keeps a
 * reference to a LayerNorm input); `saved` is that call's saved buffer and
 * params the same parameters.  Writes dx [B,T,D] and every gradient in
 * `grads` (all 14 must be non-null).  ws: scratch of >= rmx_workspace_bytes.
 * Parameter gradients reduce over the rows that used them: w1, b1, wout,
 * bout over b for each token t; the LayerNorm gammas/betas/weights/biases
 * over all B*T rows.  The reductions run in a fixed order, so repeated calls
 * are bitwise identical. */
rmx_status rmx_backward(const rmx_config* cfg, const void* x, const void* dy, const void* saved,
                        size_t saved_bytes, const rmx_params* params, void* dx,
                        const rmx_grads* grads, void* ws, size_t ws_bytes,
                        rmx_stream stream);

/* Host-memory staging for rmx_step_host.  Host buffers should be pinned
 * (page-locked) for the copies to be asynchronous. */
typedef struct { const void* x; const void* dy; void* y; void* dx; } rmx_host_io;
typedef struct { void* x; void* dy; void* y; void* dx; } rmx_device_io;

/* One end-to-end step from host memory: copies x and dy host->device into
 * `dev` (device, [B,T,D] each), runs rmx_forward and rmx_backward, and copies
 * y and dx device->host.  Parameters and gradients stay on the device.  The
 * copies run on a copy stream the library keeps per device, joined to
 * `stream` by events, so that they overlap the compute: x in four chunks of
 * samples, the forward running on the first half of the samples as soon as
 * their chunks have landed and on the second half after that (every forward
 * result is computed row by row, so it equals rmx_forward's bit for bit),
 * then dy (needed only by the backward); y once the forward is done
 * (during the backward) and dx once it is final (during the weight
 * gradients).  Returns once enqueued; everything the call does is ordered
 * before later work on `stream`, so the caller synchronises `stream` before
 * reading host y/dx.  The overlap needs pinned host buffers. */
rmx_status rmx_step_host(const rmx_config* cfg, const rmx_host_io* host,
                         const rmx_device_io* dev, const rmx_params* params,
                         const rmx_grads* grads, void* saved, size_t saved_bytes,
                         void* ws, size_t ws_bytes, rmx_stream stream);

/* CUDA-graph replay of one whole step (rmx_forward then rmx_backward) on
 * fixed buffers.  rmx_graph_create captures the step's kernel launches, with
 * the arguments given here, into an executable graph (nothing runs yet);
 * rmx_graph_launch replays it on `stream`, which computes exactly what the
 * two calls would (same kernels, same order, same results); the launches keep
 * their programmatic dependencies as graph edges.  Replaying saves the host
 * cost of the launches, which dominates small blocks.  The buffers, shapes
 * and parameter pointers are those of the capture: to change any of them,
 * create a new graph (the values in the buffers may change between replays:
 * new x, dy or parameters).  The library allocates nothing on the device;
 * the handle (host memory) lives until rmx_graph_destroy.  Per-kernel
 * profiling (rmx_profile_enable) does not apply inside a graph. */
typedef struct rmx_graph_st* rmx_graph;
rmx_status rmx_graph_create(const rmx_config* cfg, const void* x, const void* dy, const rmx_params* params,
                            void* saved, size_t saved_bytes, void* y, void* dx, const rmx_grads* grads, void* ws,
                            size_t ws_bytes, rmx_graph* out);
rmx_status rmx_graph_launch(rmx_graph g, rmx_stream stream);
rmx_status rmx_graph_destroy(rmx_graph g);

/* Synchronises `stream`, then reads and clears the library's device error
 * word.  Returns RMX_ERR_TIMEOUT if a bounded wait in a kernel gave up since
 * the last check, RMX_ERR_CUDA if the stream reported an error, else RMX_OK. */
rmx_status rmx_check(rmx_stream stream);

/* Human-readable name of a status code (static string). */
const char* rmx_status_str(rmx_status s);

/* Library version, e.g. 100 for 0.1.0. */
int rmx_version(void);

/* Number of kernel launches this library has enqueued since load (host-side
 * counter, all threads). */
long long rmx_launch_count(void);

/* Per-kernel timing.  When enabled, every launch is bracketed by CUDA events
 * recorded on the launching stream.  rmx_profile_read synchronises on the
 * recorded events, fills up to `cap` entries (name, launches, total ms) and
 * returns how many kernel names were seen; it then resets the counters. */
rmx_status rmx_profile_enable(int on);
int rmx_profile_read(const char** names, long long* launches, double* total_ms, int cap);
/* Restricts the per-kernel timing to launches of the kernel called `name`
 * (a name rmx_profile_read reports); NULL or "" times every launch again.
 * Timing one kernel brackets only its launches with events, so the others
 * run back to back as they do unprofiled.  The name is copied. */
rmx_status rmx_profile_select(const char* name);

/* Test hook (no production use): launches one tiny kernel that waits on an
 * mbarrier that nothing will ever complete, with a limit of `limit_us`
 * microseconds, so that the bounded-wait path can be exercised without a
 * hang.  The timeout is then reported by rmx_check(). */
rmx_status rmx_test_bounded_wait(int limit_us, rmx_stream stream);

/* Test hook: one grouped GEMM of the kind the block uses, without the rest of
 * the block, on device buffers in the config's storage dtype.  kind 0 =
 * forward (C[g] = A[g] @ W[g], A rows strided by G*K, W [G,K,N]);
 * kind 1 = dgrad (C[g] = A[g] @ W[g]^T, W [G,N,K]); kind 2 = wgrad
 * (C[g] = A[g]^T @ Bm[g], A [R,G,M], Bm [R,G,N], C [G,M,N]).  For kinds 0/1
 * A is [M,G,K] and C is [M,G,N].  dtype is an rmx_dtype; RMX_F32_TF32 runs
 * kind 1 on the tensor cores (the other kinds, whose operands are not both
 * K-major, run in strict float32).  Used to check the GEMM engine in
 * isolation. */
rmx_status rmx_test_gemm(int kind, int dtype, int M, int N, int K, int G, const void* A,
                         const void* Bm, void* C, rmx_stream stream);

/* No-allocation variant of the norm2 backward.  The pages have no
 * counterpart: this entry point exists for callers that cannot provide
 * scratch memory -- a host framework that owns all device memory through its
 * own pool and passes a plugin only its inputs and outputs, or a deployment
 * that must keep a fixed memory footprint with no allocation after start-up.
 *
 * Computes, for y = norm2(s2): ds2 [B,T,D] = the gradient w.r.t. s2 for
 * upstream dy [B,T,D], and the gradients dgamma2 [D], dbeta2 [D] (summed over
 * all B*T rows) and dbout [T,D] (summed over b), all in the config's storage
 * dtype -- the same values rmx_backward produces for these tensors.  s2,
 * mean2 and rstd2 are norm2's input and float32 row statistics [B*T] as
 * rmx_forward stores them in its saved buffer (s2 is the fourth tensor,
 * mean2/rstd2 the fifth and sixth statistic vectors).
 *
 * Scratch: the partial sums live in a fixed device array of 16 MiB inside
 * the library, reserved on each GPU when the library is first used there and
 * held until the process exits.  This call allocates nothing.  Shapes whose
 * partial sums (3 * ceil(B/64) * T * D floats) exceed 16 MiB, and B == 0,
 * are rejected (RMX_ERR_UNSUPPORTED / RMX_ERR_INVALID_ARG) before any
 * launch.  The first call on each device looks up the array's device address
 * with the device current; make that first call before any stream capture.
 * Every call uses the same array: calls that overlap on the GPU (on
 * different streams, or from several threads) race and must be serialised
 * by the caller.  Each call writes every scratch value it reads, so nothing
 * carries over from a previous call. */
rmx_status rmx_ln2_backward_noalloc(const rmx_config* cfg, const void* dy, const void* s2,
                                    const float* mean2, const float* rstd2, const void* gamma2,
                                    void* ds2, void* dgamma2, void* dbeta2, void* dbout,
                                    rmx_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* RMX_H */
