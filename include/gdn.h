/*
 * gdn.h -- C ABI of the gated delta rule training kernels (forward with chunk
 * checkpoints, and the reverse-time vector-Jacobian product), for NVIDIA GB300
 * (sm_103a).
 *
 * The operation (mlx issue #4614 "mx.fast.gated_delta_update VJP: wrong gradient
 * w.r.t. g ...", section "Recurrence used for the references"): for every batch row b
 * and value head h, with kv head hk = h / (Hv / Hk), a state S of shape [Dv, Dk]
 * evolves over t = 0 .. T-1 as
 *
 *     S <- g_t * S
 *     S <- S + outer(beta_t * (v_t - S k_t), k_t)
 *     y_t = S q_t
 *
 * starting from S_0 (zeros unless given). The training path (mlx-lm PR #1217 "Add
 * Metal VJP kernel for gated_delta_update", section "What this PR adds") runs the
 * forward once, saving the state at the start of every chunk of C steps, and a
 * reverse sweep that re-runs each chunk from its checkpoint to return the gradients.
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are device pointers to contiguous, row-major arrays,
 *     16-byte aligned, owned by the caller. The library allocates nothing and keeps
 *     no state between calls (gdn_bwd_noalloc's fixed scratch array is the one
 *     exception; see there).
 *   - Layouts: q, k, dq, dk       [B, T, Hk, Dk]
 *              v, y, dy, dv       [B, T, Hv, Dv]
 *              g, beta, dg, dbeta [B, T, Hv]
 *              S0, S_T, dS_T, dS0 [B, Hv, Dv, Dk]      (float32, row index = Dv index)
 *              ckpt               [B, Hv, NC, Dv, Dk]  (float32, NC = ceil(T / C))
 *   - q, k, v, g, beta, dy and every output except the states and checkpoints have
 *     the element type `shape->dtype` (float32 or bfloat16). Arithmetic and state are
 *     float32; outputs are rounded to nearest even.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and the call returns without waiting for it.
 *   - Every argument check runs on the host before anything is enqueued: a call
 *     that returns an error has launched nothing and written nothing.
 *   - Results are bitwise deterministic: no atomics; every reduction (over rows,
 *     over the value heads that share a kv head) runs in a fixed order that depends
 *     only on the problem, not on the grid or the GPU's SM count, and a batch row's
 *     results do not depend on the other rows (B = 8 gives, bit for bit, what eight
 *     B = 1 calls give).
 *   - There is no host fallback: if the GPU cannot run a kernel the call returns
 *     GDN_ERR_CUDA.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_VERSION 2

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

typedef enum {
    GDN_F32 = 0,  /* IEEE float32 */
    GDN_BF16 = 1  /* bfloat16 */
} gdn_dtype;

typedef struct {
    int B, T, Hk, Hv, Dk, Dv; /* batch rows, steps, kv heads, value heads, key dim, value dim */
    int chunk;                /* checkpoint interval C, 1..128; 0 selects 64 */
    int dtype;                /* a gdn_dtype */
} gdn_shape;

/* Return codes. */
enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = -1,       /* NULL shape or required pointer, a size <= 0, bad dtype */
    GDN_ERR_MISALIGNED = -2,        /* a pointer not 16-byte aligned */
    GDN_ERR_UNSUPPORTED_SHAPE = -3, /* Hv % Hk != 0, Dk not in {32,64,96,128,160,192,224,256},
                                       Dv % 4 != 0 or Dv > 4096, chunk outside 1..128,
                                       B or Hv > 65535, or a tensor too large to index */
    GDN_ERR_BUFFER_TOO_SMALL = -4,  /* ckpt_bytes < gdn_ckpt_bytes(shape), or workspace_bytes <
                                       gdn_bwd_workspace_bytes(shape) */
    GDN_ERR_WORKSPACE_TOO_SMALL = GDN_ERR_BUFFER_TOO_SMALL,
    GDN_ERR_CUDA = -5,              /* the CUDA runtime reported an error (see gdn_last_error) */
    GDN_ERR_TIMEOUT = -6,           /* a bounded device-side wait ran out (gdn_device_status) */
    GDN_ERR_SCRATCH_LIMIT = -7      /* gdn_bwd_noalloc: the problem needs more scratch than
                                       GDN_BWD_NOALLOC_SCRATCH_BYTES */
};

/* Bytes of the saved-for-backward buffer `ckpt` that gdn_fwd writes: the chunk-start states
 * (B*Hv*NC*Dv*Dk*4 bytes, rounded up to a multiple of 256) followed by the per-step
 * residuals v_t - u_t (B*T*Hv*Dv*4 bytes). For bf16 inputs with chunk 64, Dk in
 * {64, 128, 192} and Dv a multiple of 64 (up to 256, shared memory permitting) the forward
 * runs in its chunkwise form on the tensor cores, and the buffer continues with that form's
 * per-chunk matrices (33024 + 128 Dk + 2 Dv Dk bytes per chunk and value head, and 256 Dk
 * bytes per chunk and kv head, each part rounded up to 256 bytes; their layout is internal).
 * 0 for an invalid shape. */
GDN_API size_t gdn_ckpt_bytes(const gdn_shape *shape);

/* Bytes of device scratch gdn_bwd needs (fp32 partial sums for the fixed-order
 * reductions, and the states or per-chunk products it re-computes). 0 for an invalid
 * shape. */
GDN_API size_t gdn_bwd_workspace_bytes(const gdn_shape *shape);

/*
 * Forward with checkpoints (or, with ckpt = NULL, without: inference and decode, where no
 * backward follows; a decode step is T = 1 with the carried state passed as S0 and read
 * back from S_T). A decode step with Dk in {64, 128, 192, 256} runs as one streaming pass
 * over the state (every state element read once and written once); for that call, and only
 * that one, S_T may be S0 itself (the state updated in place).
 *   in : q, k, v, g, beta            (dtype)
 *        S0                          (float32, may be NULL: zeros)
 *   out: y                           (dtype)
 *        S_T                         (float32, may be NULL: not written)
 *        ckpt, ckpt_bytes            (float32; ckpt_bytes is the size of the buffer that ckpt
 *                                    points to, at least gdn_ckpt_bytes(shape), else the call
 *                                    returns GDN_ERR_BUFFER_TOO_SMALL before anything is
 *                                    enqueued; 16-byte aligned; ckpt may be NULL: nothing
 *                                    saved, ckpt_bytes ignored):
 *                                    ckpt[b, h, c] = state before step c*C, [B,Hv,NC,Dv,Dk];
 *                                    then, from the next 256-byte boundary, the residuals
 *                                    r[b, t, h, :] = v_t - u_t, u_t = g_t S_{t-1} k_t,
 *                                    [B,T,Hv,Dv] (what the backward re-computes from)
 * Returns GDN_OK or an error code.
 */
GDN_API int gdn_fwd(const gdn_shape *shape, const void *q, const void *k, const void *v,
                    const void *g, const void *beta, const float *S0, void *y, float *S_T,
                    float *ckpt, size_t ckpt_bytes, void *stream);

/*
 * Reverse-time VJP. Gradients of L = <dy, y> + <dS_T, S_T> with respect to q, k, v, g,
 * beta and S0, for the forward defined by the same inputs. The pages print no backward
 * formula; this is the chain rule applied to the recurrence above, in reverse time.
 *   in : q, k, v, g, beta, dy        (dtype)
 *        ckpt, ckpt_bytes            (float32) as written by gdn_fwd for the same inputs,
 *                                    shape and S0; ckpt_bytes is the buffer's size, at least
 *                                    gdn_ckpt_bytes(shape) (else GDN_ERR_BUFFER_TOO_SMALL)
 *        dS_T                        (float32, may be NULL: zeros)
 *   out: dq, dk                      (dtype) summed over the value heads of each kv head,
 *                                    in ascending value-head order
 *        dv, dg, dbeta               (dtype)
 *        dS0                         (float32, may be NULL: not written)
 *   scratch: workspace of at least gdn_bwd_workspace_bytes(shape) bytes (device,
 *            16-byte aligned, owned by the caller); its contents on entry do not matter.
 *            Two calls that overlap on the GPU must not share a workspace.
 * Returns GDN_OK or an error code.
 */
GDN_API int gdn_bwd(const gdn_shape *shape, const void *q, const void *k, const void *v,
                    const void *g, const void *beta, const float *ckpt, size_t ckpt_bytes,
                    const void *dy, const float *dS_T, void *dq, void *dk, void *dv, void *dg,
                    void *dbeta, float *dS0, void *workspace, size_t workspace_bytes,
                    void *stream);

/*
 * Backward without any allocation (no counterpart on the pages: it is a convenience of this
 * library). Same operation, arguments, results and checks as gdn_bwd, but without the
 * workspace arguments: the scratch lives in a fixed array of GDN_BWD_NOALLOC_SCRATCH_BYTES
 * bytes that the library keeps in device memory.
 *
 * Who needs it: callers that may not call cudaMalloc or any other allocator -- for example
 * code hosted inside a runtime that owns all device memory and hands out no allocator,
 * code that must not add device memory after start-up, or code for which the implicit
 * device-wide synchronisation of cudaMalloc/cudaFree is not acceptable. They pass only
 * inputs and outputs.
 *
 * Limits and behaviour:
 *   - The scratch array exists once per GPU that loads the library and stays allocated until
 *     the process exits (a fixed GDN_BWD_NOALLOC_SCRATCH_BYTES per GPU).
 *   - Problems whose gdn_bwd_workspace_bytes(shape) exceeds GDN_BWD_NOALLOC_SCRATCH_BYTES are
 *     rejected with GDN_ERR_SCRATCH_LIMIT before anything is enqueued.
 *   - The first call on a device (with that device current) looks up the array's device
 *     address once (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call on a device uses the same array. Nothing in it has to start at zero (each
 *     scratch value is written before it is read within a call), but two calls that overlap
 *     on the GPU (different streams, or different host threads) race on it: serialise them.
 *   - The work is enqueued on `stream`, which must belong to the current device.
 */
#define GDN_BWD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
GDN_API int gdn_bwd_noalloc(const gdn_shape *shape, const void *q, const void *k, const void *v,
                            const void *g, const void *beta, const float *ckpt, size_t ckpt_bytes,
                            const void *dy, const float *dS_T, void *dq, void *dk, void *dv,
                            void *dg, void *dbeta, float *dS0, void *stream);

/*
 * Sequence-parallel form (mlx-lm PR #1217, "Scope", names prefix scans as later work). The
 * state map of a run of chunks is affine, S -> S M + C (M a Dk x Dk matrix); splitting the
 * sequence into `segments` equal runs of whole chunks, one sweep takes every segment from a zero
 * state to its end state (C) and through its map (M) -- the state alone, none of the other
 * outputs -- then a scan over the segments gives their start states (X_0 = S0, X_s = X_{s-1}
 * M_{s-1} + C_{s-1}), and the segments are swept again from them, now writing y and the saved
 * buffer. The backward runs the reverse sweep from zero end adjoints, the reverse scan (with the
 * transposed maps), then the backward proper. Same results as gdn_fwd / gdn_bwd within the
 * bf16 tolerance; it pays where the plain sweep leaves SMs idle (few heads, long sequences).
 *   shape     bf16, chunk 64, a shape the tensor-core path takes both ways (else
 *             GDN_ERR_UNSUPPORTED_SHAPE), T a multiple of 64 * segments, segments >= 1.
 *   saved     ckpt of gdn_seg_ckpt_bytes(shape, segments) bytes: the saved buffer of the
 *             problem seen as B * segments rows of T / segments steps (view row b * segments
 *             + s is segment s of row b: the chunk-start states of segment s of row b, value
 *             head h, are ckpt[(b * segments + s), h, c] for its chunks c), then the maps
 *             [B * segments][Hv][Dk][Dk] float32 (from a 256-byte boundary) and their
 *             transposes (the same layout, right after them).
 *   scratch   workspace of gdn_seg_workspace_bytes(shape, segments) bytes (device, 16-byte
 *             aligned; contents on entry do not matter): two [B * segments][Hv][Dv][Dk]
 *             float32 arrays, then the backward's workspace of the viewed problem.
 * Other arguments as for gdn_fwd / gdn_bwd (S0, S_T, dS_T, dS0 may be NULL). Returns GDN_OK or an
 * error code; a size query returns 0 for a shape or segment count it does not take.
 */
/* The segment count for a GPU of `sm_count` SMs: the largest power of two P (T a multiple of
 * 64 P) whose sweeps' grid, (Dv / 64) * Hv * B * P CTAs of one SM each, still fits the GPU;
 * 1 (the plain calls) where the plain sweeps already fill it or the shape is not taken.
 * Host logic only. */
GDN_API int gdn_seg_choose(const gdn_shape *shape, int sm_count);
GDN_API size_t gdn_seg_ckpt_bytes(const gdn_shape *shape, int segments);
GDN_API size_t gdn_seg_workspace_bytes(const gdn_shape *shape, int segments);
GDN_API int gdn_fwd_seg(const gdn_shape *shape, int segments, const void *q, const void *k, const void *v,
                        const void *g, const void *beta, const float *S0, void *y, float *S_T, float *ckpt,
                        size_t ckpt_bytes, void *workspace, size_t workspace_bytes, void *stream);
GDN_API int gdn_bwd_seg(const gdn_shape *shape, int segments, const void *q, const void *k, const void *v,
                        const void *g, const void *beta, const float *ckpt, size_t ckpt_bytes, const void *dy,
                        const float *dS_T, void *dq, void *dk, void *dv, void *dg, void *dbeta, float *dS0,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Inference forward on the tensor cores (no backward follows): for a shape the chunkwise forward
 * takes (bf16, chunk 64, Dk in {64, 128, 192}, Dv a multiple of 64; else
 * GDN_ERR_UNSUPPORTED_SHAPE), the forward with its per-chunk products in `workspace`
 * (gdn_infer_workspace_bytes(shape) bytes, device, 16-byte aligned, contents on entry do not
 * matter) and nothing saved: y and S_T as gdn_fwd gives them (the same bits), without the
 * checkpoints, the bf16 states or v - u, so faster. gdn_fwd with ckpt = NULL, which has no
 * workspace, runs the sequential kernels instead (or, for T = 1, the decode step). Returns GDN_OK
 * or an error code; the size query returns 0 for a shape it does not take.
 */
GDN_API size_t gdn_infer_workspace_bytes(const gdn_shape *shape);
GDN_API int gdn_fwd_infer(const gdn_shape *shape, const void *q, const void *k, const void *v, const void *g,
                          const void *beta, const float *S0, void *y, float *S_T, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Re-computation mode (mlx-lm PR #1217, "What this PR adds": checkpoints on fixed-size chunks,
 * the forward recomputed within each chunk during the reverse sweep). For a shape the
 * chunkwise tensor-core kernels take both ways (bf16, chunk 64; else
 * GDN_ERR_UNSUPPORTED_SHAPE), the saved buffer holds only what the method saves -- the fp32
 * chunk-start states and the residuals v_t - u_t, the layout gdn_fwd describes, without the
 * chunkwise form's per-chunk products -- and gdn_bwd_rc forms those products again from q, k,
 * g, beta (and the checkpoints' bf16 operand copies) before its reverse sweep. Results equal
 * those of gdn_fwd / gdn_bwd bit for bit.
 *   ckpt       gdn_rc_ckpt_bytes(shape) bytes: [B,Hv,NC,Dv,Dk] fp32 states, then from the next
 *              256-byte boundary [B,T,Hv,Dv] fp32 residuals.
 *   workspace  gdn_rc_fwd_workspace_bytes / gdn_rc_bwd_workspace_bytes bytes (device, 16-byte
 *              aligned, contents on entry do not matter): the per-chunk products, and for the
 *              backward then its own workspace. Two calls that overlap on the GPU must not
 *              share one.
 * Other arguments as for gdn_fwd / gdn_bwd (S0, S_T, dS_T, dS0 may be NULL). Returns GDN_OK or an
 * error code; a size query returns 0 for a shape it does not take.
 */
GDN_API size_t gdn_rc_ckpt_bytes(const gdn_shape *shape);
GDN_API size_t gdn_rc_fwd_workspace_bytes(const gdn_shape *shape);
GDN_API size_t gdn_rc_bwd_workspace_bytes(const gdn_shape *shape);
GDN_API int gdn_fwd_rc(const gdn_shape *shape, const void *q, const void *k, const void *v, const void *g,
                       const void *beta, const float *S0, void *y, float *S_T, float *ckpt, size_t ckpt_bytes,
                       void *workspace, size_t workspace_bytes, void *stream);
GDN_API int gdn_bwd_rc(const gdn_shape *shape, const void *q, const void *k, const void *v, const void *g,
                       const void *beta, const float *ckpt, size_t ckpt_bytes, const void *dy, const float *dS_T,
                       void *dq, void *dk, void *dv, void *dg, void *dbeta, float *dS0, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Gates of the layer: the decay g and write strength beta from its raw gate inputs, and the
 * VJP back to them (mlx-lm PR #1217, "Correctness", trains through q, k, v, a, b, A_log,
 * dt_bias and the state; no page prints the gate map, and the one taken is the public
 * mlx-lm Qwen3-Next / Qwen3.5 linear-attention layer's). For every b, t and value head h:
 *     log g = -exp(A_log[h]) * softplus(a[b,t,h] + dt_bias[h]),  g = exp(log g)
 *     beta  = sigmoid(b[b,t,h])
 * The VJP goes through log g (d log g = g dg), with da, db elementwise and dA_log[h],
 * ddt_bias[h] summed over all b, t in a fixed order (deterministic).
 *   a, b, g, beta, dg, dbeta, da, db   [B, T, Hv]  (dtype)
 *   A_log, dt_bias, dA_log, ddt_bias   [Hv]        (float32)
 * The shape is the layer's (the same as for gdn_fwd; Hk, Dk, Dv are checked but unused).
 * All pointers are device pointers, 16-byte aligned, owned by the caller. The arithmetic is
 * fp32 (the parameter sums fp64). Returns GDN_OK or an error code (checks as for gdn_fwd;
 * B*T above 2^31-1 is GDN_ERR_UNSUPPORTED_SHAPE).
 */
GDN_API int gdn_gates_fwd(const gdn_shape *shape, const void *a, const void *b, const float *A_log,
                          const float *dt_bias, void *g, void *beta, void *stream);
GDN_API int gdn_gates_bwd(const gdn_shape *shape, const void *a, const void *b, const float *A_log,
                          const float *dt_bias, const void *dg, const void *dbeta, void *da,
                          void *db, float *dA_log, float *ddt_bias, void *stream);

/* Static description of a return code. */
GDN_API const char *gdn_strerror(int code);

/* Text of the last CUDA error seen by a gdn_* call on this host thread ("" if none). */
GDN_API const char *gdn_last_error(void);

/* Reads and clears the status word of the current device. Kernels never spin without a
 * bound: a wait inside a kernel that runs out records GDN_ERR_TIMEOUT here and the kernel
 * stops early (its outputs are then incomplete). Returns GDN_OK, GDN_ERR_TIMEOUT, or
 * GDN_ERR_CUDA if the word cannot be read. Synchronises with the device. */
GDN_API int gdn_device_status(void);

/* GDN_VERSION of the library that was loaded. */
GDN_API int gdn_version(void);

/* Per-kernel timing, a diagnostic (off by default). While it is on, every kernel that
 * gdn_fwd, gdn_bwd and the gate calls launch is bracketed by two CUDA events recorded on
 * the caller's stream, so the times are device times of each kernel on that stream. */
typedef struct gdn_kernel_time {
    char name[48];   /* kernel family, e.g. "chunk_grad" */
    int launches;    /* launches recorded since the last read */
    double ms;       /* their summed device time in milliseconds */
} gdn_kernel_time;

/* Turns per-kernel timing on (on != 0) or off; turning it off drops what was recorded.
 * Returns GDN_OK. */
GDN_API int gdn_timing_enable(int on);

/* Waits for the recorded events (host-side wait), writes up to max_entries entries (one
 * per kernel family, in order of first launch) to out, and clears the record. Returns the
 * number of families recorded (which may exceed max_entries; out may then be NULL with
 * max_entries 0), or GDN_ERR_CUDA. */
GDN_API int gdn_timing_read(gdn_kernel_time *out, int max_entries);

/* ---- Diagnostics (no counterpart on the pages). */

/* Exercises the timeout path of the library's bounded device-side waits without faulting or
 * hanging anything: enqueues on `stream` one CTA that allocates tensor memory, arms an mbarrier
 * for bytes that no copy will ever deliver (so nothing is in flight), polls it `polls` times
 * (1 .. 2^24), records GDN_ERR_TIMEOUT in the device status word (gdn_device_status), frees its
 * tensor memory and exits, exactly as a kernel of the library does when a wait runs out. The
 * GPU context stays usable. Returns GDN_OK (launched), GDN_ERR_INVALID_ARG (polls out of range)
 * or GDN_ERR_CUDA. */
GDN_API int gdn_debug_wait_probe(unsigned polls, void *stream);

/* Measured FP32 fused multiply-add rate of the current device in TFLOP/s (2 flops per FMA and
 * lane): scalar FFMA (packed = 0) or the packed two-lane f32x2 form (packed = 1) that the
 * sequential kernels use, from independent chains whose only distinct register operand is
 * the accumulator, on 8 CTAs of 256 threads per SM, best of three timed launches on a
 * private stream. Synchronises with that stream. Returns GDN_OK or GDN_ERR_CUDA. */
GDN_API int gdn_diag_fma_tflops(int packed, double *tflops);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
