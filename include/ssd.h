/*
 * libssd -- forward Mamba-2 SSD (structured state-space duality) scan on one
 * NVIDIA GB300 (sm_103a).  Plain C ABI: host or device pointers, sizes and a
 * CUDA stream handle; no framework types.
 *
 * The operation (per batch row b and head h, for t = 0 .. L-1):
 *
 *   dt_t  = softplus(dt_raw[b,t,h] + dt_bias[h])
 *   A_h   = -exp(A_log[h])                        A_log stores log(-A)
 *   h_t   = exp(dt_t * A_h) * h_{t-1} + dt_t * B[b,t,g] x[b,t,h]^T      (N x P)
 *   y[b,t,h] = C[b,t,g]^T h_t + D[h] * x[b,t,h]
 *
 * with g = h * G / H (contiguous blocks of H/G heads share a group) and h_{-1}
 * the initial state (zero when none is given).  Defined by the SSD module of
 * @seanhogg/builderforce-memory-engine 2026.6.18 (package/dist/kernels/
 * ssd.js and ssd.d.ts, module header: scalar decay per head, MIMO state per
 * head, chunked evaluation with a carried state, buffer layouts), taken with
 * A = -exp(A_log), input term dt * B x^T and a readout per channel p.  The
 * chunked evaluation (chunks of Q steps, chunk states passed from chunk to
 * chunk) follows the chunked-scan structure of mamba-rs 0.2.1
 * src/mamba3_siso/gpu/mamba3_gpu.rs (parallel branch of the forward layer:
 * decay cumsum, chunk state, state passing, chunk scan) applied to the
 * Mamba-2 recurrence above.
 *
 * Layouts: row-major and contiguous.
 *   x, y                   [B, L, H, P]   dtype (bf16 or fp32)
 *   dt_raw                 [B, L, H]      fp32
 *   B, C                   [B, L, G, N]   dtype
 *   dt_bias, A_log, D      [H]            fp32
 *   init_state, final_state [B, H, P, N]  fp32 (state stored P-major, N-minor)
 */
#ifndef LIBSSD_SSD_H
#define LIBSSD_SSD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_ABI_VERSION 2

typedef enum ssd_dtype {
    SSD_DTYPE_F32 = 0,   /* x, B, C, y are fp32 */
    SSD_DTYPE_BF16 = 1   /* x, B, C, y are bf16; arithmetic accumulates in fp32 */
} ssd_dtype_t;

typedef enum ssd_status {
    SSD_OK = 0,
    SSD_ERR_INVALID_DIMS = 1,   /* a size is negative/zero where it may not be, H % G != 0, overflow */
    SSD_ERR_NULL_PTR = 2,       /* a required pointer is NULL */
    SSD_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned */
    SSD_ERR_UNSUPPORTED = 4,    /* shape or requested path not supported */
    SSD_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed; nothing further enqueued */
    SSD_ERR_TIMEOUT = 6,        /* a kernel gave up a bounded wait (read via ssd_get_device_error) */
    SSD_ERR_ALIASING = 7,       /* y overlaps an input, or the two states overlap partially */
    SSD_ERR_SCRATCH_LIMIT = 8,  /* the scratch needed exceeds the buffer the call may use (the fixed
                                   array of ssd_scan_fwd_noalloc, the workspace of ssd_scan_fwd_ws) */
    SSD_ERR_UNSUPPORTED_DTYPE = 9   /* dims->dtype is not an ssd_dtype_t, or the path requested (or,
                                       for ssd_scan_fwd_noalloc, the only path it has) does not take it:
                                       the chunked tcgen05 path takes bf16 only */
} ssd_status_t;

/* Kernel path selection, in ssd_dims_t.flags (low 4 bits). */
#define SSD_PATH_AUTO 0u        /* decode step for seqlen 1, else the chunked tensor-core path where
                                   supported, else sequential */
#define SSD_PATH_SEQUENTIAL 1u  /* direct recurrence, fp32 FFMA (any P, N up to 2048; fp32 or bf16) */
#define SSD_PATH_CHUNKED 2u     /* chunked tcgen05 path: bf16, P = 64, N = 128, Q % 64 == 0, (H/G) even */
#define SSD_PATH_DECODE 3u      /* one step (seqlen 1), fp32 FFMA: any P, N % 4 == 0 and N <= 512; fp32 or
                                   bf16.  SSD_PATH_AUTO takes it whenever seqlen == 1 and it applies */
#define SSD_PATH_MASK 0xFu
/* Diagnostic, in ssd_dims_t.flags: on the chunked path, the first unit of every
 * chain waits for a state handoff that nothing publishes, with the bounded waits
 * shortened to 20 ms.  The launch then records SSD_ERR_TIMEOUT (read with
 * ssd_get_device_error), stops every warp, drains its own copies and MMAs and
 * returns; y and final_state are undefined.  It exercises the failure path
 * without faulting the GPU.  Ignored by the sequential path. */
#define SSD_DIAG_STALL_HANDOFF 0x100u
/* In ssd_dims_t.flags of ssd_scan_bwd only: run the chunk form's fp32
 * contractions even where its tensor-core gradient pass applies (bf16 inputs,
 * P = 64, N = 128).  The tensor-core pass rounds the masked decay products
 * and the chunk states to bf16 operands; the fp32 form does not. */
#define SSD_BWD_FP32_FORM 0x200u
/* In ssd_dims_t.flags of ssd_scan_bwd only: where the tensor-core form applies,
 * compute the chunk states and link them in two launches (every chunk at once,
 * then the chains) rather than in one launch that walks each (b, h) through its
 * chunks with the running state in TMEM.  The library takes the one-launch walk
 * when 2 B H fills the GPU's SMs or the sequence has at most 8 chunks of 64
 * steps.  Both give the same chunk states up to the order of fp32 additions. */
#define SSD_BWD_SPLIT_STATES 0x400u

/* Schedules of the chunked path (see ssd_chunk_schedule).  One may be requested
 * in ssd_dims_t.flags as (SSD_SCHEDULE_x << SSD_SCHEDULE_SHIFT); 0 there lets
 * the library choose.  A split request for a sequence of a single chunk runs
 * the range schedule (there is nothing to split).  Ignored by the sequential
 * path. */
#define SSD_SCHEDULE_NONE 0
#define SSD_SCHEDULE_RANGES 1
#define SSD_SCHEDULE_PIECES 2
#define SSD_SCHEDULE_SPLIT 3
#define SSD_SCHEDULE_SHIFT 4
#define SSD_SCHEDULE_REQUEST_MASK 0x30u

typedef struct ssd_dims {
    int64_t batch;     /* B >= 0 */
    int64_t seqlen;    /* L >= 0; need not be a multiple of chunk (ragged last chunk) */
    int32_t nheads;    /* H >= 1 */
    int32_t headdim;   /* P >= 1 */
    int32_t dstate;    /* N >= 1 */
    int32_t ngroups;   /* G >= 1, H % G == 0 */
    int32_t chunk;     /* Q >= 1: chunk length of the chunked evaluation (ignored by the sequential path) */
    int32_t dtype;     /* ssd_dtype_t of x, B, C and y */
    uint32_t flags;    /* SSD_PATH_* | optional schedule request | optional SSD_DIAG_STALL_HANDOFF */
    uint32_t reserved; /* must be 0 */
} ssd_dims_t;

/*
 * ssd_scan_fwd -- the forward scan on device memory.
 *
 * All array arguments are DEVICE pointers of the current device, owned by the
 * caller, contiguous in the layouts above and 16-byte aligned.  init_state may
 * be NULL (zero initial state); final_state may be NULL (not returned).
 * init_state and final_state may be the same pointer (in-place state update)
 * but must not overlap otherwise; y must not overlap any input.
 * `stream` is a cudaStream_t (NULL = legacy default stream).  The call only
 * enqueues work on `stream`: it never synchronises, and returns before the
 * results are ready.  Scratch memory (chunk-handoff flags, and chunk states
 * when final_state is NULL) is taken stream-ordered from a library-owned
 * memory pool and released stream-ordered after the kernel.
 * Errors: returns a status; on any status other than SSD_OK nothing was
 * enqueued, except SSD_ERR_CUDA raised by a launch itself.  A kernel that
 * exceeds a bounded wait (about 2 s) records SSD_ERR_TIMEOUT in a device
 * error word, stops, and leaves y undefined; read it with
 * ssd_get_device_error.
 */
ssd_status_t ssd_scan_fwd(const void *x, const float *dt_raw, const float *dt_bias,
                          const float *A_log, const void *B, const void *C, const float *D,
                          const float *init_state, void *y, float *final_state,
                          const ssd_dims_t *dims, void *stream);

/*
 * ssd_scan_fwd_host -- the same scan on HOST buffers (end-to-end use).
 *
 * Arguments as ssd_scan_fwd but every array is a host pointer (pinned memory
 * gives asynchronous copies; pageable works).  The call allocates device
 * buffers stream-ordered, copies the inputs in, runs the scan, copies y (and
 * final_state when non-NULL) back, releases the buffers, and synchronises
 * `stream` before returning, so the host outputs are ready on SSD_OK.
 * Calls of 32 MiB or more with several batch rows run in up to 8 pieces of
 * whole rows through three library-owned streams (copies in, scan, copies
 * out), ordered after and joined back into `stream` by events, so that the
 * two copy directions and the scan overlap.  Every piece takes the schedule
 * the whole batch would, and the results are bitwise those of ssd_scan_fwd.
 */
ssd_status_t ssd_scan_fwd_host(const void *x, const float *dt_raw, const float *dt_bias,
                               const float *A_log, const void *B, const void *C,
                               const float *D, const float *init_state, void *y,
                               float *final_state, const ssd_dims_t *dims, void *stream);

/*
 * ssd_scan_fwd_workspace_size -- bytes of scratch that ssd_scan_fwd_ws needs for
 * these dims on the current device, in *bytes (0 when the call needs none:
 * empty work or the sequential path).  The chunked path's scratch holds the
 * chunk-unit handoff flags and, when a chain is split into several units,
 * the handed-over states (the inter-chunk state passing of the chunked
 * evaluation; @seanhogg/builderforce-memory-engine, dist/kernels/ssd.js, module
 * header: chunked evaluation with a carried state).  The schedule, and so the
 * size, depends on the device's SM count.  Host only; launches nothing.
 * Returns SSD_OK, or an error for invalid or unsupported dims (as
 * ssd_select_path), or SSD_ERR_NULL_PTR.
 */
ssd_status_t ssd_scan_fwd_workspace_size(const ssd_dims_t *dims, uint64_t *bytes);

/*
 * ssd_scan_fwd_ws -- ssd_scan_fwd with caller-provided scratch.
 *
 * Arguments as ssd_scan_fwd, plus `workspace`: a DEVICE buffer of
 * `workspace_bytes` bytes, owned by the caller, 16-byte aligned, overlapping
 * no other argument.  It must hold ssd_scan_fwd_workspace_size(dims) bytes
 * (it may be NULL when that is 0); its contents on entry do not matter and
 * are undefined afterwards.  The call allocates nothing.  Two calls whose
 * kernels may overlap in time must not share a workspace.
 * Errors as ssd_scan_fwd, plus SSD_ERR_SCRATCH_LIMIT when workspace_bytes is
 * smaller than needed (nothing enqueued); a misaligned or overlapping
 * workspace gives SSD_ERR_MISALIGNED or SSD_ERR_ALIASING before any CUDA call.
 */
ssd_status_t ssd_scan_fwd_ws(const void *x, const float *dt_raw, const float *dt_bias,
                             const float *A_log, const void *B, const void *C, const float *D,
                             const float *init_state, void *y, float *final_state,
                             void *workspace, uint64_t workspace_bytes, const ssd_dims_t *dims,
                             void *stream);

/*
 * ssd_scan_fwd_noalloc -- ssd_scan_fwd on the chunked path without any
 * device-memory allocation.
 *
 * No counterpart in the paper: an engineering variant for callers that cannot
 * let a library allocate device memory during a call (a process that reserves
 * the device up front in an arena of its own, or a driver or virtualised
 * device without stream-ordered memory pools).
 *
 * Arguments, layouts and ownership as ssd_scan_fwd.  Runs the same chunked
 * tcgen05 kernel with its scratch in a fixed 32 MiB array that the library
 * module holds per device.  The array's device address is looked up on the
 * first call on a device, with that device current, and again after the
 * device's context has changed (cudaDeviceReset); make that first call before
 * any stream capture.  The call calls no allocator.
 * Errors as ssd_scan_fwd, plus:
 *   SSD_ERR_UNSUPPORTED    the chunked path does not support these dims, or
 *                          dims->flags requests a path other than
 *                          SSD_PATH_AUTO or SSD_PATH_CHUNKED (the sequential
 *                          and decode paths need no scratch: call ssd_scan_fwd),
 *                          or requests SSD_SCHEDULE_SPLIT;
 *   SSD_ERR_UNSUPPORTED_DTYPE  dims->dtype is not bf16;
 *   SSD_ERR_SCRATCH_LIMIT  the kernel would need more than 32 MiB of scratch;
 *                          nothing is enqueued.  The call never takes
 *                          SSD_SCHEDULE_SPLIT, and takes SSD_SCHEDULE_PIECES
 *                          (one 64 KiB state slot and 64 B of flags per SM)
 *                          wherever the schedule ssd_scan_fwd would take needs
 *                          more than the array, so only a device of more than
 *                          about 500 SMs gets this error;
 *   SSD_ERR_CUDA           the array's address could not be obtained.
 * Concurrency: the array is shared by all calls on a device.  Calls whose
 * kernels may overlap in time on one device (different streams, or threads
 * without ordering between them) race on it and give wrong results or time
 * out; calls ordered on one stream are safe.
 */
ssd_status_t ssd_scan_fwd_noalloc(const void *x, const float *dt_raw, const float *dt_bias,
                                  const float *A_log, const void *B, const void *C,
                                  const float *D, const float *init_state, void *y,
                                  float *final_state, const ssd_dims_t *dims, void *stream);

/*
 * ssd_trap_scan_fwd -- the trapezoidal (Mamba-3 SISO) scan, forward.
 *
 * The Mamba-3 SISO GPU forward of the pages (mamba-rs 0.2.1,
 * mamba3_siso/gpu/mamba3_gpu.rs) replaces the exponential recurrence by a
 * trapezoidal one in three coefficients and keeps the last step's k and v as
 * extra carried state (module header of its forward pass; step F5b:
 * alpha = exp(a dt), beta = alpha dt (1 - trap), gamma = trap dt).  Per batch row b and head h, with v = x, k = B, q = C of
 * the head's group g = h / (H/G):
 *   h_t = alpha_t h_{t-1} + beta_t k_{t-1} v_{t-1}^T + gamma_t k_t v_t^T
 *   y_t = q_t^T h_t + D_h v_t
 * where k_{-1}, v_{-1} are the carried k_state and v_state.  The pages print
 * the coefficients and the k/v states but not the recurrence; the form above
 * is the reading they support.  The coefficient step is fused: the call takes
 * dt, a and trap per token.
 *
 * Arguments are DEVICE pointers of the current device, owned by the caller,
 * contiguous, 16-byte aligned; dims as for ssd_scan_fwd (dtype: x, B, C, y
 * and the k/v states).  flags: a path and, for the chunked kernel, a schedule
 * request as for ssd_scan_fwd.  SSD_PATH_CHUNKED is the chunked tcgen05 kernel
 * in a trapezoidal mode (same limits and schedules as for ssd_scan_fwd: bf16,
 * P = 64, N = 128, chunk % 64 == 0, (H/G) even; scratch from the library pool;
 * one more small launch writes k_final / v_final).  The mode evaluates the
 * recurrence on the shifted state h~_t = h_t + (beta_{t+1}/alpha_{t+1})
 * k_t v_t^T, which is linear with decay alpha_t, so the split schedule applies
 * unchanged; its first pass starts each chain from h0 + dt_0 (1 - trap_0)
 * k0 v0^T.  SSD_PATH_SEQUENTIAL is a
 * sequential kernel (fp32 arithmetic).  SSD_PATH_AUTO takes the chunked kernel
 * where it applies and seqlen > 1, else the sequential one.
 *   v     [B,L,H,P]   k, q [B,L,G,N]   (dtype)
 *   dt, a, trap [B,L,H] fp32: step size (> 0), per-token decay rate (a <= 0 for
 *                       a decaying state), mixing weight in [0, 1]
 *   D [H] fp32
 *   h0, h_final [B,H,P,N] fp32; k0, k_final [B,H,N] (dtype); v0, v_final
 *                       [B,H,P] (dtype).  Inputs may be NULL (zero), outputs
 *                       NULL (not written).  Each output may be the same
 *                       pointer as its input (in place) but must not
 *                       overlap anything else.  k_final[b,h] = k[b,L-1,g] and
 *                       v_final[b,h] = v[b,L-1,h]: the next call continues
 *                       from (h_final, k_final, v_final).
 *   y [B,L,H,P] (dtype), overlapping no input.
 * The sequential kernel supports N % 4 == 0, N <= 512; P <= 128 for
 * N <= 128, P <= 64 for N <= 256, P <= 32 for N <= 512; fp32 or bf16.
 * Returns SSD_OK, or an error as ssd_scan_fwd (SSD_ERR_INVALID_DIMS also for
 * flags other than a path or a schedule request; SSD_ERR_UNSUPPORTED for
 * another path or an unsupported shape); nothing is enqueued on error.
 * seqlen 0 passes the states through.  Enqueues on `stream` only; never
 * synchronises.
 */
ssd_status_t ssd_trap_scan_fwd(const void *v, const void *k, const void *q, const float *dt,
                               const float *a, const float *trap, const float *D,
                               const float *h0, const void *k0, const void *v0, void *y,
                               float *h_final, void *k_final, void *v_final,
                               const ssd_dims_t *dims, void *stream);

/*
 * ssd_conv1d_silu_fwd -- the causal depthwise conv1d + SiLU that precedes the
 * scan in the Mamba blocks of the pages (the builderforce Mamba2Block runs one
 * causal conv1d over the fused x, B and C projection channels; the conv1d
 * kernel page: y[b,t,d] = sum_k weight[d,k] x[b,t-k,d] + bias[d], zero before
 * the sequence; the mamba-rs 0.4.0 S6 forward applies SiLU in the same
 * kernel as the conv and carries the conv state from call to call).  Over
 * the fused channels c of xbc = [x (H*P) | B (G*N) | C (G*N)]:
 *   u[b,t,c] = SiLU(bias[c] + sum_{k<K} weight[c,k] xbc[b,t-k,c])
 * with xbc before t = 0 taken from conv_state (zero when NULL), and u written
 * split into the scan's x [B,L,H,P], B and C [B,L,G,N].
 *   xbc [B,L,C], conv_state and conv_state_out [B,K-1,C] (oldest step
 *     first) in dims->dtype; weight [C,K] and bias [C] (NULL: none) fp32.
 *   conv_state_out (NULL: not written) receives the last K-1 inputs, from
 *     which a following call continues; it must not overlap conv_state.
 * DEVICE pointers, 16-byte aligned, caller-owned; outputs overlap no input.
 * dims: batch, seqlen, nheads, headdim, dstate, ngroups, dtype as for
 * ssd_scan_fwd; chunk is ignored (>= 1); flags must be 0.  Supported:
 * kernel_size 2..4, H*P and G*N multiples of 8, batch <= 65535.  Errors as
 * ssd_scan_fwd (SSD_ERR_UNSUPPORTED for an unsupported size).  seqlen 0
 * passes the conv state through.  Enqueues on `stream` only.
 */
ssd_status_t ssd_conv1d_silu_fwd(const void *xbc, const float *weight, const float *bias,
                                 const void *conv_state, void *x, void *B, void *C,
                                 void *conv_state_out, int32_t kernel_size,
                                 const ssd_dims_t *dims, void *stream);

/*
 * ssd_conv_scan_fwd -- ssd_conv1d_silu_fwd followed by ssd_scan_fwd, in one call,
 * with the conv of the x channels done inside the chunked scan kernel (the
 * builderforce Mamba2Block runs the causal conv1d over the fused x, B, C
 * projection channels, then the SSD module, on one layer's buffers; the mamba-rs
 * 0.4.0 S6 forward carries the conv state between calls).  The scan reads the
 * raw x channels of xbc and applies the conv and SiLU to each tile in shared
 * memory, so the conv's x never goes through device memory; the B and C
 * channels (shared by every head of a group) are convolved once by a small
 * kernel beforehand.
 *   u = SiLU(conv(xbc)) split into x [B,L,H,P], B and C [B,L,G,N] as
 *   ssd_conv1d_silu_fwd defines it; then y, final_state as ssd_scan_fwd
 *   defines them for (x, dt_raw, dt_bias, A_log, B, C, D, init_state).
 * xbc [B,L,H*P + 2*G*N], conv_state and conv_state_out [B,K-1,H*P + 2*G*N]
 * (bf16); conv_weight [H*P + 2*G*N, K] and conv_bias (NULL: none) fp32;
 * kernel_size K in 2..4; the scan's arguments as for ssd_scan_fwd.  Nullable:
 * conv_bias, conv_state (zero), init_state (zero), final_state and
 * conv_state_out (not written).  DEVICE pointers of the current device,
 * caller-owned, 16-byte aligned; outputs overlap no input and each other
 * (conv_state_out must not overlap conv_state).
 * Supported: the chunked path's shapes (bf16, P = 64, N = 128, chunk % 64 == 0,
 * (H/G) even; GB300-class device); flags: SSD_PATH_AUTO or SSD_PATH_CHUNKED,
 * optionally a schedule request.  Scratch (the convolved B and C, and the
 * chunked path's) comes stream-ordered from the library pool.  Errors as
 * ssd_scan_fwd; SSD_ERR_UNSUPPORTED_DTYPE for fp32.  seqlen 0 passes both
 * states through.  Enqueues on `stream` only; never synchronises.
 */
ssd_status_t ssd_conv_scan_fwd(const void *xbc, const float *conv_weight, const float *conv_bias,
                               const void *conv_state, int32_t kernel_size, const float *dt_raw,
                               const float *dt_bias, const float *A_log, const float *D,
                               const float *init_state, void *y, float *final_state,
                               void *conv_state_out, const ssd_dims_t *dims, void *stream);

/*
 * ssd_gated_rmsnorm_fwd -- the gated output norm after the scan (the Mamba-3
 * forward of the pages, step F7 with its norm: RMSNorm(y) * weight * SiLU(z)),
 * per token over its H*P channels:
 *   out = y / sqrt(mean_c(y^2) + eps) * weight * SiLU(z)
 *   y, z, out [B,L,H,P] (dims->dtype); weight [H*P] fp32; eps >= 0.
 * DEVICE pointers, 16-byte aligned, caller-owned; out overlaps no input.
 * dims as for ssd_conv1d_silu_fwd (dstate, ngroups, chunk ignored beyond their
 * validation).  Supported: H*P a multiple of 8, at most 16384.  Errors as
 * ssd_scan_fwd.
 */
ssd_status_t ssd_gated_rmsnorm_fwd(const void *y, const void *z, const float *weight, float eps,
                                   void *out, const ssd_dims_t *dims, void *stream);

/*
 * ssd_complex_scan_fwd -- the complex-valued scan with exponential-trapezoidal
 * (ET) discretisation: the Mamba-3 complex SSD module of the pages, as its
 * header defines it (complex_ssd.ts).  Per batch row and head, with
 * A = exp(log|A| + i arg A) and dt_t = softplus(dt_raw_t + dt_bias):
 *   A_bar_t = exp(dt_t A),  B_bar_t = (A_bar_t - 1) A^-1 B_t  (the exact hold)
 *   h_t = A_bar_t h_{t-1} + B_bar_t x_t^T,  y_t = Re(C_t^T h_t) + D x_t
 * (The page's printed kernel exponentiates dt (log|A| + i arg A) and reads out
 * Re(conj(C) h); its header's statement is the one implemented.)
 * x, y [B,L,H,P] and B, C [B,L,G,N] in dims->dtype; B and C hold N/2 complex
 * numbers as (re, im) pairs along N; A_polar [H,2] fp32 = (log|A|, arg A);
 * dt_raw [B,L,H], dt_bias, D [H] fp32; init_state (NULL: zero) and
 * final_state (NULL: not written) [B,H,P,N] fp32, complex as (re, im) pairs
 * along N; final_state may be init_state (in place).  DEVICE pointers, 16-byte
 * aligned; y overlaps no input.  flags: SSD_PATH_SEQUENTIAL (one sequential
 * kernel; seqlen 1 is a decode step), SSD_PATH_CHUNKED (the chunk form on the
 * tensor cores: chunks of 64 steps, two batch rows per CTA, bf16 operands and
 * fp32 accumulation; bf16 with P = 64, N = 128 and seqlen >= 2 only, else
 * SSD_ERR_UNSUPPORTED) or SSD_PATH_AUTO (the chunk form where it applies, else
 * the sequential kernel).  The sequential kernel supports N % 4 == 0,
 * N <= 512; P <= 128 for N <= 128, P <= 64 for N <= 256, P <= 32 for
 * N <= 512; fp32 or bf16.  seqlen 0 copies the state through.  Errors as
 * ssd_scan_fwd.
 */
ssd_status_t ssd_complex_scan_fwd(const void *x, const float *dt_raw, const float *dt_bias,
                                  const float *A_polar, const void *B, const void *C, const float *D,
                                  const float *init_state, void *y, float *final_state,
                                  const ssd_dims_t *dims, void *stream);

/*
 * ssd_scan_bwd -- the backward of ssd_scan_fwd: the gradients of a loss with
 * respect to every input, given dy = dL/dy and d_final = dL/d final_state.
 * They are the derivatives of the recurrence ssd_scan_fwd evaluates (the
 * SSD module's forward, direct form).  The gradient of the state runs in
 * reverse:
 *   G_{L-1} = d_final + C_{L-1} dy_{L-1}^T,  G_t = dA_{t+1} G_{t+1} + C_t dy_t^T
 *   dx_t = D dy_t + dt_t G_t^T B_t,  dB_t = dt_t G_t x_t,  dC_t = h_t dy_t
 *   ddt_raw_t = sigmoid(dt_raw_t + dt_bias) sum G_t o (a dA_t h_{t-1} + B_t x_t^T)
 *   dA_log = a sum_t sum G_t o (dt_t dA_t h_{t-1}),  dD = sum_t dy_t . x_t,
 *   d_init = dA_0 G_0
 * with dB, dC summed over the heads of each group and the per-head gradients
 * over batch rows and steps, in a fixed order (deterministic).
 * Inputs as ssd_scan_fwd, plus dy [B,L,H,P] (dims->dtype) and d_final
 * [B,H,P,N] fp32 (NULL: zero).  Outputs, all fp32, caller-owned, overlapping
 * no input and each other: dx [B,L,H,P], ddt_raw [B,L,H], ddt_bias [H],
 * dA_log [H], dB and dC [B,L,G,N], dD [H], d_init [B,H,P,N] (NULL: not
 * written).  DEVICE pointers, 16-byte aligned.  flags: a path, plus
 * SSD_BWD_FP32_FORM and SSD_BWD_SPLIT_STATES (above).
 * SSD_PATH_CHUNKED: the chunk form (chunks of 64 steps in parallel: local
 * chunk states and state gradients, a pass over the chunks that links them,
 * then every gradient of a chunk as dense contractions); supported for
 * P <= 64, N <= 128, B*H <= 65535.  For bf16 with P = 64 and N = 128 its
 * contractions run on the tensor cores (bf16 operands, fp32 accumulation;
 * the chunk states enter as two bf16 terms), and the chunk states and their
 * links may be computed in one walk per (b, h) (SSD_BWD_SPLIT_STATES);
 * otherwise, or with SSD_BWD_FP32_FORM, as fp32 FFMA.  SSD_PATH_SEQUENTIAL: one sequential
 * kernel per (b, h) that recomputes the forward states segment by segment;
 * supported for N % 4 == 0, N <= 128, P <= 128.  SSD_PATH_AUTO takes the
 * chunk form where it applies, else the sequential kernel.  Scratch (chunk
 * states and gradients, or checkpoints; per-head gradients of B and C; the
 * per-head partial sums) comes stream-ordered from the library pool.  Errors
 * as ssd_scan_fwd.  Empty work writes nothing.
 */
ssd_status_t ssd_scan_bwd(const void *x, const float *dt_raw, const float *dt_bias, const float *A_log,
                          const void *B, const void *C, const float *D, const float *init_state,
                          const void *dy, const float *d_final, float *dx, float *ddt_raw,
                          float *ddt_bias, float *dA_log, float *dB, float *dC, float *dD,
                          float *d_init, const ssd_dims_t *dims, void *stream);

/* Which path SSD_PATH_AUTO resolves to for these dims on the current device
 * (SSD_PATH_SEQUENTIAL, SSD_PATH_CHUNKED or SSD_PATH_DECODE), or
 * -(ssd_status_t) if the dims are
 * invalid or unsupported.  Host only; launches nothing. */
int32_t ssd_select_path(const ssd_dims_t *dims);

/* Kernel launches one ssd_scan_fwd call makes for these dims (0 for empty
 * work), or -(ssd_status_t).  Host only. */
int32_t ssd_launches_per_call(const ssd_dims_t *dims);

/* How the chunked path orders its work for these dims and flags on the
 * current device (the SM count enters the choice), as ssd_scan_fwd would run
 * it:
 *   SSD_SCHEDULE_NONE    no chunked work (empty, or the sequential path);
 *   SSD_SCHEDULE_RANGES  chains cut into units of whole chunks, dealt to the CTAs
 *                        in turn; a unit takes its entering state from the unit
 *                        before it in its chain (one launch);
 *   SSD_SCHEDULE_PIECES  the chains' 128-step sub-chunks, chain after chain, cut
 *                        into one run of equal length per CTA; a chain cut
 *                        between two CTAs hands its state across (one launch);
 *   SSD_SCHEDULE_SPLIT   units of whole chunks or (where a chunk is a whole
 *                        number of 128-step sub-chunks) of whole sub-chunks:
 *                        every unit's end state from zero, a combine of those
 *                        states along each chain, then every unit from its
 *                        combined entering state (three launches; two where a
 *                        chain has at most 4 units and the scan has no conv or
 *                        trapezoidal mode: each unit then combines its
 *                        predecessors' end states itself).
 * All three evaluate the chunked recurrence with the state carried from chunk
 * to chunk; they differ only in which CTA computes what, and when.
 * ssd_scan_fwd_noalloc may choose differently (see there).  Returns -(ssd_status_t)
 * for invalid or unsupported dims.  Host only; launches nothing. */
int32_t ssd_chunk_schedule(const ssd_dims_t *dims);

/* Total kernel launches this library has made in this process. */
uint64_t ssd_launch_count(void);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device into *code (0 = none, else an ssd_status_t such as
 * SSD_ERR_TIMEOUT).  Returns SSD_OK, or SSD_ERR_CUDA if the read failed. */
ssd_status_t ssd_get_device_error(void *stream, uint32_t *code);

/* Static description of a status code.  Never NULL (an unknown value gives
 * "unknown status"). */
const char *ssd_status_string(ssd_status_t status);

/* SSD_ABI_VERSION of the loaded library. */
int32_t ssd_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBSSD_SSD_H */
