/*
 * csscan.h -- C ABI of the forward selective scan of a diagonal, complex-valued,
 * input-dependent linear recurrence, on one NVIDIA B300 (sm_103a).
 *
 * What it computes. Per batch b, channel d and state n, starting from a zero state:
 *
 *   a_t      = exp(dt[b,t,d] * A[d,n] + i * theta[b,t,n])
 *   exp-Euler         h_t = a_t h_{t-1} + dt_t Bc[b,t,n] x[b,t,d]
 *   exp-trapezoidal   h_t = a_t h_{t-1} + (1 - lam_t) dt_t a_t Bc[b,t-1,n] x[b,t-1,d]
 *                                       + lam_t dt_t Bc[b,t,n] x[b,t,d],  with Bc_{-1} x_{-1} = 0
 *   zero-order hold   h_t = a_t h_{t-1} + dt_t (a_t - 1) / z_t Bc[b,t,n] x[b,t,d],
 *                     z_t = dt_t A[d,n] + i theta[b,t,n]  (a_t = e^{z_t})
 *   y[b,t,d] = Re(sum_n Cc[b,t,n] h_t[n]) + Dskip[d] x[b,t,d]
 *
 * Sources (pages of the reference material, by title and section):
 *   - "Complex parallel scan" (fengwang.github.io), section 并行扫描的数学本质: the step
 *     h_t = A_t h_{t-1} + B_t x_t as an operator, its associative combine, and its validity
 *     for complex coefficients (the basis of the chunked carry used inside);
 *   - "Mamba-3 paper story" (ai.tomabc.com): the discretisation table (Exp-Euler row:
 *     alpha = exp(dt A), gamma = dt; Exp-Trapezoidal row: beta = (1 - lam) dt exp(dt A),
 *     gamma = lam dt) and the complex-state section (real decay A, input-dependent phase
 *     e^{i theta});
 *   - "状态空间模型的对偶谱理论 2026" (blog.lonae.com), section 3.2 (pseudocode listing): the sequential loop, y read
 *     from the updated state and summed over the state index;
 *   - "Mamba-3: 选择性状态空间模型的下一代架构" (metaphor-xennon), section 2.2: y = C h + D x.
 *   The exponential in beta is read as the full complex a_t of the current step, and theta
 *   is not scaled by dt.
 *
 * Layout (every tensor contiguous, row-major, last index fastest; complex values stored
 * interleaved (re, im) in a trailing dimension of 2):
 *   x, delta        (B, L, D)      input dtype
 *   Bc, Cc          (B, L, N, 2)   input dtype
 *   theta           (B, L, N)      input dtype
 *   lambda          (B, L)         input dtype (trapezoid mode only)
 *   A               (D, N)         float32, real (one decay per channel and state)
 *   Dskip           (D)            float32
 *   y               (B, L, D)      float32 output
 * The input dtype is float32 or bf16 (CSSCAN_F32 / CSSCAN_BF16). Arithmetic is float32 with
 * the complex state held in registers; the (B, L, D, N) state never reaches device memory.
 *
 * Ownership. Every pointer is caller-owned DEVICE memory of the current CUDA device; the
 * library never frees it. The library owns one internal workspace per (device, stream)
 * that it grows with cudaMalloc on first use and when a larger problem arrives (the first
 * call on a stream must therefore not be inside a stream capture); csscan_release_workspace
 * frees all of them.
 *
 * Asynchrony. Calls enqueue work on `stream` (0 = the legacy default stream) and return; y
 * is valid once the stream reaches that point. Calls on one stream are ordered; calls on
 * different streams use different workspaces and may overlap.
 *
 * Errors. Every function returns an int status (CSSCAN_OK = 0) and throws nothing. Argument
 * checks run on the host before any launch, so a rejected call touches no device memory.
 */
#ifndef CSSCAN_H
#define CSSCAN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  CSSCAN_OK = 0,
  CSSCAN_ERR_INVALID_ARG = 1,      /* null pointer, negative size, N == 0, bad mode/dtype,
                                      lambda == NULL in trapezoid mode, bad option */
  CSSCAN_ERR_MISALIGNED = 2,       /* x or delta not 16-byte aligned, or D * sizeof(dtype) not a
                                      multiple of 16 bytes (the tile copies need both) */
  CSSCAN_ERR_UNSUPPORTED = 3,      /* N not in {2, 4, 8, 16, 32, 64}, or sizes beyond 2^31 */
  CSSCAN_ERR_CUDA = 4,             /* a CUDA runtime/driver call or a launch failed */
  CSSCAN_ERR_LOOKBACK_TIMEOUT = 5, /* device: a chunk waited past its limit for its
                                      predecessor's carry (reported by csscan_get_device_status;
                                      the outputs of that call are not valid) */
  CSSCAN_ERR_PIPELINE_TIMEOUT = 6, /* device: a tile copy did not arrive within its limit */
  CSSCAN_ERR_SCRATCH_LIMIT = 7,    /* csscan_forward_noalloc: the problem needs more scratch than
                                      its fixed CSSCAN_NOALLOC_SCRATCH_BYTES array holds */
  CSSCAN_ERR_BOUNDS = 8            /* device, bounds-checked builds only (CSSCAN_BOUNDS_CHECK): a
                                      kernel index fell outside its array; the access was redirected
                                      to the array's first element and the outputs are not valid */
};

/* Discretisation of the injection ("Mamba-3 paper story", discretisation table):
 *   EXP_EULER     gamma_t = dt_t
 *   EXP_TRAPEZOID beta_t = (1 - lam_t) dt_t a_t on Bc_{t-1} x_{t-1}, gamma_t = lam_t dt_t
 *   ZOH           gamma_t = dt_t (e^{z_t} - 1) / z_t with z_t = dt_t A + i theta_t (the table's
 *                 A^{-1}(exp(dt A) - I) with the complex exponent of a_t in place of dt A);
 *                 the scans (csscan_forward, _ex, _state, _noalloc; every N),
 *                 csscan_decode_step and csscan_backward (N <= 32); not the MIMO scan */
typedef enum { CSSCAN_MODE_EXP_EULER = 0, CSSCAN_MODE_EXP_TRAPEZOID = 1, CSSCAN_MODE_ZOH = 2 } csscan_mode_t;
typedef enum { CSSCAN_F32 = 0, CSSCAN_BF16 = 1 } csscan_dtype_t;

/*
 * Forward scan. Computes y from x, delta, A, Bc, Cc, theta, lambda and Dskip as above.
 *   x, delta, Bc, Cc, theta, lambda : device pointers in `dtype`; lambda may be NULL in
 *                                     exp-Euler mode and is required in trapezoid mode
 *   A, Dskip                        : device float32
 *   y                               : device float32, written in full (B*L*D values)
 *   B, L, D, N                      : sizes; B, L or D == 0 is a no-op returning CSSCAN_OK
 *   mode                            : csscan_mode_t
 *   dtype                           : csscan_dtype_t
 *   stream                          : CUDA stream to enqueue on
 * Alignment: x and delta 16-byte aligned and D * sizeof(dtype) a multiple of 16 (D % 4 == 0
 * for float32, D % 8 == 0 for bf16); other pointers need only their natural alignment.
 */
int csscan_forward(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                   const void* theta, const void* lambda, const float* Dskip, float* y,
                   int64_t B, int64_t L, int64_t D, int64_t N, int mode, int dtype, cudaStream_t stream);

/*
 * Launch options for csscan_forward_ex. Zero-initialise and set only what you need.
 *   cta_warps     : reserved, must be 0 (a block is 4 warps; in the exp-Euler and trapezoid
 *                   modes a thread owns one channel and 8 or 16 of its states, in the
 *                   zero-order-hold mode two channels and 8 states)
 *   chunk_len     : sequence chunk per thread block (multiple of 32); 0 = automatic
 *   carry         : 0 automatic, 1 serial (each chunk waits for its predecessor's final state),
 *                   2 decoupled (each chunk first computes its own aggregate, then looks back)
 *   silent_chunk  : test hook; -1 normally. Chunks with this index never publish their carry,
 *                   so their successors run into the bounded wait and report
 *                   CSSCAN_ERR_LOOKBACK_TIMEOUT through csscan_get_device_status
 *   poll_limit    : maximum polls of one carry wait (about 0.5 us each); 0 = default (about 2 s)
 *   scan_begin,
 *   scan_end      : optional CUDA events (NULL = none), recorded on `stream` right before and
 *                   right after the scan kernel, to time it apart from the small table kernel
 */
typedef struct {
  int32_t cta_warps;
  int32_t chunk_len;
  int32_t carry;
  int32_t silent_chunk;
  int64_t poll_limit;
  cudaEvent_t scan_begin;
  cudaEvent_t scan_end;
} csscan_options_t;

/* csscan_forward with explicit launch options (opts may be NULL = automatic). */
int csscan_forward_ex(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                      const void* theta, const void* lambda, const float* Dskip, float* y,
                      int64_t B, int64_t L, int64_t D, int64_t N, int mode, int dtype,
                      const csscan_options_t* opts, cudaStream_t stream);

/*
 * Forward scan that continues from a given state and returns the final state, so that a long
 * sequence can be scanned in pieces (or a prompt prefilled before single-step decoding): the
 * recurrent, constant-state form of the model that "Mamba-3 paper story" contrasts with
 * attention's growing cache, and the associativity of the step operator ("Complex parallel
 * scan", section 并行扫描的数学本质) that makes the pieces compose exactly.
 * Arguments as csscan_forward, plus:
 *   h0      : device float32 (B, D, N, 2), the state h_{-1} before the first step, or NULL for zero
 *   x_prev, Bc_prev : trapezoid mode only (ignored in the exp-Euler and zero-order-hold modes): the step before the first,
 *             x (B, D) and Bc (B, N, 2) in `dtype`, which the first step's beta term uses;
 *             both NULL means there is no previous step (Bc_{-1} x_{-1} = 0); one NULL is invalid
 *   h_last  : device float32 (B, D, N, 2), receives h_{L-1}, or NULL
 * h0 and h_last must be 16-byte aligned and may not overlap. Scanning [0, t0) and then [t0, L)
 * with h0 = the first call's h_last and (x_prev, Bc_prev) = its last step's x and Bc gives the
 * same y and final state as one call over [0, L).
 */
int csscan_forward_state(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                         const void* theta, const void* lambda, const float* Dskip, float* y, const float* h0,
                         const void* x_prev, const void* Bc_prev, float* h_last, int64_t B, int64_t L, int64_t D,
                         int64_t N, int mode, int dtype, cudaStream_t stream);

/*
 * One decode step for B x D sequences whose state lives in device memory (the single-token,
 * constant-state regime of "Mamba-3 paper story"; one step of the recurrence above):
 *   x, delta          : (B, D) in `dtype`, this step's input and step size
 *   Bc, Cc            : (B, N, 2) in `dtype`;  theta : (B, N) in `dtype`
 *   lambda            : (B) in `dtype`, trapezoid mode only (may be NULL in exp-Euler mode)
 *   A, Dskip          : device float32 (D, N) and (D)
 *   y                 : device float32 (B, D), written
 *   h                 : device float32 (B, D, N, 2), the state, updated in place (16-byte aligned)
 *   x_prev, Bc_prev   : trapezoid mode: the previous step's x (B, D) and Bc (B, N, 2), both NULL
 *                       for the first step of a sequence; ignored in the other modes
 *   mode              : any csscan_mode_t (zero-order hold included, every N)
 * The caller keeps the previous step's x and Bc for the trapezoid rule. One kernel launch; the
 * state is read and written once, so the step is bound by memory bandwidth.
 */
int csscan_decode_step(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                       const void* theta, const void* lambda, const float* Dskip, float* y, float* h,
                       const void* x_prev, const void* Bc_prev, int64_t B, int64_t D, int64_t N, int mode, int dtype,
                       cudaStream_t stream);

/*
 * MIMO scan: each of H heads holds one complex state of N values shared by its P channels.
 * "Mamba-3 paper story" (MIMO section) widens B and C from N-vectors to N x P matrices so that
 * a state serves P input and output channels; its formulas were lost from the page, and the
 * reading here carries the single-input sharing over:
 *   a_t     = exp(dt[b,t,h] A[h,n] + i theta[b,t,n])
 *   v_t[n]  = sum_p Bm[b,t,n,p] x[b,t,h,p]
 *   exp-Euler   h_t = a_t h_{t-1} + dt_t v_t
 *   trapezoid   h_t = a_t h_{t-1} + (1 - lam_t) dt_t a_t v_{t-1} + lam_t dt_t v_t   (v_{-1} = 0)
 *   y[b,t,h,p] = Re(sum_n Cm[b,t,n,p] h_t[n]) + Dskip[h,p] x[b,t,h,p]
 * With P = 1 it is csscan_forward with D = H.
 *   x       : (B, L, H, P) in `dtype`          delta : (B, L, H) in `dtype`
 *   Bm, Cm  : (B, L, N, P, 2) in `dtype`, complex entries (re, im), shared by all heads
 *   theta   : (B, L, N) in `dtype`             lambda : (B, L) in `dtype` (trapezoid mode only)
 *   A       : device float32 (H, N)            Dskip : device float32 (H, P)
 *   y       : device float32 (B, L, H, P), written in full
 *   mode    : CSSCAN_MODE_EXP_EULER or CSSCAN_MODE_EXP_TRAPEZOID (ZOH: CSSCAN_ERR_UNSUPPORTED)
 * N must be 2, 4, 8, 16 or 32, P 1, 2, 4 or 8 and B <= 65535 (CSSCAN_ERR_UNSUPPORTED otherwise). Pointers
 * need their element alignment, Bm and Cm that of one complex entry. Starts from the zero
 * state. Uses the per-stream workspace like csscan_forward.
 */
int csscan_forward_mimo(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm,
                        const void* theta, const void* lambda, const float* Dskip, float* y, int64_t B, int64_t L,
                        int64_t H, int64_t P, int64_t N, int mode, int dtype, cudaStream_t stream);

/*
 * Backward pass of csscan_forward (sequence from the zero state, no step -1 halo): the
 * gradients of l = sum_{b,t,d} dy[b,t,d] y[b,t,d] with respect to every input. The pages call
 * for this pass and for regenerating the states during it instead of storing them ("Complex
 * parallel scan", sections 一个问题，两种命运 and 硬件落地的挑战); the formulas are reverse-mode
 * differentiation of the recurrence above. States are recomputed from checkpoints taken every
 * 8 steps; the (B, L, D, N) state is never stored.
 *   x .. Dskip, B, L, D, N, mode, dtype : exactly as passed to csscan_forward
 *   dy      : device float32 (B, L, D), the gradient of the loss with respect to y
 * Outputs (device float32, caller-owned, fully written by the call, any alignment of 4 bytes):
 *   dx, ddelta : (B, L, D)          dA : (D, N)          dDskip : (D)
 *   dBc, dCc   : (B, L, N, 2), (d/dRe, d/dIm) of each complex entry
 *   dtheta     : (B, L, N)          dlambda : (B, L), trapezoid mode only (may be NULL in exp-Euler mode)
 * Inputs need their element alignment, Bc and Cc that of one complex entry (no 16-byte rule;
 * inputs that also meet csscan_forward's 16-byte rule let the library take the checkpoints from
 * the scan kernel, otherwise from a slower pass of its own; the zero-order hold, whose
 * injection weight is complex per element, always takes the slower path). N must be 2, 4, 8, 16 or 32
 * (CSSCAN_ERR_UNSUPPORTED otherwise) and B <= 65535. The library grows its per-stream
 * workspace to B*L*N*8 + B*ceil(L/8)*D*N*8 bytes (rotation table and checkpoints). Sums over
 * rows use float32 atomic adds, so the summed gradients (dA, dBc, dCc, dtheta, dlambda,
 * dDskip) can differ in the last bits from run to run.
 */
int csscan_backward(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                    const void* theta, const void* lambda, const float* Dskip, const float* dy, float* dx,
                    float* ddelta, float* dA, float* dBc, float* dCc, float* dtheta, float* dlambda, float* dDskip,
                    int64_t B, int64_t L, int64_t D, int64_t N, int mode, int dtype, cudaStream_t stream);

/*
 * Backward pass of csscan_forward_mimo (from the zero state): the gradients of
 * l = sum_{b,t,h,p} dy[b,t,h,p] y[b,t,h,p] with respect to every input, by reverse-mode
 * differentiation of the MIMO recurrence above, the states regenerated from checkpoints taken
 * every 8 steps ("Complex parallel scan", sections 一个问题，两种命运 and 硬件落地的挑战).
 *   x .. Dskip, B, L, H, P, N, mode, dtype : exactly as passed to csscan_forward_mimo
 *   dy      : device float32 (B, L, H, P), the gradient of the loss with respect to y
 * Outputs (device float32, caller-owned, fully written by the call, any alignment of 4 bytes):
 *   dx : (B, L, H, P)   ddelta : (B, L, H)   dA : (H, N)   dDskip : (H, P)
 *   dBm, dCm : (B, L, N, P, 2), (d/dRe, d/dIm) of each complex entry
 *   dtheta : (B, L, N)   dlambda : (B, L), trapezoid mode only (may be NULL in exp-Euler mode)
 * mode: CSSCAN_MODE_EXP_EULER or CSSCAN_MODE_EXP_TRAPEZOID (ZOH: CSSCAN_ERR_UNSUPPORTED). N must be
 * 2, 4, 8, 16 or 32, P 1, 2, 4 or 8 and B <= 65535 (CSSCAN_ERR_UNSUPPORTED otherwise); pointers
 * need their element alignment, Bm and Cm that of one complex entry. One thread walks the whole
 * sequence of each (b, head, state), so the call is fastest with many heads. The library grows
 * its per-stream workspace to B*L*N*8 + B*ceil(L/8)*H*N*8 bytes. Sums over rows use float32
 * atomic adds (the summed gradients can differ in the last bits from run to run).
 */
int csscan_backward_mimo(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm,
                         const void* theta, const void* lambda, const float* Dskip, const float* dy, float* dx,
                         float* ddelta, float* dA, float* dBm, float* dCm, float* dtheta, float* dlambda,
                         float* dDskip, int64_t B, int64_t L, int64_t H, int64_t P, int64_t N, int mode, int dtype,
                         cudaStream_t stream);

/*
 * Synchronises `stream`, then returns the device-side status of the calls made on it since
 * the last query (CSSCAN_OK, CSSCAN_ERR_LOOKBACK_TIMEOUT or CSSCAN_ERR_PIPELINE_TIMEOUT), or
 * CSSCAN_ERR_CUDA if the stream reports an error. Clears the device status.
 */
int csscan_get_device_status(cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* csscan_status_string(int status);

/*
 * Forward scan that allocates no device memory. The reference pages have no counterpart:
 * this entry point exists for callers that cannot call cudaMalloc -- for example a serving
 * loop that must not allocate after start-up (cudaMalloc can synchronise the device and has
 * no latency bound), or a host program whose device memory is entirely owned by another
 * allocator or a fixed budget. It computes exactly what csscan_forward computes, with the
 * same arguments, layouts and alignment rules, but its scratch space (the per-chunk carry
 * records and the rotation tables) lives in one fixed array of CSSCAN_NOALLOC_SCRATCH_BYTES
 * compiled into the library, which every GPU that loads the library holds until the
 * process exits.
 *
 *   device_status : optional (NULL = none) caller-owned DEVICE pointer to one uint32_t; when
 *                   the stream reaches the end of the call it holds this call's device-side
 *                   status bits (0 = ok, 1 = a carry wait timed out, 2 = a tile copy timed out)
 *
 * Returns CSSCAN_ERR_SCRATCH_LIMIT, before any launch, when the problem needs more scratch
 * than the fixed array holds (roughly B*L*N*16 bytes of tables, 32 in the zero-order-hold mode,
 * plus 8 to 16 bytes per state
 * of every chunk); csscan_forward has no such limit. The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress, which may load the library's GPU code on
 * that device), so make that first call before any stream capture. All calls share the one
 * array, whose contents persist from call to call; the call resets the parts that must start
 * at zero. Calls that can overlap on the GPU (other streams, other threads) race on the
 * array: issue them one after another on a single stream.
 */
#define CSSCAN_NOALLOC_SCRATCH_BYTES (32u << 20)
int csscan_forward_noalloc(const void* x, const void* delta, const float* A, const void* Bc, const void* Cc,
                           const void* theta, const void* lambda, const float* Dskip, float* y,
                           int64_t B, int64_t L, int64_t D, int64_t N, int mode, int dtype,
                           uint32_t* device_status, cudaStream_t stream);

/* Frees every internal workspace after synchronising its device. Returns CSSCAN_OK or
 * CSSCAN_ERR_CUDA. Safe to call at any time outside stream capture. */
int csscan_release_workspace(void);

#ifdef __cplusplus
}
#endif

#endif /* CSSCAN_H */
