/*
 * ssm_scan.h -- C ABI of the B300 (sm_103a) selective-scan library, libssm_scan.so.
 *
 * The operation (Mamba's selective scan; "Understanding Mamba" s2.2-s2.3, Eqs. (2)-(3); the aiwiki
 * "Selective State Space Models" reference loop for shapes and A = -exp(A_log)):
 *
 *   for every batch element b and channel d, with A[n] = -exp(A_log[d, n]) and h = h0[b, d, :] (or 0):
 *     for t = 0 .. L-1, for n = 0 .. N-1:
 *       Abar   = exp(delta[b,t,d] * A[n])
 *       Bbar x = delta[b,t,d] * B[b,t,n] * x[b,t,d]                          (SSM_DISC_EULER)
 *              = (exp(delta[b,t,d] A[n]) - 1) / A[n] * B[b,t,n] * x[b,t,d]   (SSM_DISC_ZOH;
 *                                                     delta * B * x where A[n] == 0)
 *       h[n]   = Abar * h[n] + Bbar x
 *     y[b,t,d] = sum_n C[b,t,n] * h[n]                   (no feedthrough term, no gate)
 *   final_state[b, d, :] = h after the last step.
 *
 * The first-order (Euler) input term keeps the exact Abar, as the pages' scalar recurrence and the
 * aiwiki reference loop do ("State Space Models & Mamba" chapter; the aiwiki entry names delta*B as the
 * form Mamba uses in practice). delta is taken as given (already made positive upstream); the _ex entry
 * points can apply softplus(delta + bias) themselves.
 *
 * Conventions shared by every entry point:
 *  - Every pointer is DEVICE memory of the current CUDA device, owned by the caller, except the data arrays
 *    of ssm_scan_fwd_host, which are host memory. No call allocates or frees memory, and none keeps a
 *    pointer after it returns (ssm_scan_fwd_host creates two streams and a few events per device on first
 *    use and keeps them for the process). The one exception: ssm_scan_bwd_noalloc
 *    uses a fixed 64 MiB scratch array compiled into the backward pass's device code. The CUDA runtime
 *    loads that code onto a device the first time a backward entry point (ssm_scan_bwd or
 *    ssm_scan_bwd_noalloc) runs there (module loading is lazy by default; with
 *    CUDA_MODULE_LOADING=EAGER it happens when the process's context on the device is created), and the
 *    64 MiB stay committed on that device until the process exits, for ssm_scan_bwd callers too.
 *  - Layouts are dense row-major in the shapes given. "dtype" arrays hold fp32 (SSM_DTYPE_F32) or
 *    bf16 (SSM_DTYPE_BF16) elements; A_log, states, h0 and final_state are always fp32.
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = the legacy default
 *    stream) and runs asynchronously; the return code covers argument checks and launch errors.
 *    ssm_check_device() synchronises the stream and reports errors raised while kernels ran.
 *  - Apart from ssm_check_device (which synchronises) and ssm_scan_fwd_host (which also uses streams of
 *    its own), a call only launches kernels on `stream`. After a first call on a device (which sets kernel
 *    attributes once), the calls can therefore be captured into a CUDA graph and replayed; and calls on
 *    different streams need no ordering between them, except ssm_scan_bwd_noalloc, whose scratch array
 *    is shared by all its calls on a device.
 *  - For the diagonal scan, N (state size) must be in [1, 16]; larger N returns SSM_ERR_UNSUPPORTED. The
 *    SSD layer has its own sizes (see ssm_ssd_fwd).
 *  - Outputs may not overlap inputs (checked on the pointer ranges: SSM_ERR_INVALID_ARG).
 *  - Any status other than SSM_OK leaves a one-line reason in ssm_last_error() (per thread).
 *  - Results are deterministic for a given shape, dtype and device (no atomics on the data path), except
 *    the sums over channels, batch and time of ssm_scan_bwd (dA_log, dB, dC), which use atomic adds whose
 *    order may change the last bits from run to run.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum, overlapping in/out ranges */
    SSM_ERR_UNSUPPORTED = 2,  /* valid but not implemented (N > 16) */
    SSM_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    SSM_ERR_TIMEOUT = 4       /* a kernel gave up a bounded wait (reported by ssm_check_device; see
                                 ssm_set_wait_limit_ns) */
} ssm_status;

typedef enum { SSM_DISC_EULER = 0, SSM_DISC_ZOH = 1 } ssm_disc;
typedef enum { SSM_DTYPE_F32 = 0, SSM_DTYPE_BF16 = 1 } ssm_dtype;

/*
 * Prefill scan over whole sequences ("Understanding Mamba" s7: discretisation, recurrence and readout
 * fused so that the [batch, L, D, N] states never leave the chip).
 *   x, delta    [batch, L, D]  dtype      input sequence and per-step step size
 *   A_log       [D, N]         fp32       A = -exp(A_log)
 *   B, C        [batch, L, N]  dtype      input / output projections, shared by all D channels
 *   h0          [batch, D, N]  fp32       initial state, or NULL for zeros
 *   y           [batch, L, D]  dtype      output (bf16 outputs are rounded to nearest even)
 *   final_state [batch, D, N]  fp32       state after step L-1 (h0 or zeros when L == 0), or NULL
 * batch, L, D >= 0 (zero sizes are no-ops apart from final_state). final_state may not overlap h0.
 */
ssm_status ssm_scan_fwd(const void *x, const void *delta, const float *A_log,
                        const void *B, const void *C, const float *h0,
                        void *y, float *final_state,
                        int64_t batch, int64_t L, int64_t D, int64_t N,
                        ssm_dtype dtype, ssm_disc disc, void *stream);

/*
 * One recurrent decode step ("Understanding Mamba" s3.2 and s10.1: the same Eq. (3) body applied
 * once to a carried state; constant work per token).
 *   state    [batch, D, N]  fp32   read and updated in place
 *   x_t, delta_t [batch, D] dtype
 *   A_log    [D, N]         fp32
 *   B_t, C_t [batch, N]     dtype
 *   y_t      [batch, D]     dtype  output
 */
ssm_status ssm_scan_step(float *state, const void *x_t, const void *delta_t, const float *A_log,
                         const void *B_t, const void *C_t, void *y_t,
                         int64_t batch, int64_t D, int64_t N,
                         ssm_dtype dtype, ssm_disc disc, void *stream);

/*
 * Prefill scan with the layer pieces the pages define around it fused in ("Understanding Mamba" s5.1
 * Eq. (6), s2.1 with Eq. (1)/(3), s8.1 Eq. (9)); every piece is optional:
 *   delta_bias     [D]            fp32   b_Delta added to delta, or NULL (0)
 *   delta_softplus                       nonzero: the scan uses softplus(delta + delta_bias[d]), where
 *                                        softplus(v) = ln(1 + e^v); zero: delta + delta_bias[d] as given
 *   D_skip         [D]            fp32   feedthrough D, or NULL (0)
 *   z              [batch, L, D]  dtype  gate input, or NULL (no gate)
 * and y[b,t,d] = (sum_n C[b,t,n] h[n] + D_skip[d] x[b,t,d]) * SiLU(z[b,t,d]), SiLU(v) = v / (1 + e^-v).
 * The other arguments, the final state (which the gate and feedthrough do not touch) and the error
 * behaviour are those of ssm_scan_fwd; z may not overlap an output. ssm_scan_fwd is this call with every
 * piece off.
 */
ssm_status ssm_scan_fwd_ex(const void *x, const void *delta, const float *A_log,
                           const void *B, const void *C, const float *h0,
                           const float *delta_bias, int delta_softplus, const float *D_skip, const void *z,
                           void *y, float *final_state,
                           int64_t batch, int64_t L, int64_t D, int64_t N,
                           ssm_dtype dtype, ssm_disc disc, void *stream);

/*
 * Prefill of ssm_scan_fwd with every data array in HOST memory: x, delta, B, C, y and final_state (and A_log,
 * h0) are host pointers, in the layouts of ssm_scan_fwd. The sequence is streamed through the device in
 * segments of seg_L steps: segment k + 1 is copied in while segment k is computed and segment k - 1's y is
 * copied out. Segments chain exactly through the state (h0 of segment k = final state of segment k - 1;
 * "Understanding Mamba" s3.2: the recurrence carries everything about the past in h), so y and final_state
 * are those of one ssm_scan_fwd over the whole sequence, computed by the same kernels. No counterpart in the
 * pages: a way to feed the path from host memory without a full-size device copy.
 *  - workspace: DEVICE memory of at least ssm_scan_fwd_host_workspace_size(batch, D, N, dtype, seg_L) bytes,
 *    owned by the caller: two segment slots (x, delta, B, C, y), two states and A_log. Too small, or seg_L < 1:
 *    SSM_ERR_INVALID_ARG.
 *  - Copies use cudaMemcpyAsync / cudaMemcpy2DAsync; they overlap compute only when the host arrays are
 *    page-locked (cudaHostAlloc / cudaHostRegister). Host arrays must stay valid, and untouched by the caller,
 *    until `stream` has completed the call's work.
 *  - Ordering: every copy and kernel is ordered after the work already on `stream` and before the work
 *    enqueued on it afterwards. Internally the uploads and downloads run on two library-owned streams per
 *    device (created on first use, kept for the life of the process) joined to `stream` by events; concurrent
 *    calls on one device are serialised while they are enqueued.
 *  - L = 0: final_state is set to h0 (or zeros) on the host before the call returns.
 *  - Errors: argument errors as for ssm_scan_fwd (host ranges of outputs may not overlap inputs), CUDA
 *    errors as SSM_ERR_CUDA; kernel-side failures are reported by ssm_check_device(stream).
 */
size_t ssm_scan_fwd_host_workspace_size(int64_t batch, int64_t D, int64_t N, ssm_dtype dtype, int64_t seg_L);
ssm_status ssm_scan_fwd_host(const void *x, const void *delta, const float *A_log,
                             const void *B, const void *C, const float *h0,
                             void *y, float *final_state,
                             void *workspace, size_t workspace_bytes, int64_t seg_L,
                             int64_t batch, int64_t L, int64_t D, int64_t N,
                             ssm_dtype dtype, ssm_disc disc, void *stream);

/*
 * One decode step with the same optional pieces (z_t [batch, D] in `dtype`): the step of ssm_scan_step on
 * delta = softplus(delta_t + delta_bias[d]) (or delta_t + delta_bias[d]), output
 * y_t = (C_t . h + D_skip[d] x_t) * SiLU(z_t).
 */
ssm_status ssm_scan_step_ex(float *state, const void *x_t, const void *delta_t, const float *A_log,
                            const void *B_t, const void *C_t,
                            const float *delta_bias, int delta_softplus, const float *D_skip, const void *z_t,
                            void *y_t, int64_t batch, int64_t D, int64_t N,
                            ssm_dtype dtype, ssm_disc disc, void *stream);

/*
 * Backward pass of the prefill scan: the gradients of
 *     J = sum_{b,t,d} dy[b,t,d] y[b,t,d] + sum_{b,d,n} dfinal[b,d,n] final_state[b,d,n]
 * with respect to every input of ssm_scan_fwd (plain scan: no softplus, feedthrough or gate). The states
 * are recomputed from the inputs rather than read from a saved copy ("State Space Models & Mamba"
 * chapter, the paragraph on the fused kernel: the backward pass recomputes h). The formulas are the
 * chain rule of the forward recurrence run backwards in time through lambda_t = dJ/dh_t.
 *   x, delta, A_log, B, C, h0   as in ssm_scan_fwd (h0 may be NULL: zero initial state)
 *   dy          [batch, L, D]  dtype   gradient of J with respect to y
 *   dfinal      [batch, D, N]  fp32    gradient with respect to final_state, or NULL (zero)
 *   dx, ddelta  [batch, L, D]  dtype   outputs (bf16 rounded to nearest even)
 *   dA_log      [D, N]         fp32    output (sums over the batch and the time axis)
 *   dB, dC      [batch, L, N]  fp32    outputs (sums over the D channels)
 *   dh0         [batch, D, N]  fp32    output, or NULL (not wanted); dfinal when L == 0
 *   workspace   device memory of at least ssm_scan_bwd_workspace_size(batch, L, D, N) bytes (may be NULL
 *               when that is 0), owned by the caller; its contents on entry do not matter and on return
 *               are unspecified. It holds the states at chunk ends between the kernel's forward
 *               recomputation and its backward walk. Two calls in flight may not share it.
 * Outputs are overwritten (dA_log, dB and dC are zeroed on the stream first, then accumulated with atomic
 * adds). No output may overlap an input, the workspace or another output. Other conventions and errors
 * as for ssm_scan_fwd; a workspace that is NULL or too small returns SSM_ERR_INVALID_ARG.
 */
ssm_status ssm_scan_bwd(const void *x, const void *delta, const float *A_log,
                        const void *B, const void *C, const float *h0,
                        const void *dy, const float *dfinal,
                        void *dx, void *ddelta, float *dA_log, float *dB, float *dC, float *dh0,
                        void *workspace, size_t workspace_bytes,
                        int64_t batch, int64_t L, int64_t D, int64_t N,
                        ssm_dtype dtype, ssm_disc disc, void *stream);

/* Bytes of workspace ssm_scan_bwd needs for these sizes (0 for sequences of at most 8 steps); 0 as well
   for invalid sizes, which ssm_scan_bwd itself rejects. */
size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t L, int64_t D, int64_t N);

/*
 * ssm_scan_bwd without a workspace argument, for callers that cannot allocate device memory themselves:
 * code running inside a host application whose memory pool owns the whole GPU and gives plugins no
 * allocator, or a service that forbids allocation once it has started serving (a cudaMalloc there can
 * stall or fail at the worst moment). It has no counterpart in the pages: it is a packaging choice of this
 * library, not part of the method.
 *
 * The chunk-end states live in a scratch array inside the library itself: 64 MiB of device memory,
 * committed on a device when the backward pass's device code is first loaded there (the first call of
 * ssm_scan_bwd or ssm_scan_bwd_noalloc on that device, unless CUDA_MODULE_LOADING=EAGER loads it with the
 * context) and held until the process exits. The call itself allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine; but that first load does take the 64 MiB from the device, so a
 * caller that may not allocate while serving should make one call at start-up, before serving and before
 * any stream capture (a call with batch, L and D all 0 and null data pointers is enough: it loads the code
 * and looks up the array's address on the current device, and computes nothing). Sizes whose ssm_scan_bwd_workspace_size() exceeds
 * 64 MiB return SSM_ERR_INVALID_ARG with a message saying so (use ssm_scan_bwd with a workspace then). All calls on a device share the one array, so two calls whose kernels may run at the
 * same time on that device (other streams, other host threads) race on it and give wrong gradients:
 * serialise them. The array needs no clearing between calls (each call writes every entry it reads).
 * Arguments, outputs and errors otherwise as for ssm_scan_bwd.
 */
ssm_status ssm_scan_bwd_noalloc(const void *x, const void *delta, const float *A_log,
                                const void *B, const void *C, const float *h0,
                                const void *dy, const float *dfinal,
                                void *dx, void *ddelta, float *dA_log, float *dB, float *dC, float *dh0,
                                int64_t batch, int64_t L, int64_t D, int64_t N,
                                ssm_dtype dtype, ssm_disc disc, void *stream);

/*
 * Mamba-2 SSD layer: the scan with A = a I, one scalar a per head, evaluated in chunks ("State Space Models
 * & Mamba" chapter, the Mamba-2 paragraph; "Mathematical Prerequisites for Mamba" s7: the recurrence is a
 * 1-semiseparable matrix product, computed as masked matrix products inside chunks on the tensor cores, with
 * the recurrence carrying the state between chunks). For head h with state S [P, N]:
 *   A_h = -exp(A_log[h]),  Abar = exp(delta[b,t,h] A_h),  coef = delta (Euler) or (Abar - 1) / A_h (ZOH)
 *   S[p][n] = Abar S[p][n] + coef B[b,t,n] x[b,t,h,p],   y[b,t,h,p] = sum_n C[b,t,n] S[p][n]
 *   x, y        [batch, L, H, P]  bf16 (dtype must be SSM_DTYPE_BF16)
 *   delta       [batch, L, H]     fp32
 *   A_log       [H]               fp32
 *   B, C        [batch, L, N]     bf16, one group shared by every head
 *   h0          [batch, H, P, N]  fp32 initial state, or NULL
 *   final_state [batch, H, P, N]  fp32, or NULL
 *   workspace   device memory of ssm_ssd_fwd_workspace_size() bytes, or NULL; its contents on entry do not
 *               matter, and two calls in flight may not share it.
 * Two implementations, the same function:
 *  - P = 64 with a workspace of at least ssm_ssd_fwd_workspace_size() bytes (256-byte aligned; h0 and
 *    final_state 16-byte aligned): chunks of 128 steps in parallel on the fifth-generation tensor cores
 *    (tcgen05 MMAs with TMEM accumulators, bulk tensor copies), in three launches on `stream` -- the chunks'
 *    own states into the workspace, the recurrence between chunks, the outputs. The second and third are
 *    programmatic dependent launches of the one before (each waits for its predecessor's writes before
 *    reading them); ordering against other work on `stream` is that of ordinary launches.
 *  - otherwise: chunks of 64 steps with warp-level MMAs, one CTA per (batch element, head, 16 channels)
 *    walking the sequence; with a workspace, long sequences are cut into segments scanned from a zero state
 *    and a second pass adds the state carried into each.
 * N must be 64 or 128 and P a multiple of 16 (else SSM_ERR_UNSUPPORTED); x, B, C and y must be 16-byte
 * aligned (else SSM_ERR_UNSUPPORTED). The products run with bf16 operands and fp32 accumulation (the
 * masked score tile and a bf16 copy of the carried state are rounded to bf16 as operands; the state itself
 * is carried in fp32; on the tensor-core path each chunk's own state, formed from bf16 operands, is stored
 * in bf16 between the first two launches). A bounded wait of the tensor-core kernels that runs out (2 s) is reported by
 * ssm_check_device() as SSM_ERR_TIMEOUT. Other conventions as for ssm_scan_fwd.
 */
ssm_status ssm_ssd_fwd(const void *x, const float *delta, const float *A_log, const void *B, const void *C,
                       const float *h0, void *y, float *final_state, void *workspace, size_t workspace_bytes,
                       int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N,
                       ssm_dtype dtype, ssm_disc disc, void *stream);

/* Bytes of workspace for ssm_ssd_fwd: for P = 64, the chunk states and the states entering each chunk (bf16)
   and each chunk's log decay (fp32) of the tensor-core path; for other P, the segment states of the warp-MMA path on the current
   device (0 when one CTA per sequence already fills it). 0 for unsupported shapes. */
size_t ssm_ssd_fwd_workspace_size(int64_t batch, int64_t L, int64_t H, int64_t P, int64_t N);

/* Synchronise `stream` and report any error raised while this library's kernels ran on it. */
ssm_status ssm_check_device(void *stream);

/*
 * Longest time, in nanoseconds, that a warp of the prefill kernel for N = 16 (the TMA-staged one) waits
 * for one staged tile of its inputs before giving up. The default is 2,000,000,000 (2 s); a healthy tile
 * arrives within microseconds. A warp that gives up stops its share of the scan and sets the library's
 * device status word, so that the next ssm_check_device() returns SSM_ERR_TIMEOUT; that launch's y and
 * final_state are then incomplete. A warp waits for the copies it still has in flight before it exits
 * (that wait keeps the fixed 2 s bound), so a launch that gives up leaves no copy writing into shared
 * memory and the device stays usable. The setting is process-wide, applies to launches made after the
 * call, and is read when each launch is enqueued. Returns the previous value. No counterpart in the
 * pages: this is the library's failure-reporting contract.
 */
uint64_t ssm_set_wait_limit_ns(uint64_t ns);

/* Static name of a status code. */
const char *ssm_status_string(ssm_status s);

/* One-line reason for the last non-OK status returned on the calling thread ("" if none). */
const char *ssm_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
