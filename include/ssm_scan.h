/*
 * ssm_scan.h -- C-ABI of the B300 (sm_103a) selective-scan library.
 *
 * Two operations of the Mamba selective state-space model (S6):
 *
 *  ssm_scan_fwd      The selective scan over a whole sequence.  For every batch
 *                    row b, channel d and state n:
 *                      Delta_t = softplus(delta_t + dt_bias[d])       (optional softplus / bias)
 *                      Abar_t  = exp(Delta_t * A[d,n])                 (zero-order hold, diagonal A)
 *                      h_t     = Abar_t * h_{t-1} + Delta_t * B_t[n] * u_t,   h_{-1} = 0
 *                      y_t     = sum_n C_t[n] * h_t[n] + D[d] * u_t  (optional D)
 *                      out_t   = y_t * silu(z_t)                       (optional gate)
 *                    and the state after the last step.
 *                    Sources: "Mamba 状态空间模型深度解析" (gsyq.cn), sections
 *                    "连续到离散的转换" (discrete recurrence, ZOH A_bar = exp(Delta A)),
 *                    "选择性机制的设计理念" (B, C, Delta = Softplus(Linear(x)) depend on the
 *                    input) and "硬件优化并行扫描算法" (A_bar = exp(Delta*A), B_bar = Delta*B,
 *                    h = scan(A_bar, B_bar*x), y = C*h); VMamba notes (genhiy.github.io),
 *                    "S4中三个矩阵的维度表示、维度变化" (one SSM per channel; B, C of shape
 *                    (B,L,N) shared by all channels; Delta of shape (B,L,D)) and
 *                    "简化的SSM架构" (the gated block that the silu(z) gate closes).
 *
 *  ssm_state_update  One decode step of the same recurrence on a stored state
 *                    (constant-memory inference: gsyq.cn page, complexity table
 *                    row "推理内存 O(d) 状态向量"; 53ai.com Mamba article, §1 on
 *                    RNN-style inference from the previous hidden state only).
 *
 *  ssm_scan_fwd_train / ssm_scan_bwd (and their _ex forms, either discretization)
 *                    The training pair: a forward that keeps chunk checkpoints of
 *                    the state, and the backward pass from them.
 *
 *  ssm_causal_conv1d_fwd / ssm_causal_conv1d_update
 *                    The depthwise causal convolution that produces the scan's
 *                    input, over whole rows and as a decode step.
 *
 * Conventions shared by every entry point
 *  - Every pointer is a DEVICE pointer owned by the caller.  The library keeps no
 *    global state between calls and allocates nothing, with one exception: a scan
 *    that runs split (SSM_FORM_SPLIT below) through an entry point without a
 *    workspace argument takes its carry buffers (4 * (dstate + 1) bytes per batch
 *    row, channel and carry segment) from the device's default memory pool with
 *    cudaMallocAsync on `stream` and returns them with cudaFreeAsync on the same
 *    stream after its last launch.  ssm_scan_fwd_ws takes them from the caller
 *    and never allocates.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  Kernel-time errors surface on the caller's next
 *    synchronisation of that stream.
 *  - All arguments are validated on the host before anything is launched.  A
 *    non-zero return means nothing was launched, except SSM_ERR_LAUNCH (the
 *    launch itself failed; see ssm_status_string).
 *  - There is no CPU fallback: every call runs the sm_103a kernels.
 *  - io dtype (SSM_F32 or SSM_BF16) applies to u/delta/z/y/B/C (scan) and to
 *    x/dt/z/out/B/C (decode).  A, D, dt_bias and the states are always float32;
 *    all arithmetic is float32.  bf16 outputs are rounded to nearest-even.
 *  - Pointers must be aligned to their element size.  Rows that are 16-byte
 *    aligned (base 16-byte aligned and a row length in bytes that is a multiple
 *    of 16) take a vectorised copy path; anything else takes an element-wise
 *    copy path inside the same kernels.  Results are identical.
 *  - dstate may be 1..16.  Sizes of zero are allowed and launch nothing (except
 *    that seqlen == 0 still writes the zero final state when last_state is given).
 */
#ifndef SSM_SCAN_H_
#define SSM_SCAN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSM_OK = 0,
  SSM_ERR_NULL = -1,        /* a required pointer is NULL */
  SSM_ERR_SHAPE = -2,       /* a size is negative, or dstate < 1 */
  SSM_ERR_DTYPE = -3,       /* io_dtype is not an ssm_dtype value */
  SSM_ERR_ALIGN = -4,       /* a pointer is not aligned to its element size */
  SSM_ERR_UNSUPPORTED = -5, /* dstate > 16, or a grid dimension would overflow */
  SSM_ERR_LAUNCH = -6,      /* the CUDA launch failed (no device, bad stream, ...) */
  SSM_ERR_TIMEOUT = -7,     /* reserved: a bounded in-kernel wait gave up */
  SSM_ERR_ARG = -8          /* an enumerated argument is out of range, or buffers alias that must not */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/*
 * How B is discretised (A is always Abar = exp(Delta A)).
 *  SSM_DISC_DELTA_B : Bbar = Delta * B, the form the scan pseudo-code uses (gsyq.cn page,
 *                     "硬件优化并行扫描算法": B_bar = Δ*B).  The default of every entry point
 *                     without a discretization argument.
 *  SSM_DISC_ZOH     : the exact zero-order hold Bbar = (Delta A)^-1 (exp(Delta A) - I) Delta B
 *                     (gsyq.cn page, "连续到离散的转换"; VMamba notes, section on the dimensions
 *                     of A, B, C), i.e. (exp(Delta A[d,n]) - 1) / A[d,n] * B[n] for the diagonal
 *                     A, with its limit Delta * B[n] where A[d,n] = 0.
 */
typedef enum { SSM_DISC_DELTA_B = 0, SSM_DISC_ZOH = 1 } ssm_discretization;

/* Version of this ABI (bumped when a signature changes, an entry point is added or a layout
 * changes): 7. */
int ssm_abi_version(void);

/*
 * Selective scan forward.
 *   u, delta, z, y : [batch][dim][seqlen], io dtype, contiguous (seqlen innermost).
 *                    delta is the raw step size before dt_bias and softplus.
 *   A              : [dim][dstate] float32, the continuous (negative) A, e.g. -exp(A_log).
 *   B, C           : [batch][dstate][seqlen], io dtype, shared by all channels of a batch row.
 *   D, dt_bias     : [dim] float32.
 *   last_state     : [batch][dim][dstate] float32, receives h after the last step.
 *   delta_softplus : non-zero applies softplus to delta + dt_bias.
 * Required: u, delta, A, B, C, y.  Nullable: D (no skip), z (no gate), dt_bias (no
 * bias), last_state (not written).  y must not overlap u, delta, z, B or C (SSM_ERR_ARG).
 * Returns an ssm_status.
 */
int ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* dt_bias, int delta_softplus, void* y, float* last_state, int batch,
                 int dim, int dstate, int seqlen, int io_dtype, void* stream);

/*
 * Selective scan forward from a given initial state h0 ([batch][dim][dstate] float32,
 * nullable = zero state).  Otherwise identical to ssm_scan_fwd.  Scanning L1 steps,
 * then L2 steps from the returned last_state, equals one scan over L1 + L2 steps:
 * the chunked streaming of long documents (gsyq.cn page, "长序列处理的最佳实践",
 * LongDocumentProcessor) at the level of one scan.  last_state may equal h0 (in place).
 */
int ssm_scan_fwd_h0(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* h0, void* y,
                    float* last_state, int batch, int dim, int dstate, int seqlen, int io_dtype, void* stream);

/*
 * ssm_scan_fwd_h0 with a choice of discretization (an ssm_discretization value; anything
 * else returns SSM_ERR_ARG).  With SSM_DISC_DELTA_B it is exactly ssm_scan_fwd_h0.
 */
int ssm_scan_fwd_ex(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* h0, void* y,
                    float* last_state, int batch, int dim, int dstate, int seqlen, int io_dtype, int discretization,
                    void* stream);

/*
 * Which kernel form a scan of these sizes launches on the current device, without launching it.
 * The plain and balanced forms compute the same recurrence in the same order per state, so their
 * results are bitwise equal; they differ in how channels are spread over SMs:
 *   SSM_FORM_PLAIN     one CTA per 32-channel block of a batch row;
 *   SSM_FORM_BALANCED  one CTA per SM holding up to three warp groups on host-planned channel
 *                      ranges (bf16, dstate 9..16, dim a multiple of 8, where the plan lowers the
 *                      busiest SM's load; SSM_SCAN_VARIANT=quad_plain in the environment turns it off).
 *   SSM_FORM_SPLIT     the balanced form with the sequence split into segments scanned side by
 *                      side, for few channels and long sequences (four segments fit the SMs'
 *                      warp groups at once: at most 3 eight-channel units per SM; or one full
 *                      group per SM plus a tail in the last batch row, when the whole rows run
 *                      first and only the tail is split; seqlen >= 8192, 16-byte aligned rows, no
 *                      checkpoints, last_state not overlapping h0).  A carry pass scans each carry segment from a zero
 *                      state (the first from h0) for its end state and step-size sum; a combine
 *                      folds them with the associative pair operator (a1, b1) o (a2, b2) =
 *                      (a1 a2, a2 b1 + b2), a segment's decay a = exp(A * sum of its Delta) (53ai.com
 *                      Mamba article, section 3.3 "Parallel Associative Scan"; gsyq.cn page,
 *                      "硬件优化并行扫描算法"); the full pass scans every segment from its combined
 *                      carry.  Results equal the unsplit scan's up to float32 rounding (the decay
 *                      of a segment is one exponential of a sum instead of a product of per-step
 *                      exponentials).  SSM_SCAN_SPLIT=off in the environment turns it off.
 * aligned_rows: non-zero when u, delta, z, B, C and y will be 16-byte aligned.  *ctas (nullable)
 * receives the grid size (of the full pass, for the split form).  Returns the form (>= 0) or a
 * negative ssm_status (SSM_ERR_LAUNCH when no device can be queried).
 */
typedef enum { SSM_FORM_PLAIN = 0, SSM_FORM_BALANCED = 1, SSM_FORM_SPLIT = 2 } ssm_scan_form;
int ssm_scan_fwd_form(int batch, int dim, int dstate, int seqlen, int io_dtype, int discretization, int aligned_rows,
                      int* ctas);

/*
 * ssm_scan_fwd_ex with caller-owned scratch: it never allocates.  A scan that runs split
 * (SSM_FORM_SPLIT) keeps its carry buffers in `workspace`: device memory, 16-byte aligned, of at
 * least the bytes ssm_scan_fwd_workspace_size reports for these sizes, overlapping no other
 * argument (SSM_ERR_ALIGN / SSM_ERR_ARG otherwise), and left alone until the scan has completed on
 * `stream`.  With a NULL workspace or fewer bytes the scan runs unsplit, with the same results as
 * SSM_SCAN_SPLIT=off.  Other arguments and the return as ssm_scan_fwd_ex.
 */
int ssm_scan_fwd_ws(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* h0, void* y,
                    float* last_state, int batch, int dim, int dstate, int seqlen, int io_dtype, int discretization,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of workspace a scan of these sizes uses on the current device (0 when it does not run
 * split); aligned_rows as for ssm_scan_fwd_form.  *bytes is required.  Returns an ssm_status
 * (SSM_ERR_LAUNCH when no device can be queried).
 */
int ssm_scan_fwd_workspace_size(int batch, int dim, int dstate, int seqlen, int io_dtype, int discretization,
                                int aligned_rows, size_t* bytes);

/*
 * Training forward: ssm_scan_fwd_h0 (Delta*B discretization) that also stores, for the backward
 * pass, the state before every SSM_SCAN_CHECKPOINT_STEPS-th step:
 *   checkpoints : [batch][ncheck][dim][dstate] float32, ncheck = ssm_scan_num_checkpoints(seqlen)
 *                 = ceil(seqlen / SSM_SCAN_CHECKPOINT_STEPS); checkpoint c holds
 *                 h_{c*SSM_SCAN_CHECKPOINT_STEPS - 1} (h0, or zero, for c = 0).  (8 bytes per
 *                 (batch, channel, step) for dstate 16: the backward restarts every 8-step
 *                 register sub-chunk from its checkpoint instead of recomputing the chunk.)
 * Required: checkpoints, plus what ssm_scan_fwd_h0 requires.  The lane-per-channel form is not
 * used for this call.  Returns an ssm_status.
 */
#define SSM_SCAN_CHECKPOINT_STEPS 8
int ssm_scan_num_checkpoints(int seqlen);
int ssm_scan_fwd_train(const void* u, const void* delta, const float* A, const void* B, const void* C,
                       const float* D, const void* z, const float* dt_bias, int delta_softplus, const float* h0,
                       void* y, float* last_state, float* checkpoints, int batch, int dim, int dstate, int seqlen,
                       int io_dtype, void* stream);

/*
 * ssm_scan_fwd_train with a choice of discretization (as ssm_scan_fwd_ex; anything else returns
 * SSM_ERR_ARG).  Pair an SSM_DISC_ZOH training forward with ssm_scan_bwd_ex(..., SSM_DISC_ZOH).
 */
int ssm_scan_fwd_train_ex(const void* u, const void* delta, const float* A, const void* B, const void* C,
                          const float* D, const void* z, const float* dt_bias, int delta_softplus, const float* h0,
                          void* y, float* last_state, float* checkpoints, int batch, int dim, int dstate, int seqlen,
                          int io_dtype, int discretization, void* stream);

/*
 * Backward pass of the scan (Delta*B discretization): the gradients of a loss given
 * dout = dLoss/dout ([batch][dim][seqlen], io dtype), from the same inputs as the forward and the
 * forward's checkpoints (ssm_scan_fwd_train).  Reverse-mode differentiation of the recurrence
 * with the adjoint state lambda_t = dy_t C_t + Abar_{t+1} lambda_{t+1}; the pages state the
 * speed-up of this layer for training (53ai.com article, sections on the hardware-aware
 * algorithm and its training speed), the steps follow from the forward definitions.
 *   du, ddelta, dz : [batch][dim][seqlen], io dtype; ddelta is with respect to the raw delta.
 *                    dz is written only when z is given (nullable).
 *   dA             : [dim][dstate] float32, summed over the batch.
 *   dB, dC         : [batch][dstate][seqlen] float32, summed over the channels.
 *   dD, ddt_bias   : [dim] float32 (written only when D / dt_bias are given; nullable).
 *   dh0            : [batch][dim][dstate] float32, the gradient of the initial state (nullable).
 * The accumulated outputs (dA, dB, dC, dD, ddt_bias) are overwritten, not added to; atomics
 * make their last bits depend on the order of the additions.  No output may alias an input.
 * Required: u, delta, A, B, C, checkpoints, dout, du, ddelta, dA, dB, dC.
 * Returns an ssm_status.
 */
int ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* dt_bias, int delta_softplus, const float* checkpoints,
                 const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz,
                 float* ddt_bias, float* dh0, int batch, int dim, int dstate, int seqlen, int io_dtype,
                 void* stream);

/*
 * ssm_scan_bwd with a choice of discretization (an ssm_discretization value; anything else
 * returns SSM_ERR_ARG).  Under SSM_DISC_ZOH the B term is c B u with c = (exp(Delta A) - 1) / A,
 * so dB and du carry c in place of Delta, dDelta gains exp(Delta A) B u in place of B u, and dA
 * gains dc/dA B u, dc/dA = (Delta exp(Delta A) - c) / A (its limit Delta^2 / 2 at A = 0).  The
 * checkpoints must come from ssm_scan_fwd_train_ex with the same discretization.  Arguments,
 * outputs and errors are otherwise those of ssm_scan_bwd, which equals this call with
 * SSM_DISC_DELTA_B.
 */
int ssm_scan_bwd_ex(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* checkpoints,
                    const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz,
                    float* ddt_bias, float* dh0, int batch, int dim, int dstate, int seqlen, int io_dtype,
                    int discretization, void* stream);

/*
 * Single-token decode step, state updated in place.
 *   state          : [batch][dim][dstate] float32, read and written.
 *   x, dt, z, out  : [batch][dim], io dtype.  dt is the raw step size.
 *   A              : [dim][dstate] float32.   B, C : [batch][dstate], io dtype.
 *   D, dt_bias     : [dim] float32.
 *   dt_softplus    : non-zero applies softplus to dt + dt_bias.
 * Required: state, x, dt, A, B, C, out.  Nullable: D, z, dt_bias.  With dt_bias
 * NULL and dt_softplus 0 the step size is dt itself.
 * Returns an ssm_status.
 */
int ssm_state_update(float* state, const void* x, const void* dt, const float* A, const void* B, const void* C,
                     const float* D, const void* z, const float* dt_bias, int dt_softplus, void* out, int batch,
                     int dim, int dstate, int io_dtype, void* stream);

/*
 * ssm_state_update with a choice of discretization (as ssm_scan_fwd_ex), so that a decode
 * continues a scan made with the same Bbar.  With SSM_DISC_DELTA_B it is exactly ssm_state_update.
 */
int ssm_state_update_ex(float* state, const void* x, const void* dt, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* dt_bias, int dt_softplus, void* out, int batch,
                        int dim, int dstate, int io_dtype, int discretization, void* stream);

/*
 * Causal depthwise conv1d, the step of the Mamba block that produces the scan's input u
 * (gsyq.cn page, SelectiveSSM sketch "卷积预处理": Conv1d(d_model, d_model, d_conv,
 * padding=d_conv-1, groups=d_model), of which the first L outputs are the causal ones;
 * datacamp tutorial, the causal-conv1d layer used inside the Mamba block).  For every
 * batch row b, channel d and step t, with W = width:
 *     out_t = act(bias[d] + sum_{k<W} weight[d,k] * x_{t-(W-1)+k}),  act = silu or identity
 * where the inputs before t = 0 are state_in (zeros when NULL).
 *   x, out             : [batch][dim][seqlen], io dtype (out must not alias x).
 *   weight             : [dim][width] float32.  bias : [dim] float32 (nullable).
 *   state_in           : [batch][dim][width-1], io dtype, the width-1 inputs before t = 0,
 *                        oldest first (nullable = zeros).
 *   state_out          : [batch][dim][width-1], io dtype, receives the width-1 last inputs of
 *                        concat(state_in, x) (nullable = not written; must not alias state_in).
 *                        Two calls carrying it equal one call over the concatenated rows.
 *   width              : 1..4 (SSM_ERR_UNSUPPORTED otherwise).  silu : non-zero applies silu.
 * Aliasing out/x or state_out/state_in returns SSM_ERR_ARG.  Returns an ssm_status.
 */
int ssm_causal_conv1d_fwd(const void* x, const float* weight, const float* bias, const void* state_in, void* out,
                          void* state_out, int batch, int dim, int seqlen, int width, int silu, int io_dtype,
                          void* stream);

/*
 * One decode step of the causal conv1d: out = act(bias + sum_{k<W-1} weight[d,k] state[k]
 * + weight[d,W-1] x), then state <- (state[1..W-2], x), in place.
 *   state : [batch][dim][width-1], io dtype (may be NULL when width == 1).
 *   x, out: [batch][dim], io dtype.  weight, bias: as ssm_causal_conv1d_fwd.
 * Returns an ssm_status.
 */
int ssm_causal_conv1d_update(void* state, const void* x, const float* weight, const float* bias, void* out,
                             int batch, int dim, int width, int silu, int io_dtype, void* stream);

/*
 * Throughput probes of the units the scan leans on (used to measure the peaks of the benchmark's
 * arithmetic rooflines on the machine it runs on).  kind:
 *   SSM_PROBE_EX2        ex2.approx alone;
 *   SSM_PROBE_FFMA       FP32 fused multiply-add alone;
 *   SSM_PROBE_FFMA2      packed f32x2 fused multiply-add alone;
 *   SSM_PROBE_EX2_FFMA2  one ex2 and one independent packed f32x2 FMA per chain step (counted in
 *                        ex2 operations): whether the special-function and FP32 pipes overlap;
 *   SSM_PROBE_RECURRENCE the scan's arithmetic per pair of states and step, with no memory
 *                        traffic: f32x2 Delta*A, two ex2, f32x2 (Delta*u)*B, f32x2 h = Abar*h + b,
 *                        f32x2 y += C*h (counted in state-steps, two per pair and step);
 *   SSM_PROBE_WAIT_TIMEOUT  the forward kernels' bounded barrier wait on a barrier that nothing
 *                        completes, with a limit of 2^20 cycles: each CTA must give up and writes
 *                        the cycles it waited (-1 if the wait completed); ops_per_cta is 0.
 * Launches nblocks CTAs (use the SM count: one CTA per SM) of independent dependency chains and
 * writes each CTA's clock cycles for the measured loop to cycles[0..nblocks-1] (device memory,
 * int64).  ssm_probe_ops_per_cta(kind) is the number of operations one CTA performs in those
 * units (lane-operations for the single-unit kinds, an f32x2 operation counting as two), so
 * ops / cycles is the rate per SM per clock.  Returns an ssm_status (SSM_ERR_ARG for an unknown
 * kind); ssm_probe_ops_per_cta returns 0 for an unknown kind.
 */
typedef enum {
  SSM_PROBE_EX2 = 0,
  SSM_PROBE_FFMA = 1,
  SSM_PROBE_FFMA2 = 2,
  SSM_PROBE_EX2_FFMA2 = 3,
  SSM_PROBE_RECURRENCE = 4,
  SSM_PROBE_WAIT_TIMEOUT = 5
} ssm_probe_kind;
int ssm_probe_cycles(int kind, long long* cycles, int nblocks, void* stream);
double ssm_probe_ops_per_cta(int kind);

/*
 * Inside the forward kernels the warps that load and prepare each chunk hand it to the warps that
 * run the recurrence through shared-memory barriers, and the decode step's bulk-copy form waits on
 * a barrier for each tile's copies.  Every such wait is bounded (about a second); a wait that gives
 * up ends the kernel early, leaving its outputs and states undefined, and is counted.  This writes the number of such waits since the library was loaded to *count (after
 * synchronising the device).  A correct build never gives up: non-zero means a defect or a device
 * that stopped a kernel's warps for over a second.  Returns SSM_OK, SSM_ERR_NULL or SSM_ERR_LAUNCH.
 */
int ssm_wait_timeouts(unsigned long long* count);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* ssm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H_ */
