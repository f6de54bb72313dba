/*
 * ssm_oracle.c -- float64 CPU oracle for the Mamba selective scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header or table with the CUDA
 * library: both sides only receive the same seeded input arrays.
 *
 * What it computes (plain definitions, no blocking, fusion or reordering):
 *
 *   Step size      Delta = softplus(delta + dt_bias[d])  (softplus optional,
 *                  dt_bias optional).  Selection makes Delta input dependent:
 *                  "Mamba 状态空间模型深度解析" (gsyq.cn), section
 *                  "选择性机制的设计理念" (Delta = Softplus(Linear(x))), and the
 *                  VMamba notes (genhiy.github.io), section
 *                  "mamba：从S4到S6的算法变化流程" (tau_Delta = softplus).
 *   Discretisation Abar = exp(Delta * A[d,n]) (zero-order hold for a diagonal
 *                  A) and Bbar*x = Delta * B[n] * u: gsyq.cn page, sections
 *                  "连续到离散的转换" and "硬件优化并行扫描算法" (A_bar =
 *                  exp(Delta*A), B_bar = Delta*B); VMamba notes, "离散化SSM".
 *                  With zoh set, Bbar is the exact zero-order hold instead:
 *                  Bbar = (Delta A)^-1 (exp(Delta A) - I) Delta B, which for a
 *                  diagonal A is (exp(Delta A[d,n]) - 1) / A[d,n] * B[n], and
 *                  Delta * B[n] where A[d,n] = 0 (its limit): gsyq.cn page,
 *                  "连续到离散的转换"; VMamba notes, section on the dimensions
 *                  of A, B, C ("S4中三个矩阵的维度表示、维度变化").
 *   Recurrence     h_t = Abar_t * h_{t-1} + Bbar_t * x_t, h_{-1} = h0 (zero
 *                  when not given): gsyq.cn page, the sequential loop in
 *                  "计算复杂度分析"; VMamba notes, "循环结构表示以快速推理".
 *   Readout        y_t = sum_n C_t[n] h_t[n] + D[d] * u_t: gsyq.cn page,
 *                  "核心数学形式" (y = C h + D x) and the D*x skip returned
 *                  by the SelectiveSSM sketch.
 *   Gate           out_t = y_t * silu(z_t), silu(z) = z / (1 + exp(-z)), the
 *                  gated-MLP merge of the Mamba block (VMamba notes,
 *                  "简化的SSM架构").
 *   Channels       every (batch, channel d) runs its own SSM; B and C are
 *                  shared by all channels of a batch row (VMamba notes,
 *                  "S4中三个矩阵的维度表示、维度变化": B, C of shape (B,L,N),
 *                  Delta of shape (B,L,D)).
 *   Decode step    the same single recurrence step applied to a stored state
 *                  (constant-memory inference: gsyq.cn page, complexity table
 *                  row "推理内存 O(d) 状态向量").
 *   Backward       reverse-mode gradients of the scan (either B discretisation) for a
 *                  loss whose gradient with respect to the outputs is dout:
 *                  the same recurrence run backwards with the adjoint state
 *                  lambda_t = dy_t C_t + Abar_{t+1} lambda_{t+1} (chain rule
 *                  through h_t = Abar_t h_{t-1} + Delta_t B_t u_t).  Training
 *                  is where the pages' speed claims are made (53ai.com
 *                  article, sections on the hardware-aware algorithm and the
 *                  training speed-up); the steps follow from the forward
 *                  definitions above and nothing else.
 *   Causal conv    depthwise causal convolution of width W over time, one
 *                  filter per channel, before the scan:
 *                    out_t = act(bias[d] + sum_k w[d,k] * x_{t-(W-1)+k}),
 *                  inputs before t = 0 taken from a carried state of the W-1
 *                  previous inputs (zeros when not given), act = silu or none.
 *                  gsyq.cn page, SelectiveSSM sketch ("卷积预处理":
 *                  Conv1d(d_model, d_model, d_conv, padding=d_conv-1,
 *                  groups=d_model), whose first L outputs are the causal
 *                  ones); datacamp tutorial, install notes (the causal-conv1d
 *                  layer used inside the Mamba block).
 *   Associative    the pair operator (a1,b1) o (a2,b2) = (a1*a2, a2*b1 + b2)
 *   scan           evaluated in tree order (53ai.com Mamba article, section
 *                  3.3 "Parallel Associative Scan": grouping does not change a
 *                  prefix result; gsyq.cn page, "硬件优化并行扫描算法").
 *
 * Layouts (all row-major, all float64, all host memory owned by the caller):
 *   u, delta, z, y          [batch][dim][seqlen]
 *   B, C                    [batch][dstate][seqlen]
 *   A                       [dim][dstate]      (continuous A, e.g. -exp(A_log))
 *   D, dt_bias              [dim]
 *   h0, last_state, state   [batch][dim][dstate]
 *   decode x, dt, z, out    [batch][dim];  decode B, C [batch][dstate]
 *
 * Channels are independent and each runs sequentially in t, so results do not
 * depend on the OpenMP thread count.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
static double softplus_f64(double x) {
  if (x > 0.0) return x + log1p(exp(-x));
  return log1p(exp(x));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
static double silu_f64(double z) { return z / (1.0 + exp(-z)); }

/* The factor Bbar / B[n] of the discretisation: Delta (Delta*B form) or the exact
 * zero-order-hold (exp(Delta*a) - 1) / a, whose limit at a = 0 is Delta. */
static double bbar_factor(double dt, double a, int zoh) {
  if (!zoh || a == 0.0) return dt;
  return expm1(dt * a) / a;
}

static double step_size(double raw, const double* dt_bias, int d, int use_softplus) {
  double v = raw;
  if (dt_bias) v += dt_bias[d];
  if (use_softplus) v = softplus_f64(v);
  return v;
}

int oracle_abi_version(void) { return 3; }

/* Selective scan over seqlen steps for every (batch, channel). */
int oracle_scan_f64(const double* u, const double* delta, const double* A, const double* B, const double* C,
                    const double* D, const double* z, const double* dt_bias, int delta_softplus, int zoh,
                    const double* h0, double* y, double* last_state, int batch, int dim, int dstate, int seqlen,
                    int nthreads) {
  if (!u || !delta || !A || !B || !C || !y) return -1;
  if (batch < 0 || dim < 0 || dstate < 1 || seqlen < 0) return -2;
  long nch = (long)batch * dim;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (long ch = 0; ch < nch; ++ch) {
    int b = (int)(ch / dim), d = (int)(ch % dim);
    double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
    for (int n = 0; n < dstate; ++n) h[n] = h0 ? h0[ch * dstate + n] : 0.0;
    const double* u_row = u + ch * seqlen;
    const double* dl_row = delta + ch * seqlen;
    const double* z_row = z ? z + ch * seqlen : NULL;
    double* y_row = y + ch * seqlen;
    for (int t = 0; t < seqlen; ++t) {
      double dt = step_size(dl_row[t], dt_bias, d, delta_softplus);
      double x = u_row[t];
      double acc = 0.0;
      for (int n = 0; n < dstate; ++n) {
        double a = A[(long)d * dstate + n];
        double abar = exp(dt * a);
        double bx = bbar_factor(dt, a, zoh) * B[((long)b * dstate + n) * seqlen + t] * x;
        h[n] = abar * h[n] + bx;
        acc += C[((long)b * dstate + n) * seqlen + t] * h[n];
      }
      if (D) acc += D[d] * x;
      if (z_row) acc *= silu_f64(z_row[t]);
      y_row[t] = acc;
    }
    if (last_state)
      for (int n = 0; n < dstate; ++n) last_state[ch * dstate + n] = h[n];
    free(h);
  }
  return 0;
}

/* One decode step: state <- Abar*state + Bbar*x in place, out = (C.state + D x) * silu(z). */
int oracle_state_update_f64(double* state, const double* x, const double* dt, const double* A, const double* B,
                            const double* C, const double* D, const double* z, const double* dt_bias,
                            int dt_softplus, int zoh, double* out, int batch, int dim, int dstate, int nthreads) {
  if (!state || !x || !dt || !A || !B || !C || !out) return -1;
  if (batch < 0 || dim < 0 || dstate < 1) return -2;
  long nch = (long)batch * dim;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
  for (long ch = 0; ch < nch; ++ch) {
    int b = (int)(ch / dim), d = (int)(ch % dim);
    double step = step_size(dt[ch], dt_bias, d, dt_softplus);
    double acc = 0.0;
    for (int n = 0; n < dstate; ++n) {
      double* s = &state[ch * dstate + n];
      double a = A[(long)d * dstate + n];
      double abar = exp(step * a);
      *s = abar * *s + bbar_factor(step, a, zoh) * B[(long)b * dstate + n] * x[ch];
      acc += C[(long)b * dstate + n] * *s;
    }
    if (D) acc += D[d] * x[ch];
    if (z) acc *= silu_f64(z[ch]);
    out[ch] = acc;
  }
  return 0;
}

/* d silu / dz = sigmoid(z) * (1 + z * (1 - sigmoid(z))). */
static double dsilu_f64(double z) {
  double sg = 1.0 / (1.0 + exp(-z));
  return sg * (1.0 + z * (1.0 - sg));
}

/*
 * Gradients of the scan (Delta*B form, or the exact zero-order hold with zoh set) given
 * dout = dLoss/dout, same layouts as the forward.  Outputs (all overwritten, summed over what the parameter is shared by):
 *   du, ddelta, dz        [batch][dim][seqlen]   (dz only when z is given; NULL skips it)
 *   dA                    [dim][dstate]          (summed over batch)
 *   dB, dC                [batch][dstate][seqlen] (summed over channels)
 *   dD, ddt_bias          [dim]                  (summed over batch and time; NULL skips)
 *   dh0                   [batch][dim][dstate]   (gradient of the initial state; NULL skips)
 * ddelta is with respect to the raw delta (before dt_bias and softplus).
 * abs_dA, abs_dB, abs_dC, abs_dD, abs_ddt_bias (each nullable, shaped like its gradient) receive
 * the sum of the absolute values of the terms that the gradient sums (for dA and d dt_bias, of
 * each term's parts): the scale that floating-point summation error is proportional to, which
 * lets a float32 result be held to a bound per element.  They do not change the gradients.
 */
int oracle_scan_bwd_f64(const double* u, const double* delta, const double* A, const double* B, const double* C,
                        const double* D, const double* z, const double* dt_bias, int delta_softplus, int zoh,
                        const double* h0, const double* dout, double* du, double* ddelta, double* dA, double* dB,
                        double* dC, double* dD, double* dz, double* ddt_bias, double* dh0, int batch, int dim,
                        int dstate, int seqlen, double* abs_dA, double* abs_dB, double* abs_dC, double* abs_dD,
                        double* abs_ddt_bias) {
  if (!u || !delta || !A || !B || !C || !dout || !du || !ddelta || !dA || !dB || !dC) return -1;
  if (batch < 0 || dim < 0 || dstate < 1 || seqlen < 0) return -2;
  long N = dstate, L = seqlen;
  for (long i = 0; i < (long)dim * N; ++i) dA[i] = 0.0;
  for (long i = 0; i < (long)batch * N * L; ++i) dB[i] = dC[i] = 0.0;
  if (dD) for (int i = 0; i < dim; ++i) dD[i] = 0.0;
  if (ddt_bias) for (int i = 0; i < dim; ++i) ddt_bias[i] = 0.0;
  if (abs_dA) for (long i = 0; i < (long)dim * N; ++i) abs_dA[i] = 0.0;
  if (abs_dB) for (long i = 0; i < (long)batch * N * L; ++i) abs_dB[i] = 0.0;
  if (abs_dC) for (long i = 0; i < (long)batch * N * L; ++i) abs_dC[i] = 0.0;
  if (abs_dD) for (int i = 0; i < dim; ++i) abs_dD[i] = 0.0;
  if (abs_ddt_bias) for (int i = 0; i < dim; ++i) abs_ddt_bias[i] = 0.0;
  double* hs = (double*)malloc(sizeof(double) * (size_t)((L + 1) * N + 1)); /* hs[(t+1)*N + n] = h_t */
  double* carry = (double*)malloc(sizeof(double) * (size_t)N);
  double* ys = (double*)malloc(sizeof(double) * (size_t)(L + 1));
  double* dts = (double*)malloc(sizeof(double) * (size_t)(L + 1));
  for (long ch = 0; ch < (long)batch * dim; ++ch) {
    int b = (int)(ch / dim), d = (int)(ch % dim);
    const double* ur = u + ch * L;
    const double* dr = delta + ch * L;
    const double* zr = z ? z + ch * L : NULL;
    const double* gr = dout + ch * L;
    /* forward, keeping every state */
    for (long n = 0; n < N; ++n) hs[n] = h0 ? h0[ch * N + n] : 0.0;
    for (long t = 0; t < L; ++t) {
      double dt = step_size(dr[t], dt_bias, d, delta_softplus);
      dts[t] = dt;
      double acc = 0.0;
      for (long n = 0; n < N; ++n) {
        double an = A[(long)d * N + n];
        double a = exp(dt * an);
        double h = a * hs[t * N + n] + bbar_factor(dt, an, zoh) * B[((long)b * N + n) * L + t] * ur[t];
        hs[(t + 1) * N + n] = h;
        acc += C[((long)b * N + n) * L + t] * h;
      }
      if (D) acc += D[d] * ur[t];
      ys[t] = acc; /* before the gate */
    }
    /* backward */
    for (long n = 0; n < N; ++n) carry[n] = 0.0;
    for (long t = L - 1; t >= 0; --t) {
      double dt = dts[t];
      double dy = zr ? gr[t] * silu_f64(zr[t]) : gr[t];
      if (zr && dz) dz[ch * L + t] = gr[t] * ys[t] * dsilu_f64(zr[t]);
      if (D && dD) dD[d] += dy * ur[t];
      if (D && abs_dD) abs_dD[d] += fabs(dy * ur[t]);
      double dut = D ? dy * D[d] : 0.0;
      double ddt = 0.0, ddt_abs = 0.0;
      for (long n = 0; n < N; ++n) {
        double an = A[(long)d * N + n];
        double a = exp(dt * an);
        double bn = B[((long)b * N + n) * L + t];
        double hp = hs[t * N + n];        /* h_{t-1} */
        double lam = dy * C[((long)b * N + n) * L + t] + carry[n];
        /* Bbar = c B with c = Delta (Delta*B form) or (exp(Delta a) - 1) / a (zero-order hold):
         * dc/dDelta = 1 or exp(Delta a); dc/da = 0 or (Delta exp(Delta a) - c) / a, whose limit
         * at Delta a -> 0 is Delta^2 (1/2 + x/3 + x^2/8 + x^3/30 + ...), x = Delta a. */
        double c = bbar_factor(dt, an, zoh), dc_ddt = 1.0, dc_da = 0.0;
        if (zoh) {
          double x = dt * an;
          dc_ddt = a;
          dc_da = fabs(x) < 1e-3 ? dt * dt * (0.5 + x / 3.0 + x * x / 8.0 + x * x * x / 30.0) : (dt * a - c) / an;
        }
        dC[((long)b * N + n) * L + t] += dy * hs[(t + 1) * N + n];
        dB[((long)b * N + n) * L + t] += lam * c * ur[t];
        dut += lam * c * bn;
        ddt += lam * (an * a * hp + dc_ddt * bn * ur[t]);
        dA[(long)d * N + n] += lam * (dt * a * hp + dc_da * bn * ur[t]);
        carry[n] = lam * a;
        if (abs_dC) abs_dC[((long)b * N + n) * L + t] += fabs(dy * hs[(t + 1) * N + n]);
        if (abs_dB) abs_dB[((long)b * N + n) * L + t] += fabs(lam * c * ur[t]);
        if (abs_dA) abs_dA[(long)d * N + n] += fabs(lam * (dt * a * hp)) + fabs(lam * (dc_da * bn * ur[t]));
        ddt_abs += fabs(lam * an * a * hp) + fabs(lam * dc_ddt * bn * ur[t]);
      }
      du[ch * L + t] = dut;
      double raw = dr[t] + (dt_bias ? dt_bias[d] : 0.0);
      double dd = delta_softplus ? ddt / (1.0 + exp(-raw)) : ddt; /* softplus' = sigmoid */
      ddelta[ch * L + t] = dd;
      if (ddt_bias && dt_bias) ddt_bias[d] += dd;
      if (abs_ddt_bias && dt_bias) abs_ddt_bias[d] += delta_softplus ? ddt_abs / (1.0 + exp(-raw)) : ddt_abs;
    }
    if (dh0)
      for (long n = 0; n < N; ++n) dh0[ch * N + n] = carry[n];
  }
  free(hs);
  free(carry);
  free(ys);
  free(dts);
  return 0;
}

/*
 * Inclusive scan of the pairs (a_t, b_t) under (a1,b1) o (a2,b2) = (a1*a2, a2*b1 + b2),
 * evaluated in tree order (recursive doubling: after round k every position holds the
 * combination of the 2^k pairs ending at it).  The b component of the result is the
 * recurrence h_t = a_t h_{t-1} + b_t from h_{-1} = 0; the a component is the running
 * product of the a's.  With a == 1 it is a plain prefix sum.
 */
int oracle_assoc_scan_pairs_f64(const double* a, const double* b, double* out_a, double* out_b, int n) {
  if (n < 0 || (n > 0 && (!a || !b || !out_a || !out_b))) return -1;
  double* pa = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* pb = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int i = 0; i < n; ++i) { out_a[i] = a[i]; out_b[i] = b[i]; }
  for (int off = 1; off < n; off *= 2) {
    for (int i = 0; i < n; ++i) { pa[i] = out_a[i]; pb[i] = out_b[i]; }
    for (int i = off; i < n; ++i) {
      /* left operand: the block ending at i-off; right operand: the block ending at i */
      double la = pa[i - off], lb = pb[i - off];
      double ra = pa[i], rb = pb[i];
      out_a[i] = la * ra;
      out_b[i] = ra * lb + rb;
    }
  }
  free(pa);
  free(pb);
  return 0;
}

/*
 * The selective scan with the recurrence evaluated by the tree-order pair scan
 * above instead of the sequential loop (same discretisation and readout).
 */
int oracle_scan_tree_f64(const double* u, const double* delta, const double* A, const double* B, const double* C,
                         const double* D, const double* z, const double* dt_bias, int delta_softplus, double* y,
                         double* last_state, int batch, int dim, int dstate, int seqlen) {
  if (!u || !delta || !A || !B || !C || !y) return -1;
  if (batch < 0 || dim < 0 || dstate < 1 || seqlen < 1) return -2;
  double* a = (double*)malloc(sizeof(double) * (size_t)seqlen);
  double* bx = (double*)malloc(sizeof(double) * (size_t)seqlen);
  double* pa = (double*)malloc(sizeof(double) * (size_t)seqlen);
  double* h = (double*)malloc(sizeof(double) * (size_t)seqlen * dstate);
  for (long ch = 0; ch < (long)batch * dim; ++ch) {
    int b = (int)(ch / dim), d = (int)(ch % dim);
    for (int n = 0; n < dstate; ++n) {
      for (int t = 0; t < seqlen; ++t) {
        double dt = step_size(delta[ch * seqlen + t], dt_bias, d, delta_softplus);
        a[t] = exp(dt * A[(long)d * dstate + n]);
        bx[t] = dt * B[((long)b * dstate + n) * seqlen + t] * u[ch * seqlen + t];
      }
      oracle_assoc_scan_pairs_f64(a, bx, pa, h + (long)n * seqlen, seqlen);
    }
    for (int t = 0; t < seqlen; ++t) {
      double acc = 0.0;
      for (int n = 0; n < dstate; ++n) acc += C[((long)b * dstate + n) * seqlen + t] * h[(long)n * seqlen + t];
      if (D) acc += D[d] * u[ch * seqlen + t];
      if (z) acc *= silu_f64(z[ch * seqlen + t]);
      y[ch * seqlen + t] = acc;
    }
    if (last_state)
      for (int n = 0; n < dstate; ++n) last_state[ch * dstate + n] = h[(long)n * seqlen + seqlen - 1];
  }
  free(a);
  free(bx);
  free(pa);
  free(h);
  return 0;
}

/*
 * Causal depthwise conv1d of width W over [batch][dim][seqlen] inputs.  state_in holds, per
 * (batch, channel), the W-1 inputs that precede t = 0 (oldest first; NULL = zeros);
 * state_out receives the W-1 last inputs of concat(state_in, x) (NULL = not written).
 * weight [dim][W], bias [dim] (NULL = 0); silu non-zero applies silu to each output.
 */
int oracle_causal_conv1d_f64(const double* x, const double* weight, const double* bias, const double* state_in,
                             double* out, double* state_out, int batch, int dim, int seqlen, int width, int silu) {
  if (!x || !weight || !out) return -1;
  if (batch < 0 || dim < 0 || seqlen < 0 || width < 1) return -2;
  int hw = width - 1;
  for (long ch = 0; ch < (long)batch * dim; ++ch) {
    int d = (int)(ch % dim);
    const double* xr = x + ch * seqlen;
    const double* sr = state_in ? state_in + ch * hw : NULL;
    for (int t = 0; t < seqlen; ++t) {
      double acc = bias ? bias[d] : 0.0;
      for (int k = 0; k < width; ++k) {
        int s = t - hw + k; /* input time index */
        double v = s >= 0 ? xr[s] : (sr ? sr[hw + s] : 0.0);
        acc += weight[(long)d * width + k] * v;
      }
      out[ch * seqlen + t] = silu ? silu_f64(acc) : acc;
    }
    if (state_out)
      for (int j = 0; j < hw; ++j) {
        int s = seqlen - hw + j; /* time index of state slot j */
        state_out[ch * hw + j] = s >= 0 ? xr[s] : (sr ? sr[hw + s] : 0.0);
      }
  }
  return 0;
}

/* Exposed for the pin tests: the scalar helpers exactly as the scan uses them. */
double oracle_softplus_f64(double x) { return softplus_f64(x); }
double oracle_silu_f64(double z) { return silu_f64(z); }
