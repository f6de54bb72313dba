// extern "C" entry points of the library: host-side validation, then the launches on the caller's
// stream.  Nothing here synchronises or keeps state between calls; the only allocation is the
// stream-ordered carry buffer of a split scan called without a workspace (ssm_scan_fwd_ws never
// allocates).
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ssm_scan.h"

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t io_size(int io) { return io == SSM_F32 ? 4 : 2; }

// Whether the byte ranges [p, p + np) and [q, q + nq) share a byte (a NULL pointer shares none).
bool overlaps(const void* p, size_t np, const void* q, size_t nq) {
  if (!p || !q || np == 0 || nq == 0) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
  return a < b + nq && b < a + np;
}

}  // namespace

extern "C" {

int ssm_abi_version(void) { return 7; }

const char* ssm_status_string(int status) {
  switch (status) {
    case SSM_OK: return "ok";
    case SSM_ERR_NULL: return "a required pointer is NULL";
    case SSM_ERR_SHAPE: return "a size is negative or dstate < 1";
    case SSM_ERR_DTYPE: return "io_dtype is not SSM_F32 or SSM_BF16";
    case SSM_ERR_ALIGN: return "a pointer is not aligned to its element size";
    case SSM_ERR_UNSUPPORTED: return "unsupported size (dstate > 16 or grid overflow)";
    case SSM_ERR_LAUNCH: return "the CUDA kernel launch failed";
    case SSM_ERR_TIMEOUT: return "a bounded in-kernel wait gave up";
    case SSM_ERR_ARG: return "an enumerated argument is out of range, or buffers alias that must not";
    default: return "unknown status";
  }
}

}  // extern "C"

namespace {

int scan_fwd_common(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* h0, void* y,
                    float* last_state, float* ckpt, int batch, int dim, int dstate, int seqlen, int io_dtype,
                    int discretization, void* stream, bool ws_given = false, void* ws = nullptr,
                    size_t ws_bytes = 0) {
  if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return SSM_ERR_SHAPE;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
  if (discretization != SSM_DISC_DELTA_B && discretization != SSM_DISC_ZOH) return SSM_ERR_ARG;
  if (dstate > 16) return SSM_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0) return SSM_OK;
  if (!A) return SSM_ERR_NULL;
  if (seqlen > 0 && (!u || !delta || !B || !C || !y)) return SSM_ERR_NULL;
  if (seqlen == 0 && !last_state) return SSM_OK;
  const size_t es = io_size(io_dtype);
  const void* io_ptrs[] = {u, delta, B, C, z, y};
  for (const void* p : io_ptrs)
    if (!aligned(p, es)) return SSM_ERR_ALIGN;
  const void* f_ptrs[] = {A, D, dt_bias, h0, last_state};
  for (const void* p : f_ptrs)
    if (!aligned(p, 4)) return SSM_ERR_ALIGN;
  if ((long long)((dim + 31) / 32) * batch > 0x7fffffffLL) return SSM_ERR_UNSUPPORTED;
  // y is written while the inputs are still being read, so it must not overlap any of them; the
  // checkpoints likewise must not overlap y, the state buffers or the inputs they are read with
  const size_t ny = size_t(batch) * dim * seqlen * es, nbc = size_t(batch) * dstate * seqlen * es;
  const size_t nst = size_t(batch) * dim * dstate * 4;
  if (overlaps(y, ny, u, ny) || overlaps(y, ny, delta, ny) || overlaps(y, ny, z, ny) || overlaps(y, ny, B, nbc) ||
      overlaps(y, ny, C, nbc))
    return SSM_ERR_ARG;
  if (ckpt) {
    const size_t nck = size_t(batch) * ssm_scan_num_checkpoints(seqlen) * dim * dstate * 4;
    if (overlaps(ckpt, nck, y, ny) || overlaps(ckpt, nck, last_state, nst) || overlaps(ckpt, nck, h0, nst) ||
        overlaps(ckpt, nck, u, ny) || overlaps(ckpt, nck, delta, ny))
      return SSM_ERR_ARG;
  }
  // the workspace is written while every other buffer is in use
  if (ws_given && ws && ws_bytes > 0) {
    if (!aligned(ws, 16)) return SSM_ERR_ALIGN;
    const size_t nA = size_t(dim) * dstate * 4, nd = size_t(dim) * 4;
    if (overlaps(ws, ws_bytes, u, ny) || overlaps(ws, ws_bytes, delta, ny) || overlaps(ws, ws_bytes, z, ny) ||
        overlaps(ws, ws_bytes, y, ny) || overlaps(ws, ws_bytes, B, nbc) || overlaps(ws, ws_bytes, C, nbc) ||
        overlaps(ws, ws_bytes, last_state, nst) || overlaps(ws, ws_bytes, h0, nst) || overlaps(ws, ws_bytes, A, nA) ||
        overlaps(ws, ws_bytes, D, nd) || overlaps(ws, ws_bytes, dt_bias, nd))
      return SSM_ERR_ARG;
  }

  ssm::ScanArgs a{};
  a.u = u, a.delta = delta, a.A = A, a.B = B, a.C = C, a.D = D, a.z = z, a.dt_bias = dt_bias, a.h0 = h0;
  a.y = y, a.last_state = last_state;
  a.batch = batch, a.dim = dim, a.dstate = dstate, a.seqlen = seqlen;
  a.softplus = delta_softplus ? 1 : 0;
  a.io = io_dtype == SSM_F32 ? ssm::kF32 : ssm::kBF16;
  a.zoh = discretization == SSM_DISC_ZOH ? 1 : 0;
  a.ckpt = ckpt;
  a.ws_given = ws_given ? 1 : 0, a.ws = ws, a.ws_bytes = ws_bytes;
  const cudaError_t err = ssm::launch_scan_fwd(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int ssm_scan_fwd_ex(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* h0, void* y,
                    float* last_state, int batch, int dim, int dstate, int seqlen, int io_dtype, int discretization,
                    void* stream) {
  return scan_fwd_common(u, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, y, last_state, nullptr, batch, dim,
                         dstate, seqlen, io_dtype, discretization, stream);
}

int ssm_scan_fwd_ws(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* h0, void* y,
                    float* last_state, int batch, int dim, int dstate, int seqlen, int io_dtype, int discretization,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return scan_fwd_common(u, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, y, last_state, nullptr, batch, dim,
                         dstate, seqlen, io_dtype, discretization, stream, true, workspace, workspace_bytes);
}

int ssm_scan_fwd_workspace_size(int batch, int dim, int dstate, int seqlen, int io_dtype, int discretization,
                                int aligned_rows, size_t* bytes) {
  if (!bytes) return SSM_ERR_NULL;
  *bytes = 0;
  if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return SSM_ERR_SHAPE;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
  if (discretization != SSM_DISC_DELTA_B && discretization != SSM_DISC_ZOH) return SSM_ERR_ARG;
  if (dstate > 16) return SSM_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0 || seqlen == 0) return SSM_OK;
  ssm::ScanArgs a{};
  a.batch = batch, a.dim = dim, a.dstate = dstate, a.seqlen = seqlen;
  a.io = io_dtype == SSM_F32 ? ssm::kF32 : ssm::kBF16;
  a.zoh = discretization == SSM_DISC_ZOH ? 1 : 0;
  const bool vec = aligned_rows != 0 && (size_t(seqlen) * io_size(io_dtype)) % 16 == 0;
  ssm::SplitPlan p{};
  if (ssm::scan_fwd_split(a, vec, p) != cudaSuccess) return SSM_ERR_LAUNCH;
  *bytes = p.segs > 0 ? p.workspace_bytes : 0;
  return SSM_OK;
}

int ssm_scan_num_checkpoints(int seqlen) {
  return seqlen > 0 ? (seqlen + SSM_SCAN_CHECKPOINT_STEPS - 1) / SSM_SCAN_CHECKPOINT_STEPS : 0;
}

int ssm_scan_fwd_train_ex(const void* u, const void* delta, const float* A, const void* B, const void* C,
                          const float* D, const void* z, const float* dt_bias, int delta_softplus, const float* h0,
                          void* y, float* last_state, float* checkpoints, int batch, int dim, int dstate, int seqlen,
                          int io_dtype, int discretization, void* stream) {
  static_assert(SSM_SCAN_CHECKPOINT_STEPS == ssm::kCkptSteps, "checkpoint interval");
  if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return SSM_ERR_SHAPE;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
  if (discretization != SSM_DISC_DELTA_B && discretization != SSM_DISC_ZOH) return SSM_ERR_ARG;
  if (dstate > 16) return SSM_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0 || seqlen == 0) {
    return ssm_scan_fwd_ex(u, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, y, last_state, batch, dim, dstate,
                           seqlen, io_dtype, discretization, stream);
  }
  if (!checkpoints) return SSM_ERR_NULL;
  if (!aligned(checkpoints, 4)) return SSM_ERR_ALIGN;
  return scan_fwd_common(u, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, y, last_state, checkpoints, batch,
                         dim, dstate, seqlen, io_dtype, discretization, stream);
}

int ssm_scan_fwd_train(const void* u, const void* delta, const float* A, const void* B, const void* C,
                       const float* D, const void* z, const float* dt_bias, int delta_softplus, const float* h0,
                       void* y, float* last_state, float* checkpoints, int batch, int dim, int dstate, int seqlen,
                       int io_dtype, void* stream) {
  return ssm_scan_fwd_train_ex(u, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, y, last_state, checkpoints,
                               batch, dim, dstate, seqlen, io_dtype, SSM_DISC_DELTA_B, stream);
}

int ssm_scan_fwd_form(int batch, int dim, int dstate, int seqlen, int io_dtype, int discretization, int aligned_rows,
                      int* ctas) {
  if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return SSM_ERR_SHAPE;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
  if (discretization != SSM_DISC_DELTA_B && discretization != SSM_DISC_ZOH) return SSM_ERR_ARG;
  if (dstate > 16) return SSM_ERR_UNSUPPORTED;
  ssm::ScanArgs a{};
  a.batch = batch, a.dim = dim, a.dstate = dstate, a.seqlen = seqlen;
  a.io = io_dtype == SSM_F32 ? ssm::kF32 : ssm::kBF16;
  a.zoh = discretization == SSM_DISC_ZOH ? 1 : 0;
  const bool vec = aligned_rows != 0 && (size_t(seqlen) * io_size(io_dtype)) % 16 == 0;
  int form = 0, n = 0;
  if (ssm::scan_fwd_form(a, vec, form, n) != cudaSuccess) return SSM_ERR_LAUNCH;
  if (ctas) *ctas = n;
  return form;
}

int ssm_scan_fwd_h0(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* h0, void* y,
                    float* last_state, int batch, int dim, int dstate, int seqlen, int io_dtype, void* stream) {
  return ssm_scan_fwd_ex(u, delta, A, B, C, D, z, dt_bias, delta_softplus, h0, y, last_state, batch, dim, dstate,
                         seqlen, io_dtype, SSM_DISC_DELTA_B, stream);
}

int ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* dt_bias, int delta_softplus, void* y, float* last_state, int batch,
                 int dim, int dstate, int seqlen, int io_dtype, void* stream) {
  return ssm_scan_fwd_h0(u, delta, A, B, C, D, z, dt_bias, delta_softplus, nullptr, y, last_state, batch, dim, dstate,
                         seqlen, io_dtype, stream);
}

int ssm_state_update_ex(float* state, const void* x, const void* dt, const float* A, const void* B, const void* C,
                        const float* D, const void* z, const float* dt_bias, int dt_softplus, void* out, int batch,
                        int dim, int dstate, int io_dtype, int discretization, void* stream) {
  if (batch < 0 || dim < 0 || dstate < 1) return SSM_ERR_SHAPE;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
  if (discretization != SSM_DISC_DELTA_B && discretization != SSM_DISC_ZOH) return SSM_ERR_ARG;
  if (dstate > 16) return SSM_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0) return SSM_OK;
  if (!state || !x || !dt || !A || !B || !C || !out) return SSM_ERR_NULL;
  const size_t es = io_size(io_dtype);
  const void* io_ptrs[] = {x, dt, B, C, z, out};
  for (const void* p : io_ptrs)
    if (!aligned(p, es)) return SSM_ERR_ALIGN;
  const void* f_ptrs[] = {state, A, D, dt_bias};
  for (const void* p : f_ptrs)
    if (!aligned(p, 4)) return SSM_ERR_ALIGN;
  if ((long long)batch * dim / 128 + 1 > 0x7fffffffLL) return SSM_ERR_UNSUPPORTED;

  ssm::UpdateArgs a{};
  a.state = state, a.x = x, a.dt = dt, a.A = A, a.B = B, a.C = C, a.D = D, a.z = z, a.dt_bias = dt_bias;
  a.out = out;
  a.batch = batch, a.dim = dim, a.dstate = dstate;
  a.softplus = dt_softplus ? 1 : 0;
  a.io = io_dtype == SSM_F32 ? ssm::kF32 : ssm::kBF16;
  a.zoh = discretization == SSM_DISC_ZOH ? 1 : 0;
  const cudaError_t err = ssm::launch_state_update(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

int ssm_state_update(float* state, const void* x, const void* dt, const float* A, const void* B, const void* C,
                     const float* D, const void* z, const float* dt_bias, int dt_softplus, void* out, int batch,
                     int dim, int dstate, int io_dtype, void* stream) {
  return ssm_state_update_ex(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, out, batch, dim, dstate, io_dtype,
                             SSM_DISC_DELTA_B, stream);
}

int ssm_scan_bwd_ex(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                    const void* z, const float* dt_bias, int delta_softplus, const float* checkpoints,
                    const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz,
                    float* ddt_bias, float* dh0, int batch, int dim, int dstate, int seqlen, int io_dtype,
                    int discretization, void* stream) {
  if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return SSM_ERR_SHAPE;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
  if (discretization != SSM_DISC_DELTA_B && discretization != SSM_DISC_ZOH) return SSM_ERR_ARG;
  if (dstate > 16) return SSM_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0) return SSM_OK;
  if (!A || !dA) return SSM_ERR_NULL;
  if (seqlen > 0 && (!u || !delta || !B || !C || !checkpoints || !dout || !du || !ddelta || !dB || !dC))
    return SSM_ERR_NULL;
  const size_t es = io_size(io_dtype);
  const void* io_ptrs[] = {u, delta, B, C, z, dout, du, ddelta, dz};
  for (const void* p : io_ptrs)
    if (!aligned(p, es)) return SSM_ERR_ALIGN;
  const void* f_ptrs[] = {A, D, dt_bias, checkpoints, dA, dB, dC, dD, ddt_bias, dh0};
  for (const void* p : f_ptrs)
    if (!aligned(p, 4)) return SSM_ERR_ALIGN;
  if ((long long)((dim + 31) / 32) * batch > 0x7fffffffLL) return SSM_ERR_UNSUPPORTED;

  ssm::ScanBwdArgs a{};
  a.u = u, a.delta = delta, a.A = A, a.B = B, a.C = C, a.D = D, a.z = z, a.dt_bias = dt_bias;
  a.ckpt = checkpoints, a.dout = dout;
  a.du = du, a.ddelta = ddelta, a.dA = dA, a.dB = dB, a.dC = dC, a.dD = dD, a.dz = dz, a.ddt_bias = ddt_bias;
  a.dh0 = dh0;
  a.batch = batch, a.dim = dim, a.dstate = dstate, a.seqlen = seqlen;
  a.softplus = delta_softplus ? 1 : 0;
  a.io = io_dtype == SSM_F32 ? ssm::kF32 : ssm::kBF16;
  a.zoh = discretization == SSM_DISC_ZOH ? 1 : 0;
  const cudaError_t err = ssm::launch_scan_bwd(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

int ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B, const void* C, const float* D,
                 const void* z, const float* dt_bias, int delta_softplus, const float* checkpoints,
                 const void* dout, void* du, void* ddelta, float* dA, float* dB, float* dC, float* dD, void* dz,
                 float* ddt_bias, float* dh0, int batch, int dim, int dstate, int seqlen, int io_dtype,
                 void* stream) {
  return ssm_scan_bwd_ex(u, delta, A, B, C, D, z, dt_bias, delta_softplus, checkpoints, dout, du, ddelta, dA, dB, dC,
                         dD, dz, ddt_bias, dh0, batch, dim, dstate, seqlen, io_dtype, SSM_DISC_DELTA_B, stream);
}

int ssm_causal_conv1d_fwd(const void* x, const float* weight, const float* bias, const void* state_in, void* out,
                          void* state_out, int batch, int dim, int seqlen, int width, int silu, int io_dtype,
                          void* stream) {
  if (batch < 0 || dim < 0 || seqlen < 0 || width < 1) return SSM_ERR_SHAPE;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
  if (width > 4) return SSM_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0) return SSM_OK;
  if (!weight) return SSM_ERR_NULL;
  if (seqlen > 0 && (!x || !out)) return SSM_ERR_NULL;
  if (seqlen == 0 && (!state_out || width == 1)) return SSM_OK;
  if (x && x == out) return SSM_ERR_ARG;
  if (state_in && state_in == state_out) return SSM_ERR_ARG;
  const size_t es = io_size(io_dtype);
  const void* io_ptrs[] = {x, out, state_in, state_out};
  for (const void* p : io_ptrs)
    if (!aligned(p, es)) return SSM_ERR_ALIGN;
  if (!aligned(weight, 4) || !aligned(bias, 4)) return SSM_ERR_ALIGN;
  // work items over 256-thread CTAs must fit a grid; formed in double, where the product cannot overflow
  if (double(batch) * double(dim) * (double(seqlen) + width) / 256.0 + 1.0 > double(0x7fffffff))
    return SSM_ERR_UNSUPPORTED;

  ssm::ConvArgs a{};
  a.x = x, a.weight = weight, a.bias = bias, a.state_in = state_in, a.out = out, a.state_out = state_out;
  a.batch = batch, a.dim = dim, a.seqlen = seqlen, a.width = width;
  a.silu = silu ? 1 : 0;
  a.io = io_dtype == SSM_F32 ? ssm::kF32 : ssm::kBF16;
  const cudaError_t err = ssm::launch_causal_conv1d(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

int ssm_causal_conv1d_update(void* state, const void* x, const float* weight, const float* bias, void* out,
                             int batch, int dim, int width, int silu, int io_dtype, void* stream) {
  if (batch < 0 || dim < 0 || width < 1) return SSM_ERR_SHAPE;
  if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
  if (width > 4) return SSM_ERR_UNSUPPORTED;
  if (batch == 0 || dim == 0) return SSM_OK;
  if (!x || !weight || !out || (width > 1 && !state)) return SSM_ERR_NULL;
  if (x == out) return SSM_ERR_ARG;
  const size_t es = io_size(io_dtype);
  const void* io_ptrs[] = {state, x, out};
  for (const void* p : io_ptrs)
    if (!aligned(p, es)) return SSM_ERR_ALIGN;
  if (!aligned(weight, 4) || !aligned(bias, 4)) return SSM_ERR_ALIGN;
  if ((long long)batch * dim / 256 + 1 > 0x7fffffffLL) return SSM_ERR_UNSUPPORTED;

  ssm::ConvUpdateArgs a{};
  a.state = state, a.x = x, a.weight = weight, a.bias = bias, a.out = out;
  a.batch = batch, a.dim = dim, a.width = width;
  a.silu = silu ? 1 : 0;
  a.io = io_dtype == SSM_F32 ? ssm::kF32 : ssm::kBF16;
  const cudaError_t err = ssm::launch_causal_conv1d_update(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

int ssm_wait_timeouts(unsigned long long* count) {
  if (!count) return SSM_ERR_NULL;
  unsigned long long n = 0, m = 0;
  if (ssm::scan_wait_timeouts(n) != cudaSuccess || ssm::decode_wait_timeouts(m) != cudaSuccess) return SSM_ERR_LAUNCH;
  *count = n + m;
  return SSM_OK;
}

int ssm_probe_cycles(int kind, long long* cycles, int nblocks, void* stream) {
  if (kind < SSM_PROBE_EX2 || kind > SSM_PROBE_WAIT_TIMEOUT) return SSM_ERR_ARG;
  if (nblocks < 0) return SSM_ERR_SHAPE;
  if (nblocks == 0) return SSM_OK;
  if (!cycles) return SSM_ERR_NULL;
  if (!aligned(cycles, 8)) return SSM_ERR_ALIGN;
  const cudaError_t err = ssm::launch_probe(kind, nblocks, cycles, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

double ssm_probe_ops_per_cta(int kind) {
  return (kind < SSM_PROBE_EX2 || kind > SSM_PROBE_WAIT_TIMEOUT) ? 0.0 : ssm::probe_ops_per_cta(kind);
}

}  // extern "C"
