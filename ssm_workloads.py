"""Seeded synthetic workloads for the selective scan and the decode step.

This module only draws inputs; it holds none of the scan's arithmetic.  Both the
CUDA path and the float64 oracle are fed from it (the tests and the benchmark
call it and hand the same arrays to each side).

Recipe (one per workload, all seeded):
  * channel parameters, float64 on the host, rounded once to float32:
      A_log[d, n] = log(n + 1),  A = -exp(A_log)          (S4D-real style init)
      dt[d]       = exp(U[ln 1e-3, ln 1e-1])              (log-uniform step size)
      dt_bias[d]  = log(expm1(dt[d]))                      (so softplus(dt_bias) = dt)
      D[d]        = N(0,1) for the tiny workload, 1.0 otherwise
  * activations u, delta_raw, z and the shared B, C rows ~ N(0, 1) (u of the long
    workload ~ N(0, 0.5^2)), drawn in float64 (host generator) or float32 (device
    generator), rounded to float32, then to bf16 (round-to-nearest-even) for the
    bf16 workloads.  The rounded values are what both sides read.
  * host generator: numpy PCG64 ``default_rng(seed)``; draw order dt, u, delta, z,
    B, C, D.  Used for the workloads small enough to materialise on the host.
  * device generator: torch's CUDA Philox generator seeded with ``seed``; used for
    the 65536-long scan and the 1024-step decode loop, whose parity tests sample
    channels and copy those inputs back to the host.
  * causal conv1d (the layer in front of the scan): x ~ N(0, 1) in the scan's io dtype and
    shape, weight[d, k] and bias[d] ~ U(-1/sqrt(W), 1/sqrt(W)) (the default init bound of a
    depthwise Conv1d, fan-in W), float32; width W = 4 (d_conv of the pages' usage example).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class ScanWorkload:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    io: str  # "f32" or "bf16"
    seed: int
    gate: bool
    D_mode: str  # "normal" or "ones"
    u_std: float = 1.0
    generator: str = "host"  # "host" or "device"

    @property
    def elements(self) -> int:
        return self.batch * self.dim * self.seqlen

    def algorithmic_bytes(self) -> int:
        """Bytes the scan must move at minimum: u, delta (and z) read once, y written once,
        B and C read once, A/D/dt_bias read once, the float32 final state written once."""
        es = 4 if self.io == "f32" else 2
        per_elem = es * (3 + (1 if self.gate else 0))
        bc = 2 * self.batch * self.dstate * self.seqlen * es
        params = self.dim * self.dstate * 4 + 2 * self.dim * 4
        state = self.batch * self.dim * self.dstate * 4
        return self.elements * per_elem + bc + params + state


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    dim: int
    dstate: int
    steps: int
    io: str
    seed: int

    def algorithmic_bytes_per_step(self) -> int:
        """State read + written (float32), x/dt/z read and out written (io dtype), B/C read,
        A/D/dt_bias read."""
        es = 4 if self.io == "f32" else 2
        bd = self.batch * self.dim
        return (2 * bd * self.dstate * 4 + 4 * bd * es + 2 * self.batch * self.dstate * es
                + self.dim * self.dstate * 4 + 2 * self.dim * 4)


TINY = ScanWorkload("tiny_f32_b1_d16_n4_l64", 1, 16, 4, 64, "f32", 0, gate=False, D_mode="normal")
SMALL = ScanWorkload("small_f32_b2_d32_n16_l64", 2, 32, 16, 64, "f32", 1, gate=True, D_mode="ones")
MID = ScanWorkload("mid_bf16_b8_d1536_n16_l2048", 8, 1536, 16, 2048, "bf16", 2, gate=True, D_mode="ones")
LONG = ScanWorkload("long_bf16_b1_d5120_n16_l65536", 1, 5120, 16, 65536, "bf16", 3, gate=True, D_mode="ones",
                    u_std=0.5, generator="device")
# One 64K-token document through a layer of the mid workload's width (d_inner 1536): few channels
# for a long sequence, the case the split scan serves.  Distributions as the long workload.
LONG_NARROW = ScanWorkload("long_bf16_b1_d1536_n16_l65536", 1, 1536, 16, 65536, "bf16", 5, gate=True,
                           D_mode="ones", u_std=0.5, generator="device")
DECODE = DecodeWorkload("decode_bf16_b256_d5120_n16_x1024", 256, 5120, 16, 1024, "bf16", 4)

SCAN_WORKLOADS = {w.name: w for w in (TINY, SMALL, MID, LONG, LONG_NARROW)}


def _io_dtype(io: str) -> torch.dtype:
    return torch.float32 if io == "f32" else torch.bfloat16


def channel_params(dim: int, dstate: int, rng: np.random.Generator):
    """A (dim, dstate) and dt_bias (dim,) as float32 torch CPU tensors (draws dt from `rng`)."""
    dt = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=dim))
    dt_bias = np.log(np.expm1(dt))
    A_log = np.log(np.arange(1, dstate + 1, dtype=np.float64))[None, :].repeat(dim, axis=0)
    A = -np.exp(A_log)
    return (torch.from_numpy(A.astype(np.float32)), torch.from_numpy(dt_bias.astype(np.float32)))


def _d_param(dim: int, rng: np.random.Generator, D_mode: str) -> torch.Tensor:
    if D_mode == "normal":
        return torch.from_numpy(rng.standard_normal(dim).astype(np.float32))
    return torch.ones(dim, dtype=torch.float32)


def _round_io(x64: np.ndarray, io: str) -> torch.Tensor:
    t = torch.from_numpy(x64.astype(np.float32))
    return t if io == "f32" else t.to(torch.bfloat16)


def scan_inputs(w: ScanWorkload, device: str | torch.device = "cpu") -> dict:
    """All inputs of a scan workload.  Host generator: drawn on the host then moved to `device`.
    Device generator: drawn on `device` (must be CUDA)."""
    rng = np.random.default_rng(w.seed)
    A, dt_bias = channel_params(w.dim, w.dstate, rng)
    shp = (w.batch, w.dim, w.seqlen)
    bshp = (w.batch, w.dstate, w.seqlen)
    if w.generator == "host":
        u = _round_io(rng.standard_normal(shp) * w.u_std, w.io)
        delta = _round_io(rng.standard_normal(shp), w.io)
        z = _round_io(rng.standard_normal(shp), w.io) if w.gate else None
        B = _round_io(rng.standard_normal(bshp), w.io)
        C = _round_io(rng.standard_normal(bshp), w.io)
        D = _d_param(w.dim, rng, w.D_mode)
        out = dict(u=u, delta=delta, z=z, B=B, C=C, A=A, D=D, dt_bias=dt_bias)
        return {k: (v.to(device) if v is not None else None) for k, v in out.items()}
    dev = torch.device(device)
    if dev.type != "cuda":
        raise ValueError(f"workload {w.name} uses the device generator; pass a CUDA device")
    D = _d_param(w.dim, rng, w.D_mode)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    dt = _io_dtype(w.io)

    def draw(shape, std=1.0):
        x = torch.empty(shape, dtype=torch.float32, device=dev)
        x.normal_(0.0, std, generator=g)
        return x.to(dt)

    u = draw(shp, w.u_std)
    delta = draw(shp)
    z = draw(shp) if w.gate else None
    B = draw(bshp)
    C = draw(bshp)
    return dict(u=u, delta=delta, z=z, B=B, C=C, A=A.to(dev), D=D.to(dev), dt_bias=dt_bias.to(dev))


def decode_params(w: DecodeWorkload, device="cpu") -> dict:
    """Channel parameters and the initial state of the decode workload (state on `device`)."""
    rng = np.random.default_rng(w.seed)
    A, dt_bias = channel_params(w.dim, w.dstate, rng)
    D = torch.ones(w.dim, dtype=torch.float32)
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    state = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device=dev)
    state.normal_(0.0, 1.0, generator=g)
    return dict(A=A.to(dev), D=D.to(dev), dt_bias=dt_bias.to(dev), state=state, generator=g)


def decode_step_inputs(w: DecodeWorkload, steps: int, generator: torch.Generator, device) -> dict:
    """x, dt, z [steps, batch, dim] and B, C [steps, batch, dstate] for `steps` consecutive
    decode steps, drawn step by step from `generator` (continuing its stream)."""
    dev = torch.device(device)
    dt_ = _io_dtype(w.io)
    bd = (steps, w.batch, w.dim)
    bn = (steps, w.batch, w.dstate)
    out = {k: torch.empty(bd, dtype=dt_, device=dev) for k in ("x", "dt", "z")}
    out.update({k: torch.empty(bn, dtype=dt_, device=dev) for k in ("B", "C")})
    tmp = torch.empty((w.batch, w.dim), dtype=torch.float32, device=dev)
    tmpn = torch.empty((w.batch, w.dstate), dtype=torch.float32, device=dev)
    for s in range(steps):
        for k in ("x", "dt", "z"):
            tmp.normal_(0.0, 1.0, generator=generator)
            out[k][s].copy_(tmp)
        for k in ("B", "C"):
            tmpn.normal_(0.0, 1.0, generator=generator)
            out[k][s].copy_(tmpn)
    return out


def random_scan_case(batch, dim, dstate, seqlen, io="f32", seed=0, gate=True, use_D=True, use_bias=True,
                     softplus=True, h0=False, u_std=1.0):
    """A small seeded case with arbitrary shapes (edge-case tests).  Host generator."""
    rng = np.random.default_rng(seed)
    shp = (batch, dim, seqlen)
    bshp = (batch, dstate, seqlen)
    A_log = rng.uniform(-1.0, 2.5, size=(dim, dstate))
    A = torch.from_numpy((-np.exp(A_log)).astype(np.float32))
    dt = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=dim))
    # with softplus the bias is log(expm1(dt)) (softplus(bias) = dt); without it the bias is dt
    # itself, so that Delta = delta + bias stays positive and the system stable
    bias = np.log(np.expm1(dt)) if softplus else dt
    dt_bias = torch.from_numpy(bias.astype(np.float32)) if use_bias else None
    u = _round_io(rng.standard_normal(shp) * u_std, io)
    delta = _round_io(rng.standard_normal(shp) if softplus else np.abs(rng.standard_normal(shp)) * 0.1, io)
    z = _round_io(rng.standard_normal(shp), io) if gate else None
    B = _round_io(rng.standard_normal(bshp), io)
    C = _round_io(rng.standard_normal(bshp), io)
    D = torch.from_numpy(rng.standard_normal(dim).astype(np.float32)) if use_D else None
    h0t = torch.from_numpy(rng.standard_normal((batch, dim, dstate)).astype(np.float32)) if h0 else None
    return dict(u=u, delta=delta, z=z, B=B, C=C, A=A, D=D, dt_bias=dt_bias, h0=h0t, softplus=softplus)


def conv_inputs(batch, dim, seqlen, width=4, io="bf16", seed=0, bias=True, state=False):
    """Seeded inputs of the causal conv1d (host generator): x [batch, dim, seqlen], weight
    [dim, width], bias [dim], and optionally a carried state [batch, dim, width-1]."""
    rng = np.random.default_rng(seed)
    bound = 1.0 / math.sqrt(width)
    x = _round_io(rng.standard_normal((batch, dim, seqlen)), io)
    weight = torch.from_numpy(rng.uniform(-bound, bound, (dim, width)).astype(np.float32))
    b = torch.from_numpy(rng.uniform(-bound, bound, dim).astype(np.float32)) if bias else None
    st = _round_io(rng.standard_normal((batch, dim, width - 1)), io) if state else None
    return dict(x=x, weight=weight, bias=b, state=st)


def to_f64(t):
    """Exact widening of a torch tensor (fp32 or bf16, any device) to a float64 numpy array."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()
