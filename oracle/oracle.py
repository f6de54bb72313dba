"""float64 CPU oracle for the Mamba selective scan -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path (the CUDA library and its
Python binding) never touches it, and it shares no code with that path: the
arithmetic lives in ``ssm_oracle.c`` (plain loops, float64, libm ``exp`` and
``log1p``), compiled here with gcc ``-O2 -fno-fast-math -ffp-contract=off``.

Every function takes numpy arrays in the layouts documented in ``ssm_oracle.c``
and returns float64 numpy arrays.  Inputs are widened to float64 exactly (fp32
and bf16 values are representable in float64), so the oracle sees the very same
numbers as the GPU.

Parity status per function (what pins it, see tests/test_oracle_pins.py):
  scan            pinned: prefix-sum worked example, closed-form y2/y3 expansions,
                  brute-force convolution form, unrolled time-varying sum, Delta->0,
                  exact halving with Delta = ln 2, softplus/silu special values.
  scan (zoh)      pinned: the exact solution of the continuous system under a held input
                  (closed form, and scipy's matrix exponential of the augmented system),
                  A = 0 equals the Delta*B form, decode steps equal the scan.
  state_update    pinned: equals the pinned scan step by step; exact halving case.
  assoc_scan      pinned: prefix-sum worked example; equals the closed-form products.
  scan_tree       pinned: equals the sequential scan (associativity).
  scan_bwd        pinned: central finite differences of <dout, out> along random directions for
                  every input (u, delta, A, B, C, D, z, dt_bias, h0; softplus on and off; both
                  discretisations, ZOH also with A near and at 0), and the closed-form gradient of
                  the prefix-sum special case.
  causal_conv1d   pinned: numpy's full convolution (first L outputs), torch's grouped Conv1d with
                  padding W-1 as the gsyq.cn sketch writes it, streaming in two pieces, impulse
                  response, silu special values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DP = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into liboracle.so next to it (OpenMP over channels)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-o", _LIB, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    return _LIB


def use_library(path: str | None) -> None:
    """Point this module at another build of ssm_oracle.c (the mutation tests use it to check
    that the pins reject planted mistakes); None restores the default build."""
    global _lib, _LIB
    with _lock:
        _lib = None
        _LIB = path if path is not None else os.path.join(_HERE, "liboracle.so")


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if _LIB == os.path.join(_HERE, "liboracle.so"):
                build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_scan_f64.restype = ctypes.c_int
            lib.oracle_scan_f64.argtypes = [_DP] * 8 + [ctypes.c_int, ctypes.c_int, _DP, _DP, _DP] + [ctypes.c_int] * 5
            lib.oracle_state_update_f64.restype = ctypes.c_int
            lib.oracle_state_update_f64.argtypes = [_DP] * 9 + [ctypes.c_int, ctypes.c_int, _DP] + [ctypes.c_int] * 4
            lib.oracle_assoc_scan_pairs_f64.restype = ctypes.c_int
            lib.oracle_assoc_scan_pairs_f64.argtypes = [_DP] * 4 + [ctypes.c_int]
            lib.oracle_scan_tree_f64.restype = ctypes.c_int
            lib.oracle_scan_tree_f64.argtypes = [_DP] * 8 + [ctypes.c_int, _DP, _DP] + [ctypes.c_int] * 4
            lib.oracle_scan_bwd_f64.restype = ctypes.c_int
            lib.oracle_scan_bwd_f64.argtypes = ([_DP] * 8 + [ctypes.c_int, ctypes.c_int] + [_DP] * 11 +
                                                [ctypes.c_int] * 4 + [_DP] * 5)
            lib.oracle_causal_conv1d_f64.restype = ctypes.c_int
            lib.oracle_causal_conv1d_f64.argtypes = [_DP] * 6 + [ctypes.c_int] * 5
            lib.oracle_softplus_f64.restype = ctypes.c_double
            lib.oracle_softplus_f64.argtypes = [ctypes.c_double]
            lib.oracle_silu_f64.restype = ctypes.c_double
            lib.oracle_silu_f64.argtypes = [ctypes.c_double]
            _lib = lib
    return _lib


def _f64(a, shape=None):
    if a is None:
        return None
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and arr.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {arr.shape}")
    return arr


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_DP)


def scan(u, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None, nthreads=0, zoh=False):
    """Selective scan.  Returns (y [batch,dim,L], last_state [batch,dim,N]).  zoh selects the exact
    zero-order-hold Bbar = (exp(Delta A) - 1) / A * B instead of Delta * B."""
    u = _f64(u)
    batch, dim, seqlen = u.shape
    A = _f64(A)
    dstate = A.shape[1]
    delta = _f64(delta, (batch, dim, seqlen))
    A = _f64(A, (dim, dstate))
    B = _f64(B, (batch, dstate, seqlen))
    C = _f64(C, (batch, dstate, seqlen))
    D = _f64(D, (dim,))
    z = _f64(z, (batch, dim, seqlen))
    dt_bias = _f64(dt_bias, (dim,))
    h0 = _f64(h0, (batch, dim, dstate))
    y = np.zeros((batch, dim, seqlen), dtype=np.float64)
    last = np.zeros((batch, dim, dstate), dtype=np.float64)
    rc = _load().oracle_scan_f64(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
                                 int(bool(delta_softplus)), int(bool(zoh)), _ptr(h0), _ptr(y), _ptr(last),
                                 batch, dim, dstate, seqlen, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_scan_f64 failed: {rc}")
    return y, last


def state_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True, nthreads=0, zoh=False):
    """One decode step.  Returns (new_state [batch,dim,N], out [batch,dim]); `state` is not modified."""
    s = np.array(state, dtype=np.float64, copy=True, order="C")
    batch, dim, dstate = s.shape
    x = _f64(x, (batch, dim))
    dt = _f64(dt, (batch, dim))
    A = _f64(A, (dim, dstate))
    B = _f64(B, (batch, dstate))
    C = _f64(C, (batch, dstate))
    D = _f64(D, (dim,))
    z = _f64(z, (batch, dim))
    dt_bias = _f64(dt_bias, (dim,))
    out = np.zeros((batch, dim), dtype=np.float64)
    rc = _load().oracle_state_update_f64(_ptr(s), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                         _ptr(dt_bias), int(bool(dt_softplus)), int(bool(zoh)), _ptr(out), batch, dim,
                                         dstate,
                                         int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_state_update_f64 failed: {rc}")
    return s, out


def assoc_scan(a, b):
    """Tree-order inclusive scan of pairs (a_t, b_t).  Returns (prod_a, h)."""
    a = _f64(a)
    b = _f64(b, a.shape)
    n = a.shape[0]
    oa = np.zeros(n, dtype=np.float64)
    ob = np.zeros(n, dtype=np.float64)
    rc = _load().oracle_assoc_scan_pairs_f64(_ptr(a), _ptr(b), _ptr(oa), _ptr(ob), n)
    if rc != 0:
        raise RuntimeError(f"oracle_assoc_scan_pairs_f64 failed: {rc}")
    return oa, ob


def scan_tree(u, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True):
    """The selective scan with the recurrence evaluated in tree order."""
    u = _f64(u)
    batch, dim, seqlen = u.shape
    A = _f64(A)
    dstate = A.shape[1]
    delta = _f64(delta, (batch, dim, seqlen))
    B = _f64(B, (batch, dstate, seqlen))
    C = _f64(C, (batch, dstate, seqlen))
    D = _f64(D, (dim,))
    z = _f64(z, (batch, dim, seqlen))
    dt_bias = _f64(dt_bias, (dim,))
    y = np.zeros((batch, dim, seqlen), dtype=np.float64)
    last = np.zeros((batch, dim, dstate), dtype=np.float64)
    rc = _load().oracle_scan_tree_f64(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                      _ptr(dt_bias), int(bool(delta_softplus)), _ptr(y), _ptr(last),
                                      batch, dim, dstate, seqlen)
    if rc != 0:
        raise RuntimeError(f"oracle_scan_tree_f64 failed: {rc}")
    return y, last


def scan_bwd(u, delta, A, B, C, dout, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None, zoh=False,
             abs_sums=False):
    """Gradients of the scan (Delta*B form, or the exact zero-order hold with zoh) for the output
    gradient dout [batch, dim, L].
    Returns a dict with du, ddelta, dA, dB, dC and, where the input is given, dD, dz,
    ddt_bias, dh0 (float64 arrays shaped like their inputs).  With abs_sums it also has abs_dA,
    abs_dB, abs_dC (and abs_dD, abs_ddt_bias where D, dt_bias are given): the sum of the absolute
    values of the terms each summed gradient adds up."""
    u = _f64(u)
    batch, dim, seqlen = u.shape
    A = _f64(A)
    dstate = A.shape[1]
    delta = _f64(delta, (batch, dim, seqlen))
    B = _f64(B, (batch, dstate, seqlen))
    C = _f64(C, (batch, dstate, seqlen))
    D = _f64(D, (dim,))
    z = _f64(z, (batch, dim, seqlen))
    dt_bias = _f64(dt_bias, (dim,))
    h0 = _f64(h0, (batch, dim, dstate))
    dout = _f64(dout, (batch, dim, seqlen))
    g = {"du": np.zeros_like(u), "ddelta": np.zeros_like(u), "dA": np.zeros_like(A), "dB": np.zeros_like(B),
         "dC": np.zeros_like(C)}
    g["dD"] = np.zeros(dim) if D is not None else None
    g["dz"] = np.zeros_like(u) if z is not None else None
    g["ddt_bias"] = np.zeros(dim) if dt_bias is not None else None
    g["dh0"] = np.zeros((batch, dim, dstate)) if h0 is not None else None
    for k in ("dA", "dB", "dC", "dD", "ddt_bias"):
        g["abs_" + k] = np.zeros_like(g[k]) if abs_sums and g[k] is not None else None
    rc = _load().oracle_scan_bwd_f64(_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                     _ptr(dt_bias), int(bool(delta_softplus)), int(bool(zoh)), _ptr(h0), _ptr(dout),
                                     _ptr(g["du"]),
                                     _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
                                     _ptr(g["dz"]), _ptr(g["ddt_bias"]), _ptr(g["dh0"]), batch, dim, dstate, seqlen,
                                     _ptr(g["abs_dA"]), _ptr(g["abs_dB"]), _ptr(g["abs_dC"]), _ptr(g["abs_dD"]),
                                     _ptr(g["abs_ddt_bias"]))
    if rc != 0:
        raise RuntimeError(f"oracle_scan_bwd_f64 failed: {rc}")
    return {k: v for k, v in g.items() if v is not None}


def causal_conv1d(x, weight, bias=None, state_in=None, silu=True):
    """Causal depthwise conv1d.  x [batch,dim,L], weight [dim,W], bias [dim], state_in
    [batch,dim,W-1] (the inputs before t = 0, oldest first).  Returns (out [batch,dim,L],
    state_out [batch,dim,W-1])."""
    x = _f64(x)
    batch, dim, seqlen = x.shape
    weight = _f64(weight)
    width = weight.shape[1]
    weight = _f64(weight, (dim, width))
    bias = _f64(bias, (dim,))
    state_in = _f64(state_in, (batch, dim, width - 1))
    out = np.zeros((batch, dim, seqlen), dtype=np.float64)
    st = np.zeros((batch, dim, width - 1), dtype=np.float64)
    rc = _load().oracle_causal_conv1d_f64(_ptr(x), _ptr(weight), _ptr(bias), _ptr(state_in), _ptr(out), _ptr(st),
                                          batch, dim, seqlen, width, int(bool(silu)))
    if rc != 0:
        raise RuntimeError(f"oracle_causal_conv1d_f64 failed: {rc}")
    return out, st


def softplus(x: float) -> float:
    return _load().oracle_softplus_f64(float(x))


def silu(x: float) -> float:
    return _load().oracle_silu_f64(float(x))
