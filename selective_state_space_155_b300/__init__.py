"""B300-native (sm_103a) selective scan of the Mamba selective state-space model.

Python binding of the C-ABI in ``include/ssm_scan.h``: the functions below only marshal
torch CUDA tensors into device pointers and the current stream, then call the library
(``libssm_scan.so``), which runs every step of the path in its own kernels.  PyTorch
provides device memory and streams; nothing is computed in Python.

    u, conv_state = causal_conv1d_fwd(x, conv_weight, conv_bias, silu=True, return_state=True)
    y, last_state = ssm_scan_fwd(u, delta, A, B, C, D, z, dt_bias, delta_softplus=True)
    u_t = causal_conv1d_update(conv_state, x_t, conv_weight, conv_bias)
    out = ssm_state_update(state, u_t, dt, A, B, C, D, z, dt_bias, dt_softplus=True)
"""
from __future__ import annotations

import torch

from . import _native
from ._native import SsmError, lib, status_string  # noqa: F401

__all__ = ["ssm_scan_fwd", "prepare_scan_fwd", "scan_fwd_form", "scan_fwd_workspace_size", "wait_timeouts", "ssm_scan_bwd", "scan_num_checkpoints", "ssm_state_update",
           "causal_conv1d_fwd", "causal_conv1d_update", "probe_unit_rates", "SsmError", "lib", "status_string",
           "io_dtype_code"]

_IO = {torch.float32: _native.SSM_F32, torch.bfloat16: _native.SSM_BF16}
_DISC = {"delta_b": _native.SSM_DISC_DELTA_B, "zoh": _native.SSM_DISC_ZOH}


def _disc(discretization: str) -> int:
    if discretization not in _DISC:
        raise ValueError(f"discretization must be one of {sorted(_DISC)}, got {discretization!r}")
    return _DISC[discretization]


def io_dtype_code(dtype: torch.dtype) -> int:
    if dtype not in _IO:
        raise TypeError(f"unsupported io dtype {dtype}; use float32 or bfloat16")
    return _IO[dtype]


def _ptr(t: torch.Tensor | None, dtype: torch.dtype | None = None, shape=None, name: str = "") -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr() or None


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream or None
    return getattr(stream, "cuda_stream", stream) or None


def scan_num_checkpoints(seqlen: int) -> int:
    """Number of state checkpoints the training forward stores for a sequence of `seqlen` steps."""
    return lib().ssm_scan_num_checkpoints(int(seqlen))


def ssm_scan_fwd(u, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, y=None, last_state=None,
                 h0=None, return_last_state=True, stream=None, discretization="delta_b", checkpoints=None,
                 workspace=None):
    """Selective scan forward (``ssm_scan_fwd`` / ``_h0`` / ``_ex`` / ``_ws`` / ``_train`` of the C-ABI).

    u, delta, z: [batch, dim, L]; B, C: [batch, dstate, L] (float32 or bfloat16, all the same);
    A: [dim, dstate], D, dt_bias: [dim], h0: [batch, dim, dstate] (float32).
    discretization: "delta_b" (Bbar = Delta B) or "zoh" (exact zero-order hold).
    checkpoints: a float32 [batch, scan_num_checkpoints(L), dim, dstate] tensor to receive the
    chunk-start states for ssm_scan_bwd (training forward, either discretization).
    workspace: a contiguous CUDA tensor (any dtype) for the carry buffers of the split form
    (``ssm_scan_fwd_ws``: the library then allocates nothing; ``scan_fwd_workspace_size`` gives
    the bytes it needs, and with fewer the scan runs unsplit).  Not with checkpoints.
    Returns (y, last_state); y has u's dtype, last_state is float32 (None if not requested).
    """
    disc = _disc(discretization)
    batch, dim, L = u.shape
    dstate = A.shape[1]
    io = io_dtype_code(u.dtype)
    if y is None:
        y = torch.empty_like(u)
    if last_state is None and return_last_state:
        last_state = torch.empty((batch, dim, dstate), dtype=torch.float32, device=u.device)
    args = [
        _ptr(u, u.dtype, (batch, dim, L), "u"),
        _ptr(delta, u.dtype, (batch, dim, L), "delta"),
        _ptr(A, torch.float32, (dim, dstate), "A"),
        _ptr(B, u.dtype, (batch, dstate, L), "B"),
        _ptr(C, u.dtype, (batch, dstate, L), "C"),
        _ptr(D, torch.float32, (dim,), "D"),
        _ptr(z, u.dtype, (batch, dim, L), "z"),
        _ptr(dt_bias, torch.float32, (dim,), "dt_bias"),
        int(bool(delta_softplus)),
    ]
    tail = [
        _ptr(y, u.dtype, (batch, dim, L), "y"),
        _ptr(last_state, torch.float32, (batch, dim, dstate), "last_state"),
        batch, dim, dstate, L, io, _stream(stream),
    ]
    h0p = _ptr(h0, torch.float32, (batch, dim, dstate), "h0")
    if workspace is not None:
        if checkpoints is not None:
            raise ValueError("workspace and checkpoints do not go together (the training forward does not split)")
        wsp = _ptr(workspace, None, None, "workspace")
        nbytes = workspace.numel() * workspace.element_size()
        _native.check("ssm_scan_fwd_ws", lib().ssm_scan_fwd_ws(*args, h0p, *tail[:-1], disc, wsp, nbytes, tail[-1]))
    elif checkpoints is not None:
        ck = _ptr(checkpoints, torch.float32, (batch, scan_num_checkpoints(L), dim, dstate), "checkpoints")
        if disc == _native.SSM_DISC_DELTA_B:
            _native.check("ssm_scan_fwd_train", lib().ssm_scan_fwd_train(*args, h0p, tail[0], tail[1], ck, *tail[2:]))
        else:
            _native.check("ssm_scan_fwd_train_ex",
                          lib().ssm_scan_fwd_train_ex(*args, h0p, tail[0], tail[1], ck, *tail[2:-1], disc, tail[-1]))
    elif disc != _native.SSM_DISC_DELTA_B:
        _native.check("ssm_scan_fwd_ex", lib().ssm_scan_fwd_ex(*args, h0p, *tail[:-1], disc, tail[-1]))
    elif h0 is None:
        _native.check("ssm_scan_fwd", lib().ssm_scan_fwd(*args, *tail))
    else:
        _native.check("ssm_scan_fwd_h0", lib().ssm_scan_fwd_h0(*args, h0p, *tail))
    return y, last_state


class PreparedCall:
    """One C-ABI call whose arguments were validated and turned into pointers once.  Calling it
    enqueues the same work again on the stream fixed at preparation, with no per-call checks: the
    tensors it was prepared from must stay alive, in place and unchanged in shape and dtype."""

    __slots__ = ("_fn", "_args", "_name", "outputs")

    def __init__(self, name: str, args: tuple, outputs: tuple):
        self._fn = getattr(lib(), name)
        self._args = args
        self._name = name
        self.outputs = outputs

    def __call__(self):
        st = self._fn(*self._args)
        if st:
            raise SsmError(self._name, st)


def prepare_scan_fwd(u, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True, y=None, last_state=None,
                     h0=None, return_last_state=True, stream=None, discretization="delta_b",
                     workspace=None) -> PreparedCall:
    """``ssm_scan_fwd_ex`` (``ssm_scan_fwd_ws`` with a workspace) with every argument checked and
    marshalled once, for callers that repeat the same scan on the same buffers (a benchmark loop, a
    fixed serving shape): the returned PreparedCall enqueues it with one foreign call and nothing
    else.  Arguments as ssm_scan_fwd; ``.outputs`` is (y, last_state)."""
    disc = _disc(discretization)
    batch, dim, L = u.shape
    dstate = A.shape[1]
    io = io_dtype_code(u.dtype)
    if y is None:
        y = torch.empty_like(u)
    if last_state is None and return_last_state:
        last_state = torch.empty((batch, dim, dstate), dtype=torch.float32, device=u.device)
    args = (
        _ptr(u, u.dtype, (batch, dim, L), "u"),
        _ptr(delta, u.dtype, (batch, dim, L), "delta"),
        _ptr(A, torch.float32, (dim, dstate), "A"),
        _ptr(B, u.dtype, (batch, dstate, L), "B"),
        _ptr(C, u.dtype, (batch, dstate, L), "C"),
        _ptr(D, torch.float32, (dim,), "D"),
        _ptr(z, u.dtype, (batch, dim, L), "z"),
        _ptr(dt_bias, torch.float32, (dim,), "dt_bias"),
        int(bool(delta_softplus)),
        _ptr(h0, torch.float32, (batch, dim, dstate), "h0"),
        _ptr(y, u.dtype, (batch, dim, L), "y"),
        _ptr(last_state, torch.float32, (batch, dim, dstate), "last_state"),
        batch, dim, dstate, L, io, disc,
    )
    if workspace is not None:
        nbytes = workspace.numel() * workspace.element_size()
        return PreparedCall("ssm_scan_fwd_ws", args + (_ptr(workspace, None, None, "workspace"), nbytes,
                                                       _stream(stream)), (y, last_state))
    return PreparedCall("ssm_scan_fwd_ex", args + (_stream(stream),), (y, last_state))


def scan_fwd_workspace_size(batch: int, dim: int, dstate: int, seqlen: int, dtype=torch.bfloat16,
                            discretization="delta_b", aligned_rows: bool = True) -> int:
    """Bytes of workspace a scan of these sizes uses on the current device (0 when it runs
    unsplit): ``ssm_scan_fwd_workspace_size``."""
    import ctypes
    n = ctypes.c_size_t(0)
    _native.check("ssm_scan_fwd_workspace_size",
                  lib().ssm_scan_fwd_workspace_size(int(batch), int(dim), int(dstate), int(seqlen), io_dtype_code(dtype),
                                                    _disc(discretization), int(bool(aligned_rows)), ctypes.byref(n)))
    return int(n.value)


def scan_fwd_form(batch: int, dim: int, dstate: int, seqlen: int, dtype=torch.bfloat16, discretization="delta_b",
                  aligned_rows: bool = True) -> tuple[str, int]:
    """(form name, CTAs) of the kernel a scan of these sizes launches on the current device
    (``ssm_scan_fwd_form``): "plain" (one CTA per 32-channel block), "balanced" (one CTA per SM
    with up to three warp groups on planned channel ranges) or "split" (the balanced form over
    segments of the sequence, linked by a carry pass; few channels and long sequences)."""
    import ctypes
    n = ctypes.c_int(0)
    st = lib().ssm_scan_fwd_form(int(batch), int(dim), int(dstate), int(seqlen), io_dtype_code(dtype),
                                 _disc(discretization), int(bool(aligned_rows)), ctypes.byref(n))
    if st < 0:
        raise SsmError("ssm_scan_fwd_form", st)
    return _native.FORM_NAMES[st], n.value


def wait_timeouts() -> int:
    """Hand-off waits inside the forward kernels that gave up since the library was loaded
    (``ssm_wait_timeouts``; synchronises the device).  0 on a healthy device."""
    import ctypes
    n = ctypes.c_ulonglong(0)
    _native.check("ssm_wait_timeouts", lib().ssm_wait_timeouts(ctypes.byref(n)))
    return int(n.value)


def ssm_scan_bwd(u, delta, A, B, C, checkpoints, dout, D=None, z=None, dt_bias=None, delta_softplus=True,
                 need_dh0=False, stream=None, discretization="delta_b"):
    """Backward pass of the scan (``ssm_scan_bwd`` / ``ssm_scan_bwd_ex`` of the C-ABI) from the
    training forward's checkpoints and dout = dLoss/dout [batch, dim, L].  discretization must be
    the training forward's.  Returns a dict of gradients: du, ddelta (and dz when z is given) in
    u's dtype; dA, dB, dC (and dD, ddt_bias, dh0 when D, dt_bias are given / need_dh0) in
    float32."""
    disc = _disc(discretization)
    batch, dim, L = u.shape
    dstate = A.shape[1]
    io = io_dtype_code(u.dtype)
    f32 = dict(dtype=torch.float32, device=u.device)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u), "dA": torch.empty((dim, dstate), **f32),
         "dB": torch.empty((batch, dstate, L), **f32), "dC": torch.empty((batch, dstate, L), **f32)}
    if D is not None:
        g["dD"] = torch.empty((dim,), **f32)
    if z is not None:
        g["dz"] = torch.empty_like(u)
    if dt_bias is not None:
        g["ddt_bias"] = torch.empty((dim,), **f32)
    if need_dh0:
        g["dh0"] = torch.empty((batch, dim, dstate), **f32)
    args = [
        _ptr(u, u.dtype, (batch, dim, L), "u"),
        _ptr(delta, u.dtype, (batch, dim, L), "delta"),
        _ptr(A, torch.float32, (dim, dstate), "A"),
        _ptr(B, u.dtype, (batch, dstate, L), "B"),
        _ptr(C, u.dtype, (batch, dstate, L), "C"),
        _ptr(D, torch.float32, (dim,), "D"),
        _ptr(z, u.dtype, (batch, dim, L), "z"),
        _ptr(dt_bias, torch.float32, (dim,), "dt_bias"),
        int(bool(delta_softplus)),
        _ptr(checkpoints, torch.float32, (batch, scan_num_checkpoints(L), dim, dstate), "checkpoints"),
        _ptr(dout, u.dtype, (batch, dim, L), "dout"),
        _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g.get("dD")),
        _ptr(g.get("dz")), _ptr(g.get("ddt_bias")), _ptr(g.get("dh0")),
        batch, dim, dstate, L, io,
    ]
    if disc == _native.SSM_DISC_DELTA_B:
        _native.check("ssm_scan_bwd", lib().ssm_scan_bwd(*args, _stream(stream)))
    else:
        _native.check("ssm_scan_bwd_ex", lib().ssm_scan_bwd_ex(*args, disc, _stream(stream)))
    return g


def ssm_state_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True, out=None, stream=None,
                     discretization="delta_b"):
    """One decode step (``ssm_state_update`` / ``ssm_state_update_ex`` of the C-ABI); `state` is
    updated in place.

    state: [batch, dim, dstate] float32; x, dt, z: [batch, dim]; B, C: [batch, dstate]
    (float32 or bfloat16); A: [dim, dstate], D, dt_bias: [dim] float32.
    discretization: "delta_b" or "zoh", as for ssm_scan_fwd.  Returns out [batch, dim].
    """
    disc = _disc(discretization)
    batch, dim, dstate = state.shape
    io = io_dtype_code(x.dtype)
    if out is None:
        out = torch.empty_like(x)
    args = [
        _ptr(state, torch.float32, (batch, dim, dstate), "state"),
        _ptr(x, x.dtype, (batch, dim), "x"),
        _ptr(dt, x.dtype, (batch, dim), "dt"),
        _ptr(A, torch.float32, (dim, dstate), "A"),
        _ptr(B, x.dtype, (batch, dstate), "B"),
        _ptr(C, x.dtype, (batch, dstate), "C"),
        _ptr(D, torch.float32, (dim,), "D"),
        _ptr(z, x.dtype, (batch, dim), "z"),
        _ptr(dt_bias, torch.float32, (dim,), "dt_bias"),
        int(bool(dt_softplus)),
        _ptr(out, x.dtype, (batch, dim), "out"),
        batch, dim, dstate, io,
    ]
    if disc != _native.SSM_DISC_DELTA_B:
        _native.check("ssm_state_update_ex", lib().ssm_state_update_ex(*args, disc, _stream(stream)))
    else:
        _native.check("ssm_state_update", lib().ssm_state_update(*args, _stream(stream)))
    return out


def causal_conv1d_fwd(x, weight, bias=None, state_in=None, silu=True, out=None, state_out=None, return_state=False,
                      stream=None):
    """Causal depthwise conv1d (``ssm_causal_conv1d_fwd`` of the C-ABI).

    x: [batch, dim, L] (float32 or bfloat16); weight: [dim, W] float32 (W <= 4); bias: [dim]
    float32; state_in: [batch, dim, W-1] (x's dtype), the inputs before t = 0.  Returns out, or
    (out, state_out) with return_state (state_out: the W-1 last inputs, for the next piece).
    """
    batch, dim, L = x.shape
    width = weight.shape[1]
    io = io_dtype_code(x.dtype)
    if out is None:
        out = torch.empty_like(x)
    if state_out is None and return_state:
        state_out = torch.empty((batch, dim, width - 1), dtype=x.dtype, device=x.device)
    st = lib().ssm_causal_conv1d_fwd(
        _ptr(x, x.dtype, (batch, dim, L), "x"),
        _ptr(weight, torch.float32, (dim, width), "weight"),
        _ptr(bias, torch.float32, (dim,), "bias"),
        _ptr(state_in, x.dtype, (batch, dim, width - 1), "state_in"),
        _ptr(out, x.dtype, (batch, dim, L), "out"),
        _ptr(state_out, x.dtype, (batch, dim, width - 1), "state_out"),
        batch, dim, L, width, int(bool(silu)), io, _stream(stream),
    )
    _native.check("ssm_causal_conv1d_fwd", st)
    return (out, state_out) if return_state else out


def causal_conv1d_update(state, x, weight, bias=None, silu=True, out=None, stream=None):
    """One decode step of the causal conv1d (``ssm_causal_conv1d_update``); `state` [batch, dim,
    W-1] is shifted in place.  x: [batch, dim].  Returns out [batch, dim]."""
    batch, dim = x.shape
    width = weight.shape[1]
    io = io_dtype_code(x.dtype)
    if out is None:
        out = torch.empty_like(x)
    st = lib().ssm_causal_conv1d_update(
        _ptr(state, x.dtype, (batch, dim, width - 1), "state") if width > 1 else None,
        _ptr(x, x.dtype, (batch, dim), "x"),
        _ptr(weight, torch.float32, (dim, width), "weight"),
        _ptr(bias, torch.float32, (dim,), "bias"),
        _ptr(out, x.dtype, (batch, dim), "out"),
        batch, dim, width, int(bool(silu)), io, _stream(stream),
    )
    _native.check("ssm_causal_conv1d_update", st)
    return out


def probe_unit_rates(device=None) -> dict:
    """Measured rates per clock per SM (``ssm_probe_cycles``), the median over one CTA per SM:
    lane-operations of ex2.approx, FP32 FMA and packed f32x2 FMA alone; ex2 operations when each
    ex2 shares its chain step with an independent f32x2 FMA (``ex2_with_ffma2``); state-steps of
    the recurrence's arithmetic mix with no memory traffic (``recurrence``)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cycles = torch.empty(sms, dtype=torch.int64, device=dev)
    out = {}
    for name, kind in (("ex2", _native.SSM_PROBE_EX2), ("ffma", _native.SSM_PROBE_FFMA),
                       ("ffma2", _native.SSM_PROBE_FFMA2), ("ex2_with_ffma2", _native.SSM_PROBE_EX2_FFMA2),
                       ("recurrence", _native.SSM_PROBE_RECURRENCE)):
        for _ in range(2):  # the first launch warms up
            _native.check("ssm_probe_cycles", lib().ssm_probe_cycles(kind, _ptr(cycles, torch.int64, None, "cycles"),
                                                                     sms, _stream(None)))
        torch.cuda.synchronize(dev)
        med = float(cycles.to("cpu").double().median())
        out[name] = lib().ssm_probe_ops_per_cta(kind) / med
    return out
