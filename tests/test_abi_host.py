"""Host-side checks of the C-ABI library (no GPU needed, nothing is launched).

The library must load on a machine without a driver, export every function that
include/ssm_scan.h declares, and reject bad arguments on the host before any launch.
"""
import ctypes
import os
import re

import pytest

import __graft_entry__
from selective_state_space_155_b300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build_library()
    return _native.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(
        ["ssm_abi_version", "ssm_scan_fwd", "ssm_scan_fwd_h0", "ssm_scan_fwd_ex", "ssm_state_update",
         "ssm_state_update_ex", "ssm_status_string", "ssm_causal_conv1d_fwd", "ssm_causal_conv1d_update",
         "ssm_scan_num_checkpoints", "ssm_scan_fwd_train", "ssm_scan_fwd_train_ex", "ssm_scan_bwd",
         "ssm_scan_bwd_ex", "ssm_probe_cycles", "ssm_probe_ops_per_cta", "ssm_scan_fwd_form", "ssm_wait_timeouts",
         "ssm_scan_fwd_ws", "ssm_scan_fwd_workspace_size"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    assert set(declared_functions()) == set(_native.SIGNATURES)


def test_status_strings(lib):
    assert lib.ssm_abi_version() == 7
    for code in range(-8, 1):
        s = lib.ssm_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.ssm_status_string(42).decode() == "unknown status"


P = 0x10000  # a fake, 64 KiB aligned "device address": validation never dereferences pointers


def scan_args(**over):
    a = dict(u=P, delta=P, A=P, B=P, C=P, D=P, z=P, dt_bias=P, softplus=1, y=P, last=P, batch=2, dim=3, dstate=16,
             seqlen=5, io=_native.SSM_F32, stream=None)
    a.update(over)
    return [a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"], a["dt_bias"], a["softplus"], a["y"],
            a["last"], a["batch"], a["dim"], a["dstate"], a["seqlen"], a["io"], a["stream"]]


@pytest.mark.parametrize("over,expected", [
    (dict(u=None), _native.SSM_ERR_NULL),
    (dict(delta=None), _native.SSM_ERR_NULL),
    (dict(A=None), _native.SSM_ERR_NULL),
    (dict(B=None), _native.SSM_ERR_NULL),
    (dict(C=None), _native.SSM_ERR_NULL),
    (dict(y=None), _native.SSM_ERR_NULL),
    (dict(batch=-1), _native.SSM_ERR_SHAPE),
    (dict(dim=-1), _native.SSM_ERR_SHAPE),
    (dict(seqlen=-1), _native.SSM_ERR_SHAPE),
    (dict(dstate=0), _native.SSM_ERR_SHAPE),
    (dict(dstate=17), _native.SSM_ERR_UNSUPPORTED),
    (dict(io=7), _native.SSM_ERR_DTYPE),
    (dict(u=P + 2), _native.SSM_ERR_ALIGN),
    (dict(A=P + 2), _native.SSM_ERR_ALIGN),
    (dict(last=P + 1), _native.SSM_ERR_ALIGN),
    (dict(io=_native.SSM_BF16, z=P + 1), _native.SSM_ERR_ALIGN),
    (dict(batch=0), _native.SSM_OK),
    (dict(dim=0, u=None, y=None), _native.SSM_OK),
    (dict(seqlen=0, u=None, delta=None, B=None, C=None, y=None, last=None), _native.SSM_OK),
])
def test_scan_validation(lib, over, expected):
    assert lib.ssm_scan_fwd(*scan_args(**over)) == expected


def test_scan_h0_validation(lib):
    args = scan_args()
    h0_args = args[:9] + [P + 2] + args[9:]
    assert lib.ssm_scan_fwd_h0(*h0_args) == _native.SSM_ERR_ALIGN
    h0_args = scan_args(u=None)[:9] + [P] + scan_args(u=None)[9:]
    assert lib.ssm_scan_fwd_h0(*h0_args) == _native.SSM_ERR_NULL


@pytest.mark.parametrize("disc,expected", [(0, _native.SSM_OK), (1, _native.SSM_OK), (2, _native.SSM_ERR_ARG),
                                            (-1, _native.SSM_ERR_ARG)])
def test_scan_ex_discretization_validation(lib, disc, expected):
    # batch 0 makes a valid call return before any launch
    args = scan_args(batch=0)
    ex_args = args[:9] + [None] + args[9:16] + [disc] + args[16:]
    assert lib.ssm_scan_fwd_ex(*ex_args) == expected


def test_scan_ex_validates_like_h0(lib):
    args = scan_args(u=None)
    assert lib.ssm_scan_fwd_ex(*(args[:9] + [None] + args[9:16] + [1] + args[16:])) == _native.SSM_ERR_NULL
    args = scan_args()
    assert lib.ssm_scan_fwd_ex(*(args[:9] + [P + 2] + args[9:16] + [1] + args[16:])) == _native.SSM_ERR_ALIGN


def update_args(**over):
    a = dict(state=P, x=P, dt=P, A=P, B=P, C=P, D=P, z=P, dt_bias=P, softplus=1, out=P, batch=2, dim=3, dstate=16,
             io=_native.SSM_BF16, stream=None)
    a.update(over)
    return [a[k] for k in ("state", "x", "dt", "A", "B", "C", "D", "z", "dt_bias", "softplus", "out", "batch", "dim",
                           "dstate", "io", "stream")]


@pytest.mark.parametrize("over,expected", [
    (dict(state=None), _native.SSM_ERR_NULL),
    (dict(x=None), _native.SSM_ERR_NULL),
    (dict(dt=None), _native.SSM_ERR_NULL),
    (dict(out=None), _native.SSM_ERR_NULL),
    (dict(B=None), _native.SSM_ERR_NULL),
    (dict(batch=-3), _native.SSM_ERR_SHAPE),
    (dict(dstate=0), _native.SSM_ERR_SHAPE),
    (dict(dstate=99), _native.SSM_ERR_UNSUPPORTED),
    (dict(io=-1), _native.SSM_ERR_DTYPE),
    (dict(state=P + 2), _native.SSM_ERR_ALIGN),
    (dict(x=P + 1), _native.SSM_ERR_ALIGN),
    (dict(batch=0), _native.SSM_OK),
])
def test_update_validation(lib, over, expected):
    assert lib.ssm_state_update(*update_args(**over)) == expected
    args = update_args(**over)
    assert lib.ssm_state_update_ex(*(args[:-1] + [1] + args[-1:])) == expected


@pytest.mark.parametrize("disc,expected", [(0, _native.SSM_OK), (1, _native.SSM_OK), (5, _native.SSM_ERR_ARG)])
def test_update_ex_discretization_validation(lib, disc, expected):
    args = update_args(batch=0)
    assert lib.ssm_state_update_ex(*(args[:-1] + [disc] + args[-1:])) == expected


def test_binding_rejects_cpu_tensors():
    import torch
    import selective_state_space_155_b300 as ssm
    u = torch.zeros(1, 2, 3)
    with pytest.raises(ValueError, match="CUDA"):
        ssm.ssm_scan_fwd(u, u, torch.zeros(2, 4), torch.zeros(1, 4, 3), torch.zeros(1, 4, 3))


def conv_args(**over):
    a = dict(x=P, weight=P, bias=P, state_in=P + 0x1000, out=P + 0x2000, state_out=P + 0x3000, batch=2, dim=3,
             seqlen=8, width=4, silu=1, io=_native.SSM_BF16, stream=None)
    a.update(over)
    return [a[k] for k in ("x", "weight", "bias", "state_in", "out", "state_out", "batch", "dim", "seqlen", "width",
                           "silu", "io", "stream")]


@pytest.mark.parametrize("over,expected", [
    (dict(x=None), _native.SSM_ERR_NULL),
    (dict(out=None), _native.SSM_ERR_NULL),
    (dict(weight=None), _native.SSM_ERR_NULL),
    (dict(width=0), _native.SSM_ERR_SHAPE),
    (dict(width=5), _native.SSM_ERR_UNSUPPORTED),
    (dict(seqlen=-1), _native.SSM_ERR_SHAPE),
    (dict(io=3), _native.SSM_ERR_DTYPE),
    (dict(out=P), _native.SSM_ERR_ARG),
    (dict(state_out=P + 0x1000), _native.SSM_ERR_ARG),
    (dict(x=P + 1), _native.SSM_ERR_ALIGN),
    (dict(weight=P + 2), _native.SSM_ERR_ALIGN),
    (dict(batch=0), _native.SSM_OK),
    (dict(seqlen=0, x=None, out=None, state_out=None), _native.SSM_OK),
])
def test_conv_validation(lib, over, expected):
    assert lib.ssm_causal_conv1d_fwd(*conv_args(**over)) == expected


@pytest.mark.parametrize("over,expected", [
    (dict(state=None), _native.SSM_ERR_NULL),
    (dict(state=None, width=1), _native.SSM_OK),
    (dict(x=None), _native.SSM_ERR_NULL),
    (dict(width=9), _native.SSM_ERR_UNSUPPORTED),
    (dict(out=P + 0x1000), _native.SSM_ERR_ARG),
    (dict(state=P + 1), _native.SSM_ERR_ALIGN),
])
def test_conv_update_validation(lib, over, expected):
    a = dict(state=P, x=P + 0x1000, weight=P, bias=None, out=P + 0x2000, batch=2, dim=3, width=4, silu=1,
             io=_native.SSM_BF16, stream=None)
    a.update(over)
    if expected == _native.SSM_OK:
        a["batch"] = 0  # a valid call that launches nothing
    args = [a[k] for k in ("state", "x", "weight", "bias", "out", "batch", "dim", "width", "silu", "io", "stream")]
    assert lib.ssm_causal_conv1d_update(*args) == expected


def test_num_checkpoints(lib):
    # one checkpoint before every 8th step (SSM_SCAN_CHECKPOINT_STEPS)
    assert [lib.ssm_scan_num_checkpoints(L) for L in (0, 1, 7, 8, 9, 2048, 65536)] == [0, 1, 1, 1, 2, 256, 8192]


def test_train_forward_validation(lib):
    args = scan_args()
    train = args[:9] + [None] + args[9:11] + [None] + args[11:]
    assert lib.ssm_scan_fwd_train(*train) == _native.SSM_ERR_NULL  # checkpoints missing
    train = args[:9] + [None] + args[9:11] + [P + 2] + args[11:]
    assert lib.ssm_scan_fwd_train(*train) == _native.SSM_ERR_ALIGN
    # the _ex form: same checks, plus the discretization code
    train = args[:9] + [None] + args[9:11] + [None] + args[11:-1]
    for disc in (_native.SSM_DISC_DELTA_B, _native.SSM_DISC_ZOH):
        assert lib.ssm_scan_fwd_train_ex(*train, disc, None) == _native.SSM_ERR_NULL
    for disc in (-1, 2):
        assert lib.ssm_scan_fwd_train_ex(*train, disc, None) == _native.SSM_ERR_ARG


def bwd_args(**over):
    a = dict(u=P, delta=P, A=P, B=P, C=P, D=P, z=P, dt_bias=P, softplus=1, ckpt=P, dout=P, du=P, ddelta=P, dA=P,
             dB=P, dC=P, dD=P, dz=P, ddt_bias=P, dh0=None, batch=2, dim=3, dstate=16, seqlen=5, io=_native.SSM_BF16,
             stream=None)
    a.update(over)
    return [a[k] for k in ("u", "delta", "A", "B", "C", "D", "z", "dt_bias", "softplus", "ckpt", "dout", "du",
                           "ddelta", "dA", "dB", "dC", "dD", "dz", "ddt_bias", "dh0", "batch", "dim", "dstate",
                           "seqlen", "io", "stream")]


@pytest.mark.parametrize("over,expected", [
    (dict(ckpt=None), _native.SSM_ERR_NULL),
    (dict(dout=None), _native.SSM_ERR_NULL),
    (dict(dB=None), _native.SSM_ERR_NULL),
    (dict(dA=None), _native.SSM_ERR_NULL),
    (dict(dstate=17), _native.SSM_ERR_UNSUPPORTED),
    (dict(io=2), _native.SSM_ERR_DTYPE),
    (dict(du=P + 1), _native.SSM_ERR_ALIGN),
    (dict(dC=P + 2), _native.SSM_ERR_ALIGN),
    (dict(batch=-1), _native.SSM_ERR_SHAPE),
    (dict(batch=0), _native.SSM_OK),
])
def test_bwd_validation(lib, over, expected):
    assert lib.ssm_scan_bwd(*bwd_args(**over)) == expected
    for disc in (_native.SSM_DISC_DELTA_B, _native.SSM_DISC_ZOH):
        assert lib.ssm_scan_bwd_ex(*bwd_args(**over)[:-1], disc, None) == expected


@pytest.mark.parametrize("disc", [-1, 2, 7])
def test_bwd_ex_rejects_unknown_discretization(lib, disc):
    assert lib.ssm_scan_bwd_ex(*bwd_args()[:-1], disc, None) == _native.SSM_ERR_ARG


def test_probe_validation(lib):
    assert lib.ssm_probe_cycles(6, P, 4, None) == _native.SSM_ERR_ARG
    assert lib.ssm_probe_cycles(-1, P, 4, None) == _native.SSM_ERR_ARG
    assert lib.ssm_probe_cycles(0, None, 4, None) == _native.SSM_ERR_NULL
    assert lib.ssm_probe_cycles(1, P + 4, 4, None) == _native.SSM_ERR_ALIGN
    assert lib.ssm_probe_cycles(2, None, 0, None) == _native.SSM_OK
    assert lib.ssm_probe_cycles(0, P, -1, None) == _native.SSM_ERR_SHAPE
    assert lib.ssm_probe_ops_per_cta(5) == 0.0  # the bounded-wait probe counts no operations
    ops = [lib.ssm_probe_ops_per_cta(k) for k in (0, 1, 2, 3, 4)]
    # lane-operations (f32x2 counts twice), ex2 operations of the mix, state-steps (two per pair)
    assert ops[0] == ops[1] == ops[3] > 0 and ops[2] == 2 * ops[1] and ops[4] == 2 * ops[1]
    assert lib.ssm_probe_ops_per_cta(7) == 0.0


def test_grid_overflow_is_refused_before_any_launch(lib):
    """Sizes whose grid would not fit a launch are refused on the host (no memory is touched)."""
    big = 2 ** 31 - 1
    assert lib.ssm_scan_fwd(*scan_args(batch=big, dim=64)) == _native.SSM_ERR_UNSUPPORTED
    assert lib.ssm_state_update(*update_args(batch=big, dim=big)) == _native.SSM_ERR_UNSUPPORTED
    assert lib.ssm_causal_conv1d_fwd(*conv_args(batch=big, dim=big)) == _native.SSM_ERR_UNSUPPORTED
    assert lib.ssm_scan_bwd(*bwd_args(batch=big, dim=64)) == _native.SSM_ERR_UNSUPPORTED
    assert lib.ssm_scan_bwd_ex(*bwd_args(batch=big, dim=64)[:-1], _native.SSM_DISC_ZOH, None) == \
        _native.SSM_ERR_UNSUPPORTED


def test_form_query_validation(lib):
    """The form query rejects bad sizes on the host; without a device it reports SSM_ERR_LAUNCH."""
    n = ctypes.c_int(-1)
    assert lib.ssm_scan_fwd_form(-1, 4, 16, 8, 1, 0, 1, ctypes.byref(n)) == _native.SSM_ERR_SHAPE
    assert lib.ssm_scan_fwd_form(1, 4, 0, 8, 1, 0, 1, ctypes.byref(n)) == _native.SSM_ERR_SHAPE
    assert lib.ssm_scan_fwd_form(1, 4, 17, 8, 1, 0, 1, ctypes.byref(n)) == _native.SSM_ERR_UNSUPPORTED
    assert lib.ssm_scan_fwd_form(1, 4, 16, 8, 7, 0, 1, ctypes.byref(n)) == _native.SSM_ERR_DTYPE
    assert lib.ssm_scan_fwd_form(1, 4, 16, 8, 1, 5, 1, ctypes.byref(n)) == _native.SSM_ERR_ARG
    st = lib.ssm_scan_fwd_form(1, 4, 16, 8, 1, 0, 1, ctypes.byref(n))
    assert st in (_native.SSM_ERR_LAUNCH, 0, 1)


def test_wait_timeouts_validation(lib):
    assert lib.ssm_wait_timeouts(None) == _native.SSM_ERR_NULL


def test_scan_output_may_not_overlap_an_input(lib):
    """y overlapping u, delta, z, B or C is refused on the host; disjoint buffers pass validation
    (and then fail to launch on a machine without a GPU)."""
    MB = 1 << 20
    disjoint = dict(u=P, delta=P + MB, z=P + 2 * MB, B=P + 3 * MB, C=P + 4 * MB, y=P + 5 * MB, last=P + 6 * MB,
                    A=P + 7 * MB, D=P + 8 * MB, dt_bias=P + 9 * MB)
    st = lib.ssm_scan_fwd(*scan_args(**disjoint))
    assert st in (_native.SSM_OK, _native.SSM_ERR_LAUNCH)
    for k in ("u", "delta", "z", "B", "C"):
        assert lib.ssm_scan_fwd(*scan_args(**{**disjoint, "y": disjoint[k]})) == _native.SSM_ERR_ARG, k
    # a partial overlap: y starting inside u's last element of float32
    n = 2 * 3 * 5 * 4
    assert lib.ssm_scan_fwd(*scan_args(**{**disjoint, "y": P + n - 4})) == _native.SSM_ERR_ARG
    assert lib.ssm_scan_fwd(*scan_args(**{**disjoint, "y": P + n})) in (_native.SSM_OK, _native.SSM_ERR_LAUNCH)


def ws_args(ws, nbytes, **over):
    """ssm_scan_fwd_ws arguments: ssm_scan_fwd's plus h0 (none), the discretization and a workspace."""
    args = scan_args(**over)
    return args[:9] + [None] + args[9:16] + [_native.SSM_DISC_DELTA_B, ws, nbytes, args[16]]


def test_workspace_scan_validation(lib):
    """ssm_scan_fwd_ws validates like ssm_scan_fwd_ex, and its workspace must be 16-byte aligned and
    overlap no other argument; a NULL workspace is allowed (the scan then runs unsplit)."""
    MB = 1 << 20
    disjoint = dict(u=P, delta=P + MB, z=P + 2 * MB, B=P + 3 * MB, C=P + 4 * MB, y=P + 5 * MB, last=P + 6 * MB,
                    A=P + 7 * MB, D=P + 8 * MB, dt_bias=P + 9 * MB)
    ws = P + 10 * MB
    assert lib.ssm_scan_fwd_ws(*ws_args(ws, MB, **disjoint)) in (_native.SSM_OK, _native.SSM_ERR_LAUNCH)
    assert lib.ssm_scan_fwd_ws(*ws_args(None, 0, **disjoint)) in (_native.SSM_OK, _native.SSM_ERR_LAUNCH)
    assert lib.ssm_scan_fwd_ws(*ws_args(ws + 8, MB, **disjoint)) == _native.SSM_ERR_ALIGN
    for k in ("u", "delta", "z", "B", "C", "y", "last", "A", "D", "dt_bias"):
        assert lib.ssm_scan_fwd_ws(*ws_args(disjoint[k], 64, **disjoint)) == _native.SSM_ERR_ARG, k
    # a workspace ending inside y's first element overlaps it; one ending right before does not
    assert lib.ssm_scan_fwd_ws(*ws_args(disjoint["y"] - 64, 65, **disjoint)) == _native.SSM_ERR_ARG
    assert lib.ssm_scan_fwd_ws(*ws_args(disjoint["y"] - 64, 64, **disjoint)) in (_native.SSM_OK,
                                                                                _native.SSM_ERR_LAUNCH)
    assert lib.ssm_scan_fwd_ws(*ws_args(ws, MB, **{**disjoint, "u": None})) == _native.SSM_ERR_NULL
    assert lib.ssm_scan_fwd_ws(*ws_args(ws, MB, **{**disjoint, "dstate": 17})) == _native.SSM_ERR_UNSUPPORTED
    args = ws_args(ws, MB, **disjoint)
    args[17] = 3  # discretization
    assert lib.ssm_scan_fwd_ws(*args) == _native.SSM_ERR_ARG


def test_workspace_size_validation(lib):
    n = ctypes.c_size_t(123)
    assert lib.ssm_scan_fwd_workspace_size(1, 64, 16, 8192, 1, 0, 1, None) == _native.SSM_ERR_NULL
    assert lib.ssm_scan_fwd_workspace_size(-1, 64, 16, 8192, 1, 0, 1, ctypes.byref(n)) == _native.SSM_ERR_SHAPE
    assert n.value == 0
    assert lib.ssm_scan_fwd_workspace_size(1, 64, 17, 8192, 1, 0, 1, ctypes.byref(n)) == _native.SSM_ERR_UNSUPPORTED
    assert lib.ssm_scan_fwd_workspace_size(1, 64, 16, 8192, 9, 0, 1, ctypes.byref(n)) == _native.SSM_ERR_DTYPE
    assert lib.ssm_scan_fwd_workspace_size(1, 64, 16, 8192, 1, 4, 1, ctypes.byref(n)) == _native.SSM_ERR_ARG
    assert lib.ssm_scan_fwd_workspace_size(0, 64, 16, 8192, 1, 0, 1, ctypes.byref(n)) == _native.SSM_OK
    assert n.value == 0
    # float32 io never splits; with no device the query of a bf16 scan reports SSM_ERR_LAUNCH
    assert lib.ssm_scan_fwd_workspace_size(1, 64, 16, 8192, 0, 0, 1, ctypes.byref(n)) == _native.SSM_OK
    assert n.value == 0
    assert lib.ssm_scan_fwd_workspace_size(1, 64, 16, 8192, 1, 0, 1, ctypes.byref(n)) in (_native.SSM_OK,
                                                                                         _native.SSM_ERR_LAUNCH)
