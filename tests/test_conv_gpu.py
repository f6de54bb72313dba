"""GPU parity of the causal depthwise conv1d (ssm_causal_conv1d_fwd / ssm_causal_conv1d_update)
against the float64 oracle, through the C-ABI.  The conv is a few multiply-adds per element, so
fp32 outputs are held to 1e-5 and bf16 outputs to their rounding (2^-8 relative)."""
import numpy as np
import pytest
import torch

import selective_state_space_155_b300 as ssm
import ssm_workloads as wl
from oracle import oracle
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
f = wl.to_f64
TOL = {"f32": 1e-5, "bf16": 8e-3}


def dev(inp):
    return {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}


def check(inp, io, silu=True, with_state=True, what=""):
    d = dev(inp)
    out, st = ssm.causal_conv1d_fwd(d["x"], d["weight"], d["bias"], d["state"] if with_state else None, silu=silu,
                                    return_state=True)
    torch.cuda.synchronize()
    ref, st_ref = oracle.causal_conv1d(f(inp["x"]), f(inp["weight"]), f(inp["bias"]),
                                       f(inp["state"]) if with_state else None, silu=silu)
    assert_close(f(out), ref, TOL[io], f"{what} out")
    np.testing.assert_array_equal(f(st), st_ref)  # the carried state is a copy of inputs: exact


def test_mid_shape_full_parity():
    """The scan's mid-size activation shape (batch 8, d_inner 1536, L 2048, bf16), width 4, silu."""
    inp = wl.conv_inputs(8, 1536, 2048, 4, "bf16", seed=2, state=True)
    check(inp, "bf16", what="mid")


@pytest.mark.parametrize("shape", [
    # (batch, dim, seqlen, width, io): vector rows, ragged rows (one element per thread),
    # rows shorter than the state, single steps, every width
    (2, 33, 64, 4, "bf16"), (2, 33, 64, 4, "f32"), (1, 7, 61, 4, "bf16"), (3, 5, 2, 4, "f32"),
    (2, 9, 1, 3, "bf16"), (2, 40, 96, 1, "bf16"), (2, 40, 96, 2, "f32"), (1, 300, 8, 3, "bf16"),
    (4, 17, 1000, 4, "f32"), (1, 1, 3, 4, "bf16"),
    # rows of an odd number of 16-byte vectors (the strided two-vector form), and of one vector
    (2, 37, 40, 4, "bf16"), (3, 9, 12, 3, "f32"), (2, 70, 8, 4, "bf16"), (1, 33, 4, 2, "f32"),
], ids=lambda s: "b{}_d{}_l{}_w{}_{}".format(*s))
@pytest.mark.parametrize("silu,with_state", [(True, True), (False, False), (True, False)])
def test_edge_shapes(shape, silu, with_state):
    batch, dim, L, W, io = shape
    inp = wl.conv_inputs(batch, dim, L, W, io, seed=batch * 31 + dim + L, state=True, bias=silu)
    check(inp, io, silu=silu, with_state=with_state, what=str(shape))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_streaming_two_pieces_equals_one_call(io):
    inp = dev(wl.conv_inputs(2, 64, 320, 4, io, seed=9))
    full = ssm.causal_conv1d_fwd(inp["x"], inp["weight"], inp["bias"])
    o1, s1 = ssm.causal_conv1d_fwd(inp["x"][..., :128].contiguous(), inp["weight"], inp["bias"], return_state=True)
    o2 = ssm.causal_conv1d_fwd(inp["x"][..., 128:].contiguous(), inp["weight"], inp["bias"], state_in=s1)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([o1, o2], dim=-1), full)


def test_empty_row_copies_the_state():
    inp = dev(wl.conv_inputs(2, 3, 0, 4, "bf16", seed=1, state=True))
    so = torch.zeros_like(inp["state"])
    ssm.causal_conv1d_fwd(inp["x"], inp["weight"], inp["bias"], inp["state"], state_out=so)
    torch.cuda.synchronize()
    assert torch.equal(so, inp["state"])


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("W", [1, 2, 4])
def test_decode_steps_equal_the_full_conv(io, W):
    """L decode steps from a carried state give the outputs and final state of one call."""
    batch, dim, L = 3, 70, 12
    inp = wl.conv_inputs(batch, dim, L, W, io, seed=W, state=True)
    d = dev(inp)
    state = d["state"].clone() if W > 1 else None
    outs = [ssm.causal_conv1d_update(state, d["x"][:, :, t].contiguous(), d["weight"], d["bias"])
            for t in range(L)]
    torch.cuda.synchronize()
    ref, st_ref = oracle.causal_conv1d(f(inp["x"]), f(inp["weight"]), f(inp["bias"]), f(inp["state"]))
    assert_close(np.stack([f(o) for o in outs], axis=-1), ref, TOL[io], "decode outs")
    if W > 1:
        np.testing.assert_array_equal(f(state), st_ref)


def test_conv_then_scan_block_prologue():
    """The block order: u = silu(conv(x)), then the scan on u, against the oracle chain."""
    w = wl.SMALL
    inp = wl.scan_inputs(w)
    cin = wl.conv_inputs(w.batch, w.dim, w.seqlen, 4, w.io, seed=5)
    d = dev(cin)
    u = ssm.causal_conv1d_fwd(d["x"], d["weight"], d["bias"])
    y, last = ssm.ssm_scan_fwd(u, *(inp[k].to(DEV) if inp[k] is not None else None
                                    for k in ("delta", "A", "B", "C", "D", "z", "dt_bias")))
    torch.cuda.synchronize()
    u_ref, _ = oracle.causal_conv1d(f(cin["x"]), f(cin["weight"]), f(cin["bias"]))
    y_ref, s_ref = oracle.scan(f(u), f(inp["delta"]), f(inp["A"]), f(inp["B"]), f(inp["C"]), f(inp["D"]),
                               f(inp["z"]), f(inp["dt_bias"]))
    assert_close(f(u), u_ref, 1e-5, "conv")
    assert_close(f(y), y_ref, 1e-4, "scan after conv")
    assert_close(f(last), s_ref, 1e-4, "state after conv")
