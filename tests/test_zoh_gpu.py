"""GPU parity of the exact zero-order-hold discretisation (ssm_scan_fwd_ex / ssm_state_update_ex
with SSM_DISC_ZOH) against the float64 oracle, through the C-ABI.

Bbar = (exp(Delta A) - 1) / A * B: the kernels evaluate it from the exponential they already
have where |Delta A| >= 1/16 and from a short series below that; the cases here put states on
both sides of that threshold, at A = 0, and at the workload sizes."""
import numpy as np
import pytest
import torch

import selective_state_space_155_b300 as ssm
import ssm_workloads as wl
from oracle import oracle
from tests.gpu_util import TOL, assert_close, io_name, oracle_scan, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
f = wl.to_f64


def run_zoh(inp, softplus=True, h0=None):
    y, last = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp.get("D"), inp.get("z"),
                               inp.get("dt_bias"), delta_softplus=softplus, h0=h0, discretization="zoh")
    torch.cuda.synchronize()
    return f(y), f(last)


def check_zoh(inp, softplus=True, h0=None, what=""):
    ty, ts = TOL[io_name(inp["u"])]
    y, last = run_zoh(inp, softplus, h0)
    y_ref, s_ref = oracle_scan(inp, softplus, h0, zoh=True)
    assert_close(y, y_ref, ty, f"{what} y")
    assert_close(last, s_ref, ts, f"{what} last_state")
    return y_ref


@pytest.mark.parametrize("w", [wl.TINY, wl.SMALL, wl.MID], ids=lambda w: w.name)
def test_zoh_workload_full_parity(w):
    inp = wl.scan_inputs(w, device=DEV)
    y_ref = check_zoh(inp, what=w.name)
    # the two discretisations really differ on these inputs
    y_eul, _ = oracle_scan(inp)
    assert np.max(np.abs(y_ref - y_eul)) > 1e-3


@pytest.mark.parametrize("shape", [(1, 1, 1, 1, "f32"), (1, 33, 16, 65, "f32"), (2, 40, 5, 63, "bf16"),
                                   (2, 65, 8, 129, "bf16"), (2, 64, 4, 300, "f32"), (1, 96, 16, 128, "bf16")],
                         ids=lambda s: "b{}_d{}_n{}_l{}_{}".format(*s))
def test_zoh_edge_shapes(shape):
    batch, dim, dstate, seqlen, io = shape
    inp = to_device(wl.random_scan_case(batch, dim, dstate, seqlen, io=io, seed=seqlen + dim + 1), DEV)
    check_zoh(inp, what=str(shape))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_both_branches_and_zero_A(io):
    """A spans 0, tiny and large magnitudes so that |Delta A| falls on both sides of the series
    threshold, including exact zeros (the limit Delta * B)."""
    inp = wl.random_scan_case(2, 64, 16, 160, io=io, seed=17)
    A = inp["A"].clone()
    g = torch.Generator().manual_seed(3)
    mags = torch.tensor([0.0, 1e-6, 1e-3, 0.05, 0.3, 1.0, 4.0, 20.0])
    A = -mags[torch.randint(0, mags.numel(), A.shape, generator=g)]
    inp["A"] = A.contiguous()
    check_zoh(to_device(inp, DEV), what="branches")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_initial_state_and_no_softplus(io):
    inp = to_device(wl.random_scan_case(2, 40, 16, 192, io=io, seed=13, h0=True, softplus=False), DEV)
    check_zoh(inp, softplus=False, h0=inp["h0"], what="h0 no-softplus")


def test_zoh_decode_steps_continue_a_zoh_scan():
    inp = wl.random_scan_case(2, 48, 16, 96, io="bf16", seed=23)
    dv = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    L1 = 64
    sl = lambda v, a, b: v[..., a:b].contiguous()
    y1, state = ssm.ssm_scan_fwd(sl(dv["u"], 0, L1), sl(dv["delta"], 0, L1), dv["A"], sl(dv["B"], 0, L1),
                                 sl(dv["C"], 0, L1), dv["D"], sl(dv["z"], 0, L1), dv["dt_bias"], discretization="zoh")
    outs = []
    for t in range(L1, 96):
        outs.append(ssm.ssm_state_update(state, dv["u"][:, :, t].contiguous(), dv["delta"][:, :, t].contiguous(),
                                         dv["A"], dv["B"][:, :, t].contiguous(), dv["C"][:, :, t].contiguous(),
                                         dv["D"], dv["z"][:, :, t].contiguous(), dv["dt_bias"],
                                         discretization="zoh"))
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.scan(f(inp["u"]), f(inp["delta"]), f(inp["A"]), f(inp["B"]), f(inp["C"]), f(inp["D"]),
                               f(inp["z"]), f(inp["dt_bias"]), zoh=True)
    assert_close(f(y1), y_ref[..., :L1], 2e-2, "zoh scan part")
    assert_close(np.stack([f(o) for o in outs], axis=-1), y_ref[..., L1:], 2e-2, "zoh decode part")
    assert_close(f(state), s_ref, 1e-4, "zoh final state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [1, 5, 16])
def test_zoh_single_decode_step(io, dstate):
    g = torch.Generator().manual_seed(dstate)
    dt_ = torch.float32 if io == "f32" else torch.bfloat16
    r = lambda *s: torch.randn(*s, generator=g)
    batch, dim = 3, 70
    A = -torch.exp(torch.rand(dim, dstate, generator=g) * 6 - 5)
    A[0, 0] = 0.0
    inp = dict(state=r(batch, dim, dstate), x=r(batch, dim).to(dt_), dt=r(batch, dim).to(dt_),
               z=r(batch, dim).to(dt_), B=r(batch, dstate).to(dt_), C=r(batch, dstate).to(dt_), A=A, D=r(dim),
               dt_bias=torch.rand(dim, generator=g) - 2.0)
    d = {k: v.to(DEV) for k, v in inp.items()}
    state = d["state"].clone()
    out = ssm.ssm_state_update(state, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                               discretization="zoh")
    torch.cuda.synchronize()
    s_ref, o_ref = oracle.state_update(f(inp["state"]), f(inp["x"]), f(inp["dt"]), f(inp["A"]), f(inp["B"]),
                                       f(inp["C"]), f(inp["D"]), f(inp["z"]), f(inp["dt_bias"]), zoh=True)
    ty, ts = TOL[io]
    assert_close(f(out), o_ref, ty, "zoh out")
    assert_close(f(state), s_ref, ts, "zoh state")


def test_zoh_binding_rejects_unknown_discretization():
    with pytest.raises(ValueError):
        ssm.ssm_scan_fwd(*(torch.empty(1, 1, 1, device=DEV),) * 2, torch.empty(1, 1, device=DEV),
                         torch.empty(1, 1, 1, device=DEV), torch.empty(1, 1, 1, device=DEV), discretization="bilinear")
