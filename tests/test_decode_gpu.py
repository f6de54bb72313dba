"""GPU parity of ssm_state_update (the decode step) against the float64 oracle (through the C-ABI)."""
import numpy as np
import pytest
import torch

import bench
import selective_state_space_155_b300 as ssm
import ssm_workloads as wl
from oracle import oracle
from tests.gpu_util import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
f = wl.to_f64


def random_step(batch, dim, dstate, io, seed, gate=True, use_D=True, use_bias=True):
    g = torch.Generator().manual_seed(seed)
    dt_ = torch.float32 if io == "f32" else torch.bfloat16
    r = lambda *s: torch.randn(*s, generator=g)
    return dict(state=r(batch, dim, dstate), x=r(batch, dim).to(dt_), dt=r(batch, dim).to(dt_),
                z=r(batch, dim).to(dt_) if gate else None, B=r(batch, dstate).to(dt_), C=r(batch, dstate).to(dt_),
                A=-torch.exp(torch.rand(dim, dstate, generator=g) * 3 - 1),
                D=r(dim) if use_D else None,
                dt_bias=torch.log(torch.expm1(torch.exp(torch.rand(dim, generator=g) * -4.6))) if use_bias else None)


@pytest.mark.parametrize("shape", [(1, 1, 1, "f32"), (3, 37, 16, "f32"), (2, 50, 5, "bf16"), (4, 129, 8, "bf16"),
                                   (2, 64, 4, "f32"), (5, 300, 16, "bf16"), (1, 7, 13, "bf16")])
@pytest.mark.parametrize("opts", [(True, True, True), (False, False, False), (True, False, True)])
def test_single_step(shape, opts):
    batch, dim, dstate, io = shape
    inp = random_step(batch, dim, dstate, io, seed=batch * dim + dstate, gate=opts[0], use_D=opts[1],
                      use_bias=opts[2])
    d = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    state = d["state"].clone()
    out = ssm.ssm_state_update(state, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                               dt_softplus=True)
    torch.cuda.synchronize()
    s_ref, o_ref = oracle.state_update(f(inp["state"]), f(inp["x"]), f(inp["dt"]), f(inp["A"]), f(inp["B"]),
                                       f(inp["C"]), f(inp["D"]), f(inp["z"]), f(inp["dt_bias"]), dt_softplus=True)
    ty, ts = TOL[io]
    assert_close(f(out), o_ref, ty, "out")
    assert_close(f(state), s_ref, ts, "state")


def test_steps_continue_a_scan():
    """scan(L1) then L2 decode steps from its last_state: every output and the final state
    match the oracle's scan over L1 + L2."""
    inp = wl.random_scan_case(2, 48, 16, 96, io="bf16", seed=21)
    dv = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    L1 = 80
    sl = lambda v, a, b: v[..., a:b].contiguous()
    y1, state = ssm.ssm_scan_fwd(sl(dv["u"], 0, L1), sl(dv["delta"], 0, L1), dv["A"], sl(dv["B"], 0, L1),
                                 sl(dv["C"], 0, L1), dv["D"], sl(dv["z"], 0, L1), dv["dt_bias"])
    outs = []
    for t in range(L1, 96):
        outs.append(ssm.ssm_state_update(state, dv["u"][:, :, t].contiguous(), dv["delta"][:, :, t].contiguous(),
                                         dv["A"], dv["B"][:, :, t].contiguous(), dv["C"][:, :, t].contiguous(),
                                         dv["D"], dv["z"][:, :, t].contiguous(), dv["dt_bias"]))
    torch.cuda.synchronize()
    y_ref, s_ref = oracle.scan(f(inp["u"]), f(inp["delta"]), f(inp["A"]), f(inp["B"]), f(inp["C"]), f(inp["D"]),
                               f(inp["z"]), f(inp["dt_bias"]))
    assert_close(f(y1), y_ref[..., :L1], 2e-2, "scan part")
    assert_close(np.stack([f(o) for o in outs], axis=-1), y_ref[..., L1:], 2e-2, "decode part")
    assert_close(f(state), s_ref, 1e-4, "final state")


def test_decode_workload_1024_steps_sampled():
    """The full decode workload (batch 256, d_inner 5120, d_state 16, 1024 steps) run as the
    benchmark runs it (one CUDA graph of 1024 in-place steps); the oracle follows 48 sampled
    channels through all 1024 steps and checks every step's output and the final state."""
    w = wl.DECODE
    run = bench.DecodeRun(w, DEV)
    rng = np.random.default_rng(4)
    bs = rng.integers(0, w.batch, 48)
    ds = rng.integers(0, w.dim, 48)
    s0 = f(run.state[bs, ds])  # [48, dstate] before the loop
    run.capture()
    run.graph.replay()
    torch.cuda.synchronize()
    inp = run.inputs
    xs, dts, zs = (f(inp[k][:, bs, ds]) for k in ("x", "dt", "z"))  # [steps, 48]
    Bs, Cs = (f(inp[k][:, bs]) for k in ("B", "C"))                  # [steps, 48, dstate]
    A, D, bias = f(run.params["A"])[ds], f(run.params["D"])[ds], f(run.params["dt_bias"])[ds]
    outs = f(run.out[:, bs, ds])
    ty, ts = TOL["bf16"]
    for i in range(len(bs)):
        # one channel followed through every step: the decode oracle iterated 1024 times equals the
        # scan oracle over those 1024 steps started from the same state (pinned on the CPU)
        y_ref, s_ref = oracle.scan(xs[:, i].reshape(1, 1, -1), dts[:, i].reshape(1, 1, -1), A[i][None, :],
                                   Bs[:, i, :].T[None], Cs[:, i, :].T[None], D[i:i + 1], zs[:, i].reshape(1, 1, -1),
                                   bias[i:i + 1], delta_softplus=True, h0=s0[i].reshape(1, 1, -1))
        assert_close(outs[:, i], y_ref.ravel(), ty, f"out of channel (b={bs[i]}, d={ds[i]})")
        assert_close(f(run.state[bs[i], ds[i]]), s_ref.ravel(), ts, f"final state of channel ({bs[i]}, {ds[i]})")


# The persistent tiled forms serve dstate 16 from 65536 channels up: tiles of 128 channels, a
# partial last tile when batch*dim is not a multiple of 128, and tiles that straddle batch rows
# when dim is not; when dim is, the tiles also stage dt_bias, D and the row's B, C, and the
# library's choice is the bulk-copy form (one bulk copy per operand range, one bulk store of the
# new states); SSM_DECODE_VARIANT=tiled forces the per-thread-copy tiled form.
TILED = [(37, 1800, "bf16"), (16, 4096, "f32"), (64, 1032, "bf16"), (32, 2048, "bf16")]


@pytest.mark.parametrize("shape", TILED, ids=lambda s: "b{}_d{}_{}".format(*s))
@pytest.mark.parametrize("opts", [(True, True, True), (False, False, False)])
@pytest.mark.parametrize("disc", ["delta_b", "zoh"])
@pytest.mark.parametrize("variant", ["auto", "tiled", "thread"])
def test_large_batch_step(shape, opts, disc, variant, monkeypatch):
    if variant == "auto":
        monkeypatch.delenv("SSM_DECODE_VARIANT", raising=False)
    else:
        monkeypatch.setenv("SSM_DECODE_VARIANT", variant)
    batch, dim, io = shape
    inp = random_step(batch, dim, 16, io, seed=batch + dim, gate=opts[0], use_D=opts[1], use_bias=opts[2])
    d = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    state = d["state"].clone()
    out = ssm.ssm_state_update(state, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"],
                               dt_softplus=True, discretization=disc)
    torch.cuda.synchronize()
    s_ref, o_ref = oracle.state_update(f(inp["state"]), f(inp["x"]), f(inp["dt"]), f(inp["A"]), f(inp["B"]),
                                       f(inp["C"]), f(inp["D"]), f(inp["z"]), f(inp["dt_bias"]), dt_softplus=True,
                                       zoh=disc == "zoh")
    ty, ts = TOL[io]
    assert_close(f(out), o_ref, ty, "out")
    assert_close(f(state), s_ref, ts, "state")


def test_tiled_and_thread_forms_agree():
    """The decode forms on the same large batch: the bulk-copy and tiled forms run the same
    per-channel arithmetic (bitwise equal); against the per-thread form the states are equal and
    the outputs agree to a bf16 rounding step (the readout sums run in different orders)."""
    inp = random_step(40, 2048, 16, "bf16", seed=77)
    d = {k: (v.to(DEV) if v is not None else None) for k, v in inp.items()}
    res = {}
    for variant in ("bulk", "tiled", "thread"):
        import os
        old = os.environ.pop("SSM_DECODE_VARIANT", None)
        if variant != "bulk":
            os.environ["SSM_DECODE_VARIANT"] = variant
        try:
            st = d["state"].clone()
            out = ssm.ssm_state_update(st, d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["z"], d["dt_bias"])
            torch.cuda.synchronize()
            res[variant] = (st, out)
        finally:
            os.environ.pop("SSM_DECODE_VARIANT", None)
            if old is not None:
                os.environ["SSM_DECODE_VARIANT"] = old
    assert torch.equal(res["bulk"][0], res["tiled"][0]) and torch.equal(res["bulk"][1], res["tiled"][1])
    assert torch.equal(res["tiled"][0], res["thread"][0])  # the update itself is identical per state
    a, b = res["tiled"][1].float(), res["thread"][1].float()
    assert float(((a - b).abs() / (1.0 + b.abs())).max()) <= 1e-2  # a bf16 rounding step at most
