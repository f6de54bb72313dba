"""GPU parity of ssm_scan_fwd / ssm_scan_fwd_h0 against the float64 oracle (through the C-ABI)."""
import numpy as np
import pytest
import torch

import selective_state_space_155_b300 as ssm
import ssm_workloads as wl
from tests.gpu_util import assert_state_rel, TOL, assert_close, io_name, oracle_scan, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(params=["auto", "quad_plain"])
def variant(request, monkeypatch):
    """Run a test with the library's choice of scan layout (balanced where its plan applies) and
    with the plain 32-channel CTAs forced."""
    if request.param != "auto":
        monkeypatch.setenv("SSM_SCAN_VARIANT", request.param)
    else:
        monkeypatch.delenv("SSM_SCAN_VARIANT", raising=False)
    return request.param


def run(inp, softplus=True, h0=None):
    y, last = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp.get("D"), inp.get("z"),
                               inp.get("dt_bias"), delta_softplus=softplus, h0=h0)
    torch.cuda.synchronize()
    assert ssm.wait_timeouts() == 0, "a hand-off wait inside the scan gave up"
    return wl.to_f64(y), wl.to_f64(last)


def check_case(inp, softplus=True, h0=None, what=""):
    ty, ts = TOL[io_name(inp["u"])]
    y, last = run(inp, softplus, h0)
    y_ref, s_ref = oracle_scan(inp, softplus, h0)
    ey = assert_close(y, y_ref, ty, f"{what} y")
    es = assert_close(last, s_ref, ts, f"{what} last_state")
    assert_state_rel(last, s_ref, f"{what} last_state")
    return ey, es


@pytest.mark.parametrize("w", [wl.TINY, wl.SMALL, wl.MID], ids=lambda w: w.name)
def test_workload_full_parity(w, variant):
    """Every output element of the tiny, small and mid-size workloads against the oracle."""
    inp = wl.scan_inputs(w, device=DEV)
    check_case(inp, what=w.name)


def test_long_workload_sampled_channels(variant):
    """The 65536-step workload at full size, in the launch configuration the benchmark times;
    the oracle recomputes 24 sampled channels (each channel is independent) end to end."""
    w = wl.LONG
    inp = wl.scan_inputs(w, device=DEV)
    y, last = run(inp)
    rng = np.random.default_rng(99)
    chans = np.unique(np.concatenate([[0, w.dim - 1], rng.choice(w.dim, 22, replace=False)]))
    ty, ts = TOL["bf16"]
    for d in chans:
        sub = dict(u=inp["u"][:, d:d + 1], delta=inp["delta"][:, d:d + 1], z=inp["z"][:, d:d + 1], B=inp["B"],
                   C=inp["C"], A=inp["A"][d:d + 1], D=inp["D"][d:d + 1], dt_bias=inp["dt_bias"][d:d + 1])
        y_ref, s_ref = oracle_scan(sub)
        assert_close(y[:, d:d + 1], y_ref, ty, f"long y channel {d}")
        assert_close(last[:, d:d + 1], s_ref, ts, f"long state channel {d}")


EDGE = [
    # (batch, dim, dstate, seqlen, io)
    (1, 1, 1, 1, "f32"),
    (1, 33, 16, 65, "f32"),
    (3, 31, 3, 100, "f32"),
    (2, 40, 5, 63, "bf16"),
    (2, 65, 8, 129, "bf16"),
    (1, 32, 12, 200, "bf16"),
    (2, 7, 16, 1, "bf16"),
    (1, 96, 16, 128, "bf16"),
    (2, 64, 4, 300, "f32"),
    (1, 50, 16, 1000, "f32"),
    (2, 100, 2, 77, "bf16"),
]


@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "b{}_d{}_n{}_l{}_{}".format(*s))
def test_edge_shapes(shape, variant):
    """Ragged lengths (scalar copy path), dim not a multiple of the CTA's 32 channels,
    dstate padded up to 4/8/16, single steps."""
    batch, dim, dstate, seqlen, io = shape
    inp = to_device(wl.random_scan_case(batch, dim, dstate, seqlen, io=io, seed=seqlen + dim), DEV)
    check_case(inp, what=str(shape))


@pytest.mark.parametrize("gate,use_D,use_bias,softplus", [
    (False, False, False, False), (True, False, True, True), (False, True, False, True), (True, True, True, False)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_optional_arguments(gate, use_D, use_bias, softplus, io, variant):
    inp = to_device(wl.random_scan_case(2, 48, 16, 136, io=io, seed=5, gate=gate, use_D=use_D, use_bias=use_bias,
                                        softplus=softplus), DEV)
    check_case(inp, softplus=softplus, what="optional args")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_initial_state_and_resume(io, variant):
    """h0 input, and scan(L1) then scan(L2) from last_state equals one scan over L1 + L2."""
    inp = to_device(wl.random_scan_case(2, 40, 16, 192, io=io, seed=3, h0=True), DEV)
    check_case(inp, h0=inp["h0"], what="h0")
    L1 = 72
    first = {k: (v[..., :L1].contiguous() if k in ("u", "delta", "z", "B", "C") else v) for k, v in inp.items()}
    second = {k: (v[..., L1:].contiguous() if k in ("u", "delta", "z", "B", "C") else v) for k, v in inp.items()}
    y1, l1 = ssm.ssm_scan_fwd(first["u"], first["delta"], first["A"], first["B"], first["C"], first["D"],
                              first["z"], first["dt_bias"])
    y2, l2 = ssm.ssm_scan_fwd(second["u"], second["delta"], second["A"], second["B"], second["C"], second["D"],
                              second["z"], second["dt_bias"], h0=l1)
    torch.cuda.synchronize()
    y_ref, s_ref = oracle_scan({k: v for k, v in inp.items() if k != "h0"})
    ty, ts = TOL[io]
    assert_close(np.concatenate([wl.to_f64(y1), wl.to_f64(y2)], axis=-1), y_ref, ty, "resumed y")
    assert_close(wl.to_f64(l2), s_ref, ts, "resumed state")


def test_in_place_state_resume():
    """last_state may be the same buffer as h0."""
    inp = to_device(wl.random_scan_case(1, 32, 16, 64, io="f32", seed=8, h0=True), DEV)
    y_ref, s_ref = oracle_scan(inp, h0=inp["h0"])
    st = inp["h0"].clone()
    y, last = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                               inp["dt_bias"], h0=st, last_state=st)
    torch.cuda.synchronize()
    assert last.data_ptr() == st.data_ptr()
    assert_close(wl.to_f64(y), y_ref, 1e-4, "y")
    assert_close(wl.to_f64(st), s_ref, 1e-4, "state in place")


def test_empty_sizes():
    A = torch.full((4, 16), -1.0, device=DEV)
    u = torch.empty((2, 4, 0), device=DEV)
    B = torch.empty((2, 16, 0), device=DEV)
    y, last = ssm.ssm_scan_fwd(u, u, A, B, B)
    torch.cuda.synchronize()
    assert y.shape == (2, 4, 0)
    assert torch.count_nonzero(last).item() == 0 and last.shape == (2, 4, 16)
    u0 = torch.empty((0, 4, 10), device=DEV)
    y, last = ssm.ssm_scan_fwd(u0, u0, A, torch.empty((0, 16, 10), device=DEV), torch.empty((0, 16, 10), device=DEV))
    assert y.shape == (0, 4, 10)


def test_delta_zero_is_skip_only_on_gpu(variant):
    """Delta = 0 (no softplus, no bias): the state never moves and y = D u, i.e. the float32
    product rounded to bf16."""
    inp = to_device(wl.random_scan_case(2, 64, 16, 256, io="bf16", seed=4, gate=False, use_bias=False,
                                        softplus=False), DEV)
    inp["delta"] = torch.zeros_like(inp["delta"])
    y, last = run(inp, softplus=False)
    ref = (inp["D"].cpu()[None, :, None] * inp["u"].cpu().float()).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(y, ref)
    assert np.count_nonzero(last) == 0


def test_misaligned_pointer_rejected():
    """A float32 pointer that is not 4-byte aligned is refused on the host (nothing launched)."""
    inp = to_device(wl.random_scan_case(1, 4, 4, 16, io="bf16", seed=1), DEV)
    y = torch.empty_like(inp["u"])
    st = ssm.lib().ssm_scan_fwd(inp["u"].data_ptr(), inp["delta"].data_ptr(), inp["A"].data_ptr() + 2,
                                inp["B"].data_ptr(), inp["C"].data_ptr(), None, None, None, 1, y.data_ptr(), None,
                                1, 4, 4, 16, 1, None)
    assert st == ssm._native.SSM_ERR_ALIGN
