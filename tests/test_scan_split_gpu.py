"""The split form of the forward scan (few channels, long sequences): segments of the sequence
scanned side by side, the state entering each one combined from carry segments by the pair
operator (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2).  Checked against the float64 oracle on every
element, against the unsplit scan (SSM_SCAN_SPLIT=off), for forced segment counts, both
discretizations, an initial state, lengths that are not a whole number of chunks, carries that
barely decay, and the form the long workload takes."""
import numpy as np
import pytest
import torch

import selective_state_space_155_b300 as ssm
import ssm_workloads as wl
from tests.gpu_util import TOL, assert_close, assert_state_rel, oracle_scan, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

# (batch, dim, dstate, seqlen): one row; two rows with a length that is not a whole number of
# 32-step chunks (one chunk per copy); padded states (dstate 12) on a length of 9000; three rows of
# 40 channels (8-channel groups)
SHAPES = [(1, 64, 16, 8192), (2, 64, 16, 8232), (1, 128, 12, 9000), (3, 40, 16, 8256)]


def set_split(monkeypatch, split):
    monkeypatch.delenv("SSM_SCAN_VARIANT", raising=False)
    if split is None:
        monkeypatch.delenv("SSM_SCAN_SPLIT", raising=False)
    else:
        monkeypatch.setenv("SSM_SCAN_SPLIT", split)


def run(inp, monkeypatch, split=None, disc="delta_b", h0=None, last_state=None):
    set_split(monkeypatch, split)
    y, last = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                               inp["dt_bias"], delta_softplus=inp.get("softplus", True), h0=h0,
                               last_state=last_state, discretization=disc)
    torch.cuda.synchronize()
    assert ssm.wait_timeouts() == 0, "a hand-off wait inside the scan gave up"
    return y, last


def form_of(inp, disc="delta_b"):
    batch, dim, L = inp["u"].shape
    return ssm.scan_fwd_form(batch, dim, inp["A"].shape[1], L, inp["u"].dtype, disc)[0]


def check_oracle(y, last, inp, disc="delta_b", h0=None, what=""):
    ty, ts = TOL["bf16"]
    y_ref, s_ref = oracle_scan(inp, inp.get("softplus", True), h0, zoh=disc == "zoh")
    assert_close(wl.to_f64(y), y_ref, ty, f"{what} y")
    assert_close(wl.to_f64(last), s_ref, ts, f"{what} last_state")
    assert_state_rel(wl.to_f64(last), s_ref, f"{what} last_state")
    return y_ref, s_ref


def test_split_form_chosen(monkeypatch):
    """The split applies to few channels and long sequences only, and the switch turns it off."""
    set_split(monkeypatch, None)
    for shape in SHAPES:
        assert ssm.scan_fwd_form(*shape)[0] == "split", shape
    assert ssm.scan_fwd_form(*shape, discretization="zoh")[0] == "split"
    assert ssm.scan_fwd_form(1, 2048, 16, 32768)[0] == "split"
    # the long workload: 640 units, one full group per SM on whole rows and its 48-unit tail split
    assert ssm.scan_fwd_form(1, 5120, 16, 65536)[0] == "split"
    assert ssm.scan_fwd_form(1, 4736, 16, 65536)[0] == "plain"  # 592 units: one full group per SM, no tail
    assert ssm.scan_fwd_form(8, 1536, 16, 2048)[0] == "balanced"  # the mid workload: many channels
    assert ssm.scan_fwd_form(1, 64, 16, 4096)[0] == "balanced"  # too short
    assert ssm.scan_fwd_form(1, 64, 16, 8192, aligned_rows=False)[0] != "split"
    assert ssm.scan_fwd_form(1, 64, 16, 8192, dtype=torch.float32)[0] == "plain"
    set_split(monkeypatch, "off")
    assert ssm.scan_fwd_form(1, 64, 16, 8192)[0] == "balanced"


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}_d{}_n{}_l{}".format(*s))
@pytest.mark.parametrize("mode", ["plain_args", "h0", "zoh", "no_gate"])
def test_split_against_oracle(shape, mode, monkeypatch):
    batch, dim, N, L = shape
    inp = to_device(wl.random_scan_case(batch, dim, N, L, io="bf16", seed=dim + L, gate=mode != "no_gate",
                                        h0=mode == "h0"), DEV)
    disc = "zoh" if mode == "zoh" else "delta_b"
    h0 = inp["h0"] if mode == "h0" else None
    set_split(monkeypatch, None)
    assert form_of(inp, disc) == "split"
    y, last = run(inp, monkeypatch, None, disc, h0)
    check_oracle(y, last, inp, disc, h0, f"split {mode}")


@pytest.mark.parametrize("disc", ["delta_b", "zoh"])
def test_split_equals_unsplit(disc, monkeypatch):
    """The split and the unsplit scan differ only in float32 rounding (a segment's decay is one
    exponential of a sum rather than a product of per-step exponentials): y within two bf16 steps,
    the state within 2e-5 relative."""
    inp = to_device(wl.random_scan_case(2, 64, 16, 8192, io="bf16", seed=21, h0=True), DEV)
    ys, ss = run(inp, monkeypatch, None, disc, inp["h0"])
    yu, su = run(inp, monkeypatch, "off", disc, inp["h0"])
    ys, yu, ss, su = (wl.to_f64(t) for t in (ys, yu, ss, su))
    assert np.max(np.abs(ys - yu) / (1.0 + np.abs(yu))) <= 2.0 ** -7
    assert np.max(np.abs(ss - su) / (1.0 + np.abs(su))) <= 2e-5


@pytest.mark.parametrize("split", ["2,1", "2,4", "3,2", "4,1", "4,4"])
def test_forced_segment_counts(split, monkeypatch):
    """Every (segments, carry segments per segment) the switch can force gives the oracle's result."""
    inp = to_device(wl.random_scan_case(1, 64, 16, 8192, io="bf16", seed=5, h0=True), DEV)
    set_split(monkeypatch, split)
    assert form_of(inp) == "split", split
    y, last = run(inp, monkeypatch, split, "delta_b", inp["h0"])
    check_oracle(y, last, inp, "delta_b", inp["h0"], f"split {split}")


@pytest.mark.parametrize("disc", ["delta_b", "zoh"])
def test_carries_that_barely_decay(disc, monkeypatch):
    """Small |A| and small steps: a segment's state reaches through every later segment (the decay
    over a whole carry segment stays near 1), so a wrong carry or a wrong combine order shows in
    every output after the first segment."""
    inp = wl.random_scan_case(1, 64, 16, 8192, io="bf16", seed=9, h0=True)
    inp["A"] = -0.01 * torch.arange(1, 17, dtype=torch.float32).repeat(64, 1)
    inp["dt_bias"] = torch.full((64,), float(np.log(np.expm1(1e-3))), dtype=torch.float32)
    inp = to_device(inp, DEV)
    y, last = run(inp, monkeypatch, "4,4", disc, inp["h0"])
    y_ref, s_ref = check_oracle(y, last, inp, disc, inp["h0"], "slow decay")
    # the carried part is large here: the state at the end is far from what the last segment alone
    # would build from zero
    assert np.max(np.abs(s_ref)) > 1.0


def test_in_place_state_is_not_split(monkeypatch):
    """last_state on the same buffer as h0 runs unsplit (a split's full pass would read h0 in one
    segment while another writes the final state) and still matches the oracle."""
    inp = to_device(wl.random_scan_case(1, 64, 16, 8192, io="bf16", seed=11, h0=True), DEV)
    y_ref, s_ref = oracle_scan(inp, True, inp["h0"])
    st = inp["h0"].clone()
    y, last = run(inp, monkeypatch, None, "delta_b", st, st)
    assert last.data_ptr() == st.data_ptr()
    assert_close(wl.to_f64(y), y_ref, TOL["bf16"][0], "y")
    assert_close(wl.to_f64(st), s_ref, TOL["bf16"][1], "state in place")


def test_split_stream_capture(monkeypatch):
    """The split's stream-ordered carry buffers work inside a captured CUDA graph, replayed twice."""
    inp = to_device(wl.random_scan_case(1, 64, 16, 8192, io="bf16", seed=13), DEV)
    set_split(monkeypatch, None)
    y = torch.empty_like(inp["u"])
    last = torch.empty((1, 64, 16), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["dt_bias"],
                     y=y, last_state=last, stream=s)  # warm-up on the capture stream
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                         inp["dt_bias"], y=y, last_state=last, stream=s)
    for _ in range(2):
        y.zero_(), last.zero_()
        g.replay()
        torch.cuda.synchronize()
        check_oracle(y, last, inp, what="graph replay")


def workspace_for(inp, disc="delta_b"):
    """A float32 workspace of the bytes the scan of `inp` reports, and that byte count."""
    batch, dim, L = inp["u"].shape
    N = inp["A"].shape[1]
    n = ssm.scan_fwd_workspace_size(batch, dim, N, L, inp["u"].dtype, disc)
    return torch.empty(n // 4, dtype=torch.float32, device=DEV), n


def test_workspace_size(monkeypatch):
    """Split shapes need 4 (dstate + 1) bytes per batch row, channel and carry segment; others none."""
    set_split(monkeypatch, None)
    for (batch, dim, N, L) in SHAPES:
        n = ssm.scan_fwd_workspace_size(batch, dim, N, L)
        assert n > 0 and n % (4 * batch * dim * (N + 1)) == 0, (batch, dim, N, L, n)
    assert ssm.scan_fwd_workspace_size(8, 1536, 16, 2048) == 0
    assert ssm.scan_fwd_workspace_size(1, 64, 16, 8192, dtype=torch.float32) == 0
    set_split(monkeypatch, "off")
    assert ssm.scan_fwd_workspace_size(1, 64, 16, 8192) == 0


@pytest.mark.parametrize("disc", ["delta_b", "zoh"])
def test_workspace_scan_equals_allocating_scan(disc, monkeypatch):
    """ssm_scan_fwd_ws with the reported workspace runs the same split, bit for bit; with one float
    too few it runs unsplit, bit for bit the SSM_SCAN_SPLIT=off result."""
    inp = to_device(wl.random_scan_case(2, 64, 16, 8232, io="bf16", seed=31, h0=True), DEV)
    ya, sa = run(inp, monkeypatch, None, disc, inp["h0"])
    ws, n = workspace_for(inp, disc)
    assert n > 0 and ws.numel() * 4 == n
    yw, sw = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                              inp["dt_bias"], h0=inp["h0"], discretization=disc, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(ya, yw) and torch.equal(sa, sw)
    small = torch.empty(n // 4 - 1, dtype=torch.float32, device=DEV)
    ys, ss = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                              inp["dt_bias"], h0=inp["h0"], discretization=disc, workspace=small)
    torch.cuda.synchronize()
    yo, so = run(inp, monkeypatch, "off", disc, inp["h0"])
    assert torch.equal(ys, yo) and torch.equal(ss, so)
    check_oracle(yw, sw, inp, disc, inp["h0"], "workspace")


def test_workspace_scan_in_a_graph(monkeypatch):
    """With a workspace the split enqueues kernels only, so a captured graph of it replays with no
    allocation node; replayed twice against the oracle."""
    inp = to_device(wl.random_scan_case(1, 64, 16, 8192, io="bf16", seed=17), DEV)
    set_split(monkeypatch, None)
    ws, n = workspace_for(inp)
    y = torch.empty_like(inp["u"])
    last = torch.empty((1, 64, 16), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    call = ssm.prepare_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["dt_bias"], y=y, last_state=last, workspace=ws, stream=s)
    torch.cuda.synchronize()
    call()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for _ in range(2):
        y.zero_(), last.zero_()
        g.replay()
        torch.cuda.synchronize()
        check_oracle(y, last, inp, what="workspace graph replay")


# Tail splits: one full 4-unit group per SM runs whole rows and the last batch row's remaining
# units are split (batch 1 with 4800 channels: a 48-unit tail; batch 2 with 2400: the tail starts
# inside the last row).
TAIL_SHAPES = [(1, 4800, 16, 8192), (2, 2400, 16, 8192)]


@pytest.mark.parametrize("shape", TAIL_SHAPES, ids=lambda s: "b{}_d{}_n{}_l{}".format(*s))
@pytest.mark.parametrize("mode", ["plain_args", "h0_zoh"])
def test_tail_split_against_oracle(shape, mode, monkeypatch):
    batch, dim, N, L = shape
    inp = to_device(wl.random_scan_case(batch, dim, N, L, io="bf16", seed=dim + 7, h0=mode == "h0_zoh"), DEV)
    disc = "zoh" if mode == "h0_zoh" else "delta_b"
    h0 = inp["h0"] if mode == "h0_zoh" else None
    set_split(monkeypatch, None)
    assert form_of(inp, disc) == "split"
    y, last = run(inp, monkeypatch, None, disc, h0)
    check_oracle(y, last, inp, disc, h0, f"tail split {mode}")
    yo, so = run(inp, monkeypatch, "off", disc, h0)
    y, yo, last, so = (wl.to_f64(t) for t in (y, yo, last, so))
    assert np.max(np.abs(y - yo) / (1.0 + np.abs(yo))) <= 2.0 ** -7
    assert np.max(np.abs(last - so) / (1.0 + np.abs(so))) <= 2e-5
