"""Out-of-bounds write detection without a sanitizer: every output buffer of every entry point is
carved out of a larger allocation whose guard regions before and after it hold a sentinel, and
the guards must be bit-identical after the launches.  Shapes are ragged (dim not a multiple of
the CTA's channels, L not a multiple of the chunk, dstate padded) so that every tail path runs."""
import pytest
import torch

import selective_state_space_155_b300 as ssm
import ssm_workloads as wl
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
GUARD = 256  # elements on each side


class Guarded:
    """A buffer of `shape` inside a larger one filled with a sentinel; `view` is the buffer."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        self.n = n
        self.base = torch.empty(n + 2 * GUARD, dtype=dtype, device=DEV)
        if dtype.is_floating_point:
            self.base.fill_(-12345.0)
        else:
            self.base.fill_(-12345)
        # keep the view 16-byte aligned: GUARD elements is a multiple of 16 bytes for every dtype used
        self.view = self.base[GUARD:GUARD + n].view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        lo, hi = self.base[:GUARD], self.base[GUARD + self.n:]
        assert bool((lo == -12345).all()) and bool((hi == -12345).all()), f"{what}: write outside the buffer"


# bf16 with dstate 9..16 and dim a multiple of 8 takes the balanced layout
SHAPES = [(2, 33, 16, 65, "bf16"), (1, 40, 5, 63, "f32"), (3, 7, 3, 100, "bf16"), (1, 65, 8, 31, "f32"),
          (2, 40, 16, 65, "bf16"), (3, 1032, 16, 70, "bf16"), (2, 40, 12, 77, "f32"), (1, 24, 9, 40, "bf16")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}_d{}_n{}_l{}_{}".format(*s))
@pytest.mark.parametrize("variant", ["default", "quad_plain"])
def test_scan_outputs_stay_in_bounds(shape, variant, monkeypatch):
    if variant == "default":  # the balanced form wherever its plan applies
        monkeypatch.delenv("SSM_SCAN_VARIANT", raising=False)
    else:
        monkeypatch.setenv("SSM_SCAN_VARIANT", variant)
    batch, dim, N, L, io = shape
    inp = to_device(wl.random_scan_case(batch, dim, N, L, io=io, seed=L, h0=True), DEV)
    y = Guarded((batch, dim, L), inp["u"].dtype)
    last = Guarded((batch, dim, N), torch.float32)
    ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["dt_bias"],
                     h0=inp["h0"], y=y.view, last_state=last.view)
    y.check("y")
    last.check("last_state")
    yz = Guarded((batch, dim, L), inp["u"].dtype)
    ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["dt_bias"],
                     y=yz.view, return_last_state=False, discretization="zoh")
    yz.check("y (zoh)")


# split forms: a full split with a ragged length (one chunk per copy), padded states and three rows
# of 40 channels, and a tail split (whole rows first, then the last row's tail)
SPLIT_SHAPES = [(2, 64, 12, 8232), (3, 40, 16, 8256), (1, 4800, 16, 8192)]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=lambda s: "b{}_d{}_n{}_l{}".format(*s))
@pytest.mark.parametrize("disc", ["delta_b", "zoh"])
def test_split_scan_writes_stay_in_bounds(shape, disc, monkeypatch):
    """The split's outputs and its caller-owned carry buffers: nothing is written outside y,
    last_state or the workspace the scan reports."""
    monkeypatch.delenv("SSM_SCAN_VARIANT", raising=False)
    monkeypatch.delenv("SSM_SCAN_SPLIT", raising=False)
    batch, dim, N, L = shape
    assert ssm.scan_fwd_form(batch, dim, N, L, discretization=disc)[0] == "split"
    inp = to_device(wl.random_scan_case(batch, dim, N, L, io="bf16", seed=L + 3, h0=True), DEV)
    nbytes = ssm.scan_fwd_workspace_size(batch, dim, N, L, discretization=disc)
    ws = Guarded((nbytes // 4,), torch.float32)
    y = Guarded((batch, dim, L), inp["u"].dtype)
    last = Guarded((batch, dim, N), torch.float32)
    ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["dt_bias"],
                     h0=inp["h0"], y=y.view, last_state=last.view, discretization=disc, workspace=ws.view)
    ws.check("workspace")
    y.check("y (split)")
    last.check("last_state (split)")


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}_d{}_n{}_l{}_{}".format(*s))
@pytest.mark.parametrize("disc", ["delta_b", "zoh"])
def test_training_pair_outputs_stay_in_bounds(shape, disc):
    batch, dim, N, L, io = shape
    inp = to_device(wl.random_scan_case(batch, dim, N, L, io=io, seed=L + 1), DEV)
    ck = Guarded((batch, ssm.scan_num_checkpoints(L), dim, N), torch.float32)
    y = Guarded((batch, dim, L), inp["u"].dtype)
    ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"], inp["dt_bias"],
                     y=y.view, checkpoints=ck.view, discretization=disc)
    ck.check("checkpoints")
    y.check("y (training forward)")
    dout = torch.randn(inp["u"].shape, device=DEV).to(inp["u"].dtype)
    g = {k: Guarded(s, t) for k, (s, t) in {
        "du": ((batch, dim, L), inp["u"].dtype), "ddelta": ((batch, dim, L), inp["u"].dtype),
        "dz": ((batch, dim, L), inp["u"].dtype), "dA": ((dim, N), torch.float32),
        "dB": ((batch, N, L), torch.float32), "dC": ((batch, N, L), torch.float32), "dD": ((dim,), torch.float32),
        "ddt_bias": ((dim,), torch.float32), "dh0": ((batch, dim, N), torch.float32)}.items()}
    p = lambda t: t.data_ptr()
    st = ssm.lib().ssm_scan_bwd_ex(p(inp["u"]), p(inp["delta"]), p(inp["A"]), p(inp["B"]), p(inp["C"]),
                                   p(inp["D"]), p(inp["z"]), p(inp["dt_bias"]), 1, p(ck.view), p(dout),
                                   p(g["du"].view), p(g["ddelta"].view), p(g["dA"].view), p(g["dB"].view),
                                   p(g["dC"].view), p(g["dD"].view), p(g["dz"].view), p(g["ddt_bias"].view),
                                   p(g["dh0"].view), batch, dim, N, L, ssm.io_dtype_code(inp["u"].dtype),
                                   1 if disc == "zoh" else 0, None)
    assert st == 0
    for k, b in g.items():
        b.check(k)


@pytest.mark.parametrize("shape", [(2, 33, 16, "bf16"), (3, 37, 5, "f32"), (1, 129, 8, "bf16"),
                                   (37, 1800, 16, "bf16"), (33, 2000, 16, "f32"), (16, 4096, 16, "bf16")])
def test_decode_outputs_stay_in_bounds(shape):
    batch, dim, N, io = shape
    dt_ = torch.float32 if io == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(dim)
    r = lambda *s: torch.randn(*s, generator=g).to(DEV)
    st = Guarded((batch, dim, N), torch.float32)
    st.view.copy_(r(batch, dim, N))
    out = Guarded((batch, dim), dt_)
    A = -torch.rand(dim, N, generator=g).to(DEV) - 0.1
    for disc in ("delta_b", "zoh"):
        ssm.ssm_state_update(st.view, r(batch, dim).to(dt_), r(batch, dim).to(dt_), A, r(batch, N).to(dt_),
                             r(batch, N).to(dt_), r(dim), r(batch, dim).to(dt_), r(dim), out=out.view,
                             discretization=disc)
        st.check(f"state ({disc})")
        out.check(f"out ({disc})")


@pytest.mark.parametrize("shape", [(2, 33, 64, 4, "bf16"), (2, 9, 61, 3, "f32"), (2, 37, 40, 4, "bf16"),
                                   (1, 5, 2, 4, "bf16")])
def test_conv_outputs_stay_in_bounds(shape):
    batch, dim, L, W, io = shape
    inp = {k: (v.to(DEV) if v is not None else None)
           for k, v in wl.conv_inputs(batch, dim, L, W, io, seed=L, state=True).items()}
    out = Guarded((batch, dim, L), inp["x"].dtype)
    so = Guarded((batch, dim, W - 1), inp["x"].dtype)
    ssm.causal_conv1d_fwd(inp["x"], inp["weight"], inp["bias"], inp["state"], out=out.view, state_out=so.view)
    out.check("out")
    so.check("state_out")
    st = Guarded((batch, dim, W - 1), inp["x"].dtype)
    st.view.copy_(inp["state"])
    o1 = Guarded((batch, dim), inp["x"].dtype)
    ssm.causal_conv1d_update(st.view, inp["x"][:, :, 0].contiguous(), inp["weight"], inp["bias"], out=o1.view)
    st.check("decode state")
    o1.check("decode out")
