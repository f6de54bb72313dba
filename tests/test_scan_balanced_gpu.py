"""The balanced forward layout (one CTA per SM, up to three warp groups on planned channel ranges)
against the plain layout (32-channel CTAs, SSM_SCAN_VARIANT=quad_plain): every channel runs the same
arithmetic, so y, the final state and the checkpoints must be bitwise equal.  The parity of the
balanced form against the float64 oracle is covered by the scan tests, which select it by default
wherever its plan applies (bf16, dstate 9..16, dim a multiple of 8), the mid and long workloads
included."""
import numpy as np
import pytest
import torch

import selective_state_space_155_b300 as ssm
import ssm_workloads as wl
from tests.gpu_util import oracle_scan, to_device, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

# (batch, dim, dstate, seqlen): split rows, 8-channel groups, ranges across batch rows, long rows
SHAPES = [(8, 1536, 16, 256), (1, 5120, 16, 384), (2, 1032, 16, 300), (7, 1544, 12, 100), (3, 40, 16, 77),
          (1, 64, 16, 64), (5, 200, 16, 129), (2, 4096, 16, 64)]


def run(inp, monkeypatch, variant, disc="delta_b", h0=None, ckpt=False):
    if variant is None:
        monkeypatch.delenv("SSM_SCAN_VARIANT", raising=False)
    else:
        monkeypatch.setenv("SSM_SCAN_VARIANT", variant)
    batch, dim, L = inp["u"].shape
    N = inp["A"].shape[1]
    ck = torch.full((batch, ssm.scan_num_checkpoints(L), dim, N), -7.0, device=DEV) if ckpt else None
    y, last = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                               inp["dt_bias"], h0=h0, discretization=disc, checkpoints=ck)
    torch.cuda.synchronize()
    return y, last, ck


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}_d{}_n{}_l{}".format(*s))
@pytest.mark.parametrize("mode", ["plain_args", "h0_ckpt", "zoh", "no_gate"])
def test_balanced_equals_plain(shape, mode, monkeypatch):
    batch, dim, N, L = shape
    inp = to_device(wl.random_scan_case(batch, dim, N, L, io="bf16", seed=dim + L, gate=mode != "no_gate",
                                        h0=mode == "h0_ckpt"), DEV)
    kw = dict(disc="zoh" if mode == "zoh" else "delta_b", h0=inp.get("h0") if mode == "h0_ckpt" else None,
              ckpt=mode == "h0_ckpt")
    yb, sb, cb = run(inp, monkeypatch, None, **kw)
    # the comparison means something only if the balanced layout is what ran (this also fails if
    # a build's register count no longer matches the kernel's register split, which turns it off)
    form, ctas = ssm.scan_fwd_form(batch, dim, N, L, inp["u"].dtype, kw["disc"])
    assert form == "balanced" and 0 < ctas <= torch.cuda.get_device_properties(0).multi_processor_count, \
        (form, ctas)
    yp, sp, cp = run(inp, monkeypatch, "quad_plain", **kw)
    assert ssm.scan_fwd_form(batch, dim, N, L, inp["u"].dtype, kw["disc"])[0] == "plain"
    assert torch.equal(yb, yp), "y differs"
    assert torch.equal(sb, sp), "final state differs"
    if cb is not None:
        assert torch.equal(cb, cp), "checkpoints differ"


def test_balanced_long_rows_against_oracle():
    """One long row set (batch 1, 5120 channels: the plan puts 32 or 8 channels on each SM) against
    the float64 oracle on every element."""
    inp = to_device(wl.random_scan_case(1, 5120, 16, 200, io="bf16", seed=3), DEV)
    y, last = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                               inp["dt_bias"])
    torch.cuda.synchronize()
    y_ref, s_ref = oracle_scan(inp)
    assert_close(wl.to_f64(y), y_ref, 2e-2, "y")
    assert_close(wl.to_f64(last), s_ref, 1e-4, "state")
