"""GPU parity of the training pair (ssm_scan_fwd_train + ssm_scan_bwd) against the float64 oracle,
through the C-ABI.

Tolerances: the per-element gradients (du, ddelta, dz) are held element-wise like the forward's
outputs (1e-4 relative for float32 io, 2e-2 for bf16 io, whose outputs are rounded to bf16).  The
gradients that are sums over many terms of both signs (dA over batch and time, dB and dC over the
channels, dD and ddt_bias) are float32 accumulations whose error scales with the size of the terms,
not of the result, so each element is held against the sum of the absolute values of its own terms
(which the oracle returns beside the gradient): |got - ref| <= KAPPA * sum|terms|.  dh0, the
adjoint state carried back to t = 0 rather than a sum, keeps the norm-wise form
max|got - ref| <= 2e-4 * max(1, max|ref|).
"""
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
ELEMENTWISE = ("du", "ddelta", "dz")
CKPT = 8  # SSM_SCAN_CHECKPOINT_STEPS: steps between the training forward's checkpoints


# Per-element bound for the summed gradients, relative to the element's absolute-term sum.  A
# float32 sum of n terms can be off by up to n * 2^-24 of that sum in the worst case (above 1e-4 for
# n > 1700, i.e. for every workload here), but the kernel adds at most 32 partials in registers
# before a float32 atomic across CTAs, so the realized error stays near sqrt(n) * 2^-24; with the
# forward recomputation's approximate exponentials (a few units in the last place per term) the
# largest ratio measured on B300 over all cases of this file is 4.2e-6.  KAPPA leaves ~25x headroom.
KAPPA = 1e-4
SUMMED = ("dA", "dB", "dC", "dD", "ddt_bias")


def term_close(got, ref, abs_sum, what):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bound = KAPPA * abs_sum
    bad = err > bound
    if np.any(bad):
        i = int(np.argmax(err / np.maximum(abs_sum, 1e-300)))
        raise AssertionError(f"{what}: {int(bad.sum())} elements with |got-ref| > {KAPPA:.0e} * sum|terms|; "
                             f"worst |got-ref| = {err.flat[i]:.3e}, sum|terms| = {abs_sum.flat[i]:.3e}")


def norm_close(got, ref, tol, what):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    scale = max(1.0, float(np.max(np.abs(ref))) if ref.size else 1.0)
    assert err <= tol * scale, f"{what}: max|got-ref| = {err:.3e} > {tol:.1e} * {scale:.3e}"


def train_step(inp, dout, softplus=True, h0=None, need_dh0=False, disc="delta_b"):
    batch, dim, L = inp["u"].shape
    N = inp["A"].shape[1]
    ck = torch.empty((batch, ssm.scan_num_checkpoints(L), dim, N), dtype=torch.float32, device=DEV)
    y, last = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp.get("D"), inp.get("z"),
                               inp.get("dt_bias"), delta_softplus=softplus, h0=h0, checkpoints=ck,
                               discretization=disc)
    g = ssm.ssm_scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], ck, dout, D=inp.get("D"),
                         z=inp.get("z"), dt_bias=inp.get("dt_bias"), delta_softplus=softplus, need_dh0=need_dh0,
                         discretization=disc)
    torch.cuda.synchronize()
    return y, last, ck, g


def check_bwd(inp, softplus=True, h0=None, seed=0, what="", disc="delta_b"):
    io = io_name(inp["u"])
    gen = torch.Generator().manual_seed(seed)
    dout = torch.randn(inp["u"].shape, generator=gen).to(inp["u"].dtype).to(DEV)
    y, last, ck, g = train_step(inp, dout, softplus, h0, need_dh0=h0 is not None, disc=disc)
    ref = oracle.scan_bwd(f(inp["u"]), f(inp["delta"]), f(inp["A"]), f(inp["B"]), f(inp["C"]), f(dout),
                          D=f(inp.get("D")), z=f(inp.get("z")), dt_bias=f(inp.get("dt_bias")),
                          delta_softplus=softplus, h0=f(h0) if h0 is not None else None, zoh=disc == "zoh",
                          abs_sums=True)
    grads = {k: v for k, v in ref.items() if not k.startswith("abs_")}
    assert set(grads) <= set(g) | ({"dh0"} if h0 is None else set()), (sorted(grads), sorted(g))
    for k, r in grads.items():
        if r is None or (k == "dh0" and h0 is None):
            continue
        got = f(g[k])
        if k in ELEMENTWISE:
            assert_close(got, r, TOL[io][0], f"{what} {k}")
        elif k in SUMMED:
            term_close(got, r, ref["abs_" + k], f"{what} {k}")
        else:
            norm_close(got, r, 2e-4, f"{what} {k}")
    return y, last, ck


@pytest.mark.parametrize("w", [wl.TINY, wl.SMALL], ids=lambda w: w.name)
def test_workload_backward_parity(w):
    inp = wl.scan_inputs(w, device=DEV)
    check_bwd(inp, what=w.name)


def test_mid_workload_backward_parity():
    """The mid-size workload (batch 8, d_inner 1536, d_state 16, L 2048, bf16): every gradient of
    every element against the float64 oracle."""
    inp = wl.scan_inputs(wl.MID, device=DEV)
    check_bwd(inp, seed=2, what="mid")


@pytest.mark.parametrize("shape", [
    # (batch, dim, dstate, seqlen, io): ragged chunk tails, dim not a multiple of 32, padded dstate,
    # single steps
    (1, 1, 1, 1, "f32"), (2, 33, 16, 65, "f32"), (3, 31, 3, 100, "f32"), (2, 40, 5, 63, "bf16"),
    (2, 65, 8, 129, "bf16"), (1, 32, 12, 31, "bf16"), (2, 7, 16, 1, "f32"), (1, 50, 16, 300, "f32"),
], ids=lambda s: "b{}_d{}_n{}_l{}_{}".format(*s))
def test_edge_shapes_backward(shape):
    batch, dim, dstate, seqlen, io = shape
    inp = to_device(wl.random_scan_case(batch, dim, dstate, seqlen, io=io, seed=seqlen * 7 + dim), DEV)
    check_bwd(inp, seed=seqlen, what=str(shape))


@pytest.mark.parametrize("gate,use_D,use_bias,softplus", [
    (False, False, False, False), (True, False, True, True), (False, True, False, True), (True, True, True, False)])
def test_optional_arguments_backward(gate, use_D, use_bias, softplus):
    inp = to_device(wl.random_scan_case(2, 48, 16, 136, io="f32", seed=5, gate=gate, use_D=use_D,
                                        use_bias=use_bias, softplus=softplus), DEV)
    check_bwd(inp, softplus=softplus, what="optional args")


def test_initial_state_gradient():
    inp = to_device(wl.random_scan_case(2, 40, 16, 96, io="f32", seed=3, h0=True), DEV)
    check_bwd(inp, h0=inp["h0"], what="h0")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_training_forward_matches_forward_and_checkpoints(io):
    """The training forward returns the same y and last_state as the plain forward, and its
    checkpoint c is the oracle's state after the first CKPT * c steps."""
    inp = to_device(wl.random_scan_case(2, 40, 16, 200, io=io, seed=9, h0=True), DEV)
    dout = torch.zeros_like(inp["u"])
    y, last, ck, _ = train_step(inp, dout, h0=inp["h0"])
    y0, last0 = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                 inp["dt_bias"], h0=inp["h0"])
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(last, last0)
    ckn = f(ck)
    np.testing.assert_array_equal(ckn[:, 0], f(inp["h0"]))
    for c in range(1, ckn.shape[1]):
        pre = {k: (v[..., :CKPT * c].contiguous() if k in ("u", "delta", "z", "B", "C") else v) for k, v in inp.items()}
        _, s_ref = oracle_scan(pre, h0=inp["h0"])
        assert_close(ckn[:, c], s_ref, 1e-4, f"checkpoint {c}")


# ---- the exact zero-order hold: the same cases, plus the decay regimes its factor branches on ----

@pytest.mark.parametrize("w", [wl.TINY, wl.SMALL], ids=lambda w: w.name)
def test_zoh_workload_backward_parity(w):
    inp = wl.scan_inputs(w, device=DEV)
    check_bwd(inp, what="zoh " + w.name, disc="zoh")


def test_zoh_mid_workload_backward_parity():
    """Batch 8, d_inner 1536, d_state 16, L 2048, bf16, under the hold: every gradient element."""
    inp = wl.scan_inputs(wl.MID, device=DEV)
    check_bwd(inp, seed=4, what="zoh mid", disc="zoh")


@pytest.mark.parametrize("shape", [
    (1, 1, 1, 1, "f32"), (2, 33, 16, 65, "f32"), (3, 31, 3, 100, "f32"), (2, 40, 5, 63, "bf16"),
    (2, 65, 8, 129, "bf16"), (2, 7, 16, 1, "f32"), (1, 50, 16, 300, "f32"),
], ids=lambda s: "b{}_d{}_n{}_l{}_{}".format(*s))
def test_zoh_edge_shapes_backward(shape):
    batch, dim, dstate, seqlen, io = shape
    inp = to_device(wl.random_scan_case(batch, dim, dstate, seqlen, io=io, seed=seqlen * 5 + dim), DEV)
    check_bwd(inp, seed=seqlen + 1, what="zoh " + str(shape), disc="zoh")


@pytest.mark.parametrize("gate,use_D,use_bias,softplus", [
    (False, False, False, False), (True, True, True, True), (True, False, True, False)])
def test_zoh_optional_arguments_backward(gate, use_D, use_bias, softplus):
    inp = to_device(wl.random_scan_case(2, 48, 16, 136, io="f32", seed=6, gate=gate, use_D=use_D,
                                        use_bias=use_bias, softplus=softplus), DEV)
    check_bwd(inp, softplus=softplus, what="zoh optional args", disc="zoh")


def test_zoh_initial_state_gradient():
    inp = to_device(wl.random_scan_case(2, 40, 16, 96, io="f32", seed=8, h0=True), DEV)
    check_bwd(inp, h0=inp["h0"], what="zoh h0", disc="zoh")


@pytest.mark.parametrize("regime", ["near_zero", "mixed"])
def test_zoh_backward_decay_regimes(regime):
    """A on both sides of the factor's series/direct switch: near_zero puts every A in [-2e-3, 0]
    with some exactly 0 (the limits Delta and Delta^2/2); mixed spreads |A| over 1e-4 .. 30, so
    Delta*A runs from about -1e-4 to beyond -50 in one channel."""
    inp = to_device(wl.random_scan_case(2, 64, 16, 160, io="f32", seed=13), DEV)
    rng = np.random.default_rng(17 if regime == "near_zero" else 19)
    if regime == "near_zero":
        A = -rng.uniform(0.0, 2e-3, tuple(inp["A"].shape))
        A[:, ::5] = 0.0
    else:
        A = -np.exp(rng.uniform(np.log(1e-4), np.log(30.0), tuple(inp["A"].shape)))
    inp["A"] = torch.from_numpy(A.astype(np.float32)).to(DEV)
    check_bwd(inp, seed=3, what="zoh " + regime, disc="zoh")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_training_forward_matches_forward_and_checkpoints(io):
    """The training forward under the hold returns the plain hold forward's y and last_state, and
    its checkpoint c is the oracle's hold state after the first CKPT * c steps."""
    inp = to_device(wl.random_scan_case(2, 40, 16, 200, io=io, seed=10, h0=True), DEV)
    dout = torch.zeros_like(inp["u"])
    y, last, ck, _ = train_step(inp, dout, h0=inp["h0"], disc="zoh")
    y0, last0 = ssm.ssm_scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["D"], inp["z"],
                                 inp["dt_bias"], h0=inp["h0"], discretization="zoh")
    torch.cuda.synchronize()
    assert torch.equal(y, y0) and torch.equal(last, last0)
    ckn = f(ck)
    np.testing.assert_array_equal(ckn[:, 0], f(inp["h0"]))
    for c in range(1, ckn.shape[1]):
        pre = {k: (v[..., :CKPT * c].contiguous() if k in ("u", "delta", "z", "B", "C") else v) for k, v in inp.items()}
        _, s_ref = oracle_scan(pre, h0=inp["h0"], zoh=True)
        assert_close(ckn[:, c], s_ref, 1e-4, f"zoh checkpoint {c}")
