"""Pins of the float64 oracle to facts fixed by the pages and by mathematics (CPU only).

Each test checks the oracle against something other than itself: a value the pages
print, a closed form the pages derive, a brute-force definition written in a
different form, or an exact special case.  Together they catch a dropped term
(D skip, gate, bias), a wrong sign (A), a wrong index or transposed operand (B, C
over batch/state/time), and a readout taken before the state update.
"""
import math
import os

import numpy as np
import pytest

from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            vals[key.strip()] = np.array([float(v) for v in rest.split(",")])
    return vals


# ---------------------------------------------------------------------------------------------
# 53ai.com Mamba article, section 3.3 "Parallel Associative Scan": the prefix-sum worked example.
# ---------------------------------------------------------------------------------------------
def test_prefix_sum_worked_example_pair_scan():
    g = _read_golden("prefix_sum_example.txt")
    prod, h = oracle.assoc_scan(np.ones_like(g["input"]), g["input"])
    np.testing.assert_array_equal(h, g["output"])
    np.testing.assert_array_equal(prod, np.ones_like(g["input"]))


def test_prefix_sum_worked_example_full_scan():
    """A = 0 (so Abar = 1), Delta = 1, B = C = 1, no D: the scan reduces to a prefix sum of u."""
    g = _read_golden("prefix_sum_example.txt")
    L = g["input"].size
    u = g["input"].reshape(1, 1, L)
    ones = np.ones((1, 1, L))
    y, last = oracle.scan(u, ones, np.zeros((1, 1)), ones, ones, delta_softplus=False)
    np.testing.assert_array_equal(y.ravel(), g["output"])
    assert last.ravel()[0] == g["output"][-1]
    y_t, _ = oracle.scan_tree(u, ones, np.zeros((1, 1)), ones, ones, delta_softplus=False)
    np.testing.assert_array_equal(y_t.ravel(), g["output"])


def test_pair_scan_running_product_and_grouping():
    """Tree-order pair scan: the a-component is the running product (numpy cumprod), and the
    b-component does not depend on how the pairs are grouped (sequential scan of the same pairs)."""
    rng = np.random.default_rng(7)
    a = rng.uniform(0.2, 1.0, size=37)
    b = rng.standard_normal(37)
    prod, h = oracle.assoc_scan(a, b)
    np.testing.assert_allclose(prod, np.cumprod(a), rtol=1e-14)
    # the same pairs through the sequential selective scan: Delta=1, A=log(a_t) cannot vary in t, so
    # instead compare with the closed form h_t = sum_s (prod_{r=s+1..t} a_r) b_s.
    ref = np.array([sum(np.prod(a[s + 1:t + 1]) * b[s] for s in range(t + 1)) for t in range(a.size)])
    np.testing.assert_allclose(h, ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# VMamba notes, "循环结构表示以快速推理": the expansion of y_2 and y_3 (the '+' signs lost in
# extraction restored), for time-invariant Abar, Bbar, C and h_{-1} = 0.
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("L", [3, 4])
def test_closed_form_y2_y3(L):
    rng = np.random.default_rng(11)
    N = 3
    A = -rng.uniform(0.3, 2.0, size=(1, N))
    delta = 0.37
    Bv = rng.standard_normal(N)
    Cv = rng.standard_normal(N)
    x = rng.standard_normal(L)
    y, _ = oracle.scan(x.reshape(1, 1, L), np.full((1, 1, L), delta), A,
                       np.repeat(Bv[None, :, None], L, axis=2), np.repeat(Cv[None, :, None], L, axis=2),
                       delta_softplus=False)
    Ab = np.exp(delta * A[0])
    Bb = delta * Bv
    y2 = np.sum(Cv * Ab * Ab * Bb) * x[0] + np.sum(Cv * Ab * Bb) * x[1] + np.sum(Cv * Bb) * x[2]
    assert y[0, 0, 2] == pytest.approx(y2, rel=1e-13, abs=1e-15)
    if L == 4:
        y3 = (np.sum(Cv * Ab * Ab * Ab * Bb) * x[0] + np.sum(Cv * Ab * Ab * Bb) * x[1]
              + np.sum(Cv * Ab * Bb) * x[2] + np.sum(Cv * Bb) * x[3])
        assert y[0, 0, 3] == pytest.approx(y3, rel=1e-13, abs=1e-15)


# ---------------------------------------------------------------------------------------------
# VMamba notes, "卷积结构表示以并行训练" and 53ai.com article §2.4: for time-invariant
# Delta, B, C the output is the convolution y = K * x with K_k = C Abar^k Bbar (+ the D skip).
# ---------------------------------------------------------------------------------------------
def test_convolution_form_time_invariant():
    rng = np.random.default_rng(3)
    batch, dim, N, L = 2, 3, 5, 48
    A = -np.exp(rng.uniform(-1.0, 1.5, size=(dim, N)))
    delta_c = rng.uniform(0.01, 0.5, size=dim)
    Bv = rng.standard_normal((batch, N))
    Cv = rng.standard_normal((batch, N))
    D = rng.standard_normal(dim)
    u = rng.standard_normal((batch, dim, L))
    delta = np.repeat(delta_c[None, :, None], L, axis=2).repeat(batch, axis=0)
    B = np.repeat(Bv[:, :, None], L, axis=2)
    C = np.repeat(Cv[:, :, None], L, axis=2)
    y, _ = oracle.scan(u, delta, A, B, C, D=D, delta_softplus=False)
    for b in range(batch):
        for d in range(dim):
            Ab = np.exp(delta_c[d] * A[d])
            K = np.array([np.sum(Cv[b] * Ab ** k * delta_c[d] * Bv[b]) for k in range(L)])
            conv = np.array([np.dot(K[:t + 1], u[b, d, t::-1]) for t in range(L)])
            np.testing.assert_allclose(y[b, d], conv + D[d] * u[b, d], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# Fully time-varying (selective) inputs: the unrolled sum
#   y_t = sum_{s<=t} sum_n C_t[n] (prod_{r=s+1..t} Abar_r[n]) Delta_s B_s[n] u_s + D u_t
# written with explicit batch/state/time indices (VMamba notes, "mamba：从S4到S6": B, C of
# shape (B, L, N) shared by channels, Delta of shape (B, L, D)).
# ---------------------------------------------------------------------------------------------
def test_unrolled_time_varying():
    rng = np.random.default_rng(5)
    batch, dim, N, L = 2, 3, 4, 11
    A = -np.exp(rng.uniform(-1.0, 1.5, size=(dim, N)))
    delta = rng.uniform(0.01, 0.6, size=(batch, dim, L))
    bias = rng.uniform(-0.005, 0.005, size=dim)
    B = rng.standard_normal((batch, N, L))
    C = rng.standard_normal((batch, N, L))
    D = rng.standard_normal(dim)
    u = rng.standard_normal((batch, dim, L))
    y, last = oracle.scan(u, delta, A, B, C, D=D, dt_bias=bias, delta_softplus=False)
    for b in range(batch):
        for d in range(dim):
            dl = delta[b, d] + bias[d]
            for t in range(L):
                acc = D[d] * u[b, d, t]
                for s in range(t + 1):
                    decay = np.exp(A[d] * dl[s + 1:t + 1].sum())
                    acc += np.sum(C[b, :, t] * decay * dl[s] * B[b, :, s]) * u[b, d, s]
                assert y[b, d, t] == pytest.approx(acc, rel=1e-11, abs=1e-12)
            hL = sum(np.exp(A[d] * dl[s + 1:].sum()) * dl[s] * B[b, :, s] * u[b, d, s] for s in range(L))
            np.testing.assert_allclose(last[b, d], hL, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------------------------
# Delta -> 0: Abar = 1 and Bbar x = 0, so the state never moves and y = C h0 + D u exactly.
# ---------------------------------------------------------------------------------------------
def test_delta_zero_gives_skip_only():
    rng = np.random.default_rng(9)
    batch, dim, N, L = 2, 4, 6, 17
    A = -np.exp(rng.standard_normal((dim, N)))
    u = rng.standard_normal((batch, dim, L))
    B = rng.standard_normal((batch, N, L))
    C = rng.standard_normal((batch, N, L))
    D = rng.standard_normal(dim)
    zero = np.zeros((batch, dim, L))
    y, last = oracle.scan(u, zero, A, B, C, D=D, delta_softplus=False)
    np.testing.assert_array_equal(y, D[None, :, None] * u)
    np.testing.assert_array_equal(last, 0.0)
    h0 = rng.standard_normal((batch, dim, N))
    y, last = oracle.scan(u, zero, A, B, C, D=D, delta_softplus=False, h0=h0)
    np.testing.assert_array_equal(last, h0)
    ref = np.einsum("bnt,bdn->bdt", C, h0) + D[None, :, None] * u
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# Zero-order hold Abar = exp(Delta A) (gsyq.cn page, "连续到离散的转换"): with Delta = ln 2 and
# A[n] = -(n+1) the state halves (n+1) times per step -- exact powers of two.
# ---------------------------------------------------------------------------------------------
def test_exact_halving_discretisation():
    N, L = 4, 9
    A = -np.arange(1, N + 1, dtype=np.float64)[None, :]
    h0 = np.ones((1, 1, N))
    C = np.ones((1, N, L))
    y, last = oracle.scan(np.ones((1, 1, L)), np.full((1, 1, L), math.log(2.0)), A, np.zeros((1, N, L)), C,
                          delta_softplus=False, h0=h0)
    n1 = np.arange(1, N + 1)
    np.testing.assert_allclose(last.ravel(), 2.0 ** (-n1 * L), rtol=1e-13)
    ref = np.array([np.sum(2.0 ** (-n1 * (t + 1))) for t in range(L)])
    np.testing.assert_allclose(y.ravel(), ref, rtol=1e-13)
    # the decode step applies the same discretisation
    s, out = oracle.state_update(h0, np.ones((1, 1)), np.full((1, 1), math.log(2.0)), A, np.zeros((1, N)),
                                 np.ones((1, N)), dt_softplus=False)
    np.testing.assert_allclose(s.ravel(), 2.0 ** (-n1), rtol=1e-14)
    assert out[0, 0] == pytest.approx(np.sum(2.0 ** (-n1)), rel=1e-14)


def test_structured_A_powers():
    """With A[n] = -(n+1) a, Abar_n = exp(-Delta a)^(n+1) for every n."""
    rng = np.random.default_rng(2)
    N, L = 16, 5
    a = 0.7
    A = (-a * np.arange(1, N + 1))[None, :]
    dl = rng.uniform(0.01, 1.0, size=(1, 1, L))
    s = np.ones((1, 1, N))
    for t in range(L):
        s, _ = oracle.state_update(s, np.zeros((1, 1)), dl[:, :, t], A, np.zeros((1, N)), np.zeros((1, N)),
                                   dt_softplus=False)
    r = np.exp(-a * dl.sum())
    np.testing.assert_allclose(s.ravel(), r ** np.arange(1, N + 1), rtol=1e-13)


# ---------------------------------------------------------------------------------------------
# Softplus (gsyq.cn page, "选择性机制的设计理念": Delta = Softplus(Linear(x))).
# ---------------------------------------------------------------------------------------------
def test_softplus_special_values():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=1e-15)
    assert oracle.softplus(math.log(math.e - 1.0)) == pytest.approx(1.0, rel=1e-15)
    for x in (-30.0, -3.0, -0.4, 0.7, 5.0, 40.0):
        assert oracle.softplus(x) - oracle.softplus(-x) == pytest.approx(x, rel=1e-14, abs=1e-15)
        assert oracle.softplus(x) > 0.0
    assert oracle.softplus(-50.0) == pytest.approx(math.exp(-50.0), rel=1e-12)
    assert oracle.softplus(700.0) == 700.0


def test_softplus_and_bias_inside_scan():
    """delta = 0 with dt_bias = ln(e-1) and softplus gives Delta = 1 exactly; with A[n] = -(n+1) ln 2
    the state halves (n+1) times per step.  Pins 'bias added before softplus'."""
    N, L = 3, 5
    A = (-math.log(2.0) * np.arange(1, N + 1))[None, :]
    bias = np.array([math.log(math.e - 1.0)])
    _, last = oracle.scan(np.ones((1, 1, L)), np.zeros((1, 1, L)), A, np.zeros((1, N, L)), np.ones((1, N, L)),
                          dt_bias=bias, delta_softplus=True, h0=np.ones((1, 1, N)))
    np.testing.assert_allclose(last.ravel(), 2.0 ** (-np.arange(1, N + 1) * L), rtol=1e-13)
    # and the Bbar x = Delta B u term with Delta = 1: one step from zero state gives h = B u
    _, last = oracle.scan(np.full((1, 1, 1), 3.0), np.zeros((1, 1, 1)), A, np.full((1, N, 1), 2.0),
                          np.ones((1, N, 1)), dt_bias=bias, delta_softplus=True)
    np.testing.assert_allclose(last.ravel(), 6.0, rtol=1e-14)


# ---------------------------------------------------------------------------------------------
# The silu(z) gate of the Mamba block (VMamba notes, "简化的SSM架构"): sigmoid(ln 3) = 3/4.
# ---------------------------------------------------------------------------------------------
def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert oracle.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    for x in (-20.0, -1.3, 0.2, 2.5, 30.0):
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, rel=1e-14, abs=1e-15)


def test_gate_inside_scan():
    """Delta = 0 makes y = D u; the gate then multiplies by silu(z): z = +-ln 3 gives 3/4 and -1/4 ln 3."""
    dim, N, L = 2, 3, 4
    u = np.arange(1, dim * L + 1, dtype=np.float64).reshape(1, dim, L)
    D = np.array([0.5, -2.0])
    z = np.empty((1, dim, L))
    z[..., 0::2] = math.log(3.0)
    z[..., 1::2] = -math.log(3.0)
    rng = np.random.default_rng(1)
    y, _ = oracle.scan(u, np.zeros((1, dim, L)), -np.ones((dim, N)), rng.standard_normal((1, N, L)),
                       rng.standard_normal((1, N, L)), D=D, z=z, delta_softplus=False)
    factor = np.where(np.arange(L) % 2 == 0, 0.75 * math.log(3.0), -0.25 * math.log(3.0))
    np.testing.assert_allclose(y, D[None, :, None] * u * factor[None, None, :], rtol=1e-14)


# ---------------------------------------------------------------------------------------------
# Associativity (53ai.com §3.3, gsyq.cn "硬件优化并行扫描算法"): sequential and tree order agree.
# ---------------------------------------------------------------------------------------------
def test_tree_order_equals_sequential():
    rng = np.random.default_rng(13)
    batch, dim, N, L = 2, 5, 16, 77
    A = -np.exp(rng.uniform(-1.0, 2.0, size=(dim, N)))
    u, delta, z = (rng.standard_normal((batch, dim, L)) for _ in range(3))
    B, C = (rng.standard_normal((batch, N, L)) for _ in range(2))
    D = rng.standard_normal(dim)
    bias = rng.uniform(-6.0, -2.0, size=dim)
    y1, l1 = oracle.scan(u, delta, A, B, C, D=D, z=z, dt_bias=bias)
    y2, l2 = oracle.scan_tree(u, delta, A, B, C, D=D, z=z, dt_bias=bias)
    np.testing.assert_allclose(y2, y1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Constant-memory decode (gsyq.cn complexity table, "推理内存 O(d) 状态向量"): L decode steps equal
# one scan over L; a scan resumed from its own last state equals the scan over the whole length.
# ---------------------------------------------------------------------------------------------
def test_decode_steps_equal_scan():
    rng = np.random.default_rng(17)
    batch, dim, N, L = 2, 3, 16, 20
    A = -np.exp(rng.uniform(-1.0, 2.0, size=(dim, N)))
    u, delta, z = (rng.standard_normal((batch, dim, L)) for _ in range(3))
    B, C = (rng.standard_normal((batch, N, L)) for _ in range(2))
    D = rng.standard_normal(dim)
    bias = rng.uniform(-6.0, -2.0, size=dim)
    y, last = oracle.scan(u, delta, A, B, C, D=D, z=z, dt_bias=bias)
    s = np.zeros((batch, dim, N))
    for t in range(L):
        s, out = oracle.state_update(s, u[:, :, t], delta[:, :, t], A, B[:, :, t], C[:, :, t], D=D, z=z[:, :, t],
                                     dt_bias=bias)
        np.testing.assert_allclose(out, y[:, :, t], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(s, last, rtol=1e-15, atol=1e-15)


def test_resume_from_last_state():
    rng = np.random.default_rng(19)
    batch, dim, N, L1, L2 = 1, 4, 8, 13, 19
    L = L1 + L2
    A = -np.exp(rng.uniform(-1.0, 2.0, size=(dim, N)))
    u, delta, z = (rng.standard_normal((batch, dim, L)) for _ in range(3))
    B, C = (rng.standard_normal((batch, N, L)) for _ in range(2))
    bias = rng.uniform(-6.0, -2.0, size=dim)
    y, last = oracle.scan(u, delta, A, B, C, z=z, dt_bias=bias)
    ya, la = oracle.scan(u[..., :L1], delta[..., :L1], A, B[..., :L1], C[..., :L1], z=z[..., :L1], dt_bias=bias)
    yb, lb = oracle.scan(u[..., L1:], delta[..., L1:], A, B[..., L1:], C[..., L1:], z=z[..., L1:], dt_bias=bias,
                         h0=la)
    np.testing.assert_array_equal(np.concatenate([ya, yb], axis=-1), y)
    np.testing.assert_array_equal(lb, last)


def test_segment_carries_combine_to_the_sequential_scan():
    """The split scan's decomposition, in float64: each segment scanned from a zero state (the first
    from h0) gives its end state, its decay is exp(A * sum of its Delta), and folding the (decay,
    end state) pairs with the pair operator (53ai.com section 3.3) gives the state entering every
    segment; scanning each segment from that state reproduces the sequential scan's y and final
    state.  The sums of Delta come from softplus(delta + dt_bias) written out here, not from the
    scan."""
    rng = np.random.default_rng(23)
    batch, dim, N, L, seg = 2, 3, 8, 96, 24
    A = -np.exp(rng.uniform(-3.0, 0.5, size=(dim, N)))  # slow decays: the carries matter
    u, delta, z = (rng.standard_normal((batch, dim, L)) for _ in range(3))
    B, C = (rng.standard_normal((batch, N, L)) for _ in range(2))
    D = rng.standard_normal(dim)
    bias = rng.uniform(-5.0, -3.0, size=dim)
    h0 = rng.standard_normal((batch, dim, N))
    y, last = oracle.scan(u, delta, A, B, C, D=D, z=z, dt_bias=bias, h0=h0)
    sl = [slice(k, k + seg) for k in range(0, L, seg)]
    ends, decays = [], []
    for j, s_ in enumerate(sl):
        _, h_end = oracle.scan(u[..., s_], delta[..., s_], A, B[..., s_], C[..., s_], D=D, z=z[..., s_],
                               dt_bias=bias, h0=h0 if j == 0 else None)
        x = delta[..., s_] + bias[None, :, None]
        dsum = np.sum(np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x))), axis=-1)  # (batch, dim)
        ends.append(h_end)
        decays.append(np.exp(A[None, :, :] * dsum[:, :, None]))
    starts = np.zeros((len(sl), batch, dim, N))
    for b in range(batch):
        for d in range(dim):
            for n in range(N):
                _, hs = oracle.assoc_scan([dk[b, d, n] for dk in decays], [ek[b, d, n] for ek in ends])
                starts[:, b, d, n] = hs  # state after segment j (segment 0 started from h0)
    ys = []
    for j, s_ in enumerate(sl):
        yj, lj = oracle.scan(u[..., s_], delta[..., s_], A, B[..., s_], C[..., s_], D=D, z=z[..., s_],
                             dt_bias=bias, h0=h0 if j == 0 else starts[j - 1])
        ys.append(yj)
    np.testing.assert_allclose(np.concatenate(ys, axis=-1), y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lj, last, rtol=1e-11, atol=1e-12)
    # the carries are not negligible here: without them the later segments differ
    y_nocarry, _ = oracle.scan(u[..., sl[-1]], delta[..., sl[-1]], A, B[..., sl[-1]], C[..., sl[-1]], D=D,
                               z=z[..., sl[-1]], dt_bias=bias)
    assert np.max(np.abs(y_nocarry - y[..., sl[-1]])) > 1e-3


def test_empty_and_thread_count_independence():
    rng = np.random.default_rng(23)
    A = -np.ones((3, 2))
    y, last = oracle.scan(np.zeros((1, 3, 0)), np.zeros((1, 3, 0)), A, np.zeros((1, 2, 0)), np.zeros((1, 2, 0)))
    assert y.shape == (1, 3, 0)
    np.testing.assert_array_equal(last, 0.0)
    u, delta = (rng.standard_normal((2, 3, 40)) for _ in range(2))
    B, C = (rng.standard_normal((2, 2, 40)) for _ in range(2))
    r1 = oracle.scan(u, delta, A, B, C, nthreads=1)
    r4 = oracle.scan(u, delta, A, B, C, nthreads=4)
    np.testing.assert_array_equal(r1[0], r4[0])
    np.testing.assert_array_equal(r1[1], r4[1])


# ---------------------------------------------------------------------------------------------
# Exact zero-order hold: gsyq.cn page, section "连续到离散的转换", and the VMamba notes print
# Bbar = (Delta A)^-1 (exp(Delta A) - I) Delta B.  Under a held input this is the exact
# solution of the continuous system h' = A h + B x sampled every Delta.
# ---------------------------------------------------------------------------------------------
def test_zoh_equals_continuous_solution_under_constant_input():
    """Constant Delta, B, C, u: h after k steps is (exp(A k Delta) - 1) / A * B u, the solution of
    h' = A h + B u from h(0) = 0 at time k*Delta (closed form)."""
    L, dt = 40, 0.37
    A = np.array([[-0.7, -2.3, 0.4]])
    Bv = np.array([1.5, -0.6, 0.9])
    Cv = np.array([0.8, 1.1, -0.3])
    u = np.full((1, 1, L), 0.75)
    delta = np.full((1, 1, L), dt)
    B = np.repeat(Bv[None, :, None], L, axis=2)
    C = np.repeat(Cv[None, :, None], L, axis=2)
    y, last = oracle.scan(u, delta, A, B, C, delta_softplus=False, zoh=True)
    k = np.arange(1, L + 1)[:, None]
    h = (np.exp(A[0][None, :] * k * dt) - 1.0) / A[0][None, :] * Bv[None, :] * 0.75
    np.testing.assert_allclose(y.ravel(), h @ Cv, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(last.ravel(), h[-1], rtol=1e-12)


def test_zoh_equals_matrix_exponential_of_augmented_system():
    """Time-varying Delta, B, u held over each step: one step of the continuous system is the
    matrix exponential of the augmented generator [[A, B u], [0, 0]] * Delta (scipy.linalg.expm),
    applied to (h, 1).  Random signs, softplus step sizes, dt_bias, D and gate all on."""
    from scipy.linalg import expm
    rng = np.random.default_rng(31)
    b_, d_, N, L = 1, 2, 3, 9
    u = rng.standard_normal((b_, d_, L))
    delta = rng.standard_normal((b_, d_, L))
    A = -np.exp(rng.uniform(-1.0, 1.0, (d_, N)))
    B = rng.standard_normal((b_, N, L))
    C = rng.standard_normal((b_, N, L))
    D = rng.standard_normal(d_)
    z = rng.standard_normal((b_, d_, L))
    bias = rng.uniform(-1.0, 0.5, d_)
    y, last = oracle.scan(u, delta, A, B, C, D=D, z=z, dt_bias=bias, delta_softplus=True, zoh=True)
    for d in range(d_):
        h = np.zeros(N)
        for t in range(L):
            dt = math.log1p(math.exp(delta[0, d, t] + bias[d]))
            for n in range(N):
                G = np.array([[A[d, n], B[0, n, t] * u[0, d, t]], [0.0, 0.0]]) * dt
                h[n] = (expm(G) @ np.array([h[n], 1.0]))[0]
            ref = (C[0, :, t] @ h + D[d] * u[0, d, t]) * z[0, d, t] / (1.0 + math.exp(-z[0, d, t]))
            assert abs(y[0, d, t] - ref) <= 1e-11 * (1.0 + abs(ref)), (d, t, y[0, d, t], ref)
        np.testing.assert_allclose(last[0, d], h, rtol=1e-11, atol=1e-13)


def test_zoh_with_A_zero_is_delta_B():
    """A = 0: (exp(Delta A) - 1) / A tends to Delta, so the two discretisations coincide exactly."""
    rng = np.random.default_rng(5)
    u = rng.standard_normal((2, 3, 12))
    delta = rng.standard_normal((2, 3, 12))
    B = rng.standard_normal((2, 4, 12))
    C = rng.standard_normal((2, 4, 12))
    A = np.zeros((3, 4))
    y0, s0 = oracle.scan(u, delta, A, B, C, delta_softplus=True)
    y1, s1 = oracle.scan(u, delta, A, B, C, delta_softplus=True, zoh=True)
    np.testing.assert_array_equal(y0, y1)
    np.testing.assert_array_equal(s0, s1)


def test_zoh_decode_steps_equal_scan():
    rng = np.random.default_rng(8)
    b_, d_, N, L = 2, 3, 4, 6
    u = rng.standard_normal((b_, d_, L))
    delta = rng.standard_normal((b_, d_, L))
    A = -np.exp(rng.standard_normal((d_, N)))
    B = rng.standard_normal((b_, N, L))
    C = rng.standard_normal((b_, N, L))
    D = rng.standard_normal(d_)
    z = rng.standard_normal((b_, d_, L))
    bias = rng.standard_normal(d_)
    y, last = oracle.scan(u, delta, A, B, C, D=D, z=z, dt_bias=bias, zoh=True)
    s = np.zeros((b_, d_, N))
    for t in range(L):
        s, out = oracle.state_update(s, u[:, :, t], delta[:, :, t], A, B[:, :, t], C[:, :, t], D=D, z=z[:, :, t],
                                     dt_bias=bias, zoh=True)
        np.testing.assert_array_equal(out, y[:, :, t])
    np.testing.assert_array_equal(s, last)


# ---------------------------------------------------------------------------------------------
# Causal depthwise conv1d before the scan: gsyq.cn page, SelectiveSSM sketch ("卷积预处理",
# Conv1d(d_model, d_model, d_conv, padding=d_conv-1, groups=d_model)); datacamp tutorial,
# install notes (the causal-conv1d layer inside the Mamba block).
# ---------------------------------------------------------------------------------------------
def _conv_case(seed, batch=2, dim=5, L=23, W=4):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((batch, dim, L)), rng.standard_normal((dim, W)), rng.standard_normal(dim))


def test_conv_equals_numpy_full_convolution():
    """Each output is numpy's full convolution of the row with the channel's filter (flipped,
    since np.convolve flips its second argument), first L outputs, plus the bias."""
    x, w, bias = _conv_case(1)
    out, _ = oracle.causal_conv1d(x, w, bias, silu=False)
    for b in range(x.shape[0]):
        for d in range(x.shape[1]):
            ref = np.convolve(x[b, d], w[d][::-1])[: x.shape[2]] + bias[d]
            np.testing.assert_allclose(out[b, d], ref, rtol=1e-13, atol=1e-13)


def test_conv_equals_torch_grouped_conv1d_as_the_sketch_writes_it():
    """torch.nn.functional.conv1d with groups = channels and padding W-1 (the sketch's layer);
    its first L outputs are the causal ones.  Then silu."""
    import torch
    x, w, bias = _conv_case(2, batch=3, dim=6, L=31, W=4)
    out, _ = oracle.causal_conv1d(x, w, bias, silu=True)
    xt = torch.from_numpy(x)
    ref = torch.nn.functional.conv1d(xt, torch.from_numpy(w)[:, None, :], torch.from_numpy(bias), padding=3,
                                     groups=6)[..., :31]
    ref = torch.nn.functional.silu(ref).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_conv_streaming_in_two_pieces(W):
    """conv(L1) then conv(L2) carrying the W-1 last inputs equals conv(L1 + L2); the carried
    state is the last W-1 inputs."""
    x, w, bias = _conv_case(3, L=40, W=W)
    full, st_full = oracle.causal_conv1d(x, w, bias)
    o1, s1 = oracle.causal_conv1d(x[..., :17], w, bias)
    o2, s2 = oracle.causal_conv1d(x[..., 17:], w, bias, state_in=s1)
    np.testing.assert_array_equal(np.concatenate([o1, o2], axis=-1), full)
    np.testing.assert_array_equal(s2, st_full)
    np.testing.assert_array_equal(st_full, x[..., 40 - (W - 1):])


def test_conv_impulse_response_and_short_rows():
    """A unit impulse at t = 0 returns the filter taps in reverse order of k (out_t = w[W-1-t]);
    with a row shorter than W-1 the carried state mixes the old state and the row."""
    w = np.array([[0.5, -1.0, 2.0, 3.0]])
    x = np.zeros((1, 1, 6))
    x[0, 0, 0] = 1.0
    out, _ = oracle.causal_conv1d(x, w, None, silu=False)
    np.testing.assert_array_equal(out.ravel(), [3.0, 2.0, -1.0, 0.5, 0.0, 0.0])
    st_in = np.array([[[7.0, 8.0, 9.0]]])
    out, st = oracle.causal_conv1d(np.array([[[1.0]]]), w, None, state_in=st_in, silu=False)
    assert out.ravel()[0] == 0.5 * 7.0 - 1.0 * 8.0 + 2.0 * 9.0 + 3.0 * 1.0
    np.testing.assert_array_equal(st.ravel(), [8.0, 9.0, 1.0])


# ---------------------------------------------------------------------------------------------
# Backward pass: gradients of <dout, out> pinned to central finite differences of the pinned
# forward oracle along random directions (float64, step 1e-5: truncation ~1e-10 relative), and
# to the closed form of the prefix-sum special case.
# ---------------------------------------------------------------------------------------------
def _bwd_case(seed, softplus=True, h0=True, gate=True, use_D=True, use_bias=True):
    rng = np.random.default_rng(seed)
    b_, d_, N, L = 2, 3, 4, 9
    case = dict(u=rng.standard_normal((b_, d_, L)), delta=rng.standard_normal((b_, d_, L)) * (1.0 if softplus else 0.3),
                A=-np.exp(rng.uniform(-1.0, 1.0, (d_, N))), B=rng.standard_normal((b_, N, L)),
                C=rng.standard_normal((b_, N, L)), D=rng.standard_normal(d_) if use_D else None,
                z=rng.standard_normal((b_, d_, L)) if gate else None,
                dt_bias=rng.uniform(-1.0, 0.5, d_) if use_bias else None,
                h0=rng.standard_normal((b_, d_, N)) if h0 else None)
    if not softplus:
        case["delta"] = np.abs(case["delta"]) + 0.05
        if use_bias:
            case["dt_bias"] = np.abs(case["dt_bias"]) * 0.1
    dout = rng.standard_normal((b_, d_, L))
    return case, dout


def _loss(case, dout, softplus, zoh=False):
    y, _ = oracle.scan(case["u"], case["delta"], case["A"], case["B"], case["C"], D=case["D"], z=case["z"],
                       dt_bias=case["dt_bias"], delta_softplus=softplus, h0=case["h0"], zoh=zoh)
    return float(np.sum(dout * y))


GRAD_OF = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
           "dt_bias": "ddt_bias", "h0": "dh0"}


@pytest.mark.parametrize("softplus", [True, False])
@pytest.mark.parametrize("name", sorted(GRAD_OF))
def test_backward_matches_finite_differences(name, softplus):
    case, dout = _bwd_case(11 + len(name), softplus=softplus)
    g = oracle.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dout, D=case["D"], z=case["z"],
                        dt_bias=case["dt_bias"], delta_softplus=softplus, h0=case["h0"])
    rng = np.random.default_rng(99)
    v = rng.standard_normal(case[name].shape)
    eps = 1e-5
    plus = dict(case)
    plus[name] = case[name] + eps * v
    minus = dict(case)
    minus[name] = case[name] - eps * v
    fd = (_loss(plus, dout, softplus) - _loss(minus, dout, softplus)) / (2 * eps)
    an = float(np.sum(g[GRAD_OF[name]] * v))
    assert abs(fd - an) <= 1e-7 * (1.0 + abs(fd)), (name, fd, an)


def test_backward_prefix_sum_closed_form():
    """A = 0, Delta = 1 (no softplus, no bias), B = C = 1, D given, no gate: out_t = sum_{s<=t} u_s
    + D u_t, so du_t = sum_{s>=t} dout_s + D dout_t, dD = sum_t dout_t u_t, and ddelta_t =
    sum_{s>=t} dout_s * u_t (Delta scales the input term only, since Abar = 1 for every Delta)."""
    L = 12
    rng = np.random.default_rng(4)
    u = rng.standard_normal((1, 1, L))
    dout = rng.standard_normal((1, 1, L))
    ones = np.ones((1, 1, L))
    D = np.array([0.7])
    g = oracle.scan_bwd(u, ones, np.zeros((1, 1)), ones, ones, dout, D=D, delta_softplus=False)
    tail = np.cumsum(dout[0, 0, ::-1])[::-1]
    np.testing.assert_allclose(g["du"][0, 0], tail + 0.7 * dout[0, 0], rtol=1e-13)
    np.testing.assert_allclose(g["dD"], [np.sum(dout * u)], rtol=1e-13)
    np.testing.assert_allclose(g["ddelta"][0, 0], tail * u[0, 0, :], rtol=1e-12, atol=1e-14)


SUMMED = ("dA", "dB", "dC", "dD", "ddt_bias")


@pytest.mark.parametrize("zoh", [False, True])
def test_backward_abs_sums_bound_the_gradients(zoh):
    """The absolute-term sums are the magnitude scale of each summed gradient (triangle inequality)
    and leave the gradients themselves bitwise unchanged."""
    case, dout = _bwd_case(5)
    kw = dict(D=case["D"], z=case["z"], dt_bias=case["dt_bias"], h0=case["h0"], zoh=zoh)
    g = oracle.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dout, **kw)
    ga = oracle.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dout, abs_sums=True, **kw)
    for k in g:
        np.testing.assert_array_equal(g[k], ga[k])
    for k in SUMMED:
        assert np.all(ga["abs_" + k] >= np.abs(ga[k]) * (1 - 1e-14)), k
        assert np.any(ga["abs_" + k] > np.abs(ga[k]) * (1 + 1e-6)), k  # mixed signs in a generic case


def test_backward_abs_sums_equal_the_gradients_when_every_term_is_nonnegative():
    """With u, B, C, D, h0, dout >= 0, A < 0, Delta > 0 and no gate every term of dA, dB, dC and
    dD is >= 0 (the adjoint stays >= 0), so each absolute-term sum is its gradient exactly: the
    sums add up the very terms the gradients do, in the same order."""
    case, dout = _bwd_case(6, gate=False)
    for k in ("u", "B", "C", "D", "h0"):
        case[k] = np.abs(case[k])
    dout = np.abs(dout)
    ga = oracle.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dout, D=case["D"],
                         dt_bias=case["dt_bias"], h0=case["h0"], abs_sums=True)
    for k in ("dA", "dB", "dC", "dD"):
        np.testing.assert_array_equal(ga["abs_" + k], ga[k])


@pytest.mark.parametrize("softplus", [True, False])
@pytest.mark.parametrize("name", sorted(GRAD_OF))
def test_zoh_backward_matches_finite_differences(name, softplus):
    """The same finite-difference pin for the exact zero-order hold; A holds one state at exactly
    0 and one at -1e-5 so that both limits of the factor's derivative are exercised."""
    case, dout = _bwd_case(23 + len(name), softplus=softplus)
    case["A"] = case["A"].copy()
    case["A"][0, 0] = 0.0
    case["A"][1, 1] = -1e-5
    g = oracle.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dout, D=case["D"], z=case["z"],
                        dt_bias=case["dt_bias"], delta_softplus=softplus, h0=case["h0"], zoh=True)
    rng = np.random.default_rng(98)
    v = rng.standard_normal(case[name].shape)
    eps = 1e-5
    plus = dict(case)
    plus[name] = case[name] + eps * v
    minus = dict(case)
    minus[name] = case[name] - eps * v
    fd = (_loss(plus, dout, softplus, zoh=True) - _loss(minus, dout, softplus, zoh=True)) / (2 * eps)
    an = float(np.sum(g[GRAD_OF[name]] * v))
    assert abs(fd - an) <= 1e-7 * (1.0 + abs(fd)), (name, fd, an)


def test_zoh_backward_small_decay_branch_matches_finite_differences():
    """Every A in [-2e-3, 0): Delta*A lands on both sides of the point where the hold factor's
    A-derivative switches from its direct form to its series, so dA is pinned on both branches."""
    case, dout = _bwd_case(41, softplus=True)
    rng = np.random.default_rng(5)
    case["A"] = -rng.uniform(0.0, 2e-3, case["A"].shape)
    g = oracle.scan_bwd(case["u"], case["delta"], case["A"], case["B"], case["C"], dout, D=case["D"], z=case["z"],
                        dt_bias=case["dt_bias"], delta_softplus=True, h0=case["h0"], zoh=True)
    for seed in range(3):
        v = np.random.default_rng(200 + seed).standard_normal(case["A"].shape)
        eps = 1e-6
        plus, minus = dict(case), dict(case)
        plus["A"] = case["A"] + eps * v
        minus["A"] = case["A"] - eps * v
        fd = (_loss(plus, dout, True, zoh=True) - _loss(minus, dout, True, zoh=True)) / (2 * eps)
        an = float(np.sum(g["dA"] * v))
        assert abs(fd - an) <= 1e-8 * (1.0 + abs(fd)), (seed, fd, an)
