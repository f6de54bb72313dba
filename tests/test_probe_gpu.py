"""GPU check of the unit-throughput probes (ssm_probe_cycles): the measured per-SM rates must be
in the range a B300 SM can physically deliver (the special-function unit is a small fraction of
the FP32 lanes; packed f32x2 cannot exceed twice the scalar lane rate)."""
import pytest
import torch

import selective_state_space_155_b300 as ssm

pytestmark = pytest.mark.gpu


def test_probe_rates_are_plausible():
    r = ssm.probe_unit_rates()
    assert 4.0 <= r["ex2"] <= 64.0, r
    assert 32.0 <= r["ffma"] <= 256.0, r
    assert 32.0 <= r["ffma2"] <= 2.0 * 256.0, r
    assert r["ex2"] < r["ffma"], r
    # the mixes cannot beat their parts: ex2 with an f32x2 FMA alongside at most at the ex2-alone
    # rate, and a state-step needs one ex2, so the recurrence at most at the ex2 rate
    assert 2.0 <= r["ex2_with_ffma2"] <= 1.05 * r["ex2"], r
    assert 2.0 <= r["recurrence"] <= 1.05 * r["ex2"], r


def test_probe_writes_one_count_per_cta():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cycles = torch.full((sms + 1,), -7, dtype=torch.int64, device="cuda")
    st = ssm.lib().ssm_probe_cycles(0, cycles.data_ptr(), sms, None)
    torch.cuda.synchronize()
    assert st == 0
    c = cycles.cpu()
    assert bool((c[:sms] > 0).all()) and int(c[sms]) == -7


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """The forward kernels' barrier wait on a barrier that nothing completes: every CTA must give
    up after its limit (2^20 cycles) instead of hanging, and the device keeps working."""
    cycles = torch.full((4,), -7, dtype=torch.int64, device="cuda")
    st = ssm.lib().ssm_probe_cycles(5, cycles.data_ptr(), 4, None)
    torch.cuda.synchronize()
    assert st == 0
    c = cycles.cpu().tolist()
    assert all(2 ** 20 <= v < 2 ** 26 for v in c), c
    x = torch.ones(16, device="cuda")
    assert float((x * 2).sum()) == 32.0
