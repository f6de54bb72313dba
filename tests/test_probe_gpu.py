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


def test_probe_writes_one_count_per_cta():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cycles = torch.full((sms + 1,), -7, dtype=torch.int64, device="cuda")
    st = ssm.lib().ssm_probe_cycles(0, cycles.data_ptr(), sms, None)
    torch.cuda.synchronize()
    assert st == 0
    c = cycles.cpu()
    assert bool((c[:sms] > 0).all()) and int(c[sms]) == -7
