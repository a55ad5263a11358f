"""The scan on the GPU at the two ends of the step size Delta, against the
oracle ("State Space Models (SSMs) & Mamba", section "The Magic of Selective
Scan": a small Delta keeps the state, a large one resets it to the current
input).

* Delta -> 0 (delta_raw + delta_bias = -200): the state is kept exactly, so
  hL equals h0 bit for bit and y_t = (C_t . h0 + D u_t) silu(z_t);
* Delta |A| >> 1 (delta_raw + delta_bias = +60): the past is forgotten and
  h_t = Delta_t B_t u_t;
* long memory: Delta three and six e-folds below the workloads' recipe over
  10,240 tokens, where the decay per token is within 1e-4 to 1e-6 of 1 and
  the forgetting rate 1 - exp(Delta A) must be accurate to its own few
  digits, not to those of 1; held to the same bars as every other case.
Each runs through the plain forward (one pass and the two-pass segmented
plan) and the decode step.
"""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import make_inputs, make_step_inputs
from tests.gpu_util import TIN, gpu_fwd, load_ssm, oracle_fwd, to_dev
from tests.parity import TOL, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _limit_inputs(dt, value, L=200):
    x = make_inputs(2, 40, 16, L, seed=61, in_dtype=dt, h0=True)
    x.delta_raw = np.zeros_like(x.delta_raw)
    x.delta_bias = np.full_like(x.delta_bias, value)
    return x


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("nseg", ["1", "2"])
def test_delta_to_zero_keeps_state_exactly(ssm, dt, nseg, monkeypatch):
    monkeypatch.setenv("SSM_FWD_NSEG", nseg)
    x = _limit_inputs(dt, -200.0)
    y, hL = gpu_fwd(ssm, x)
    assert np.array_equal(hL, x.h0), "hL differs from h0 with delta = softplus(-200)"
    yo, ho = oracle_fwd(x)
    assert np.array_equal(ho.astype(np.float32), x.h0)
    assert_close(y, yo, TOL[dt], "y")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("nseg", ["1", "2"])
def test_large_delta_forgets_state(ssm, dt, nseg, monkeypatch):
    monkeypatch.setenv("SSM_FWD_NSEG", nseg)
    x = _limit_inputs(dt, 60.0)
    y, hL = gpu_fwd(ssm, x)
    yo, ho = oracle_fwd(x)
    # the final state is Delta B_L u_L (Delta = 60): nothing of h0 is left
    mem = 60.0 * x.Bm[:, None, :, -1].astype(np.float64) * x.u[:, :, -1:].astype(np.float64)
    assert_close(ho, mem, 1e-12, "oracle hL vs Delta B u")
    assert_close(hL, ho, TOL[dt], "hL")
    assert_close(y, yo, TOL[dt], "y")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("value", [-200.0, 60.0])
def test_decode_step_delta_limits(ssm, dt, value):
    s = make_step_inputs(3, 256, 16, seed=62, in_dtype=dt)
    s["delta_raw"] = np.zeros_like(s["delta_raw"])
    s["delta_bias"] = np.full_like(s["delta_bias"], value)
    tin, f32 = TIN[dt], torch.float32
    st = to_dev(s["state"], f32)
    y = ssm.ssm_scan_step(to_dev(s["u"], tin), to_dev(s["delta_raw"], tin), to_dev(s["A"], f32),
                          to_dev(s["Bm"], tin), to_dev(s["Cm"], tin), st, to_dev(s["Dv"], f32),
                          to_dev(s["z"], tin), to_dev(s["delta_bias"], f32),
                          out_dtype=torch.float32)
    torch.cuda.synchronize()
    yo, so = oracle.scan_step(s["u"], s["delta_raw"], s["A"], s["Bm"], s["Cm"], s["state"],
                              s["Dv"], s["z"], s["delta_bias"])
    if value < 0:
        assert np.array_equal(st.cpu().numpy(), s["state"])
    assert_close(st.cpu().numpy(), so, TOL[dt], "state")
    assert_close(y.cpu().numpy(), yo, TOL[dt], "y")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("efolds", [3.0, 6.0])
@pytest.mark.parametrize("nseg", ["1", "2"])
def test_small_delta_long_memory(ssm, dt, efolds, nseg, monkeypatch):
    """Delta e^-3 and e^-6 times the recipe's over 10,240 tokens."""
    monkeypatch.setenv("SSM_FWD_NSEG", nseg)
    x = make_inputs(1, 40, 16, 64 * 160, seed=63, in_dtype=dt, h0=True)
    x.delta_bias = (x.delta_bias - np.float32(efolds)).astype(np.float32)
    tol = TOL[dt]
    y, hL = gpu_fwd(ssm, x)
    yo, ho = oracle_fwd(x)
    assert_close(hL, ho, tol, "hL")
    assert_close(y, yo, tol, "y")
