"""Single-token decode step on the GPU against the oracle, and chained steps
against the forward scan (recurrent inference: "State Space Models (SSMs) &
Mamba", section "The Payoff: Linear Scaling and Lightning-Fast Inference")."""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import WORKLOADS, make_inputs, make_step_inputs
from tests.gpu_util import TIN, gpu_fwd, load_ssm, to_dev
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _step(ssm, s, dt, out_dtype=torch.float32, state=None):
    tin = TIN[dt]
    f32 = torch.float32
    st = to_dev(s["state"] if state is None else state, f32)
    y = ssm.ssm_scan_step(to_dev(s["u"], tin), to_dev(s["delta_raw"], tin), to_dev(s["A"], f32),
                          to_dev(s["Bm"], tin), to_dev(s["Cm"], tin), st, to_dev(s["Dv"], f32),
                          to_dev(s["z"], tin), to_dev(s["delta_bias"], f32), out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), st.cpu().numpy()


@pytest.mark.parametrize("shape", [(3, 50, 16), (2, 33, 5), (4, 17, 1), (1, 9, 64), (2, 12, 32)])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_step_small(ssm, shape, dt):
    Bt, D, N = shape
    s = make_step_inputs(Bt, D, N, seed=20 + D, in_dtype=dt)
    y, st = _step(ssm, s, dt)
    yo, so = oracle.scan_step(s["u"], s["delta_raw"], s["A"], s["Bm"], s["Cm"], s["state"],
                              s["Dv"], s["z"], s["delta_bias"])
    assert_close(y, yo, TOL[dt], "y")
    assert_close(st, so, TOL[dt], "state")


# Shapes that reach each decode kernel: N = 16 with D a multiple of 128 (one
# thread per channel, 128-channel tiles), D a multiple of 64 with N in
# {8, 16, 32} (64-channel tiles), and the per-element kernel otherwise.
# (64, 1280, 16) has more 128-channel tiles than six per CTA of any grid the
# launch picks, so the tile ring wraps.
@pytest.mark.parametrize("shape", [(3, 256, 16), (1, 128, 16), (64, 1280, 16), (2, 192, 16),
                                   (2, 128, 8), (3, 64, 32), (2, 320, 4)])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_step_tiled_paths(ssm, shape, dt):
    Bt, D, N = shape
    s = make_step_inputs(Bt, D, N, seed=30 + D + N, in_dtype=dt)
    y, st = _step(ssm, s, dt)
    yo, so = oracle.scan_step(s["u"], s["delta_raw"], s["A"], s["Bm"], s["Cm"], s["state"],
                              s["Dv"], s["z"], s["delta_bias"])
    assert_close(y, yo, TOL[dt], "y")
    assert_close(st, so, TOL[dt], "state")


@pytest.mark.parametrize("shape", [(2, 256, 16), (2, 192, 16), (2, 40, 16)])
@pytest.mark.parametrize("absent", ["z", "Dv", "delta_bias", "all"])
def test_step_optional_inputs_absent(ssm, shape, absent):
    Bt, D, N = shape
    s = make_step_inputs(Bt, D, N, seed=40 + D, in_dtype="bf16")
    for k in (("z", "Dv", "delta_bias") if absent == "all" else (absent,)):
        s[k] = None
    tin, f32 = TIN["bf16"], torch.float32
    opt = lambda v, t: None if v is None else to_dev(v, t)
    st = to_dev(s["state"], f32)
    y = ssm.ssm_scan_step(to_dev(s["u"], tin), to_dev(s["delta_raw"], tin), to_dev(s["A"], f32),
                          to_dev(s["Bm"], tin), to_dev(s["Cm"], tin), st, opt(s["Dv"], f32),
                          opt(s["z"], tin), opt(s["delta_bias"], f32), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    yo, so = oracle.scan_step(s["u"], s["delta_raw"], s["A"], s["Bm"], s["Cm"], s["state"],
                              s["Dv"], s["z"], s["delta_bias"])
    assert_bf16_output(y.float().cpu().numpy(), yo, TOL["bf16"], "y")
    assert_close(st.cpu().numpy(), so, TOL["bf16"], "state")


def test_step_decode_workload_all_channels(ssm):
    w = WORKLOADS["decode_step"]
    s = make_step_inputs(w["Bt"], w["D"], w["N"], seed=w["seed"], in_dtype="bf16")
    y, st = _step(ssm, s, "bf16")
    yo, so = oracle.scan_step(s["u"], s["delta_raw"], s["A"], s["Bm"], s["Cm"], s["state"],
                              s["Dv"], s["z"], s["delta_bias"])
    assert_close(y, yo, TOL["bf16"], "y")
    assert_close(st, so, TOL["bf16"], "state")


def test_steps_reproduce_forward(ssm):
    x = make_inputs(2, 24, 16, 40, seed=21, in_dtype="bf16", h0=True)
    yf, hf = gpu_fwd(ssm, x)
    state = x.h0.copy()
    ys = []
    for t in range(x.u.shape[-1]):
        s = dict(u=x.u[..., t], delta_raw=x.delta_raw[..., t], z=x.z[..., t], Bm=x.Bm[..., t],
                 Cm=x.Cm[..., t], A=x.A, Dv=x.Dv, delta_bias=x.delta_bias)
        yt, state = _step(ssm, s, "bf16", state=state)
        ys.append(yt)
    yo, ho = oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    assert_close(np.stack(ys, -1), yo, TOL["bf16"], "stepped y vs oracle")
    assert_close(state, ho, TOL["bf16"], "stepped state vs oracle")
    assert_close(np.stack(ys, -1), yf, TOL["bf16"], "stepped y vs GPU forward")


@pytest.mark.parametrize("shape", [(2, 256, 16), (2, 192, 16), (2, 40, 16)])
def test_step_status_word(ssm, shape):
    """A status word passed to the decode step stays SSM_OK on a normal step
    (each decode kernel path), the result is unchanged, and ssm_get_status
    reads it back."""
    Bt, D, N = shape
    s = make_step_inputs(Bt, D, N, seed=50 + D, in_dtype="bf16")
    tin, f32 = TIN["bf16"], torch.float32
    status = torch.zeros(64, dtype=torch.int32, device="cuda")
    st = to_dev(s["state"], f32)
    y = ssm.ssm_scan_step(to_dev(s["u"], tin), to_dev(s["delta_raw"], tin), to_dev(s["A"], f32),
                          to_dev(s["Bm"], tin), to_dev(s["Cm"], tin), st, to_dev(s["Dv"], f32),
                          to_dev(s["z"], tin), to_dev(s["delta_bias"], f32),
                          out_dtype=torch.float32, status=status)
    assert ssm.ssm_get_status(status) == ssm.SSM_OK
    yo, so = oracle.scan_step(s["u"], s["delta_raw"], s["A"], s["Bm"], s["Cm"], s["state"],
                              s["Dv"], s["z"], s["delta_bias"])
    assert_close(y.cpu().numpy(), yo, TOL["bf16"], "y")
    assert_close(st.cpu().numpy(), so, TOL["bf16"], "state")
