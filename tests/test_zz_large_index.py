"""Parity past 2^31 elements per tensor: forward and backward calls whose
per-token tensors (batch x channels x tokens) hold more than 2^31 elements,
so that every offset into u, delta_raw, z, dy, y, du, ddelta_raw, dz and
into the workspace's per-token arrays must be 64-bit.  Sampled channels of
every batch row, always including the last row of the last batch (whose
offsets lie beyond 2^31), are compared with the oracle (channels are
independent given the shared B and C).  The forward runs both on whole rows
(the planner's segmented plan turned off) and with the planner's choice; the
backward takes the planner's choice (segments over the long row).  The
decode step runs on a state of more than 2^31 fp32 values (its rows, batch x
channels, stay below 2^31).

Collected after the other parity files and before test_zz_no_alloc.py.
"""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import device_inputs
from tests.gpu_util import load_ssm, rows_to_host
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu

L_LONG = 1 << 20


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _sample_channels(D, rng, k):
    ds = np.sort(rng.choice(D, size=k, replace=False))
    ds[0] = 0
    ds[-1] = D - 1
    return ds


@pytest.mark.parametrize("whole_rows", [True, False], ids=["whole_rows", "planner"])
def test_forward_past_2_31_elements(ssm, whole_rows, monkeypatch):
    Bt, D, N, L = 2, 1040, 16, L_LONG
    assert Bt * D * L > 2 ** 31
    if whole_rows:
        monkeypatch.setenv("SSM_FWD_NSEG", "1")
    out_dtype = torch.bfloat16 if whole_rows else torch.float32
    a = device_inputs(Bt, D, N, L, seed=4242, in_dtype="bf16", h0=True)
    y, hL = ssm.ssm_scan_fwd(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["Dv"], a["z"],
                             a["delta_bias"], a["h0"], out_dtype=out_dtype)
    torch.cuda.synchronize()
    rng = np.random.default_rng(31)
    for b in range(Bt):
        ds = _sample_channels(D, rng, 4)
        bi = [b]
        host = lambda t: rows_to_host(t, bi, ds)
        yo, ho = oracle.scan_fwd(host(a["u"]), host(a["delta_raw"]), a["A"][ds].cpu().numpy(),
                                 a["Bm"][bi].float().cpu().numpy(), a["Cm"][bi].float().cpu().numpy(),
                                 a["Dv"][ds].cpu().numpy(), host(a["z"]),
                                 a["delta_bias"][ds].cpu().numpy(), host(a["h0"]))
        yg = y[bi][:, ds].float().cpu().numpy()
        what = "forward past 2^31 (%s) b=%d" % ("whole rows" if whole_rows else "planner", b)
        if out_dtype == torch.bfloat16:
            assert_bf16_output(yg, yo, TOL["bf16"], what + " y")
        else:
            assert_close(yg, yo, TOL["bf16"], what + " y")
        assert_close(hL[bi][:, ds].cpu().numpy(), ho, TOL["bf16"], what + " hL")
    del a, y, hL
    torch.cuda.empty_cache()


def test_backward_past_2_31_elements(ssm):
    """Every token's du, ddelta_raw and dz and the per-channel dA, dD,
    ddelta_bias and dh0 of sampled channels (dB and dC sum over all channels;
    they are compared in full at the Mamba-2.8B shape)."""
    Bt, D, N, L = 1, 2100, 16, L_LONG
    assert Bt * D * L > 2 ** 31
    a = device_inputs(Bt, D, N, L, seed=4343, in_dtype="bf16", h0=True, dy=True)
    dhL = torch.randn(Bt, D, N, generator=torch.Generator(device="cuda").manual_seed(7),
                      device="cuda")
    g = ssm.ssm_scan_bwd(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["dy"], a["Dv"],
                         a["z"], a["delta_bias"], a["h0"], dhL, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ds = _sample_channels(D, np.random.default_rng(32), 4)
    bi = [0]
    host = lambda t: rows_to_host(t, bi, ds)
    o = oracle.scan_bwd(host(a["u"]), host(a["delta_raw"]), a["A"][ds].cpu().numpy(),
                        a["Bm"].float().cpu().numpy(), a["Cm"].float().cpu().numpy(),
                        host(a["dy"]), a["Dv"][ds].cpu().numpy(), host(a["z"]),
                        a["delta_bias"][ds].cpu().numpy(), host(a["h0"]), host(dhL))
    tol = TOL["bf16"]
    for k in ("du", "ddelta_raw", "dz", "dh0"):
        assert_close(g[k][bi][:, ds].cpu().numpy(), o[k], tol, "backward past 2^31 " + k)
    for k in ("dA", "dD", "ddelta_bias"):
        assert_close(g[k][ds].cpu().numpy(), o[k], tol, "backward past 2^31 " + k)
    del a, g, dhL
    torch.cuda.empty_cache()


def test_decode_step_state_past_2_31_elements(ssm):
    """One decode step on (27,000, 5,120, 16): the state holds 2.2e9 fp32 values,
    updated in place; sampled (batch row, channel) pairs against the oracle's step."""
    Bt, D, N = 27000, 5120, 16
    assert Bt * D * N > 2 ** 31
    a = device_inputs(Bt, D, N, 1, seed=4444, in_dtype="bf16", h0=True)
    step = {k: a[k][:, :, 0].contiguous() for k in ("u", "delta_raw", "z", "Bm", "Cm")}
    state = a["h0"]
    bsel = [0, 13331, Bt - 1]
    dsel = np.array([0, 2047, D - 1])
    state0 = state[bsel][:, dsel].cpu().numpy()
    y = ssm.ssm_scan_step(step["u"], step["delta_raw"], a["A"], step["Bm"], step["Cm"], state,
                          a["Dv"], step["z"], a["delta_bias"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    sub = lambda t: t[bsel][:, dsel].float().cpu().numpy()
    yo, so = oracle.scan_step(sub(step["u"]), sub(step["delta_raw"]), a["A"][dsel].cpu().numpy(),
                              step["Bm"][bsel].float().cpu().numpy(),
                              step["Cm"][bsel].float().cpu().numpy(), state0,
                              a["Dv"][dsel].cpu().numpy(), sub(step["z"]),
                              a["delta_bias"][dsel].cpu().numpy())
    assert_close(y[bsel][:, dsel].cpu().numpy(), yo, TOL["bf16"], "decode past 2^31 y")
    assert_close(state[bsel][:, dsel].cpu().numpy(), so, TOL["bf16"], "decode past 2^31 state")
    del a, step, state, y
    torch.cuda.empty_cache()
