"""Backward scan on the GPU against the fp64 oracle's reverse mode, element
by element.

Small and ragged shapes (several 64-token tiles plus a ragged tail, channel
counts that do not fill a CTA, state sizes from 1 to 64, absent optional
terms, an upstream gradient of the final state, both load paths), the tiny
fp32 workload, bf16 outputs, the empty sequence, and the Mamba-2.8B layer
shape in full: there every channel is compared, and dB and dC -- sums over
all 5120 channels -- are compared against the oracle run channel-chunk by
channel-chunk and summed.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle
from scan_inputs import WORKLOADS, device_inputs, make_inputs
from tests.gpu_util import TIN, device_args, load_ssm, oracle_bwd_chunk, to_dev
from tests.parity import TOL, assert_bf16_output, assert_close, rel_err

pytestmark = pytest.mark.gpu

PER_TOKEN = ("du", "ddelta_raw", "dz")
OUTS = ("du", "ddelta_raw", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _gpu_bwd(ssm, x, dhL, out_dtype):
    a = device_args(x)
    g = ssm.ssm_scan_bwd(a["u"], a["delta_raw"], a["A"], a["B"], a["C"], to_dev(x.dy, TIN[x.in_dtype]),
                         a["D"], a["z"], a["delta_bias"], a["h0"], to_dev(dhL, torch.float32),
                         out_dtype=out_dtype)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.float().cpu().numpy()) for k, v in g.items()}


def _check(ssm, x, dhL=None, out_dtype=torch.float32):
    tol = TOL[x.in_dtype]
    g = _gpu_bwd(ssm, x, dhL, out_dtype)
    o = oracle.scan_bwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z, x.delta_bias, x.h0,
                        dhL)
    for k in OUTS:
        if k == "dz" and x.z is None:
            assert g[k] is None
            continue
        if out_dtype == torch.bfloat16 and k in PER_TOKEN:
            assert_bf16_output(g[k], o[k], tol, k)
        else:
            assert_close(g[k], o[k], tol, k)


def _dhL(x, seed):
    Bt, D, N, L = x.shape
    return np.random.default_rng(seed).standard_normal((Bt, D, N)).astype(np.float32)


def test_tiny_fp32_workload(ssm):
    w = WORKLOADS["tiny_fp32"]
    x = make_inputs(w["Bt"], w["D"], w["N"], w["L"], seed=w["seed"], in_dtype="f32",
                    a_jitter=False, dy=True)
    _check(ssm, x)


CASES = [
    # (Bt, D, N, L, dtype, options, with dhL)
    (2, 40, 16, 200, "bf16", {}, False),           # ragged D and ragged last tile, TMA path
    (1, 70, 16, 77, "bf16", {"h0": True}, True),   # rows not 16-byte aligned: plain loads
    (2, 20, 8, 96, "f32", {}, True),               # fp32 TMA path
    (3, 33, 4, 130, "f32", {"h0": True}, True),    # fp32 plain loads, N padded to 8
    (2, 64, 16, 128, "bf16", {"h0": True}, True),
    (1, 128, 16, 64, "bf16", {"with_z": False}, False),
    (1, 96, 16, 192, "bf16", {"with_D": False, "with_bias": False}, True),
    (2, 10, 1, 100, "bf16", {}, True),
    (1, 50, 5, 256, "bf16", {"h0": True}, False),
    (1, 36, 32, 160, "bf16", {}, True),
    (1, 24, 64, 136, "bf16", {"h0": True}, True),
    (1, 17, 16, 1, "bf16", {"h0": True}, True),    # a single token
    (1, 17, 16, 65, "f32", {"h0": True}, True),
    (4, 300, 16, 320, "bf16", {}, False),
    (1, 40, 16, 1000, "f32", {"h0": True}, True),  # long fp32 sequence (suffix sums)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%dx%dx%dx%d-%s" % c[:5])
def test_small_shapes(ssm, case):
    Bt, D, N, L, dt, opt, with_dhL = case
    x = make_inputs(Bt, D, N, L, seed=300 + D + L, in_dtype=dt, dy=True, **opt)
    _check(ssm, x, _dhL(x, 7) if with_dhL else None)


@pytest.mark.parametrize("nt", ["2", "4"])
def test_threads_per_channel_variants(ssm, nt, monkeypatch):
    monkeypatch.setenv("SSM_BWD_NT", nt)
    x = make_inputs(2, 90, 16, 330, seed=17, in_dtype="bf16", h0=True, dy=True)
    _check(ssm, x, _dhL(x, 8))
    x = make_inputs(1, 30, 16, 96, seed=18, in_dtype="f32", dy=True)
    _check(ssm, x)


@pytest.mark.parametrize("nt,w", [("2", "7"), ("4", "9")])
def test_plan_override_that_does_not_fit(ssm, nt, w, monkeypatch):
    """A tile-shape override too large for the shared memory falls back to
    the planner's own choice and the result stays correct."""
    monkeypatch.setenv("SSM_BWD_NT", nt)
    monkeypatch.setenv("SSM_BWD_W", w)
    x = make_inputs(2, 100, 16, 200, seed=77, in_dtype="bf16", dy=True)
    _check(ssm, x)


def test_bf16_outputs(ssm):
    x = make_inputs(2, 64, 16, 256, seed=19, in_dtype="bf16", dy=True)
    _check(ssm, x, out_dtype=torch.bfloat16)


def test_empty_sequence_passes_dhL_through(ssm):
    x = make_inputs(2, 8, 16, 1, seed=20, in_dtype="bf16", dy=True)
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dt)
    e = torch.empty(2, 8, 0, dtype=torch.bfloat16, device="cuda")
    eb = torch.empty(2, 16, 0, dtype=torch.bfloat16, device="cuda")
    dhL = dev(_dhL(x, 3), torch.float32)
    g = ssm.ssm_scan_bwd(e, e, dev(x.A, torch.float32), eb, eb, e, dev(x.Dv, torch.float32),
                         e, dev(x.delta_bias, torch.float32), None, dhL)
    torch.cuda.synchronize()
    assert torch.equal(g["dh0"], dhL)
    for k in ("dA", "dD", "ddelta_bias"):
        assert torch.count_nonzero(g[k]) == 0, k


def test_full_size_mamba2p8b(ssm):
    """Every output of the Mamba-2.8B layer backward (batch 2, D 5120, N 16,
    L 8192) against the oracle, channel chunk by channel chunk."""
    w = WORKLOADS["mamba2p8b_fwdbwd"]
    Bt, D, N, L = w["Bt"], w["D"], w["N"], w["L"]
    a = device_inputs(Bt, D, N, L, seed=w["seed"], in_dtype="bf16", dy=True)
    g = ssm.ssm_scan_bwd(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["dy"], a["Dv"],
                         a["z"], a["delta_bias"], None, None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    Bh = a["Bm"].float().cpu().numpy()
    Ch = a["Cm"].float().cpu().numpy()
    step = 256
    jobs = []
    for d0 in range(0, D, step):
        sl = slice(d0, d0 + step)
        h = lambda t: t[:, sl].float().cpu().numpy()
        jobs.append((h(a["u"]), h(a["delta_raw"]), a["A"][sl].cpu().numpy(), Bh, Ch, h(a["dy"]),
                     a["Dv"][sl].cpu().numpy(), h(a["z"]), a["delta_bias"][sl].cpu().numpy()))
    with mp.get_context("spawn").Pool(min(8, os.cpu_count() or 1)) as pool:
        res = pool.map(oracle_bwd_chunk, jobs)
    tol = TOL["bf16"]
    worst = {}
    dB = np.zeros((Bt, N, L))
    dC = np.zeros((Bt, N, L))
    for i, o in enumerate(res):
        sl = slice(i * step, (i + 1) * step)
        for k in ("du", "ddelta_raw", "dz"):
            worst[k] = max(worst.get(k, 0.0), rel_err(g[k][:, sl].cpu().numpy(), o[k]))
        for k in ("dA", "dD", "ddelta_bias"):
            worst[k] = max(worst.get(k, 0.0), rel_err(g[k][sl].cpu().numpy(), o[k]))
        worst["dh0"] = max(worst.get("dh0", 0.0), rel_err(g["dh0"][:, sl].cpu().numpy(), o["dh0"]))
        dB += o["dB"]
        dC += o["dC"]
    worst["dB"] = rel_err(g["dB"].cpu().numpy(), dB)
    worst["dC"] = rel_err(g["dC"].cpu().numpy(), dC)
    print("mamba2p8b backward, max normalised errors:", worst)
    for k, e in worst.items():
        assert e <= tol, "%s: %.3e > %.1e" % (k, e, tol)
