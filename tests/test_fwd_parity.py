"""Forward scan on the GPU against the fp64 oracle, element by element.

Small and ragged shapes (several 64-token tiles plus a ragged tail, channel
counts that do not fill a CTA, odd state sizes, absent optional terms, both
load paths), the tiny fp32 workload exactly, the segmented plan, and every
full-size forward workload on sampled channels (channels are independent
given the shared B and C, so any subset is checked exactly).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from scan_inputs import WORKLOADS, device_inputs, make_inputs
from tests.gpu_util import gpu_fwd, load_ssm, oracle_fwd, rows_to_host
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _check(ssm, x, out_dtype=torch.float32):
    tol = TOL[x.in_dtype]
    y, hL = gpu_fwd(ssm, x, out_dtype)
    yo, ho = oracle_fwd(x)
    if out_dtype == torch.bfloat16:
        assert_bf16_output(y, yo, tol, "y")
    else:
        assert_close(y, yo, tol, "y")
    assert_close(hL, ho, tol, "hL")


def test_tiny_fp32_workload(ssm):
    w = WORKLOADS["tiny_fp32"]
    x = make_inputs(w["Bt"], w["D"], w["N"], w["L"], seed=w["seed"], in_dtype="f32",
                    a_jitter=False)
    _check(ssm, x)


CASES = [
    # (Bt, D, N, L, dtype, options)
    (2, 40, 16, 200, "bf16", {}),              # ragged D and ragged last tile, TMA path
    (1, 70, 16, 77, "bf16", {}),               # rows not 16-byte aligned: plain-load path
    (2, 20, 8, 96, "f32", {}),                 # fp32 TMA path (two boxes per tile)
    (3, 33, 4, 130, "f32", {"h0": True}),      # fp32 plain-load path, initial state
    (2, 64, 16, 128, "bf16", {"h0": True}),
    (1, 128, 16, 64, "bf16", {"with_z": False}),
    (1, 96, 16, 192, "bf16", {"with_D": False, "with_bias": False}),
    (2, 10, 1, 100, "bf16", {}),
    (1, 50, 5, 256, "bf16", {"h0": True}),
    (1, 36, 32, 160, "bf16", {}),
    (1, 24, 64, 136, "bf16", {"h0": True}),
    (1, 17, 16, 1, "bf16", {"h0": True}),      # a single token
    (1, 17, 16, 65, "f32", {}),
    (4, 300, 16, 320, "bf16", {}),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%dx%dx%dx%d-%s" % c[:5])
def test_small_shapes(ssm, case):
    Bt, D, N, L, dt, opt = case
    x = make_inputs(Bt, D, N, L, seed=100 + D + L, in_dtype=dt, **opt)
    _check(ssm, x)


@pytest.mark.parametrize("nt", ["1", "2", "4"])
def test_threads_per_channel_variants(ssm, nt, monkeypatch):
    monkeypatch.setenv("SSM_FWD_NT", nt)
    x = make_inputs(2, 90, 16, 330, seed=7, in_dtype="bf16", h0=True)
    _check(ssm, x)
    x = make_inputs(1, 30, 16, 96, seed=8, in_dtype="f32")
    _check(ssm, x)


@pytest.mark.parametrize("nseg", ["2", "3", "7"])
def test_segmented_plan(ssm, nseg, monkeypatch):
    """Two passes and a carry across segments reproduce the single pass."""
    monkeypatch.setenv("SSM_FWD_NSEG", nseg)
    x = make_inputs(2, 70, 16, 64 * 29 + 13, seed=9, in_dtype="bf16", h0=True)
    _check(ssm, x)
    x = make_inputs(1, 20, 16, 64 * 30, seed=10, in_dtype="f32", h0=True)
    _check(ssm, x)


@pytest.mark.parametrize("dt,L,bias_shift", [("bf16", 64 * 160, 0.0), ("bf16", 64 * 160, 3.0),
                                             ("bf16", 64 * 40, -1.0), ("f32", 64 * 160, 3.0),
                                             ("f32", 64 * 64, 0.0)])
def test_segmented_plan_long_segments(ssm, dt, L, bias_shift, monkeypatch):
    """Two segments of 1280 to 5120 tokens: with the recipe's delta, with a
    larger one (+3 on the bias: the decay over a segment underflows to zero,
    so the carry passes on the segment's own summary alone) and with a
    smaller one (-1: long memory across the segment boundary).  fp32 inputs
    over these lengths are held to the long-sequence fp32 bar."""
    monkeypatch.setenv("SSM_FWD_NSEG", "2")
    x = make_inputs(1, 40, 16, L, seed=13, in_dtype=dt, h0=True)
    x.delta_bias = (x.delta_bias + np.float32(bias_shift)).astype(np.float32)
    tol = TOL[dt]
    y, hL = gpu_fwd(ssm, x)
    yo, ho = oracle_fwd(x)
    assert_close(y, yo, tol, "y")
    assert_close(hL, ho, tol, "hL")


def test_bf16_output(ssm):
    x = make_inputs(2, 64, 16, 256, seed=11, in_dtype="bf16")
    _check(ssm, x, out_dtype=torch.bfloat16)


def test_empty_sequence_returns_initial_state(ssm):
    x = make_inputs(2, 8, 16, 1, seed=12, in_dtype="bf16", h0=True)
    dev = lambda a, dt: torch.from_numpy(a).cuda().to(dt)
    u = torch.empty(2, 8, 0, dtype=torch.bfloat16, device="cuda")
    Bm = torch.empty(2, 16, 0, dtype=torch.bfloat16, device="cuda")
    h0 = dev(x.h0, torch.float32)
    y, hL = ssm.ssm_scan_fwd(u, u, dev(x.A, torch.float32), Bm, Bm, h0=h0)
    torch.cuda.synchronize()
    assert y.shape == (2, 8, 0)
    assert torch.equal(hL, h0)
    _, hL0 = ssm.ssm_scan_fwd(u, u, dev(x.A, torch.float32), Bm, Bm)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hL0) == 0


# ------------------------------------------------------------------ full size
def _sampled_full(ssm, name, samples_per_batch=6, out_dtype=torch.float32):
    w = WORKLOADS[name]
    Bt, D, N, L = w["Bt"], w["D"], w["N"], w["L"]
    a = device_inputs(Bt, D, N, L, seed=w["seed"], in_dtype="bf16")
    y, hL = ssm.ssm_scan_fwd(a["u"], a["delta_raw"], a["A"], a["Bm"],
                             a["Cm"], a["Dv"], a["z"], a["delta_bias"], a["h0"],
                             out_dtype=out_dtype)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1234)
    for b in range(Bt):
        ds = np.sort(rng.choice(D, size=samples_per_batch, replace=False))
        ds[0] = 0
        ds[-1] = D - 1
        bi = [b]
        host = lambda t: rows_to_host(t, bi, ds)
        yo, ho = oracle.scan_fwd(host(a["u"]), host(a["delta_raw"]), a["A"][ds].cpu().numpy(),
                                 a["Bm"][bi].float().cpu().numpy(),
                                 a["Cm"][bi].float().cpu().numpy(), a["Dv"][ds].cpu().numpy(),
                                 host(a["z"]), a["delta_bias"][ds].cpu().numpy(), None)
        yg = y[bi][:, ds].float().cpu().numpy()
        hg = hL[bi][:, ds].cpu().numpy()
        if out_dtype == torch.bfloat16:
            assert_bf16_output(yg, yo, TOL["bf16"], "%s y b=%d" % (name, b))
        else:
            assert_close(yg, yo, TOL["bf16"], "%s y b=%d" % (name, b))
        assert_close(hg, ho, TOL["bf16"], "%s hL b=%d" % (name, b))
    del a, y, hL
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["mamba130m_fwd", "mamba1p4b_fwd", "mamba2p8b_fwdbwd"])
def test_full_size_sampled(ssm, name):
    _sampled_full(ssm, name)


def test_full_size_bf16_output_sampled(ssm):
    _sampled_full(ssm, "mamba1p4b_fwd", out_dtype=torch.bfloat16)


def test_million_length_sampled(ssm):
    _sampled_full(ssm, "million_fwd", samples_per_batch=4)
