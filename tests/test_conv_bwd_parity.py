"""Reverse mode of the scan fed by the block's conv prologue ("Mamba
Architecture Explained", section "The Architecture in Practice": the branch's
Conv1D and SiLU before the selective SSM) on the GPU against the oracle's
scan_bwd_conv, element by element: dx, dconv_w, dconv_b and every gradient
of the scan itself, at small and ragged shapes (several 64-token tiles and a
ragged last channel tile), widths 1 to 4, with and without the conv bias,
the gate, h0 and dhL, both input precisions and bf16 gradients; and at the
Mamba-1.4B layer shape on sampled channels."""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import device_inputs, make_inputs
from tests.gpu_util import TIN, device_args, load_ssm, rows_to_host, to_dev
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu

PER_TOKEN = ("dx", "ddelta_raw", "dz")
OUTS = ("dx", "ddelta_raw", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0", "dconv_w",
        "dconv_b")


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _conv(D, K, seed, with_bias=True):
    rng = np.random.default_rng(seed)
    w = (0.5 * rng.standard_normal((D, K))).astype(np.float32)
    b = (0.1 * rng.standard_normal(D)).astype(np.float32) if with_bias else None
    return w, b


def _run(ssm, x, K, seed, with_bias=True, dhL=None, out_dtype=torch.float32):
    Bt, D, N, L = x.shape
    w, b = _conv(D, K, seed, with_bias)
    a = device_args(x)
    g = ssm.ssm_scan_bwd_conv(a["u"], to_dev(w, torch.float32), to_dev(b, torch.float32),
                              a["delta_raw"], a["A"], a["B"], a["C"], to_dev(x.dy, TIN[x.in_dtype]),
                              a["D"], a["z"], a["delta_bias"], a["h0"], to_dev(dhL, torch.float32),
                              out_dtype=out_dtype)
    torch.cuda.synchronize()
    o = oracle.scan_bwd_conv(x.u, w, b, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z,
                             x.delta_bias, x.h0, dhL)
    tol = TOL[x.in_dtype]
    for k in OUTS:
        if (k == "dz" and x.z is None) or (k == "dconv_b" and b is None):
            assert g[k] is None, k
            continue
        got = g[k].float().cpu().numpy()
        if out_dtype == torch.bfloat16 and k in PER_TOKEN:
            assert_bf16_output(got, o[k], tol, k)
        else:
            assert_close(got, o[k], tol, k)


CASES = [
    # (Bt, D, N, L, dtype, K, conv bias, options, dhL)
    (2, 40, 16, 200, "bf16", 4, True, {"h0": True}, True),
    (1, 70, 16, 136, "bf16", 3, False, {}, False),
    (2, 24, 16, 96, "f32", 4, True, {"h0": True}, True),
    (1, 33, 12, 132, "f32", 2, True, {}, True),
    (2, 48, 16, 64, "bf16", 1, True, {"with_z": False}, False),
    (1, 32, 16, 320, "bf16", 4, True, {"with_D": False, "with_bias": False}, True),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_conv_backward_matches_oracle(ssm, case):
    Bt, D, N, L, dtype, K, cb, opts, with_dhL = case
    x = make_inputs(Bt, D, N, L, seed=800 + L + K, in_dtype=dtype, dy=True, **opts)
    dhL = (np.random.default_rng(801).standard_normal((Bt, D, N)).astype(np.float32)
           if with_dhL else None)
    _run(ssm, x, K, 802 + K, cb, dhL)


def test_conv_backward_bf16_gradients(ssm):
    x = make_inputs(2, 40, 16, 256, seed=810, in_dtype="bf16", dy=True, h0=True)
    _run(ssm, x, 4, 811, True, None, out_dtype=torch.bfloat16)


def test_conv_backward_unsupported_shape(ssm):
    """Rows that are not a multiple of 16 bytes are refused before anything
    is enqueued."""
    x = make_inputs(1, 16, 16, 100, seed=820, in_dtype="bf16", dy=True)
    with pytest.raises(ssm.SSMError):
        _run(ssm, x, 4, 821)


def test_conv_backward_full_size_sampled(ssm):
    """The Mamba-1.4B layer shape (batch 4, D 4096, N 16, L 4096, width 4),
    sampled channels of every batch row: dx, ddelta_raw, dz, and the
    per-channel dA, dD, ddelta_bias, dconv_w, dconv_b (sums over all batch
    rows and tokens of those channels)."""
    Bt, D, N, L = 4, 4096, 16, 4096
    a = device_inputs(Bt, D, N, L, seed=2, in_dtype="bf16", dy=True)
    g0 = torch.Generator(device="cuda")
    g0.manual_seed(1002)
    w = 0.5 * torch.randn(D, 4, generator=g0, device="cuda")
    b = 0.1 * torch.randn(D, generator=g0, device="cuda")
    g = ssm.ssm_scan_bwd_conv(a["u"], w, b, a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["dy"],
                              a["Dv"], a["z"], a["delta_bias"], None, None,
                              out_dtype=torch.float32)
    torch.cuda.synchronize()
    ds = np.array([0, 1234, 2047, 3001, D - 1])
    bi = list(range(Bt))
    host = lambda t: rows_to_host(t, bi, ds)
    o = oracle.scan_bwd_conv(host(a["u"]), w[ds].cpu().numpy(), b[ds].cpu().numpy(),
                             host(a["delta_raw"]), a["A"][ds].cpu().numpy(),
                             a["Bm"].float().cpu().numpy(), a["Cm"].float().cpu().numpy(),
                             host(a["dy"]), a["Dv"][ds].cpu().numpy(), host(a["z"]),
                             a["delta_bias"][ds].cpu().numpy(), None, None)
    tol = TOL["bf16"]
    for k in ("dx", "ddelta_raw", "dz", "dh0"):
        assert_close(g[k][:, ds].cpu().numpy(), o[k], tol, "conv backward " + k)
    for k in ("dA", "dD", "ddelta_bias", "dconv_w", "dconv_b"):
        assert_close(g[k][ds].cpu().numpy(), o[k], tol, "conv backward " + k)
    del a, g
    torch.cuda.empty_cache()
