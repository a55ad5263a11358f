"""The scan fed by the block's conv prologue ("Mamba Architecture Explained",
section "The Architecture in Practice": Conv1D and SiLU before the selective
SSM) on the GPU against the oracle: conv_silu then the scan, in fp64."""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import make_inputs
from tests.gpu_util import device_args, load_ssm, to_dev
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _conv_params(D, K, seed, with_bias=True):
    rng = np.random.default_rng(seed)
    w = (0.5 * rng.standard_normal((D, K))).astype(np.float32)
    b = (0.1 * rng.standard_normal(D)).astype(np.float32) if with_bias else None
    return w, b


def _check(ssm, x, w, b, out_dtype=torch.float32, tol=None):
    a = device_args(x)
    y, hL = ssm.ssm_scan_fwd_conv(a["u"], to_dev(w, torch.float32), to_dev(b, torch.float32),
                                  a["delta_raw"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                  a["delta_bias"], a["h0"], out_dtype=out_dtype)
    torch.cuda.synchronize()
    yo, ho = oracle.scan_fwd_conv(x.u, w, b, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z,
                                  x.delta_bias, x.h0)
    tol = TOL[x.in_dtype] if tol is None else tol
    if out_dtype == torch.bfloat16:
        assert_bf16_output(y.float().cpu().numpy(), yo, tol, "y")
    else:
        assert_close(y.float().cpu().numpy(), yo, tol, "y")
    assert_close(hL.cpu().numpy(), ho, tol, "hL")


CASES = [
    # (Bt, D, N, L, dtype, K, options, conv bias)
    (2, 70, 16, 64 * 5 + 8, "bf16", 4, {"h0": True}, True),   # ragged channels and last chunk
    (1, 40, 16, 256, "f32", 2, {}, False),
    (3, 33, 12, 200, "bf16", 3, {"with_z": False}, True),     # 12 states padded to 16
    (2, 64, 16, 128, "bf16", 1, {"with_D": False, "with_bias": False}, True),
    (1, 24, 16, 64, "bf16", 4, {}, True),                      # one chunk
    (4, 300, 16, 320, "bf16", 4, {}, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%dx%dx%dx%d-%s-k%d" % c[:6])
def test_conv_prologue_small(ssm, case):
    Bt, D, N, L, dt, K, opts, with_b = case
    x = make_inputs(Bt, D, N, L, seed=60 + D, in_dtype=dt, **opts)
    w, b = _conv_params(D, K, 61 + D, with_b)
    _check(ssm, x, w, b)


def test_conv_prologue_bf16_output(ssm):
    x = make_inputs(2, 64, 16, 256, seed=70, in_dtype="bf16")
    w, b = _conv_params(64, 4, 71)
    _check(ssm, x, w, b, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("nt", ["1", "2", "4"])
def test_conv_prologue_lanes_per_channel(ssm, nt, monkeypatch):
    monkeypatch.setenv("SSM_FWD_NT", nt)
    x = make_inputs(2, 50, 16, 64 * 3 + 16, seed=72, in_dtype="bf16", h0=True)
    w, b = _conv_params(50, 4, 73)
    _check(ssm, x, w, b)


@pytest.mark.parametrize("nseg", ["2", "3"])
def test_conv_prologue_segmented(ssm, nseg, monkeypatch):
    """Segments start inside the sequence: each reads the 3 inputs before it."""
    monkeypatch.setenv("SSM_FWD_NSEG", nseg)
    x = make_inputs(1, 50, 16, 64 * 30, seed=74, in_dtype="bf16", h0=True)
    w, b = _conv_params(50, 4, 75)
    _check(ssm, x, w, b)
    monkeypatch.setenv("SSM_FWD_NSEG", "2")
    x = make_inputs(1, 40, 16, 64 * 160, seed=76, in_dtype="bf16")
    w, b = _conv_params(40, 4, 77)
    _check(ssm, x, w, b)


@pytest.mark.parametrize("N,L", [(32, 64), (16, 201)])
def test_conv_prologue_unsupported_shape(ssm, N, L):
    """More than 16 states, or token rows that are not a multiple of 16
    bytes: the call returns SSM_ERR_UNSUPPORTED before any launch."""
    x = make_inputs(1, 16, N, L, seed=78, in_dtype="bf16")
    w, b = _conv_params(16, 4, 79)
    with pytest.raises(ssm.SSMError):
        _check(ssm, x, w, b)
