"""The bidirectional scan on the GPU against the oracle ("Mamba Architecture
Explained", section "Frequently Asked Questions": bidirectional SSM
variants): a left-to-right and a right-to-left selective scan over the same
input and gate, each with its own parameters, summed."""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import make_inputs
from tests.gpu_util import TIN, load_ssm, to_dev
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _dirs(Bt, D, N, L, seed, dt, **kw):
    """Two independent parameter sets drawn with the same recipe; u and z
    from the first."""
    return (make_inputs(Bt, D, N, L, seed=seed, in_dtype=dt, **kw),
            make_inputs(Bt, D, N, L, seed=seed + 1, in_dtype=dt, **kw))


def _host(x):
    return dict(delta_raw=x.delta_raw, A=x.A, Bm=x.Bm, Cm=x.Cm, Dv=x.Dv, delta_bias=x.delta_bias,
                h0=x.h0)


def _dev(x):
    t = TIN[x.in_dtype]
    return dict(delta_raw=to_dev(x.delta_raw, t), A=to_dev(x.A, torch.float32), B=to_dev(x.Bm, t),
                C=to_dev(x.Cm, t), D=to_dev(x.Dv, torch.float32),
                delta_bias=to_dev(x.delta_bias, torch.float32), h0=to_dev(x.h0, torch.float32))


def _run(ssm, xf, xr, out_dtype=torch.float32, tol=None, tied=False):
    t = TIN[xf.in_dtype]
    rev_h, rev_d = (_host(xf), _dev(xf)) if tied else (_host(xr), _dev(xr))
    y, hL, hL_r = ssm.ssm_scan_fwd_bidir(to_dev(xf.u, t), to_dev(xf.z, t), _dev(xf), rev_d,
                                         out_dtype=out_dtype)
    torch.cuda.synchronize()
    yo, ho, hro = oracle.scan_fwd_bidir(xf.u, xf.z, _host(xf), rev_h)
    tol = TOL[xf.in_dtype] if tol is None else tol
    if out_dtype == torch.bfloat16:
        assert_bf16_output(y.float().cpu().numpy(), yo, tol, "y")
    else:
        assert_close(y.cpu().numpy(), yo, tol, "y")
    assert_close(hL.cpu().numpy(), ho, tol, "hL")
    assert_close(hL_r.cpu().numpy(), hro, tol, "hL_r")


CASES = [
    # (Bt, D, N, L, dtype, options)
    (2, 70, 16, 64 * 5 + 8, "bf16", {"h0": True}),   # ragged channels, ragged last chunk
    (1, 40, 16, 200, "f32", {"h0": True}),
    (3, 33, 12, 136, "bf16", {"with_z": False}),
    (2, 64, 16, 64, "bf16", {"with_D": False, "with_bias": False}),
    (4, 300, 16, 256, "bf16", {}),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%dx%dx%dx%d-%s" % c[:5])
def test_bidir_small(ssm, case):
    Bt, D, N, L, dt, opts = case
    xf, xr = _dirs(Bt, D, N, L, 100 + D, dt, **opts)
    _run(ssm, xf, xr)


def test_bidir_bf16_output_and_tied(ssm):
    xf, xr = _dirs(2, 64, 16, 256, 110, "bf16")
    _run(ssm, xf, xr, out_dtype=torch.bfloat16)
    _run(ssm, xf, xr, tied=True)


@pytest.mark.parametrize("nt", ["1", "2", "4"])
def test_bidir_lanes_per_channel(ssm, nt, monkeypatch):
    monkeypatch.setenv("SSM_FWD_NT", nt)
    xf, xr = _dirs(2, 50, 16, 64 * 3 + 16, 112, "bf16", h0=True)
    _run(ssm, xf, xr)


def test_bidir_long_sequence(ssm, monkeypatch):
    """A long row in one segment per direction."""
    monkeypatch.setenv("SSM_FWD_NSEG", "1")
    xf, xr = _dirs(1, 24, 16, 64 * 40, 114, "f32")
    _run(ssm, xf, xr)
    xf, xr = _dirs(1, 40, 16, 64 * 100, 116, "bf16")
    _run(ssm, xf, xr)


@pytest.mark.parametrize("nseg", ["2", "3", "7"])
def test_bidir_segmented(ssm, nseg, monkeypatch):
    """The two-pass split of a row in both directions: the right-to-left
    summaries run from each segment's right end and its carry from the last
    segment down; initial states of both directions, a ragged last chunk,
    fp32 and bf16."""
    monkeypatch.setenv("SSM_FWD_NSEG", nseg)
    xf, xr = _dirs(1, 40, 16, 64 * 29 + 8, 130, "bf16", h0=True)
    _run(ssm, xf, xr)
    xf, xr = _dirs(2, 24, 16, 64 * 30, 132, "f32", h0=True)
    _run(ssm, xf, xr)


@pytest.mark.parametrize("shift", [-1.0, 3.0])
def test_bidir_segmented_long_segments(ssm, shift, monkeypatch):
    """Two segments of 5,120 tokens with smaller and larger delta (long memory
    across the segment boundary in both directions; decay to zero)."""
    monkeypatch.setenv("SSM_FWD_NSEG", "2")
    xf, xr = _dirs(1, 40, 16, 64 * 160, 134, "bf16", h0=True)
    for x in (xf, xr):
        x.delta_bias = (x.delta_bias + np.float32(shift)).astype(np.float32)
    _run(ssm, xf, xr)


def test_bidir_unsupported_shape(ssm):
    xf, xr = _dirs(1, 16, 16, 201, 118, "bf16")
    with pytest.raises(ssm.SSMError):
        _run(ssm, xf, xr)
