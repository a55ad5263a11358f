"""Reverse mode of the bidirectional scan on the GPU against the oracle
("Mamba Architecture Explained", section "Frequently Asked Questions":
bidirectional variants run a second scan right to left).  du and dz are the
sums of the two directions' gradients; every other gradient belongs to one
direction.  Ragged channel counts and last chunks, rows that are not
16-byte multiples (plain loads in the sweeps), fp32 and bf16 inputs, bf16
outputs, upstream gradients of both final states, no gate, tied weights."""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import make_inputs
from tests.gpu_util import TIN, load_ssm, to_dev
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu

PER_TOKEN = ("du", "dz", "ddelta_raw")


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _host(x):
    return dict(delta_raw=x.delta_raw, A=x.A, Bm=x.Bm, Cm=x.Cm, Dv=x.Dv, delta_bias=x.delta_bias,
                h0=x.h0)


def _dev(x):
    t = TIN[x.in_dtype]
    f32 = torch.float32
    return dict(delta_raw=to_dev(x.delta_raw, t), A=to_dev(x.A, f32), B=to_dev(x.Bm, t),
                C=to_dev(x.Cm, t), D=to_dev(x.Dv, f32), delta_bias=to_dev(x.delta_bias, f32),
                h0=to_dev(x.h0, f32))


def _cmp(g, o, tol, name, bf16_out):
    g = g.float().cpu().numpy()
    if bf16_out and name.split(".")[-1] in PER_TOKEN:
        assert_bf16_output(g, o, tol, name)
    else:
        assert_close(g, o, tol, name)


def _run(ssm, Bt, D, N, L, dt, seed, out_dtype=torch.float32, gate=True, dhl=True, tied=False,
         h0=True):
    xf = make_inputs(Bt, D, N, L, seed=seed, in_dtype=dt, h0=h0, dy=True, with_z=gate)
    xr = xf if tied else make_inputs(Bt, D, N, L, seed=seed + 1, in_dtype=dt, h0=h0)
    rng = np.random.default_rng(seed + 2)
    dhL = rng.standard_normal((Bt, D, N)).astype(np.float32) if dhl else None
    dhL_r = rng.standard_normal((Bt, D, N)).astype(np.float32) if dhl else None
    t = TIN[dt]
    shared, gf, gr = ssm.ssm_scan_bwd_bidir(to_dev(xf.u, t), to_dev(xf.z, t), _dev(xf), _dev(xr),
                                            to_dev(xf.dy, t), to_dev(dhL, torch.float32),
                                            to_dev(dhL_r, torch.float32), out_dtype=out_dtype)
    torch.cuda.synchronize()
    so, of, orr = oracle.scan_bwd_bidir(xf.u, xf.z, _host(xf), _host(xr), xf.dy, dhL, dhL_r)
    tol = TOL[dt]
    bf = out_dtype == torch.bfloat16
    _cmp(shared["du"], so["du"], tol, "du", bf)
    if gate:
        _cmp(shared["dz"], so["dz"], tol, "dz", bf)
    else:
        assert shared["dz"] is None
    for tag, g, o in (("fwd", gf, of), ("rev", gr, orr)):
        for k in ("ddelta_raw", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0"):
            _cmp(g[k], o[k], tol, tag + "." + k, bf)


CASES = [
    # (Bt, D, N, L, dtype)
    (2, 40, 16, 200, "bf16"),     # ragged channels and last chunk, TMA path
    (1, 33, 16, 130, "bf16"),     # rows not a multiple of 16 bytes: plain loads
    (2, 20, 8, 96, "f32"),
    (1, 17, 16, 65, "f32"),
    (1, 24, 4, 64, "bf16"),
    (1, 12, 32, 72, "bf16"),
    (1, 9, 16, 1, "bf16"),        # a single token
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "%dx%dx%dx%d-%s" % c)
def test_bidir_bwd_shapes(ssm, case):
    Bt, D, N, L, dt = case
    _run(ssm, Bt, D, N, L, dt, seed=500 + D + L)


def test_bidir_bwd_bf16_output(ssm):
    _run(ssm, 2, 48, 16, 256, "bf16", seed=520, out_dtype=torch.bfloat16)


def test_bidir_bwd_no_gate_no_upstream_state(ssm):
    _run(ssm, 1, 40, 16, 192, "bf16", seed=530, gate=False, dhl=False, h0=False)


def test_bidir_bwd_tied_weights(ssm):
    _run(ssm, 2, 32, 16, 128, "f32", seed=540, tied=True)


def test_bidir_bwd_long_rows(ssm):
    """Many chunks per row (the sweeps' chunk re-anchoring) in both directions."""
    _run(ssm, 1, 24, 16, 64 * 30 + 8, "f32", seed=550)
    _run(ssm, 1, 40, 16, 64 * 40, "bf16", seed=552)
