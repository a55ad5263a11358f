"""The backward's segmented plan (long sequences with few channels) on the GPU
against the fp64 oracle's reverse mode ("Mamba: Linear-Time Sequence Modeling
with Selective State Spaces", section "Key points": sequences up to a million
tokens).  The sequence is cut into segments run side by side: every segment
starts from the forward carry's state, takes the adjoint entering at its
right end from the adjoint summary and its carry, and the dA terms of the
tangent crossing segment boundaries come from the tangent carry.  The
results must equal the oracle's whole-sequence reverse mode, including where
a boundary falls inside a segment's last chunk, where segments are ragged,
and in the long-memory and forgetting regimes of delta."""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import make_inputs
from tests.gpu_util import TIN, device_args, load_ssm, to_dev
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu

PER_TOKEN = ("du", "ddelta_raw", "dz")
OUTS = ("du", "ddelta_raw", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _state(x, seed):
    Bt, D, N, L = x.shape
    return np.random.default_rng(seed).standard_normal((Bt, D, N)).astype(np.float32)


def _check(ssm, x, dhL, out_dtype=torch.float32):
    a = device_args(x)
    g = ssm.ssm_scan_bwd(a["u"], a["delta_raw"], a["A"], a["B"], a["C"], to_dev(x.dy, TIN[x.in_dtype]),
                         a["D"], a["z"], a["delta_bias"], a["h0"], to_dev(dhL, torch.float32),
                         out_dtype=out_dtype)
    torch.cuda.synchronize()
    o = oracle.scan_bwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z, x.delta_bias, x.h0, dhL)
    tol = TOL[x.in_dtype]
    for k in OUTS:
        got = None if g[k] is None else g[k].float().cpu().numpy()
        if k == "dz" and x.z is None:
            assert got is None
            continue
        if out_dtype == torch.bfloat16 and k in PER_TOKEN:
            assert_bf16_output(got, o[k], tol, k)
        else:
            assert_close(got, o[k], tol, k)


@pytest.mark.parametrize("nseg", [2, 3, 7])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_segments_match_whole_sequence(ssm, monkeypatch, nseg, dtype):
    """40 chunks cut into 2, 3 and 7 segments (7: ragged, the last segment
    shorter), with h0, dhL, the gate, D and the bias."""
    monkeypatch.setenv("SSM_BWD_NSEG", str(nseg))
    x = make_inputs(1, 40, 16, 64 * 40, seed=700 + nseg, in_dtype=dtype, dy=True, h0=True)
    _check(ssm, x, _state(x, 701 + nseg))


@pytest.mark.parametrize("nt", ["2", "4"])
def test_segments_lanes_per_channel(ssm, monkeypatch, nt):
    """Two and four lanes per channel, a ragged last chunk, no initial state,
    no dhL, bf16 gradients."""
    monkeypatch.setenv("SSM_BWD_NSEG", "4")
    monkeypatch.setenv("SSM_BWD_NT", nt)
    x = make_inputs(2, 24, 16, 64 * 24 + 40, seed=710 + int(nt), in_dtype="bf16", dy=True)
    _check(ssm, x, None, out_dtype=torch.bfloat16)


def test_segments_without_optional_terms(ssm, monkeypatch):
    monkeypatch.setenv("SSM_BWD_NSEG", "5")
    x = make_inputs(1, 32, 16, 64 * 30, seed=720, in_dtype="bf16", dy=True, with_z=False,
                    with_D=False, with_bias=False)
    _check(ssm, x, _state(x, 721))


@pytest.mark.parametrize("nseg", [1, 6])
@pytest.mark.parametrize("shift", [-3.0, 0.0, 4.0])
def test_segments_memory_regimes(ssm, monkeypatch, shift, nseg):
    """delta far below the recipe (the state and the adjoint carry across
    every segment), at it, and far above it (the decay across a segment is
    below fp32 resolution: the carries pass nothing on); the whole-row plan
    on the same inputs (fp32: the forward sweep's compensated state keeps
    dz, dC and ddelta_raw within 1e-5 where the state remembers thousands of
    tokens)."""
    monkeypatch.setenv("SSM_BWD_NSEG", str(nseg))
    x = make_inputs(1, 16, 16, 64 * 36, seed=730, in_dtype="f32", dy=True, h0=True)
    x.delta_bias = (x.delta_bias + np.float32(shift)).astype(np.float32)
    _check(ssm, x, _state(x, 731))


def test_planner_segments_few_channels(ssm):
    """Without an override the planner cuts a few-channel long sequence into
    segments (48 channels, 16,384 tokens); the result is the whole-sequence
    reverse mode."""
    x = make_inputs(1, 48, 16, 16384, seed=740, in_dtype="bf16", dy=True, h0=True)
    _check(ssm, x, _state(x, 741))
