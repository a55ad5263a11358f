"""Reverse mode over packed variable-length sequences on the GPU against the
oracle ("Mamba Architecture Explained", section "Problem 3: Ecosystem
maturity": sequence packing).  Every sequence has its own reverse mode: dh0
per sequence, dhL per sequence, nothing crossing a start; dA, dD, ddelta_bias
summed over the sequences, dB and dC over the channels."""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import make_inputs, packed_seqlens
from tests.gpu_util import TIN, device_args, load_ssm, to_dev
from tests.parity import TOL, assert_bf16_output, assert_close

pytestmark = pytest.mark.gpu

OUTS = ("du", "ddelta_raw", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0")
PER_TOKEN = ("du", "ddelta_raw", "dz")


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _state(nseq, Bt, D, N, seed):
    return np.random.default_rng(seed).standard_normal((nseq, Bt, D, N)).astype(np.float32)


def _run(ssm, x, cu, h0=None, dhL=None, out_dtype=torch.float32, tol=None):
    a = device_args(x)
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    g = ssm.ssm_scan_bwd_varlen(a["u"], cu_d, a["delta_raw"], a["A"], a["B"], a["C"],
                                to_dev(x.dy, TIN[x.in_dtype]), a["D"], a["z"], a["delta_bias"],
                                to_dev(h0, torch.float32), to_dev(dhL, torch.float32),
                                out_dtype=out_dtype)
    torch.cuda.synchronize()
    o = oracle.scan_bwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, cu, x.Dv, x.z,
                               x.delta_bias, h0, dhL)
    tol = TOL[x.in_dtype] if tol is None else tol
    for k in OUTS:
        if k == "dz" and x.z is None:
            assert g[k] is None
            continue
        got = g[k].float().cpu().numpy()
        if out_dtype == torch.bfloat16 and k in PER_TOKEN:
            assert_bf16_output(got, o[k], tol, k)
        else:
            assert_close(got, o[k], tol, k)


# boundaries inside super-blocks (and inside one lane's 8 tokens), on chunk
# and super-block starts, empty sequences at the start, middle and end,
# one-token sequences
CUTS = [0, 0, 1, 5, 16, 17, 64, 64, 100, 191, 192, 250, 256, 300, 317, 320, 320]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("states", ["none", "h0", "h0+dhL"])
def test_varlen_bwd_boundaries(ssm, dtype, states):
    Bt, D, N, L = 2, 70, 16, 320
    x = make_inputs(Bt, D, N, L, seed=600, in_dtype=dtype, dy=True)
    ns = len(CUTS) - 1
    h0 = _state(ns, Bt, D, N, 601) if states != "none" else None
    dhL = _state(ns, Bt, D, N, 602) if states == "h0+dhL" else None
    _run(ssm, x, CUTS, h0, dhL)


def test_varlen_bwd_dense_starts(ssm):
    """A start at nearly every token of some super-blocks (several restarts
    inside one lane's run of the suffix sum)."""
    Bt, D, N, L = 1, 40, 16, 256
    x = make_inputs(Bt, D, N, L, seed=610, in_dtype="bf16", dy=True)
    cuts = sorted(set([0, 2, 3, 4, 6, 7, 8, 9, 11, 14, 15, 16, 17, 31, 32, 33, 62, 63, 64, 65,
                       127, 128, 129, 200, 254, 255, 256]))
    ns = len(cuts) - 1
    _run(ssm, x, cuts, _state(ns, Bt, D, N, 611), _state(ns, Bt, D, N, 612))


def test_varlen_bwd_one_sequence_matches_plain_backward(ssm):
    """One sequence covering the row is the plain backward."""
    x = make_inputs(2, 48, 16, 192, seed=620, in_dtype="bf16", dy=True, h0=True)
    dhL = _state(1, 2, 48, 16, 621)
    _run(ssm, x, [0, 192], x.h0[None], dhL)


def test_varlen_bwd_all_empty_but_one(ssm):
    x = make_inputs(1, 16, 16, 64, seed=630, in_dtype="bf16", dy=True)
    _run(ssm, x, [0, 0, 0, 64, 64], _state(4, 1, 16, 16, 631), _state(4, 1, 16, 16, 632))


def test_varlen_bwd_no_gate_bf16_output(ssm):
    Bt, D, N, L = 2, 64, 16, 256
    x = make_inputs(Bt, D, N, L, seed=640, in_dtype="bf16", dy=True, with_z=False)
    cuts = [0, 30, 64, 65, 200, 256]
    ns = len(cuts) - 1
    _run(ssm, x, cuts, _state(ns, Bt, D, N, 641), _state(ns, Bt, D, N, 642),
         out_dtype=torch.bfloat16)


def test_varlen_bwd_packed_recipe_long_row(ssm):
    """The packed workload's length mix (log-uniform lengths) over many
    chunks, fp32 and bf16."""
    L = 64 * 48
    cu = packed_seqlens(L, seed=650, lo=16, hi=1024)
    for dt, seed in (("f32", 651), ("bf16", 652)):
        x = make_inputs(1, 40, 16, L, seed=seed, in_dtype=dt, dy=True)
        ns = len(cu) - 1
        _run(ssm, x, cu, _state(ns, 1, 40, 16, seed + 10), _state(ns, 1, 40, 16, seed + 20))


def test_varlen_bwd_bad_starts_reported(ssm):
    """Starts out of order or not ending at L: the call runs (no access
    outside the buffers) and the workspace status says SSM_ERR_SEQLENS."""
    x = make_inputs(1, 16, 16, 128, seed=660, in_dtype="bf16", dy=True)
    a = device_args(x)
    dy = to_dev(x.dy, torch.bfloat16)
    shape = ssm.make_shape(1, 16, 16, 128, ssm.SSM_BF16, ssm.SSM_F32)
    ws = torch.empty(ssm.ssm_scan_workspace_bytes(shape, True), dtype=torch.uint8, device="cuda")
    for cu in ([0, 70, 50, 128], [0, 64, 127], [1, 64, 128], [0, 64, 200]):
        cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
        ssm.ssm_scan_bwd_varlen(a["u"], cu_d, a["delta_raw"], a["A"], a["B"], a["C"], dy,
                                out_dtype=torch.float32, workspace=ws)
        assert ssm.ssm_get_status(ws) == ssm.SSM_ERR_SEQLENS, cu
    cu_d = torch.tensor([0, 64, 128], dtype=torch.int32, device="cuda")
    ssm.ssm_scan_bwd_varlen(a["u"], cu_d, a["delta_raw"], a["A"], a["B"], a["C"], dy,
                            out_dtype=torch.float32, workspace=ws)
    assert ssm.ssm_get_status(ws) == ssm.SSM_OK


def test_varlen_bwd_unsupported_shape(ssm):
    x = make_inputs(1, 16, 8, 100, seed=670, in_dtype="bf16", dy=True)
    with pytest.raises(ssm.SSMError):
        _run(ssm, x, [0, 50, 100])


@pytest.mark.parametrize("nt", ["2", "4"])
def test_varlen_bwd_lanes_per_channel(ssm, nt, monkeypatch):
    """Two and four lanes per channel (32-token super-blocks: restarts in
    four lanes' runs of the suffix sum)."""
    monkeypatch.setenv("SSM_BWD_NT", nt)
    Bt, D, N, L = 1, 50, 16, 320
    x = make_inputs(Bt, D, N, L, seed=680 + int(nt), in_dtype="bf16", dy=True)
    ns = len(CUTS) - 1
    _run(ssm, x, CUTS, _state(ns, Bt, D, N, 690), _state(ns, Bt, D, N, 691))
    xf = make_inputs(Bt, D, N, L, seed=685 + int(nt), in_dtype="f32", dy=True)
    _run(ssm, xf, CUTS, _state(ns, Bt, D, N, 692), _state(ns, Bt, D, N, 693))


# segment boundaries of the forced segmented plans below: 12 chunks in 3
# segments start at tokens 256 and 512; in 4 segments at 192, 384 and 576
SEG_CUTS = [0, 100, 192, 256, 300, 383, 384, 511, 512, 512, 600, 700, 768]


@pytest.mark.parametrize("nseg", ["3", "4"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_varlen_bwd_segments(ssm, nseg, dtype, monkeypatch):
    """The segmented plan over packed sequences: starts on segment
    boundaries (a sequence ending with a segment's last token), inside
    segments, an empty sequence on a boundary, and sequences spanning two
    segments; h0 and dhL per sequence."""
    monkeypatch.setenv("SSM_BWD_NSEG", nseg)
    Bt, D, N, L = 2, 40, 16, 768
    x = make_inputs(Bt, D, N, L, seed=700 + int(nseg), in_dtype=dtype, dy=True)
    ns = len(SEG_CUTS) - 1
    _run(ssm, x, SEG_CUTS, _state(ns, Bt, D, N, 701), _state(ns, Bt, D, N, 702))


def test_varlen_bwd_segments_long_sequences(ssm, monkeypatch):
    """Few sequences, each spanning several segments (the carries pass the
    state, the adjoint and the dA tangent across boundaries inside a
    sequence), and a last sequence that starts inside the last segment."""
    monkeypatch.setenv("SSM_BWD_NSEG", "6")
    Bt, D, N, L = 1, 32, 16, 64 * 30
    cuts = [0, 64 * 11 + 5, 64 * 27 + 30, L]
    x = make_inputs(Bt, D, N, L, seed=710, in_dtype="bf16", dy=True)
    ns = len(cuts) - 1
    _run(ssm, x, cuts, _state(ns, Bt, D, N, 711), _state(ns, Bt, D, N, 712))


def test_varlen_bwd_packed_recipe_planner_segments(ssm):
    """The packed workload's length mix over a long row with few channels:
    the planner cuts it into segments by itself."""
    L = 64 * 256
    cu = packed_seqlens(L, seed=720, lo=16, hi=4096)
    x = make_inputs(1, 48, 16, L, seed=721, in_dtype="bf16", dy=True)
    ns = len(cu) - 1
    _run(ssm, x, cu, _state(ns, 1, 48, 16, 722), _state(ns, 1, 48, 16, 723))
