"""Packed variable-length sequences on the GPU against the oracle ("Mamba
Architecture Explained", section "Problem 3: Ecosystem maturity": sequence
packing): every sequence restarts from its own initial state (and, with the
conv prologue, from a zero conv window); final states per sequence."""
import numpy as np
import pytest
import torch

import oracle
from scan_inputs import make_inputs, packed_seqlens
from tests.gpu_util import device_args, load_ssm, to_dev
from tests.parity import TOL, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _run(ssm, x, cu, h0=None, conv=None, tol=None, ws=None):
    a = device_args(x)
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    cw = cb = None
    if conv is not None:
        cw, cb = to_dev(conv[0], torch.float32), to_dev(conv[1], torch.float32)
    y, hL = ssm.ssm_scan_fwd_varlen(a["u"], cu_d, a["delta_raw"], a["A"], a["B"], a["C"], a["D"],
                                    a["z"], a["delta_bias"], to_dev(h0, torch.float32),
                                    conv_w=cw, conv_b=cb, out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    yo, ho = oracle.scan_fwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, cu, x.Dv, x.z, x.delta_bias,
                                    h0, None if conv is None else conv[0],
                                    None if conv is None else conv[1])
    tol = TOL[x.in_dtype] if tol is None else tol
    assert_close(y.cpu().numpy(), yo, tol, "y")
    assert_close(hL.cpu().numpy(), ho, tol, "hL")


def _h0(nseq, Bt, D, N, seed):
    return np.random.default_rng(seed).standard_normal((nseq, Bt, D, N)).astype(np.float32)


def _conv(D, seed, K=4):
    r = np.random.default_rng(seed)
    return ((0.5 * r.standard_normal((D, K))).astype(np.float32),
            (0.1 * r.standard_normal(D)).astype(np.float32))


# boundaries inside super-blocks, on chunk and super-block starts, empty
# sequences at the start, middle and end, one-token sequences
CUTS = [0, 0, 1, 5, 16, 17, 64, 64, 100, 191, 192, 250, 256, 300, 317, 320, 320]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("with_h0", [False, True])
def test_varlen_boundaries(ssm, dtype, with_h0):
    Bt, D, N, L = 2, 70, 16, 320
    x = make_inputs(Bt, D, N, L, seed=80, in_dtype=dtype)
    h0 = _h0(len(CUTS) - 1, Bt, D, N, 81) if with_h0 else None
    _run(ssm, x, CUTS, h0)


@pytest.mark.parametrize("with_h0", [False, True])
def test_varlen_conv(ssm, with_h0):
    """The conv window restarts at every sequence start (sequences of 1, 2
    and 3 tokens see fewer than 3 predecessors)."""
    Bt, D, N, L = 2, 70, 16, 320
    x = make_inputs(Bt, D, N, L, seed=82, in_dtype="bf16", with_z=False)
    cuts = [0, 1, 3, 6, 7, 15, 16, 18, 63, 64, 65, 66, 130, 320]
    h0 = _h0(len(cuts) - 1, Bt, D, N, 83) if with_h0 else None
    _run(ssm, x, cuts, h0, conv=_conv(D, 84))


@pytest.mark.parametrize("nt", ["1", "2", "4"])
def test_varlen_lanes_per_channel(ssm, nt, monkeypatch):
    monkeypatch.setenv("SSM_FWD_NT", nt)
    x = make_inputs(1, 50, 12, 256, seed=85, in_dtype="bf16")
    cuts = [0, 3, 40, 41, 128, 200, 256]
    _run(ssm, x, cuts, _h0(len(cuts) - 1, 1, 50, 12, 86), conv=_conv(50, 87, K=3))


@pytest.mark.parametrize("nseg", ["2", "5"])
def test_varlen_segmented(ssm, nseg, monkeypatch):
    """Segments of the two-pass plan: a sequence start inside a segment cuts
    the carried state off; sequences span segment edges."""
    monkeypatch.setenv("SSM_FWD_NSEG", nseg)
    L = 64 * 40
    x = make_inputs(1, 40, 16, L, seed=88, in_dtype="bf16")
    cuts = [0, 100, 640, 641, 1280, 1900, 1901, 2500, L]
    _run(ssm, x, cuts, _h0(len(cuts) - 1, 1, 40, 16, 89), conv=_conv(40, 90))
    _run(ssm, x, [0, 1000, L])
    xf = make_inputs(1, 24, 16, L, seed=91, in_dtype="f32")
    _run(ssm, xf, cuts)


def test_varlen_packed_recipe(ssm):
    """The packed workload's length mix on a short row: many sequences."""
    L = 64 * 64
    cu = packed_seqlens(L, seed=92, lo=16, hi=512)
    x = make_inputs(1, 64, 16, L, seed=92, in_dtype="bf16")
    _run(ssm, x, cu)


def test_varlen_all_empty_and_single(ssm):
    x = make_inputs(1, 16, 16, 64, seed=93, in_dtype="bf16", h0=True)
    _run(ssm, x, [0, 64], x.h0[None])
    _run(ssm, x, [0, 0, 0, 64, 64], _h0(4, 1, 16, 16, 94))


def test_varlen_bad_starts_reported(ssm):
    """Starts out of order or not ending at L: the call runs (no access
    outside the buffers) and the workspace status says SSM_ERR_SEQLENS."""
    x = make_inputs(1, 16, 16, 128, seed=95, in_dtype="bf16")
    a = device_args(x)
    shape = ssm.make_shape(1, 16, 16, 128, ssm.SSM_BF16, ssm.SSM_F32)
    ws = torch.empty(ssm.ssm_scan_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    for cu in ([0, 70, 50, 128], [0, 64, 127], [1, 64, 128], [0, 64, 200]):
        cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
        ssm.ssm_scan_fwd_varlen(a["u"], cu_d, a["delta_raw"], a["A"], a["B"], a["C"],
                                out_dtype=torch.float32, workspace=ws)
        assert ssm.ssm_get_status(ws) == ssm.SSM_ERR_SEQLENS, cu
    # and a good call afterwards clears it
    cu_d = torch.tensor([0, 64, 128], dtype=torch.int32, device="cuda")
    ssm.ssm_scan_fwd_varlen(a["u"], cu_d, a["delta_raw"], a["A"], a["B"], a["C"],
                            out_dtype=torch.float32, workspace=ws)
    assert ssm.ssm_get_status(ws) == ssm.SSM_OK
