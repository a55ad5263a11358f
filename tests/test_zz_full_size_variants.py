"""Full-size sampled parity of the forward variants, each at the size and in
the launch configuration the bench times: the conv prologue (Mamba-1.4B shape,
width 4), packed sequences (Mamba-1.4B channels, one 65,536-token row of 17
sequences, four segments) and the bidirectional scan (Mamba-1.4B shape, two
parameter sets), and the backward of the packed row, of the bidirectional
scan and of the million-token sequence (segmented plan).  Sampled channels
of every batch row are compared with the oracle (channels are independent).  The smaller parity cases of each variant
live in test_conv_parity.py, test_varlen_parity.py and test_bidir_parity.py;
this file is collected after them.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from scan_inputs import device_inputs, packed_seqlens
from tests.gpu_util import load_ssm, rows_to_host, to_dev
from tests.parity import TOL, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssm():
    return load_ssm()


def _conv_params(D, K, seed):
    rng = np.random.default_rng(seed)
    return ((0.5 * rng.standard_normal((D, K))).astype(np.float32),
            (0.1 * rng.standard_normal(D)).astype(np.float32))


def test_conv_full_size_sampled(ssm):
    """The bench's conv workload (Mamba-1.4B shape, width 4) on sampled
    channels of every batch row, in the launch configuration the bench times."""
    w = bench.WORKLOADS["mamba1p4b_conv_fwd"]
    Bt, D, N, L, K = w["Bt"], w["D"], w["N"], w["L"], w["conv"]
    a = device_inputs(Bt, D, N, L, seed=w["seed"], in_dtype="bf16")
    cw, cb = _conv_params(D, K, 7)
    y, hL = ssm.ssm_scan_fwd_conv(a["u"], to_dev(cw, torch.float32), to_dev(cb, torch.float32),
                                  a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["Dv"], a["z"],
                                  a["delta_bias"], None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1235)
    for b in range(Bt):
        ds = np.sort(rng.choice(D, size=6, replace=False))
        ds[0], ds[-1] = 0, D - 1
        host = lambda t: rows_to_host(t, [b], ds)
        yo, ho = oracle.scan_fwd_conv(host(a["u"]), cw[ds], cb[ds], host(a["delta_raw"]),
                                      a["A"][ds].cpu().numpy(), a["Bm"][[b]].float().cpu().numpy(),
                                      a["Cm"][[b]].float().cpu().numpy(), a["Dv"][ds].cpu().numpy(),
                                      host(a["z"]), a["delta_bias"][ds].cpu().numpy(), None)
        assert_close(y[[b]][:, ds].cpu().numpy(), yo, TOL["bf16"], "y b=%d" % b)
        assert_close(hL[[b]][:, ds].cpu().numpy(), ho, TOL["bf16"], "hL b=%d" % b)
    del a, y, hL
    torch.cuda.empty_cache()


def test_varlen_full_size_sampled(ssm):
    """The bench's packed workload (Mamba-1.4B channels, one 65,536-token row
    of 17 sequences, four segments) on sampled channels."""
    w = bench.WORKLOADS["packed_mamba1p4b_fwd"]
    Bt, D, N, L = w["Bt"], w["D"], w["N"], w["L"]
    a = device_inputs(Bt, D, N, L, seed=w["seed"], in_dtype="bf16")
    cu = packed_seqlens(L, seed=w["seed"])
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    y, hL = ssm.ssm_scan_fwd_varlen(a["u"], cu_d, a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["Dv"],
                                    a["z"], a["delta_bias"], None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ds = np.sort(np.random.default_rng(1236).choice(D, size=6, replace=False))
    ds[0], ds[-1] = 0, D - 1
    host = lambda t: rows_to_host(t, [0], ds)
    yo, ho = oracle.scan_fwd_varlen(host(a["u"]), host(a["delta_raw"]), a["A"][ds].cpu().numpy(),
                                    a["Bm"][[0]].float().cpu().numpy(),
                                    a["Cm"][[0]].float().cpu().numpy(), cu, a["Dv"][ds].cpu().numpy(),
                                    host(a["z"]), a["delta_bias"][ds].cpu().numpy())
    assert_close(y[[0]][:, ds].cpu().numpy(), yo, TOL["bf16"], "y")
    assert_close(hL[:, [0]][:, :, ds].cpu().numpy(), ho, TOL["bf16"], "hL")
    del a, y, hL
    torch.cuda.empty_cache()


def test_bidir_full_size_sampled(ssm):
    """The bench's bidirectional workload (Mamba-1.4B shape, two parameter
    sets) on sampled channels of every batch row."""
    w = bench.WORKLOADS["bidir_mamba1p4b_fwd"]
    Bt, D, N, L = w["Bt"], w["D"], w["N"], w["L"]
    a = device_inputs(Bt, D, N, L, seed=w["seed"], in_dtype="bf16")
    r = device_inputs(Bt, D, N, L, seed=w["seed"] + 1, in_dtype="bf16")

    def dev_dir(x):
        return dict(delta_raw=x["delta_raw"], A=x["A"], B=x["Bm"], C=x["Cm"], D=x["Dv"],
                    delta_bias=x["delta_bias"])
    y, hL, hL_r = ssm.ssm_scan_fwd_bidir(a["u"], a["z"], dev_dir(a), dev_dir(r),
                                         out_dtype=torch.float32)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1237)
    for b in range(Bt):
        ds = np.sort(rng.choice(D, size=6, replace=False))
        ds[0], ds[-1] = 0, D - 1
        host = lambda t: rows_to_host(t, [b], ds)

        def host_dir(x):
            return dict(delta_raw=host(x["delta_raw"]), A=x["A"][ds].cpu().numpy(),
                        Bm=x["Bm"][[b]].float().cpu().numpy(), Cm=x["Cm"][[b]].float().cpu().numpy(),
                        Dv=x["Dv"][ds].cpu().numpy(), delta_bias=x["delta_bias"][ds].cpu().numpy())
        yo, ho, hro = oracle.scan_fwd_bidir(host(a["u"]), host(a["z"]), host_dir(a), host_dir(r))
        assert_close(y[[b]][:, ds].cpu().numpy(), yo, TOL["bf16"], "y b=%d" % b)
        assert_close(hL[[b]][:, ds].cpu().numpy(), ho, TOL["bf16"], "hL b=%d" % b)
        assert_close(hL_r[[b]][:, ds].cpu().numpy(), hro, TOL["bf16"], "hL_r b=%d" % b)
    del a, r, y, hL, hL_r
    torch.cuda.empty_cache()


def test_packed_backward_long_row(ssm):
    """The packed backward over the packed workload's row (65,536 tokens cut
    by the bench's length recipe) on 256 channels: every output against the
    oracle (dB and dC are sums over all channels, so no channel sampling)."""
    from scan_inputs import make_inputs
    w = bench.WORKLOADS["packed_mamba1p4b_fwdbwd"]
    L = w["L"]
    cu = packed_seqlens(L, seed=w["seed"])
    x = make_inputs(1, 256, 16, L, seed=w["seed"], in_dtype="bf16", dy=True)
    nseq = len(cu) - 1
    rng = np.random.default_rng(71)
    h0 = rng.standard_normal((nseq, 1, 256, 16)).astype(np.float32)
    dhL = rng.standard_normal((nseq, 1, 256, 16)).astype(np.float32)
    t, f32 = torch.bfloat16, torch.float32
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    g = ssm.ssm_scan_bwd_varlen(to_dev(x.u, t), cu_d, to_dev(x.delta_raw, t), to_dev(x.A, f32),
                                to_dev(x.Bm, t), to_dev(x.Cm, t), to_dev(x.dy, t), to_dev(x.Dv, f32),
                                to_dev(x.z, t), to_dev(x.delta_bias, f32), to_dev(h0, f32),
                                to_dev(dhL, f32), out_dtype=f32)
    torch.cuda.synchronize()
    o = oracle.scan_bwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, cu, x.Dv, x.z,
                               x.delta_bias, h0, dhL)
    for k in o:
        assert_close(g[k].float().cpu().numpy(), o[k], TOL["bf16"], k)


def test_bidir_backward_long_rows(ssm):
    """The bidirectional backward at the Mamba-1.4B sequence length (4,096
    tokens) on 128 channels, both directions' parameters, every output
    against the oracle."""
    from scan_inputs import make_inputs
    Bt, D, N, L = 1, 128, 16, 4096
    xf = make_inputs(Bt, D, N, L, seed=72, in_dtype="bf16", dy=True, h0=True)
    xr = make_inputs(Bt, D, N, L, seed=73, in_dtype="bf16", h0=True)
    rng = np.random.default_rng(74)
    dhL = rng.standard_normal((Bt, D, N)).astype(np.float32)
    dhL_r = rng.standard_normal((Bt, D, N)).astype(np.float32)
    t, f32 = torch.bfloat16, torch.float32
    dev = lambda x: dict(delta_raw=to_dev(x.delta_raw, t), A=to_dev(x.A, f32), B=to_dev(x.Bm, t),
                         C=to_dev(x.Cm, t), D=to_dev(x.Dv, f32),
                         delta_bias=to_dev(x.delta_bias, f32), h0=to_dev(x.h0, f32))
    host = lambda x: dict(delta_raw=x.delta_raw, A=x.A, Bm=x.Bm, Cm=x.Cm, Dv=x.Dv,
                          delta_bias=x.delta_bias, h0=x.h0)
    shared, gf, gr = ssm.ssm_scan_bwd_bidir(to_dev(xf.u, t), to_dev(xf.z, t), dev(xf), dev(xr),
                                            to_dev(xf.dy, t), to_dev(dhL, f32), to_dev(dhL_r, f32),
                                            out_dtype=f32)
    torch.cuda.synchronize()
    so, of, orr = oracle.scan_bwd_bidir(xf.u, xf.z, host(xf), host(xr), xf.dy, dhL, dhL_r)
    for k in so:
        assert_close(shared[k].cpu().numpy(), so[k], TOL["bf16"], k)
    for tag, gg, oo in (("fwd", gf, of), ("rev", gr, orr)):
        for k in oo:
            assert_close(gg[k].cpu().numpy(), oo[k], TOL["bf16"], tag + "." + k)


def test_million_length_backward_sampled(ssm):
    """The reverse mode of the million-token sequence (batch 1, D 1536, N 16,
    L 2^20; the planner's segmented plan) against the oracle on sampled
    channels: every token's du, ddelta_raw and dz, and dA, dD, ddelta_bias and
    dh0 of those channels.  (dB and dC sum over all 1,536 channels; the
    segmented plan's dB and dC are compared in full at smaller sizes.)"""
    w = bench.WORKLOADS["million_fwd"]
    Bt, D, N, L = w["Bt"], w["D"], w["N"], w["L"]
    a = device_inputs(Bt, D, N, L, seed=w["seed"], in_dtype="bf16", dy=True)
    g = ssm.ssm_scan_bwd(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["dy"], a["Dv"],
                         a["z"], a["delta_bias"], None, None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ds = np.array([0, 517, 1103, D - 1])
    bi = [0]
    host = lambda t: rows_to_host(t, bi, ds)
    o = oracle.scan_bwd(host(a["u"]), host(a["delta_raw"]), a["A"][ds].cpu().numpy(),
                        a["Bm"].float().cpu().numpy(), a["Cm"].float().cpu().numpy(),
                        host(a["dy"]), a["Dv"][ds].cpu().numpy(), host(a["z"]),
                        a["delta_bias"][ds].cpu().numpy(), None, None)
    tol = TOL["bf16"]
    for k in ("du", "ddelta_raw", "dz", "dh0"):
        assert_close(g[k][bi][:, ds].cpu().numpy(), o[k], tol, "million backward " + k)
    for k in ("dA", "dD", "ddelta_bias"):
        assert_close(g[k][ds].cpu().numpy(), o[k], tol, "million backward " + k)
    del a, g
    torch.cuda.empty_cache()
