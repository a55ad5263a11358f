"""What fp32 arithmetic of the method's own formula reaches, and so why the
kernel's fp32-input path carries a compensated state.

The parity bar for fp32 inputs is 1e-5 in the metric of tests/parity.py.
This file evaluates the oracle's loop with every operation rounded to fp32
in the oracle's order (softplus, exp(delta A), the state update, the
read-out sum, the gate; the reverse mode likewise), in numpy float32, on the
long fp32 cases the GPU tests run, and compares it with the fp64 oracle:

* on the cases with the workloads' recipe for Delta (and larger Delta) it
  stays under 1e-5, so 1e-5 is attainable there and the GPU is held to it;
* in the long-memory regime (Delta three and six e-folds below the recipe,
  10,240 tokens) it misses 1e-5 by an order of magnitude: exp(delta A)
  rounded to fp32 keeps only the relative accuracy of 1, not that of the
  small forgetting rate 1 - exp(delta A), and the rounding of a state that
  barely changes piles up over the ~1/(delta |A|) tokens it remembers.  The
  kernel's fp32 path therefore carries the state as two floats and the
  decay as 2^x - 1, which meets 1e-5 there as well (tests/test_delta_regimes.py).

The inputs are drawn exactly as the GPU tests draw them (same shapes, seeds
and shifts of the bias).
"""
import numpy as np
import pytest

import oracle
from scan_inputs import make_inputs
from tests.parity import TOL, rel_err

F = np.float32


def _softplus32(x):
    x = x.astype(F)
    return np.where(x > 0, x + np.log1p(np.exp(-np.abs(x))), np.log1p(np.exp(np.minimum(x, 0))))


def _silu32(z):
    z = z.astype(F)
    return z * (F(1) / (F(1) + np.exp(-z)))


def _fwd32(u, dr, A, Bm, Cm, Dv, z, bias, h0):
    """oracle.scan_fwd with every operation in float32, rows vectorised."""
    Bt, D, L = u.shape
    N = A.shape[1]
    y = np.empty((Bt, D, L), F)
    hL = np.empty((Bt, D, N), F)
    bias = np.zeros(D, F) if bias is None else bias.astype(F)
    Dv = np.zeros(D, F) if Dv is None else Dv.astype(F)
    A = A.astype(F)
    for b in range(Bt):
        h = np.zeros((D, N), F) if h0 is None else h0[b].astype(F).copy()
        for t in range(L):
            ut = u[b, :, t].astype(F)
            delta = _softplus32(dr[b, :, t].astype(F) + bias)
            ys = np.zeros(D, F)
            for n in range(N):
                a = np.exp(delta * A[:, n])
                h[:, n] = a * h[:, n] + (delta * F(Bm[b, n, t])) * ut
                ys = ys + F(Cm[b, n, t]) * h[:, n]
            ys = ys + Dv * ut
            y[b, :, t] = ys * _silu32(z[b, :, t]) if z is not None else ys
        hL[b] = h
    return y, hL


def _bwd32(u, dr, A, Bm, Cm, dy, Dv, z, bias, h0, dhL):
    """oracle.scan_bwd with every operation in float32, rows vectorised."""
    Bt, D, L = u.shape
    N = A.shape[1]
    A = A.astype(F)
    bias = np.zeros(D, F) if bias is None else bias.astype(F)
    Dv = np.zeros(D, F) if Dv is None else Dv.astype(F)
    out = {k: np.zeros(s, F) for k, s in
           (("du", (Bt, D, L)), ("ddelta_raw", (Bt, D, L)), ("dz", (Bt, D, L)), ("dA", (D, N)),
            ("dB", (Bt, N, L)), ("dC", (Bt, N, L)), ("dD", (D,)), ("ddelta_bias", (D,)),
            ("dh0", (Bt, D, N)))}
    for b in range(Bt):
        hs = np.zeros((L + 1, D, N), F)
        as_ = np.zeros((L, D, N), F)
        dl = np.zeros((L, D), F)
        ys = np.zeros((L, D), F)
        if h0 is not None:
            hs[0] = h0[b].astype(F)
        for t in range(L):
            ut = u[b, :, t].astype(F)
            delta = _softplus32(dr[b, :, t].astype(F) + bias)
            dl[t] = delta
            acc = np.zeros(D, F)
            for n in range(N):
                a = np.exp(delta * A[:, n])
                as_[t, :, n] = a
                hs[t + 1, :, n] = a * hs[t, :, n] + (delta * F(Bm[b, n, t])) * ut
                acc = acc + F(Cm[b, n, t]) * hs[t + 1, :, n]
            ys[t] = acc + Dv * ut
        lam = np.zeros((D, N), F) if dhL is None else dhL[b].astype(F).copy()
        for t in range(L - 1, -1, -1):
            ut = u[b, :, t].astype(F)
            zt = z[b, :, t].astype(F) if z is not None else None
            gate = _silu32(zt) if z is not None else np.ones(D, F)
            g = dy[b, :, t].astype(F) * gate
            if z is not None:
                s = F(1) / (F(1) + np.exp(-zt))
                out["dz"][b, :, t] = dy[b, :, t].astype(F) * ys[t] * s * (F(1) + zt * (F(1) - s))
            out["dD"] += g * ut
            delta = dl[t]
            du_t = g * Dv
            ddelta = np.zeros(D, F)
            for n in range(N):
                Cv, Bv = F(Cm[b, n, t]), F(Bm[b, n, t])
                lam[:, n] = lam[:, n] + g * Cv
                a, hprev = as_[t, :, n], hs[t, :, n]
                out["dC"][b, n, t] += np.sum(g * hs[t + 1, :, n], dtype=F)
                out["dB"][b, n, t] += np.sum(lam[:, n] * delta * ut, dtype=F)
                du_t = du_t + lam[:, n] * delta * Bv
                ddelta = ddelta + lam[:, n] * (A[:, n] * a * hprev + Bv * ut)
                out["dA"][:, n] += lam[:, n] * delta * a * hprev
                lam[:, n] = lam[:, n] * a
            out["du"][b, :, t] = du_t
            ddr = ddelta * (F(1) / (F(1) + np.exp(-(dr[b, :, t].astype(F) + bias))))
            out["ddelta_raw"][b, :, t] = ddr
            out["ddelta_bias"] += ddr
        out["dh0"][b] = lam
    return out


def _fwd_err(x):
    y, hL = _fwd32(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    yo, ho = oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    return max(rel_err(y, yo), rel_err(hL, ho))


def _shifted(Bt, D, N, L, seed, shift, h0=True):
    x = make_inputs(Bt, D, N, L, seed=seed, in_dtype="f32", h0=h0)
    x.delta_bias = (x.delta_bias + np.float32(shift)).astype(np.float32)
    return x


# builders of the plain fp32 evaluation's error, one per long fp32 case
def _segmented_long(L, shift):
    return lambda: _fwd_err(_shifted(1, 40, 16, L, 13, shift))


def _small_delta(efolds):
    return lambda: _fwd_err(_shifted(1, 40, 16, 64 * 160, 63, -efolds))


def _varlen_segmented():
    L = 64 * 40
    x = make_inputs(1, 24, 16, L, seed=91, in_dtype="f32")
    cuts = [0, 100, 640, 641, 1280, 1900, 1901, 2500, L]
    ys, hs = [], []
    for s0, s1 in zip(cuts[:-1], cuts[1:]):
        sl = slice(s0, s1)
        y, h = _fwd32(x.u[..., sl], x.delta_raw[..., sl], x.A, x.Bm[..., sl], x.Cm[..., sl],
                      x.Dv, x.z[..., sl], x.delta_bias, None)
        ys.append(y)
        hs.append(h)
    yo, ho = oracle.scan_fwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, cuts, x.Dv, x.z,
                                    x.delta_bias)
    return max(rel_err(np.concatenate(ys, -1), yo), rel_err(np.stack(hs), ho))


def _bidir_long():
    L = 64 * 40
    xf = make_inputs(1, 24, 16, L, seed=114, in_dtype="f32")
    xr = make_inputs(1, 24, 16, L, seed=115, in_dtype="f32")
    fl = lambda a: None if a is None else np.ascontiguousarray(a[..., ::-1])
    yf, hf = _fwd32(xf.u, xf.delta_raw, xf.A, xf.Bm, xf.Cm, xf.Dv, xf.z, xf.delta_bias, xf.h0)
    yr, hr = _fwd32(fl(xf.u), fl(xr.delta_raw), xr.A, fl(xr.Bm), fl(xr.Cm), xr.Dv, fl(xf.z),
                    xr.delta_bias, xr.h0)
    y = yf + yr[..., ::-1]
    host = lambda x: dict(delta_raw=x.delta_raw, A=x.A, Bm=x.Bm, Cm=x.Cm, Dv=x.Dv,
                          delta_bias=x.delta_bias, h0=x.h0)
    yo, ho, hro = oracle.scan_fwd_bidir(xf.u, xf.z, host(xf), host(xr))
    return max(rel_err(y, yo), rel_err(hf, ho), rel_err(hr, hro))


def _bwd_long():
    x = make_inputs(1, 40, 16, 1000, seed=300 + 40 + 1000, in_dtype="f32", dy=True, h0=True)
    Bt, D, N, L = x.shape
    dhL = np.random.default_rng(7).standard_normal((Bt, D, N)).astype(np.float32)
    g = _bwd32(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z, x.delta_bias, x.h0, dhL)
    o = oracle.scan_bwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z, x.delta_bias, x.h0,
                        dhL)
    return max(rel_err(g[k], o[k]) for k in o)


# every long fp32 case of the GPU tests: True where the plain fp32
# evaluation misses 1e-5 (the long-memory regime)
CASES = {
    "segmented_long_segments L=10240 bias+3": (_segmented_long(64 * 160, 3.0), False),
    "segmented_long_segments L=4096 bias+0": (_segmented_long(64 * 64, 0.0), False),
    "small_delta_long_memory e^-3": (_small_delta(3.0), True),
    "small_delta_long_memory e^-6": (_small_delta(6.0), True),
    "varlen_segmented L=2560": (_varlen_segmented, False),
    "bidir_long_sequence L=2560": (_bidir_long, False),
    "bwd 1000 tokens": (_bwd_long, False),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_plain_fp32_evaluation(name):
    fn, misses = CASES[name]
    err = fn()
    if misses:
        assert err > 5 * TOL["f32"], "%s: plain fp32 error %.3e" % (name, err)
    else:
        assert err < 0.5 * TOL["f32"], "%s: plain fp32 error %.3e" % (name, err)
