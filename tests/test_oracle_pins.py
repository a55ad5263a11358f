"""Pins for the fp64 oracle, against facts fixed outside of the oracle itself.

Each test names the passage or the mathematics that fixes the expected value:
  * the LTI special case -- with Delta, B, C constant in time a state space
    model is a causal convolution ("Mamba: How Selective State Spaces Achieve
    5x Faster Inference Than Transformers", section "State space models before
    Mamba: HiPPO and S4"; "Mamba Architecture Explained", section "How State
    Space Models Work"), checked by brute force and by a library FFT;
  * the materialised time-varying kernel y = M u (the scan unrolled), which
    pins which token's B, C and Delta enter each term;
  * closed forms (L = 1, geometric series), the remember / forget limits of
    Delta ("State Space Models (SSMs) & Mamba", section "The Magic of
    Selective Scan: Content-Aware Memory");
  * library routines for softplus and the sigmoid;
  * central finite differences and the adjoint identity for the backward.
A plausible slip in the oracle (a dropped term, a sign, an off-by-one in t, B
and C swapped, the gate applied before the D term) fails at least one of them.
"""
import numpy as np
import pytest
from scipy.signal import fftconvolve
from scipy.special import expit

import oracle
from scan_inputs import make_inputs

RTOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _softplus_lib(x):
    return np.logaddexp(0.0, x)


def _silu_lib(z):
    return z * expit(z)


def test_softplus_and_silu_match_library():
    xs = np.concatenate([np.linspace(-60, 60, 241), [-745.0, -30.5, 0.0, 1e-8, 700.0]])
    for x in xs:
        assert oracle.softplus(x) == pytest.approx(_softplus_lib(x), rel=1e-14, abs=1e-300)
        assert oracle.silu(x) == pytest.approx(_silu_lib(x), rel=1e-14, abs=1e-300)


def _lti_problem(rng, Bt, D, N, L, with_h0):
    """Delta, B, C constant in t (per channel / batch), u and z varying."""
    u = rng.standard_normal((Bt, D, L))
    z = rng.standard_normal((Bt, D, L))
    draw = np.repeat(rng.standard_normal((Bt, D, 1)), L, axis=2)
    bias = rng.uniform(-4, 0, D)
    A = -rng.uniform(0.1, 3.0, (D, N))
    Bc = rng.standard_normal((Bt, N))
    Cc = rng.standard_normal((Bt, N))
    Bm = np.repeat(Bc[:, :, None], L, axis=2)
    Cm = np.repeat(Cc[:, :, None], L, axis=2)
    Dv = rng.standard_normal(D)
    h0 = rng.standard_normal((Bt, D, N)) if with_h0 else None
    return u, z, draw, bias, A, Bc, Cc, Bm, Cm, Dv, h0


@pytest.mark.parametrize("with_h0", [False, True])
def test_lti_equals_bruteforce_causal_convolution(with_h0):
    """Constant Delta, B, C: y = (K * u + D u) silu(z), K_k = sum_n C_n e^{delta A_n k} delta B_n,
    plus the free response sum_n C_n e^{delta A_n (t+1)} h0_n."""
    rng = _rng(11)
    Bt, D, N, L = 2, 3, 4, 37
    u, z, draw, bias, A, Bc, Cc, Bm, Cm, Dv, h0 = _lti_problem(rng, Bt, D, N, L, with_h0)
    y, hL = oracle.scan_fwd(u, draw, A, Bm, Cm, Dv=Dv, z=z, delta_bias=bias, h0=h0)
    for b in range(Bt):
        for d in range(D):
            delta = _softplus_lib(draw[b, d, 0] + bias[d])
            lam = np.exp(delta * A[d])                     # (N,)
            k = np.arange(L)
            K = (Cc[b] * delta * Bc[b] * lam[None, :] ** k[:, None]).sum(1)
            ys = np.array([sum(K[j] * u[b, d, t - j] for j in range(t + 1)) for t in range(L)])
            if with_h0:
                ys += (Cc[b] * h0[b, d] * lam[None, :] ** (k[:, None] + 1)).sum(1)
            ys += Dv[d] * u[b, d]
            np.testing.assert_allclose(y[b, d], ys * _silu_lib(z[b, d]), rtol=1e-11, atol=1e-12)
            # final state: h_L = sum_s lam^{L-1-s} delta B u_s (+ lam^L h0)
            hexp = (lam[None, :] ** (L - 1 - k)[:, None] * delta * Bc[b] * u[b, d][:, None]).sum(0)
            if with_h0:
                hexp += lam ** L * h0[b, d]
            np.testing.assert_allclose(hL[b, d], hexp, rtol=1e-11, atol=1e-12)


def test_lti_long_sequence_equals_fft_convolution():
    """Same view at L = 4096 through a library FFT convolution (no gate, no D)."""
    rng = _rng(12)
    Bt, D, N, L = 1, 2, 16, 4096
    u, z, draw, bias, A, Bc, Cc, Bm, Cm, Dv, _ = _lti_problem(rng, Bt, D, N, L, False)
    y, _ = oracle.scan_fwd(u, draw, A, Bm, Cm, delta_bias=bias)
    for d in range(D):
        delta = _softplus_lib(draw[0, d, 0] + bias[d])
        lam = np.exp(delta * A[d])
        k = np.arange(L)
        K = (Cc[0] * delta * Bc[0] * np.exp(np.outer(k, np.log(lam)))).sum(1)
        ref = fftconvolve(u[0, d], K)[:L]
        scale = np.sqrt(np.mean(ref ** 2))
        np.testing.assert_allclose(y[0, d], ref, rtol=0, atol=1e-9 * scale)


def test_time_varying_kernel_materialised():
    """The scan unrolled: ys_t = sum_{s<=t} sum_n C_t[n] exp(A_n (S_t - S_s)) delta_s B_s[n] u_s
    + D u_t with S_t = sum_{r<=t} delta_r.  Pins which token's B, C and Delta enter."""
    rng = _rng(13)
    Bt, D, N, L = 1, 2, 3, 24
    u = rng.standard_normal((Bt, D, L))
    z = rng.standard_normal((Bt, D, L))
    draw = rng.standard_normal((Bt, D, L))
    bias = rng.uniform(-3, 0, D)
    A = -rng.uniform(0.2, 2.0, (D, N))
    Bm = rng.standard_normal((Bt, N, L))
    Cm = rng.standard_normal((Bt, N, L))
    Dv = rng.standard_normal(D)
    y, _ = oracle.scan_fwd(u, draw, A, Bm, Cm, Dv=Dv, z=z, delta_bias=bias)
    for d in range(D):
        delta = _softplus_lib(draw[0, d] + bias[d])
        S = np.cumsum(delta)
        M = np.zeros((L, L))
        for t in range(L):
            for s in range(t + 1):
                M[t, s] = np.sum(Cm[0, :, t] * np.exp(A[d] * (S[t] - S[s])) * delta[s] * Bm[0, :, s])
        ys = M @ u[0, d] + Dv[d] * u[0, d]
        np.testing.assert_allclose(y[0, d], ys * _silu_lib(z[0, d]), rtol=1e-10, atol=1e-12)


def test_single_token_closed_form():
    """L = 1: h_1 = e^{delta A} h0 + delta B u, y = (C.h_1 + D u) silu(z)."""
    rng = _rng(14)
    D, N = 5, 4
    u, draw, z = rng.standard_normal((3, 1, D, 1))
    A = -rng.uniform(0.5, 4, (D, N))
    Bm, Cm = rng.standard_normal((2, 1, N, 1))
    Dv, bias = rng.standard_normal(D), rng.uniform(-5, 1, D)
    h0 = rng.standard_normal((1, D, N))
    y, hL = oracle.scan_fwd(u, draw, A, Bm, Cm, Dv=Dv, z=z, delta_bias=bias, h0=h0)
    delta = np.logaddexp(0.0, draw[0, :, 0] + bias)
    h1 = np.exp(delta[:, None] * A) * h0[0] + delta[:, None] * Bm[0, :, 0] * u[0, :, 0][:, None]
    ref = (h1 @ Cm[0, :, 0] + Dv * u[0, :, 0]) * _silu_lib(z[0, :, 0])
    np.testing.assert_allclose(y[0, :, 0], ref, rtol=1e-13)
    np.testing.assert_allclose(hL[0], h1, rtol=1e-13)


def test_constant_input_geometric_series():
    """N = 1, u = 1, constant delta, B, C, h0 = 0: h_t = delta B (1 - a^{t+1}) / (1 - a)."""
    L = 200
    a_coef, Bv, Cv, draw = -0.7, 1.3, -0.4, 0.25
    u = np.ones((1, 1, L))
    y, hL = oracle.scan_fwd(u, np.full((1, 1, L), draw), np.array([[a_coef]]),
                            np.full((1, 1, L), Bv), np.full((1, 1, L), Cv))
    delta = np.log1p(np.exp(draw))
    a = np.exp(delta * a_coef)
    t = np.arange(L)
    h = delta * Bv * (1 - a ** (t + 1)) / (1 - a)
    np.testing.assert_allclose(y[0, 0], Cv * h, rtol=1e-12)
    np.testing.assert_allclose(hL[0, 0, 0], h[-1], rtol=1e-12)


def test_delta_to_zero_remembers_state():
    """Delta_raw + bias = -200: delta ~ e^-200, the state is kept ("selectively
    remember") and y_t = (C_t . h0 + D u_t) silu(z_t)."""
    rng = _rng(15)
    Bt, D, N, L = 1, 3, 4, 50
    u, z = rng.standard_normal((2, Bt, D, L))
    draw = np.full((Bt, D, L), -200.0)
    A = -rng.uniform(0.5, 16, (D, N))
    Bm, Cm = rng.standard_normal((2, Bt, N, L))
    Dv = rng.standard_normal(D)
    h0 = rng.standard_normal((Bt, D, N))
    y, hL = oracle.scan_fwd(u, draw, A, Bm, Cm, Dv=Dv, z=z, delta_bias=np.zeros(D), h0=h0)
    np.testing.assert_allclose(hL, h0, rtol=1e-80, atol=0)
    ref = (np.einsum("dn,nt->dt", h0[0], Cm[0]) + Dv[:, None] * u[0]) * _silu_lib(z[0])
    np.testing.assert_allclose(y[0], ref, rtol=1e-12)


def test_large_delta_forgets_state():
    """delta |A| >> 1: the past decays away ("selectively forget") and
    h_t = delta_t B_t u_t exactly to double precision."""
    rng = _rng(16)
    Bt, D, N, L = 1, 2, 3, 30
    u = rng.standard_normal((Bt, D, L))
    draw = 60.0 + rng.uniform(0, 1, (Bt, D, L))
    A = -rng.uniform(1.0, 5.0, (D, N))
    Bm, Cm = rng.standard_normal((2, Bt, N, L))
    h0 = rng.standard_normal((Bt, D, N))
    y, hL = oracle.scan_fwd(u, draw, A, Bm, Cm, h0=h0)
    delta = draw[0]                                   # softplus(x) = x + O(e^-60)
    ref = np.einsum("nt,nt->t", Cm[0], Bm[0])[None, :] * delta * u[0]
    np.testing.assert_allclose(y[0], ref, rtol=1e-12)
    np.testing.assert_allclose(hL[0], delta[:, -1:] * Bm[0, :, -1][None, :] * u[0, :, -1:],
                               rtol=1e-12)


def _small_random(seed, Bt=2, D=3, N=4, L=40, h0=True):
    x = make_inputs(Bt, D, N, L, seed=seed, in_dtype="f32", h0=h0, dy=True)
    return x


def test_split_and_carry_reproduces_unsplit():
    x = _small_random(3)
    y, hL = oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    for L1 in (1, 17, 39):
        ya, ha = oracle.scan_fwd(x.u[..., :L1], x.delta_raw[..., :L1], x.A, x.Bm[..., :L1],
                                 x.Cm[..., :L1], x.Dv, x.z[..., :L1], x.delta_bias, x.h0)
        yb, hb = oracle.scan_fwd(x.u[..., L1:], x.delta_raw[..., L1:], x.A, x.Bm[..., L1:],
                                 x.Cm[..., L1:], x.Dv, x.z[..., L1:], x.delta_bias, ha)
        np.testing.assert_allclose(np.concatenate([ya, yb], -1), y, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(hb, hL, rtol=1e-12, atol=1e-14)


def test_linear_in_u_and_causal():
    x = _small_random(4, h0=False)
    rng = _rng(17)
    u2 = rng.standard_normal(x.u.shape)
    f = lambda uu: oracle.scan_fwd(uu, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias)[0]
    np.testing.assert_allclose(f(2.0 * x.u - 3.0 * u2), 2.0 * f(x.u) - 3.0 * f(u2),
                               rtol=1e-10, atol=1e-12)
    t0 = 23
    up = x.u.copy()
    up[..., t0] += 5.0
    y0, y1 = f(x.u), f(up)
    np.testing.assert_array_equal(y0[..., :t0], y1[..., :t0])
    assert np.all(np.abs(y0[..., t0] - y1[..., t0]) > 0)


def test_channels_are_independent():
    x = _small_random(5)
    y, hL = oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    d = 1
    y1, h1 = oracle.scan_fwd(x.u[:, d:d + 1], x.delta_raw[:, d:d + 1], x.A[d:d + 1], x.Bm,
                             x.Cm, x.Dv[d:d + 1], x.z[:, d:d + 1], x.delta_bias[d:d + 1],
                             x.h0[:, d:d + 1])
    np.testing.assert_array_equal(y1[:, 0], y[:, d])
    np.testing.assert_array_equal(h1[:, 0], hL[:, d])


def test_decode_steps_reproduce_forward():
    """Recurrent inference ("State Space Models (SSMs) & Mamba", section "The Payoff"):
    L single-token steps from h0 equal the forward scan over L tokens."""
    x = _small_random(6, L=12)
    y, hL = oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    st = x.h0.copy()
    for t in range(x.u.shape[-1]):
        yt, st = oracle.scan_step(x.u[..., t], x.delta_raw[..., t], x.A, x.Bm[..., t],
                                  x.Cm[..., t], st, x.Dv, x.z[..., t], x.delta_bias)
        np.testing.assert_allclose(yt, y[..., t], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(st, hL, rtol=1e-13)


def test_decode_step_closed_form():
    rng = _rng(18)
    Bt, D, N = 3, 4, 5
    u, draw, z = rng.standard_normal((3, Bt, D))
    A = -rng.uniform(0.5, 4, (D, N))
    Bm, Cm = rng.standard_normal((2, Bt, N))
    Dv, bias = rng.standard_normal(D), rng.uniform(-5, 1, D)
    st = rng.standard_normal((Bt, D, N))
    y, st2 = oracle.scan_step(u, draw, A, Bm, Cm, st, Dv, z, bias)
    delta = np.logaddexp(0.0, draw + bias[None, :])
    h = np.exp(delta[..., None] * A[None]) * st + delta[..., None] * Bm[:, None, :] * u[..., None]
    np.testing.assert_allclose(st2, h, rtol=1e-13)
    ref = (np.einsum("bdn,bn->bd", h, Cm) + Dv[None] * u) * _silu_lib(z)
    np.testing.assert_allclose(y, ref, rtol=1e-13)


# ---------------------------------------------------------------- backward ---

def _loss(x, dy, dhL, **over):
    args = dict(u=x.u, delta_raw=x.delta_raw, A=x.A, Bm=x.Bm, Cm=x.Cm, Dv=x.Dv, z=x.z,
                delta_bias=x.delta_bias, h0=x.h0)
    args.update(over)
    y, hL = oracle.scan_fwd(**args)
    return float(np.sum(dy * y) + np.sum(dhL * hL))


_BWD_NAMES = [("u", "du"), ("delta_raw", "ddelta_raw"), ("A", "dA"), ("Bm", "dB"),
              ("Cm", "dC"), ("Dv", "dD"), ("z", "dz"), ("delta_bias", "ddelta_bias"),
              ("h0", "dh0")]


def test_backward_matches_central_finite_differences():
    x = make_inputs(1, 2, 2, 5, seed=7, in_dtype="f32", h0=True, dy=True)
    for k in ("u", "delta_raw", "A", "Bm", "Cm", "Dv", "z", "delta_bias", "h0", "dy"):
        setattr(x, k, getattr(x, k).astype(np.float64))
    rng = _rng(19)
    dy = x.dy
    dhL = rng.standard_normal(x.h0.shape)
    g = oracle.scan_bwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, dy, Dv=x.Dv, z=x.z,
                        delta_bias=x.delta_bias, h0=x.h0, dhL=dhL)
    eps = 1e-6
    for name, gname in _BWD_NAMES:
        base = getattr(x, name)
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            p = base.copy(); p[idx] += eps
            m = base.copy(); m[idx] -= eps
            fd[idx] = (_loss(x, dy, dhL, **{name: p}) - _loss(x, dy, dhL, **{name: m})) / (2 * eps)
        np.testing.assert_allclose(g[gname], fd, rtol=2e-6, atol=2e-8, err_msg=gname)


def test_backward_adjoint_identity():
    """<dy, J v> = <J^T dy, v> for a random direction v over all inputs (J by
    a central difference along v)."""
    x = make_inputs(2, 3, 4, 16, seed=8, in_dtype="f32", h0=True, dy=True)
    rng = _rng(20)
    names = [n for n, _ in _BWD_NAMES]
    base = {n: getattr(x, n).astype(np.float64) for n in names}
    v = {n: rng.standard_normal(base[n].shape) for n in names}
    dy = x.dy.astype(np.float64)
    dhL = np.zeros(x.h0.shape)
    g = oracle.scan_bwd(base["u"], base["delta_raw"], base["A"], base["Bm"], base["Cm"], dy,
                        Dv=base["Dv"], z=base["z"], delta_bias=base["delta_bias"],
                        h0=base["h0"], dhL=dhL)
    eps = 1e-5
    plus = {n: base[n] + eps * v[n] for n in names}
    minus = {n: base[n] - eps * v[n] for n in names}
    yp, _ = oracle.scan_fwd(**plus)
    ym, _ = oracle.scan_fwd(**minus)
    lhs = np.sum(dy * (yp - ym)) / (2 * eps)
    rhs = sum(np.sum(g[gn] * v[n]) for n, gn in _BWD_NAMES)
    assert lhs == pytest.approx(rhs, rel=1e-7)


def test_backward_closed_form_dD():
    """dD = sum_{b,t} dy silu(z) u, a direct consequence of y = (... + D u) silu(z)."""
    x = make_inputs(2, 3, 4, 16, seed=9, in_dtype="f32", h0=False, dy=True)
    g = oracle.scan_bwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, Dv=x.Dv, z=x.z,
                        delta_bias=x.delta_bias)
    z = x.z.astype(np.float64)
    ref = np.sum(x.dy.astype(np.float64) * _silu_lib(z) * x.u, axis=(0, 2))
    np.testing.assert_allclose(g["dD"], ref, rtol=1e-12)


# ----- the block's conv prologue ("Mamba Architecture Explained", section
# "The Architecture in Practice": Conv1D then SiLU before the selective SSM)

def _silu(v):
    return v * expit(v)


@pytest.mark.parametrize("K", [1, 2, 4])
def test_conv_silu_matches_library_convolution(K):
    """Causal depthwise convolution = numpy's full convolution with the
    reversed kernel, cut to the first L outputs (left zero padding)."""
    rng = np.random.default_rng(40 + K)
    Bt, D, L = 2, 5, 37
    x = rng.standard_normal((Bt, D, L))
    w = rng.standard_normal((D, K))
    b = rng.standard_normal(D)
    u = oracle.conv_silu(x, w, b)
    ref = np.empty_like(u)
    for bb in range(Bt):
        for d in range(D):
            ref[bb, d] = _silu(b[d] + np.convolve(x[bb, d], w[d, ::-1])[:L])
    np.testing.assert_allclose(u, ref, rtol=1e-13, atol=1e-13)


def test_conv_silu_impulse_and_bias():
    """An impulse at t = 0 reads the kernel out backwards over the first K
    tokens (w[K-1] at t = 0 ... w[0] at t = K-1) and only the bias after;
    without a bias the output there is silu(0) = 0."""
    K, L = 4, 9
    w = np.array([[0.5, -1.0, 2.0, 0.25]])
    x = np.zeros((1, 1, L))
    x[0, 0, 0] = 1.0
    b = np.array([0.3])
    u = oracle.conv_silu(x, w, b)[0, 0]
    for t in range(L):
        pre = 0.3 + (w[0, K - 1 - t] if t < K else 0.0)
        assert u[t] == pytest.approx(_silu(pre), abs=1e-15)
    u0 = oracle.conv_silu(x, w, None)[0, 0]
    assert np.all(u0[K:] == 0.0)


def test_scan_fwd_conv_is_scan_of_conv_output():
    """The prologue feeds u: scanning conv_silu(x) equals scan_fwd_conv."""
    rng = np.random.default_rng(44)
    x = make_inputs(2, 6, 4, 30, seed=44, in_dtype="f32", h0=True)
    w = rng.standard_normal((6, 4))
    b = rng.standard_normal(6)
    y1, h1 = oracle.scan_fwd_conv(x.u, w, b, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z,
                                  x.delta_bias, x.h0)
    u = oracle.conv_silu(x.u, w, b)
    y2, h2 = oracle.scan_fwd(u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(h1, h2)


# ---- packed sequences ("Mamba Architecture Explained", section "Problem 3:
# Ecosystem maturity": sequence packing)

def _pack(rows):
    """Concatenate per-sequence arrays (Bt, X, Ls) along the token axis."""
    return np.concatenate(rows, axis=2)


@pytest.mark.parametrize("conv", [False, True])
def test_varlen_equal_lengths_match_batched_rows(conv):
    """Four equal-length sequences packed into one row give what the batched
    scan gives with each sequence as its own batch row (a different loop of
    the oracle: the batch dimension, not slicing)."""
    S, D, N, Ls = 4, 5, 4, 13
    x = make_inputs(S, D, N, Ls, seed=50, in_dtype="f32", h0=True)
    rng = np.random.default_rng(51)
    w = rng.standard_normal((D, 3)) if conv else None
    b = rng.standard_normal(D) if conv else None
    rows = lambda a: _pack([a[s:s + 1] for s in range(S)])
    cu = [Ls * s for s in range(S + 1)]
    y, hL = oracle.scan_fwd_varlen(rows(x.u), rows(x.delta_raw), x.A, rows(x.Bm), rows(x.Cm), cu,
                                   x.Dv, rows(x.z), x.delta_bias, x.h0[:, None], w, b)
    u = oracle.conv_silu(x.u, w, b) if conv else x.u
    yb, hb = oracle.scan_fwd(u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    np.testing.assert_allclose(y[0], np.concatenate(list(yb), axis=1), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hL[:, 0], hb, rtol=1e-13, atol=1e-13)


def test_varlen_one_sequence_is_the_plain_scan():
    x = make_inputs(2, 4, 4, 29, seed=52, in_dtype="f32", h0=True)
    y, hL = oracle.scan_fwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, [0, 29], x.Dv, x.z,
                                   x.delta_bias, x.h0[None])
    y2, h2 = oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(hL[0], h2)


def test_varlen_sequences_do_not_see_each_other():
    """Changing one sequence's inputs changes no other sequence's outputs;
    empty sequences return their initial state and change nothing."""
    x = make_inputs(1, 3, 4, 40, seed=53, in_dtype="f32")
    cu = [0, 0, 11, 11, 25, 40, 40]
    h0 = np.random.default_rng(54).standard_normal((6, 1, 3, 4))
    y, hL = oracle.scan_fwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, cu, x.Dv, x.z,
                                   x.delta_bias, h0)
    u2 = x.u.copy()
    u2[:, :, 11:25] += 1.0
    y2, h2 = oracle.scan_fwd_varlen(u2, x.delta_raw, x.A, x.Bm, x.Cm, cu, x.Dv, x.z,
                                    x.delta_bias, h0)
    assert np.array_equal(y[:, :, :11], y2[:, :, :11]) and np.array_equal(y[:, :, 25:], y2[:, :, 25:])
    assert not np.allclose(y[:, :, 11:25], y2[:, :, 11:25])
    for s in (0, 1, 4, 5):
        np.testing.assert_array_equal(hL[s], h2[s])
    for s in (0, 2, 5):                   # empty sequences
        np.testing.assert_array_equal(hL[s], h0[s])
    # a sequence boundary is a reset: zero B*u in front of sequence 3 leaves it unchanged
    y3, _ = oracle.scan_fwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, [0, 25, 40], x.Dv, x.z,
                                   x.delta_bias, None)
    y4, _ = oracle.scan_fwd(x.u[:, :, 25:], x.delta_raw[:, :, 25:], x.A, x.Bm[:, :, 25:],
                            x.Cm[:, :, 25:], x.Dv, x.z[:, :, 25:], x.delta_bias, None)
    np.testing.assert_array_equal(y3[:, :, 25:], y4)


# ---- bidirectional scan ("Mamba Architecture Explained", section "Frequently
# Asked Questions": bidirectional SSM variants)

def test_bidirectional_materialised_kernels():
    """y = silu(z) * ((M_f + M_r) u + (D_f + D_r) u): M_f lower triangular
    with prefix sums of delta (left-to-right scan), M_r upper triangular with
    suffix sums P_t = sum_{r>=t} delta_r of the other direction's delta,
    M_r[t,s] = sum_n C_t[n] exp(A_n (P_t - P_s)) delta_s B_s[n] for s >= t."""
    rng = _rng(60)
    Bt, D, N, L = 1, 2, 3, 21
    u = rng.standard_normal((Bt, D, L))
    z = rng.standard_normal((Bt, D, L))

    def params():
        return dict(delta_raw=rng.standard_normal((Bt, D, L)), A=-rng.uniform(0.2, 2.0, (D, N)),
                    Bm=rng.standard_normal((Bt, N, L)), Cm=rng.standard_normal((Bt, N, L)),
                    Dv=rng.standard_normal(D), delta_bias=rng.uniform(-3, 0, D))
    f, r = params(), params()
    y, _, _ = oracle.scan_fwd_bidir(u, z, f, r)
    for d in range(D):
        M = np.zeros((L, L))
        df = _softplus_lib(f["delta_raw"][0, d] + f["delta_bias"][d])
        S = np.cumsum(df)
        for t in range(L):
            for s in range(t + 1):
                M[t, s] += np.sum(f["Cm"][0, :, t] * np.exp(f["A"][d] * (S[t] - S[s])) * df[s]
                                  * f["Bm"][0, :, s])
        dr = _softplus_lib(r["delta_raw"][0, d] + r["delta_bias"][d])
        P = np.cumsum(dr[::-1])[::-1]
        for t in range(L):
            for s in range(t, L):
                M[t, s] += np.sum(r["Cm"][0, :, t] * np.exp(r["A"][d] * (P[t] - P[s])) * dr[s]
                                  * r["Bm"][0, :, s])
        ys = M @ u[0, d] + (f["Dv"][d] + r["Dv"][d]) * u[0, d]
        np.testing.assert_allclose(y[0, d], ys * _silu_lib(z[0, d]), rtol=1e-10, atol=1e-12)


def test_bidirectional_final_states_and_mirror():
    """The right-to-left scan's final state is the state after token 0, and
    mirroring every input swaps the two directions."""
    x = make_inputs(2, 3, 4, 17, seed=61, in_dtype="f32", h0=True)
    f = dict(delta_raw=x.delta_raw, A=x.A, Bm=x.Bm, Cm=x.Cm, Dv=x.Dv, delta_bias=x.delta_bias, h0=x.h0)
    x2 = make_inputs(2, 3, 4, 17, seed=62, in_dtype="f32", h0=True)
    r = dict(delta_raw=x2.delta_raw, A=x2.A, Bm=x2.Bm, Cm=x2.Cm, Dv=x2.Dv, delta_bias=x2.delta_bias,
             h0=x2.h0)
    y, hf, hr = oracle.scan_fwd_bidir(x.u, x.z, f, r)
    # the state after token 0 of the right-to-left scan: one step from its
    # state after token 1, by the single-token closed form
    _, h1 = oracle.scan_fwd(x.u[..., ::-1][..., :16].copy(), x2.delta_raw[..., ::-1][..., :16].copy(),
                            x2.A, x2.Bm[..., ::-1][..., :16].copy(), x2.Cm[..., ::-1][..., :16].copy(),
                            x2.Dv, None, x2.delta_bias, x2.h0)
    f64 = lambda a: np.asarray(a, np.float64)
    delta0 = _softplus_lib(f64(x2.delta_raw[..., 0]) + f64(x2.delta_bias)[None, :])
    step = np.exp(delta0[..., None] * f64(x2.A)[None]) * h1 + \
        (delta0 * f64(x.u[..., 0]))[..., None] * f64(x2.Bm)[:, None, :, 0]
    np.testing.assert_allclose(hr, step, rtol=1e-12, atol=1e-12)
    flip = lambda a: np.ascontiguousarray(a[..., ::-1])
    fm = {k: (flip(v) if k in ("delta_raw", "Bm", "Cm") else v) for k, v in f.items()}
    rm = {k: (flip(v) if k in ("delta_raw", "Bm", "Cm") else v) for k, v in r.items()}
    ym, hfm, hrm = oracle.scan_fwd_bidir(flip(x.u), flip(x.z), rm, fm)
    np.testing.assert_allclose(flip(ym), y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hfm, hr, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hrm, hf, rtol=1e-12, atol=1e-12)


def test_varlen_backward_equal_lengths_match_batched_rows():
    """Packed equal-length sequences: the reverse mode equals the batched
    reverse mode with one sequence per batch row (the channel sums dA, dD,
    ddelta_bias match the sums over batch rows)."""
    S, D, N, Ls = 3, 4, 3, 9
    x = make_inputs(S, D, N, Ls, seed=63, in_dtype="f32", h0=True, dy=True)
    dhL = _rng(64).standard_normal((S, D, N))
    rows = lambda a: _pack([a[s:s + 1] for s in range(S)])
    cu = [Ls * s for s in range(S + 1)]
    g = oracle.scan_bwd_varlen(rows(x.u), rows(x.delta_raw), x.A, rows(x.Bm), rows(x.Cm),
                               rows(x.dy), cu, x.Dv, rows(x.z), x.delta_bias, x.h0[:, None],
                               dhL[:, None])
    r = oracle.scan_bwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z, x.delta_bias, x.h0, dhL)
    for k in ("du", "ddelta_raw", "dB", "dC", "dz"):
        np.testing.assert_allclose(g[k][0], np.concatenate(list(r[k]), axis=1), rtol=1e-12,
                                   atol=1e-13, err_msg=k)
    for k in ("dA", "dD", "ddelta_bias"):
        np.testing.assert_allclose(g[k], r[k], rtol=1e-12, atol=1e-13, err_msg=k)
    np.testing.assert_allclose(g["dh0"][:, 0], r["dh0"], rtol=1e-12, atol=1e-13)


def test_varlen_backward_adjoint_identity():
    """<dy, J v> + <dhL, J_h v> = <J^T (dy, dhL), v> through the packed forward,
    with empty sequences and a one-token sequence among them."""
    x = make_inputs(1, 3, 4, 20, seed=65, in_dtype="f32", dy=True)
    cu = [0, 0, 1, 9, 9, 20]
    nseq = len(cu) - 1
    rng = _rng(66)
    names = ["u", "delta_raw", "A", "Bm", "Cm", "Dv", "z", "delta_bias"]
    base = {n: getattr(x, n).astype(np.float64) for n in names}
    base["h0"] = rng.standard_normal((nseq, 1, 3, 4))
    v = {n: rng.standard_normal(base[n].shape) for n in base}
    dy = x.dy.astype(np.float64)
    dhL = rng.standard_normal((nseq, 1, 3, 4))

    def fwd(p):
        return oracle.scan_fwd_varlen(p["u"], p["delta_raw"], p["A"], p["Bm"], p["Cm"], cu,
                                      p["Dv"], p["z"], p["delta_bias"], p["h0"])
    g = oracle.scan_bwd_varlen(base["u"], base["delta_raw"], base["A"], base["Bm"], base["Cm"],
                               dy, cu, base["Dv"], base["z"], base["delta_bias"], base["h0"], dhL)
    eps = 1e-5
    yp, hp = fwd({n: base[n] + eps * v[n] for n in base})
    ym, hm = fwd({n: base[n] - eps * v[n] for n in base})
    lhs = (np.sum(dy * (yp - ym)) + np.sum(dhL * (hp - hm))) / (2 * eps)
    gn = dict(u="du", delta_raw="ddelta_raw", A="dA", Bm="dB", Cm="dC", Dv="dD", z="dz",
              delta_bias="ddelta_bias", h0="dh0")
    rhs = sum(np.sum(g[gn[n]] * v[n]) for n in base)
    assert lhs == pytest.approx(rhs, rel=1e-7)
    np.testing.assert_array_equal(g["dh0"][0], dhL[0])   # empty sequences pass dhL through
    np.testing.assert_array_equal(g["dh0"][3], dhL[3])


def test_bidirectional_backward_adjoint_identity():
    """<dy, J v> + <dhL, J_f v> + <dhL_r, J_r v> = <J^T (dy, dhL, dhL_r), v>
    over both directions' parameters and the shared u, z."""
    rng = _rng(67)
    Bt, D, N, L = 2, 3, 4, 11
    u = rng.standard_normal((Bt, D, L))
    z = rng.standard_normal((Bt, D, L))

    def params():
        return dict(delta_raw=rng.standard_normal((Bt, D, L)), A=-rng.uniform(0.2, 2.0, (D, N)),
                    Bm=rng.standard_normal((Bt, N, L)), Cm=rng.standard_normal((Bt, N, L)),
                    Dv=rng.standard_normal(D), delta_bias=rng.uniform(-3, 0, D),
                    h0=rng.standard_normal((Bt, D, N)))
    f, r = params(), params()
    dy = rng.standard_normal((Bt, D, L))
    dhL, dhL_r = rng.standard_normal((Bt, D, N)), rng.standard_normal((Bt, D, N))
    vu, vz = rng.standard_normal(u.shape), rng.standard_normal(z.shape)
    vf = {k: rng.standard_normal(np.shape(a)) for k, a in f.items()}
    vr = {k: rng.standard_normal(np.shape(a)) for k, a in r.items()}
    eps = 1e-5

    def at(sign):
        return oracle.scan_fwd_bidir(u + sign * eps * vu, z + sign * eps * vz,
                                     {k: a + sign * eps * vf[k] for k, a in f.items()},
                                     {k: a + sign * eps * vr[k] for k, a in r.items()})
    (yp, hp, hrp), (ym, hm, hrm) = at(1), at(-1)
    lhs = (np.sum(dy * (yp - ym)) + np.sum(dhL * (hp - hm)) + np.sum(dhL_r * (hrp - hrm))) / (2 * eps)
    shared, gf, gr = oracle.scan_bwd_bidir(u, z, f, r, dy, dhL, dhL_r)
    names = dict(delta_raw="ddelta_raw", A="dA", Bm="dB", Cm="dC", Dv="dD",
                 delta_bias="ddelta_bias", h0="dh0")
    rhs = np.sum(shared["du"] * vu) + np.sum(shared["dz"] * vz)
    rhs += sum(np.sum(gf[names[k]] * vf[k]) for k in f) + sum(np.sum(gr[names[k]] * vr[k]) for k in r)
    assert lhs == pytest.approx(rhs, rel=1e-7)


# ----- reverse mode of the conv prologue

def _conv_loss(x, cw, cb, dy, dhL, xin=None, w=None, b=None):
    y, hL = oracle.scan_fwd_conv(x.u if xin is None else xin, cw if w is None else w,
                                 cb if b is None else b, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z,
                                 x.delta_bias, x.h0)
    return float(np.sum(dy * y) + np.sum(dhL * hL))


@pytest.mark.parametrize("K", [1, 2, 4])
def test_conv_backward_matches_central_finite_differences(K):
    """dx, dconv_w and dconv_b of scan_bwd_conv against central differences of
    sum(dy * y) + sum(dhL * hL), y and hL from scan_fwd_conv (the tensor in
    the u slot is the branch input x)."""
    x = make_inputs(2, 2, 3, 7, seed=30 + K, in_dtype="f32", h0=True, dy=True)
    rng = _rng(31 + K)
    cw = rng.standard_normal((2, K)) * 0.7
    cb = rng.standard_normal(2) * 0.3
    dhL = rng.standard_normal(x.h0.shape)
    dy = x.dy.astype(np.float64)
    g = oracle.scan_bwd_conv(x.u, cw, cb, x.delta_raw, x.A, x.Bm, x.Cm, dy, x.Dv, x.z,
                             x.delta_bias, x.h0, dhL)
    eps = 1e-6
    for name, base, gname in (("xin", x.u.astype(np.float64), "dx"), ("w", cw, "dconv_w"),
                              ("b", cb, "dconv_b")):
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            p = base.copy(); p[idx] += eps
            m = base.copy(); m[idx] -= eps
            fd[idx] = (_conv_loss(x, cw, cb, dy, dhL, **{name: p}) -
                       _conv_loss(x, cw, cb, dy, dhL, **{name: m})) / (2 * eps)
        np.testing.assert_allclose(g[gname], fd, rtol=2e-6, atol=2e-8, err_msg=gname)


def test_conv_backward_width_one_is_the_silu_derivative():
    """K = 1, weight 1, no bias: u = silu(x), so dx = du silu'(x) with
    silu'(x) = s + x s (1 - s), s the logistic function, and dconv_w =
    sum du silu'(x) x."""
    rng = _rng(40)
    x = rng.standard_normal((2, 3, 11))
    du = rng.standard_normal((2, 3, 11))
    dx, dw, db = oracle.conv_silu_bwd(x, np.ones((3, 1)), None, du)
    s = expit(x)
    ref = du * (s + x * s * (1.0 - s))
    np.testing.assert_allclose(dx, ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dw[:, 0], np.sum(ref * x, axis=(0, 2)), rtol=1e-12)
    assert db is None


def test_conv_backward_rest_is_the_scan_backward_on_u():
    """Every output besides dx, dconv_w, dconv_b is scan_bwd's on u = conv_silu(x)."""
    x = make_inputs(1, 3, 4, 20, seed=41, in_dtype="f32", h0=True, dy=True)
    cw = _rng(42).standard_normal((3, 4)) * 0.5
    g = oracle.scan_bwd_conv(x.u, cw, None, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z,
                             x.delta_bias, x.h0)
    u = oracle.conv_silu(x.u, cw, None)
    r = oracle.scan_bwd(u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z, x.delta_bias, x.h0)
    for k in ("ddelta_raw", "dA", "dB", "dC", "dD", "dz", "ddelta_bias", "dh0"):
        np.testing.assert_array_equal(g[k], r[k], err_msg=k)
