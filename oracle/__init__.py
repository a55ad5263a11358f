"""fp64 CPU oracle for the selective scan -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and it imports nothing from the product.

The arithmetic lives in ``ssm_oracle.c`` (plain C, fp64, one loop per
definition); this module only builds that file with gcc, loads it with ctypes
and converts numpy arrays to contiguous float64.

Every function here is pinned by tests outside of itself (see
``tests/test_oracle_pins.py``): the LTI convolution view of "Mamba: How
Selective State Spaces Achieve 5x Faster Inference Than Transformers"
(section "State space models before Mamba: HiPPO and S4") and "Mamba
Architecture Explained" (section "How State Space Models Work"), closed forms,
the remember/forget limits of "State Space Models (SSMs) & Mamba" (section
"The Magic of Selective Scan"), and finite differences for the backward.
The packed-sequence form (``scan_fwd_varlen``) is pinned against the batched
scan with one sequence per batch row, and by the independence of sequences;
the bidirectional form (``scan_fwd_bidir``) against its materialised upper-
and lower-triangular time-varying kernels.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_HDR = os.path.join(_HERE, "ssm_oracle.h")
_LIB = os.path.join(_HERE, "libssmoracle.so")
_lock = threading.Lock()
_lib = None

# -O3 without -ffast-math: exp/log1p keep their libm semantics.  No
# -march=native: the built library travels to hosts with other CPUs.
CFLAGS = ["-O3", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into libssmoracle.so (in place) if stale."""
    stale = force or not os.path.exists(_LIB) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def bind(lib):
    """Declare the C functions' argument types on a loaded oracle library."""
    P = ctypes.c_void_p
    I = ctypes.c_int64
    lib.oracle_softplus.argtypes = [ctypes.c_double]
    lib.oracle_softplus.restype = ctypes.c_double
    lib.oracle_conv_silu.argtypes = [I, I, I, I, P, P, P, P]
    lib.oracle_conv_silu.restype = None
    lib.oracle_conv_silu_bwd.argtypes = [I, I, I, I, P, P, P, P, P, P, P]
    lib.oracle_conv_silu_bwd.restype = None
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_scan_fwd.argtypes = [I, I, I, I] + [P] * 11
    lib.oracle_scan_fwd.restype = None
    lib.oracle_scan_step.argtypes = [I, I, I] + [P] * 10
    lib.oracle_scan_step.restype = None
    lib.oracle_scan_bwd.argtypes = [I, I, I, I] + [P] * 20
    lib.oracle_scan_bwd.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(ctypes.CDLL(build()))
    return _lib


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def softplus(x: float) -> float:
    return _load().oracle_softplus(float(x))


def silu(x: float) -> float:
    return _load().oracle_silu(float(x))


def conv_silu(x, conv_w, conv_b=None):
    """Causal depthwise convolution of width K = conv_w.shape[1] with left
    zero padding, then SiLU: u[b,d,t] = silu(conv_b[d] + sum_k conv_w[d,k] *
    x[b,d,t-(K-1)+k]).  x (Bt,D,L) -> u (Bt,D,L)."""
    x, conv_w = _f64(x), _f64(conv_w)
    conv_b = _f64(conv_b)
    Bt, D, L = x.shape
    K = conv_w.shape[1]
    assert conv_w.shape == (D, K)
    u = np.empty((Bt, D, L), np.float64)
    _load().oracle_conv_silu(Bt, D, L, K, _ptr(x), _ptr(conv_w), _ptr(conv_b), _ptr(u))
    return u


def scan_fwd_conv(x, conv_w, conv_b, delta_raw, A, Bm, Cm, Dv=None, z=None, delta_bias=None,
                  h0=None):
    """The scan fed by the block's conv prologue: scan_fwd(conv_silu(x), ...)."""
    return scan_fwd(conv_silu(x, conv_w, conv_b), delta_raw, A, Bm, Cm, Dv, z, delta_bias, h0)


def conv_silu_bwd(x, conv_w, conv_b, du):
    """Reverse mode of conv_silu given du = dLoss/du: returns (dx, dconv_w,
    dconv_b) (dconv_b None when conv_b is None)."""
    x, conv_w, du = _f64(x), _f64(conv_w), _f64(du)
    conv_b = _f64(conv_b)
    Bt, D, L = x.shape
    K = conv_w.shape[1]
    assert conv_w.shape == (D, K) and du.shape == (Bt, D, L)
    dx = np.empty((Bt, D, L), np.float64)
    dw = np.empty((D, K), np.float64)
    db = np.empty((D,), np.float64) if conv_b is not None else None
    _load().oracle_conv_silu_bwd(Bt, D, L, K, _ptr(x), _ptr(conv_w), _ptr(conv_b), _ptr(du),
                                 _ptr(dx), _ptr(dw), _ptr(db))
    return dx, dw, db


def scan_bwd_conv(x, conv_w, conv_b, delta_raw, A, Bm, Cm, dy, Dv=None, z=None,
                  delta_bias=None, h0=None, dhL=None):
    """Reverse mode of scan_fwd_conv: scan_bwd on u = conv_silu(x), then the
    prologue's reverse mode on its du.  Returns scan_bwd's dict with du
    replaced by dx, plus dconv_w and dconv_b."""
    u = conv_silu(x, conv_w, conv_b)
    out = scan_bwd(u, delta_raw, A, Bm, Cm, dy, Dv, z, delta_bias, h0, dhL)
    dx, dw, db = conv_silu_bwd(x, conv_w, conv_b, out.pop("du"))
    out["dx"] = dx
    out["dconv_w"] = dw
    out["dconv_b"] = db
    return out


def scan_fwd_varlen(u, delta_raw, A, Bm, Cm, cu_seqlens, Dv=None, z=None, delta_bias=None,
                    h0=None, conv_w=None, conv_b=None):
    """Packed sequences ("Mamba Architecture Explained", section "Problem 3:
    Ecosystem maturity": several sequences packed into one row): every batch
    row holds nseq = len(cu_seqlens) - 1 sequences, sequence s at tokens
    [cu_seqlens[s], cu_seqlens[s+1]).  Each is an independent sequence: its
    state starts at h0[s] (zeros when h0 is None), its conv window (conv_w
    given) starts from zeros, and its final state is returned.  Shapes as in
    scan_fwd, with h0 and the returned final states (nseq, Bt, D, N); an empty
    sequence's final state is its initial state."""
    u, delta_raw, Bm, Cm, z = map(_f64, (u, delta_raw, Bm, Cm, z))
    cu = [int(v) for v in cu_seqlens]
    Bt, D, L = u.shape
    N = A.shape[1]
    nseq = len(cu) - 1
    assert nseq >= 1 and cu[0] == 0 and cu[-1] == L
    assert all(cu[s] <= cu[s + 1] for s in range(nseq))
    h0 = None if h0 is None else _f64(h0)
    assert h0 is None or h0.shape == (nseq, Bt, D, N)
    y = np.empty((Bt, D, L), np.float64)
    hL = np.empty((nseq, Bt, D, N), np.float64)
    for s in range(nseq):
        lo, hi = cu[s], cu[s + 1]
        hs = None if h0 is None else h0[s]
        if hi == lo:
            hL[s] = 0.0 if hs is None else hs
            continue
        us = u[:, :, lo:hi]
        if conv_w is not None:
            us = conv_silu(us, conv_w, conv_b)
        ys, hL[s] = scan_fwd(us, delta_raw[:, :, lo:hi], A, Bm[:, :, lo:hi], Cm[:, :, lo:hi], Dv,
                             None if z is None else z[:, :, lo:hi], delta_bias, hs)
        y[:, :, lo:hi] = ys
    return y, hL


def scan_bwd_varlen(u, delta_raw, A, Bm, Cm, dy, cu_seqlens, Dv=None, z=None, delta_bias=None,
                    h0=None, dhL=None):
    """Reverse mode of scan_fwd_varlen (without the conv prologue): each
    packed sequence's own reverse mode (scan_bwd on its token range, from its
    h0[s] and with its dhL[s]); the per-token gradients land in the sequence's
    range and the per-channel ones (dA, dD, ddelta_bias) are summed over the
    sequences.  dh0 is (nseq, Bt, D, N); an empty sequence passes dhL[s]
    straight to dh0[s]."""
    u, delta_raw, Bm, Cm, dy, z = map(_f64, (u, delta_raw, Bm, Cm, dy, z))
    cu = [int(v) for v in cu_seqlens]
    Bt, D, L = u.shape
    N = A.shape[1]
    nseq = len(cu) - 1
    assert nseq >= 1 and cu[0] == 0 and cu[-1] == L
    assert all(cu[s] <= cu[s + 1] for s in range(nseq))
    h0 = None if h0 is None else _f64(h0)
    dhL = None if dhL is None else _f64(dhL)
    out = {
        "du": np.zeros((Bt, D, L)), "ddelta_raw": np.zeros((Bt, D, L)),
        "dA": np.zeros((D, N)), "dB": np.zeros((Bt, N, L)), "dC": np.zeros((Bt, N, L)),
        "dD": np.zeros((D,)), "dz": np.zeros((Bt, D, L)), "ddelta_bias": np.zeros((D,)),
        "dh0": np.zeros((nseq, Bt, D, N)),
    }
    for s in range(nseq):
        lo, hi = cu[s], cu[s + 1]
        if hi == lo:
            if dhL is not None:
                out["dh0"][s] = dhL[s]
            continue
        cut = lambda a: None if a is None else a[:, :, lo:hi]
        g = scan_bwd(cut(u), cut(delta_raw), A, cut(Bm), cut(Cm), cut(dy), Dv, cut(z),
                     delta_bias, None if h0 is None else h0[s], None if dhL is None else dhL[s])
        for k in ("du", "ddelta_raw", "dB", "dC", "dz"):
            out[k][:, :, lo:hi] = g[k]
        for k in ("dA", "dD", "ddelta_bias"):
            out[k] += g[k]
        out["dh0"][s] = g["dh0"]
    if z is None:
        out["dz"][:] = 0.0
    return out


def scan_fwd_bidir(u, z, fwd, rev):
    """Bidirectional scan ("Mamba Architecture Explained", section "Frequently
    Asked Questions": bidirectional SSM variants beside the causal scan): the
    sum of two selective scans over the same input u and gate z, one over
    t = 0 .. L-1 and one over t = L-1 .. 0.  `fwd` and `rev` are dicts with
    each direction's delta_raw, A, Bm, Cm and optional Dv, delta_bias, h0.
    Returns (y, hL of the left-to-right scan (state after token L-1), hL of the
    right-to-left scan (state after token 0))."""
    def one(d, flip):
        f = (lambda a: None if a is None else np.ascontiguousarray(np.asarray(a)[..., ::-1])) \
            if flip else (lambda a: a)
        y, h = scan_fwd(f(u), f(d["delta_raw"]), d["A"], f(d["Bm"]), f(d["Cm"]), d.get("Dv"),
                        f(z), d.get("delta_bias"), d.get("h0"))
        return f(y), h
    yf, hf = one(fwd, False)
    yr, hr = one(rev, True)
    return yf + yr, hf, hr


def scan_bwd_bidir(u, z, fwd, rev, dy, dhL=None, dhL_r=None):
    """Reverse mode of scan_fwd_bidir: each direction's reverse mode (the
    right-to-left one on mirrored tensors, mirrored back); du and dz are the
    sums of the two directions'.  Returns (shared, grads_fwd, grads_rev):
    shared = {du, dz}; each grads dict holds ddelta_raw, dA, dB, dC, dD,
    ddelta_bias, dh0 for its direction."""
    def one(d, flip, dh):
        f = (lambda a: None if a is None else np.ascontiguousarray(np.asarray(a)[..., ::-1])) \
            if flip else (lambda a: a)
        g = scan_bwd(f(u), f(d["delta_raw"]), d["A"], f(d["Bm"]), f(d["Cm"]), f(dy), d.get("Dv"),
                     f(z), d.get("delta_bias"), d.get("h0"), dh)
        for k in ("du", "ddelta_raw", "dB", "dC", "dz"):
            g[k] = f(g[k])
        return g
    gf = one(fwd, False, dhL)
    gr = one(rev, True, dhL_r)
    shared = {"du": gf.pop("du") + gr.pop("du"), "dz": gf.pop("dz") + gr.pop("dz")}
    return shared, gf, gr


def scan_fwd(u, delta_raw, A, Bm, Cm, Dv=None, z=None, delta_bias=None, h0=None):
    """Forward selective scan.  Shapes: u, delta_raw, z (Bt,D,L); Bm, Cm (Bt,N,L);
    A (D,N); Dv, delta_bias (D); h0 (Bt,D,N).  Returns (y (Bt,D,L), hL (Bt,D,N))."""
    u, delta_raw, A, Bm, Cm = map(_f64, (u, delta_raw, A, Bm, Cm))
    Dv, z, delta_bias, h0 = map(_f64, (Dv, z, delta_bias, h0))
    Bt, D, L = u.shape
    N = A.shape[1]
    assert delta_raw.shape == u.shape and A.shape == (D, N)
    assert Bm.shape == (Bt, N, L) and Cm.shape == (Bt, N, L)
    assert z is None or z.shape == u.shape
    assert h0 is None or h0.shape == (Bt, D, N)
    y = np.empty((Bt, D, L), np.float64)
    hL = np.empty((Bt, D, N), np.float64)
    _load().oracle_scan_fwd(Bt, D, N, L, _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(Bm),
                            _ptr(Cm), _ptr(Dv), _ptr(z), _ptr(delta_bias), _ptr(h0),
                            _ptr(y), _ptr(hL))
    return y, hL


def scan_step(u, delta_raw, A, Bm, Cm, state, Dv=None, z=None, delta_bias=None):
    """One decode step.  u, delta_raw, z (Bt,D); Bm, Cm (Bt,N); state (Bt,D,N).
    Returns (y (Bt,D), new_state (Bt,D,N)); the input state is not modified."""
    u, delta_raw, A, Bm, Cm = map(_f64, (u, delta_raw, A, Bm, Cm))
    Dv, z, delta_bias = map(_f64, (Dv, z, delta_bias))
    st = np.array(state, dtype=np.float64, copy=True, order="C")
    Bt, D = u.shape
    N = A.shape[1]
    assert st.shape == (Bt, D, N) and Bm.shape == (Bt, N) and Cm.shape == (Bt, N)
    y = np.empty((Bt, D), np.float64)
    _load().oracle_scan_step(Bt, D, N, _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(Bm),
                             _ptr(Cm), _ptr(Dv), _ptr(z), _ptr(delta_bias), _ptr(st),
                             _ptr(y))
    return y, st


def scan_bwd(u, delta_raw, A, Bm, Cm, dy, Dv=None, z=None, delta_bias=None, h0=None,
             dhL=None):
    """Reverse mode of scan_fwd.  Returns a dict with du, ddelta_raw, dA, dB, dC,
    dD, dz, ddelta_bias, dh0 (all float64)."""
    u, delta_raw, A, Bm, Cm, dy = map(_f64, (u, delta_raw, A, Bm, Cm, dy))
    Dv, z, delta_bias, h0, dhL = map(_f64, (Dv, z, delta_bias, h0, dhL))
    Bt, D, L = u.shape
    N = A.shape[1]
    out = {
        "du": np.empty((Bt, D, L)), "ddelta_raw": np.empty((Bt, D, L)),
        "dA": np.empty((D, N)), "dB": np.empty((Bt, N, L)), "dC": np.empty((Bt, N, L)),
        "dD": np.empty((D,)), "dz": np.empty((Bt, D, L)), "ddelta_bias": np.empty((D,)),
        "dh0": np.empty((Bt, D, N)),
    }
    _load().oracle_scan_bwd(Bt, D, N, L, _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(Bm),
                            _ptr(Cm), _ptr(Dv), _ptr(z), _ptr(delta_bias), _ptr(h0),
                            _ptr(dy), _ptr(dhL), _ptr(out["du"]), _ptr(out["ddelta_raw"]),
                            _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
                            _ptr(out["dD"]), _ptr(out["dz"]), _ptr(out["ddelta_bias"]),
                            _ptr(out["dh0"]))
    return out
