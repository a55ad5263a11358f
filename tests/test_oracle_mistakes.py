"""Mistakes planted in the oracle, on the CPU, must each fail at least one
pin of tests/test_oracle_pins.py: a dropped term, a wrong sign or index, a
swapped operand.  C mistakes are planted in a copy of ssm_oracle.c built
into a temporary library; mistakes in the Python-level forms (packed
sequences, bidirectional) in a copy of the oracle module's source."""
import ctypes
import inspect
import itertools
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

C_SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")
PY_SRC = oracle.__file__

# (name, text in ssm_oracle.c, replacement)
C_MISTAKES = [
    ("exp sign", "double a = exp(delta * A[n]);", "double a = exp(-delta * A[n]);"),
    ("dropped delta in the input term", "h[n] = a * h[n] + delta * Bv[n * bc_stride] * u;",
     "h[n] = a * h[n] + Bv[n * bc_stride] * u;"),
    ("read-out before the update",
     "        h[n] = a * h[n] + delta * Bv[n * bc_stride] * u;\n        ys += Cv[n * bc_stride] * h[n];",
     "        ys += Cv[n * bc_stride] * h[n];\n        h[n] = a * h[n] + delta * Bv[n * bc_stride] * u;"),
    ("B and C swapped",
     "        h[n] = a * h[n] + delta * Bv[n * bc_stride] * u;\n        ys += Cv[n * bc_stride] * h[n];",
     "        h[n] = a * h[n] + delta * Cv[n * bc_stride] * u;\n        ys += Bv[n * bc_stride] * h[n];"),
    ("dropped D skip", "return ys + Dskip * u;", "return ys;"),
    ("gate before the D skip", "y[row + t] = z ? ys * oracle_silu(z[row + t]) : ys;",
     "y[row + t] = z ? (ys - Dskip * u[row + t]) * oracle_silu(z[row + t]) + Dskip * u[row + t] : ys;"),
    ("dropped delta bias", "double delta = oracle_softplus(dr + bias);",
     "double delta = oracle_softplus(dr);"),
    ("softplus without log1p", "    return log1p(exp(x));\n}", "    return exp(x);\n}"),
    ("h0 ignored", "for (int64_t n = 0; n < N; ++n) h[n] = h0 ? h0[(b * D + d) * N + n] : 0.0;",
     "for (int64_t n = 0; n < N; ++n) h[n] = 0.0;"),
    ("conv window one token late",
     "const int64_t tt = t - (K - 1) + k;\n                    if (tt >= 0) s += ",
     "const int64_t tt = t - K + k;\n                    if (tt >= 0) s += "),
    ("conv taps reversed", "if (tt >= 0) s += conv_w[d * K + k] * x[row + tt];",
     "if (tt >= 0) s += conv_w[d * K + (K - 1 - k)] * x[row + tt];"),
    ("dA sign", "dA[d * N + n] += lam[n] * delta * a * hprev;",
     "dA[d * N + n] -= lam[n] * delta * a * hprev;"),
    ("dB from g instead of lambda", "dB[(b * N + n) * L + t] += lam[n] * delta * u[row + t];",
     "dB[(b * N + n) * L + t] += g * Cv * delta * u[row + t];"),
    ("dz formula", "dz[row + t] = dy[row + t] * ys[t] * s * (1.0 + zt * (1.0 - s));",
     "dz[row + t] = dy[row + t] * ys[t] * s * (1.0 + zt * s);"),
    ("conv backward: silu' without its second term",
     "dpre[t] = du[row + t] * sg * (1.0 + p * (1.0 - sg));", "dpre[t] = du[row + t] * sg;"),
    ("conv backward: dx taps not mirrored", "const int64_t tt = t + (K - 1) - k;",
     "const int64_t tt = t + k;"),
    ("conv backward: dconv_w against the unshifted input",
     "if (tt >= 0) dconv_w[d * K + k] += dpre[t] * x[row + tt];",
     "if (tt >= 0) dconv_w[d * K + k] += dpre[t] * x[row + t];"),
    ("conv backward: dconv_b dropped", "if (dconv_b) dconv_b[d] += dpre[t];", ""),
    ("dh0 without the last decay", "lam[n] *= a; /* becomes a_t lambda_t, the carry into t-1 */",
     "if (t > 0) lam[n] *= a;"),
]

# (name, text in oracle/__init__.py, replacement)
PY_MISTAKES = [
    ("packed sequence one token too long",
     "        lo, hi = cu[s], cu[s + 1]\n        hs = None if h0 is None else h0[s]\n",
     "        lo, hi = cu[s], min(cu[s + 1] + 1, L)\n        hs = None if h0 is None else h0[s]\n"),
    ("packed h0 of the first sequence", "        hs = None if h0 is None else h0[s]\n",
     "        hs = None if h0 is None else h0[0]\n"),
    ("packed conv window across starts",
     "        us = u[:, :, lo:hi]\n        if conv_w is not None:\n            us = conv_silu(us, conv_w, conv_b)\n",
     "        us = (u if conv_w is None else conv_silu(u, conv_w, conv_b))[:, :, lo:hi]\n"),
    ("right-to-left output not mirrored back", "        return f(y), h\n", "        return y, h\n"),
    ("right-to-left scan with the left-to-right parameters", "    yr, hr = one(rev, True)\n",
     "    yr, hr = one(fwd, True)\n"),
    ("packed backward: channel gradients of the last sequence only", "            out[k] += g[k]\n",
     "            out[k] = g[k]\n"),
    ("packed backward: dh0 into the first sequence", "        out[\"dh0\"][s] = g[\"dh0\"]\n",
     "        out[\"dh0\"][0] = g[\"dh0\"]\n"),
    ("packed backward: the first sequence's dhL", "None if dhL is None else dhL[s])",
     "None if dhL is None else dhL[0])"),
    ("bidirectional backward: right-to-left gradients not mirrored back",
     "        for k in (\"du\", \"ddelta_raw\", \"dB\", \"dC\", \"dz\"):\n            g[k] = f(g[k])\n", ""),
    ("bidirectional backward: dz of one direction", "\"dz\": gf.pop(\"dz\") + gr.pop(\"dz\")",
     "\"dz\": gf.pop(\"dz\") + 0.0 * gr.pop(\"dz\")"),
    ("bidirectional backward: the other direction's dhL", "    gr = one(rev, True, dhL_r)\n",
     "    gr = one(rev, True, dhL)\n"),
    ("conv backward: the scan's du not passed through the prologue",
     "    dx, dw, db = conv_silu_bwd(x, conv_w, conv_b, out.pop(\"du\"))\n",
     "    dx, dw, db = conv_silu_bwd(x, conv_w, conv_b, 0.0 * out.pop(\"du\") + 1.0)\n"),
    ("right-to-left output not gated",
     "        y, h = scan_fwd(f(u), f(d[\"delta_raw\"]), d[\"A\"], f(d[\"Bm\"]), f(d[\"Cm\"]), d.get(\"Dv\"),\n                        f(z),",
     "        y, h = scan_fwd(f(u), f(d[\"delta_raw\"]), d[\"A\"], f(d[\"Bm\"]), f(d[\"Cm\"]), d.get(\"Dv\"),\n                        None if flip else f(z),"),
]

PUBLIC = ("softplus", "silu", "conv_silu", "scan_fwd_conv", "scan_fwd_varlen", "scan_bwd_varlen",
          "scan_fwd_bidir", "scan_bwd_bidir", "scan_fwd", "scan_step", "scan_bwd", "conv_silu_bwd",
          "scan_bwd_conv")


def _pin_calls():
    """Every pin with each of its parameter sets, as zero-argument callables."""
    calls = []
    for name, f in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        sets = [{}]
        for m in getattr(f, "pytestmark", []):
            if m.name != "parametrize":
                continue
            names = [s.strip() for s in m.args[0].split(",")]
            vals = [v if len(names) > 1 else (v,) for v in m.args[1]]
            sets = [dict(a, **dict(zip(names, v))) for a, v in itertools.product(sets, vals)]
        calls += [(name, (lambda f=f, kw=kw: f(**kw))) for kw in sets]
    return calls


def _caught():
    """Names of the pins that fail."""
    failed = []
    for name, call in _pin_calls():
        try:
            call()
        except Exception:          # an assertion, or a crash on the wrong shapes
            failed.append(name)
            break
    return failed


def _plant(text, old, new):
    assert text.count(old) == 1, "the planted mistake no longer matches the oracle: %r" % old
    return text.replace(old, new)


@pytest.mark.parametrize("mistake", C_MISTAKES, ids=[m[0] for m in C_MISTAKES])
def test_c_mistake_fails_a_pin(mistake, tmp_path, monkeypatch):
    _, old, new = mistake
    src = tmp_path / "ssm_oracle.c"
    src.write_text(_plant(open(C_SRC).read(), old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, "-I", os.path.dirname(C_SRC), str(src),
                           "-o", str(lib), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.bind(ctypes.CDLL(str(lib))))
    assert _caught(), "no pin catches: " + mistake[0]


@pytest.mark.parametrize("mistake", PY_MISTAKES, ids=[m[0] for m in PY_MISTAKES])
def test_python_mistake_fails_a_pin(mistake, monkeypatch):
    _, old, new = mistake
    ns = {"__name__": "oracle_planted", "__file__": PY_SRC}
    exec(compile(_plant(open(PY_SRC).read(), old, new), PY_SRC, "exec"), ns)
    for name in PUBLIC:
        monkeypatch.setattr(oracle, name, ns[name])
    assert _caught(), "no pin catches: " + mistake[0]


def test_unplanted_oracle_passes_every_pin():
    assert not _caught()
