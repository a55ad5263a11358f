"""Seeded synthetic inputs for the selective scan.

This module is shared by the oracle tests, the GPU parity tests and the
bench.  It holds random-number plumbing and the value recipes only -- none of
the scan's arithmetic.

Recipes (the workloads named for the Mamba layer shapes; the pages name the
model scales, "Mamba: How Selective State Spaces Achieve 5x Faster Inference
Than Transformers", section "What the numbers show"):
  u, z, B, C, D_skip, delta_raw ~ N(0, 1)
  A[d, n] = -(n + 1)               (S4D-real), plus U[0, 0.1) jitter when asked
  delta_bias[d] = log(expm1(dt_d)),  dt_d = exp(U[ln 1e-3, ln 1e-1))
      i.e. the bias for which softplus(bias) = dt_d, log-uniform in [1e-3, 1e-1];
      delta_raw ~ N(0,1) is added to it unscaled.
  h0 = 0 unless asked; the decode state ~ N(0, 1); dy ~ N(0, 1).
bf16 tensors are drawn in fp32 and rounded to nearest-even bf16; the returned
float32 arrays hold exactly the bf16 values, so the oracle sees exactly what the
GPU sees.

Host generation is per row: every (tensor, row) pair has its own Philox key,
so any subset of channels can be regenerated alone (used for sampled parity at
full size).  ``device_inputs`` draws the same recipe with torch's seeded CUDA
generator for large workloads; callers copy sampled rows back for the oracle.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence

import numpy as np

# tensor ids (part of the Philox key)
_U, _DR, _Z, _B, _C, _DSKIP, _AJIT, _DT, _H0, _DY = range(10)


def _rng(seed: int, tensor: int, row: int) -> np.random.Generator:
    key = np.array([np.uint64(seed), np.uint64((tensor << 40) | row)], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    r = ((bits + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    # NaN/Inf are not produced by these recipes; keep them as they are anyway
    bad = ~np.isfinite(x)
    if bad.any():
        out = out.copy()
        out[bad] = x[bad]
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are exactly bf16."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert not np.any(b & 0xFFFF), "value is not bf16-representable"
    return (b >> 16).astype(np.uint16)


def _rows_normal(seed, tensor, rows: Sequence[int], n: int) -> np.ndarray:
    out = np.empty((len(rows), n), np.float32)
    for i, r in enumerate(rows):
        out[i] = _rng(seed, tensor, r).standard_normal(n, dtype=np.float32)
    return out


@dataclasses.dataclass
class ScanInputs:
    """One problem instance (float32 arrays; bf16 tensors hold bf16 values)."""
    u: np.ndarray            # (Bt, D, L)
    delta_raw: np.ndarray    # (Bt, D, L)
    A: np.ndarray            # (D, N)   fp32
    Bm: np.ndarray           # (Bt, N, L)
    Cm: np.ndarray           # (Bt, N, L)
    Dv: Optional[np.ndarray]          # (D)   fp32
    z: Optional[np.ndarray]           # (Bt, D, L)
    delta_bias: Optional[np.ndarray]  # (D)   fp32
    h0: Optional[np.ndarray]          # (Bt, D, N) fp32
    dy: Optional[np.ndarray] = None   # (Bt, D, L)
    in_dtype: str = "f32"             # dtype of u, delta_raw, z, Bm, Cm, dy

    @property
    def shape(self):
        Bt, D, L = self.u.shape
        return Bt, D, self.A.shape[1], L


def make_inputs(Bt: int, D: int, N: int, L: int, *, seed: int, in_dtype: str = "bf16",
                a_jitter: bool = True, with_D: bool = True, with_z: bool = True,
                with_bias: bool = True, h0: bool = False, dy: bool = False,
                channels: Optional[Sequence[int]] = None) -> ScanInputs:
    """Generate the recipe on the host.

    ``channels`` restricts the per-channel tensors (u, delta_raw, z, dy, A,
    D_skip, delta_bias, h0) to that subset of d; B and C are always full.
    The values for a given (seed, b, d) do not depend on the subset.
    """
    chans = list(range(D)) if channels is None else [int(c) for c in channels]
    Dc = len(chans)
    rnd = round_bf16 if in_dtype == "bf16" else (lambda a: a.astype(np.float32))

    def per_channel_seq(tensor):
        rows = [b * D + d for b in range(Bt) for d in chans]
        return rnd(_rows_normal(seed, tensor, rows, L).reshape(Bt, Dc, L))

    u = per_channel_seq(_U)
    dr = per_channel_seq(_DR)
    z = per_channel_seq(_Z) if with_z else None
    Bm = rnd(_rows_normal(seed, _B, range(Bt * N), L).reshape(Bt, N, L))
    Cm = rnd(_rows_normal(seed, _C, range(Bt * N), L).reshape(Bt, N, L))
    Dv = (np.array([_rng(seed, _DSKIP, d).standard_normal(dtype=np.float32) for d in chans],
                   np.float32) if with_D else None)
    A = np.empty((Dc, N), np.float32)
    for i, d in enumerate(chans):
        base = -(np.arange(N, dtype=np.float32) + 1.0)
        if a_jitter:
            base = base + _rng(seed, _AJIT, d).uniform(0.0, 0.1, N).astype(np.float32)
        A[i] = base
    bias = None
    if with_bias:
        lo, hi = np.log(1e-3), np.log(1e-1)
        dt = np.array([np.exp(_rng(seed, _DT, d).uniform(lo, hi)) for d in chans])
        bias = np.log(np.expm1(dt)).astype(np.float32)
    h = None
    if h0:
        rows = [b * D + d for b in range(Bt) for d in chans]
        h = _rows_normal(seed, _H0, rows, N).reshape(Bt, Dc, N)
    g = per_channel_seq(_DY) if dy else None
    return ScanInputs(u=u, delta_raw=dr, A=A, Bm=Bm, Cm=Cm, Dv=Dv, z=z, delta_bias=bias,
                      h0=h, dy=g, in_dtype=in_dtype)


def make_step_inputs(Bt: int, D: int, N: int, *, seed: int, in_dtype: str = "bf16",
                     channels: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """Single-token decode inputs: u, delta_raw, z (Bt,D); Bm, Cm (Bt,N);
    A (D,N) with jitter; Dv, delta_bias (D); state (Bt,D,N) ~ N(0,1)."""
    x = make_inputs(Bt, D, N, 1, seed=seed, in_dtype=in_dtype, h0=True, channels=channels)
    return dict(u=x.u[:, :, 0].copy(), delta_raw=x.delta_raw[:, :, 0].copy(),
                z=x.z[:, :, 0].copy(), Bm=x.Bm[:, :, 0].copy(), Cm=x.Cm[:, :, 0].copy(),
                A=x.A, Dv=x.Dv, delta_bias=x.delta_bias, state=x.h0)


def packed_seqlens(L: int, *, seed: int, lo: int = 256, hi: int = 16384) -> list:
    """Start offsets (nseq + 1 ints, 0 first, L last) of sequences packed into
    one row of L tokens: lengths log-uniform in [lo, hi], drawn until the row
    is full, the last one cut to fit (documents of mixed length packed for
    one pass, "Mamba Architecture Explained", section "Problem 3: Ecosystem
    maturity")."""
    g = np.random.default_rng(np.random.SeedSequence([seed, 0x5EC]))
    cu = [0]
    while cu[-1] < L:
        n = int(np.exp(g.uniform(np.log(lo), np.log(hi))))
        cu.append(min(L, cu[-1] + max(1, n)))
    return cu


# ----------------------------------------------------------------------------
# The five workloads (shape, dtype and recipe switches).
# ----------------------------------------------------------------------------
WORKLOADS = {
    # tiny fp32 forward; A without jitter; h0 = 0
    "tiny_fp32": dict(Bt=1, D=16, N=4, L=64, in_dtype="f32", a_jitter=False, seed=0),
    # Mamba-130M layer: d_model 768, expand 2
    "mamba130m_fwd": dict(Bt=8, D=1536, N=16, L=2048, in_dtype="bf16", seed=1),
    # Mamba-1.4B layer: d_model 2048, expand 2
    "mamba1p4b_fwd": dict(Bt=4, D=4096, N=16, L=4096, in_dtype="bf16", seed=2),
    # Mamba-2.8B layer: d_model 2560, expand 2; forward and backward
    "mamba2p8b_fwdbwd": dict(Bt=2, D=5120, N=16, L=8192, in_dtype="bf16", seed=3, dy=True),
    # million-length forward
    "million_fwd": dict(Bt=1, D=1536, N=16, L=1 << 20, in_dtype="bf16", seed=4),
    # single-token decode from a random state
    "decode_step": dict(Bt=256, D=5120, N=16, L=1, in_dtype="bf16", seed=4),
}


def device_inputs(Bt: int, D: int, N: int, L: int, *, seed: int, in_dtype: str = "bf16",
                  a_jitter: bool = True, h0: bool = False, dy: bool = False,
                  device="cuda"):
    """The same recipe drawn on the device with torch's seeded generator (for
    workloads too large to draw on the host).  Returns a dict of torch tensors:
    u, delta_raw, z, Bm, Cm in ``in_dtype``; A, Dv, delta_bias, h0 in fp32."""
    import math
    import torch
    dt = torch.bfloat16 if in_dtype == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def normal(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(dt)

    out = {
        "u": normal(Bt, D, L), "delta_raw": normal(Bt, D, L), "z": normal(Bt, D, L),
        "Bm": normal(Bt, N, L), "Cm": normal(Bt, N, L),
        "Dv": torch.randn(D, generator=g, device=device),
    }
    A = -(torch.arange(N, device=device, dtype=torch.float32) + 1.0).repeat(D, 1)
    if a_jitter:
        A = A + 0.1 * torch.rand(D, N, generator=g, device=device)
    out["A"] = A.contiguous()
    lo, hi = math.log(1e-3), math.log(1e-1)
    dts = torch.exp(lo + (hi - lo) * torch.rand(D, generator=g, device=device,
                                                dtype=torch.float64))
    out["delta_bias"] = torch.log(torch.expm1(dts)).float()
    out["h0"] = torch.randn(Bt, D, N, generator=g, device=device) if h0 else None
    out["dy"] = normal(Bt, D, L) if dy else None
    return out
