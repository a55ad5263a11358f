"""GPU-side plumbing shared by the parity tests: moving seeded inputs to the
device, running the library through its binding, and the oracle beside it."""
from __future__ import annotations

import numpy as np
import torch

import oracle

TIN = {"bf16": torch.bfloat16, "f32": torch.float32}


def load_ssm():
    from tests.buildlib import ensure_built
    ensure_built()
    import selective_state_space_123_b300 as m
    return m


def to_dev(a, dtype):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(dtype)


def device_args(x):
    """ScanInputs (host) -> dict of device tensors for the binding."""
    tin = TIN[x.in_dtype]
    f32 = torch.float32
    return dict(u=to_dev(x.u, tin), delta_raw=to_dev(x.delta_raw, tin), A=to_dev(x.A, f32),
                B=to_dev(x.Bm, tin), C=to_dev(x.Cm, tin), D=to_dev(x.Dv, f32),
                z=to_dev(x.z, tin), delta_bias=to_dev(x.delta_bias, f32),
                h0=to_dev(x.h0, f32))


def gpu_fwd(ssm, x, out_dtype=torch.float32):
    a = device_args(x)
    y, hL = ssm.ssm_scan_fwd(a["u"], a["delta_raw"], a["A"], a["B"], a["C"], a["D"], a["z"],
                             a["delta_bias"], a["h0"], out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), hL.cpu().numpy()


def oracle_fwd(x):
    return oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)


def rows_to_host(t, b_idx, d_idx):
    """Gather rows [b, d, :] of a device tensor to a float32 numpy array (Bsel, Dsel, ...)."""
    sub = t[b_idx][:, d_idx]
    return sub.float().cpu().numpy()


def oracle_bwd_chunk(args):
    """Worker for chunked oracle runs (spawned process): the reverse mode on a
    subset of channels.  Returns the oracle's outputs for those channels."""
    (u, dr, A, Bm, Cm, dy, Dv, z, bias) = args
    return oracle.scan_bwd(u, dr, A, Bm, Cm, dy, Dv, z, bias, None, None)
