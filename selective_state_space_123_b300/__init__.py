"""Python binding of libssmscan.so -- the selective scan on B300 (sm_103a).

The functions here carry the C-ABI names (include/ssm_scan.h) and only
marshal arguments: they check torch tensors (device, dtype, shape,
contiguity), allocate outputs and the workspace with torch, pass raw device
pointers and the current CUDA stream to the library, and turn a non-zero
status into an exception.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.  If the library is not built or
cannot be loaded, importing this package raises.

Computed (per batch b, channel d, state n, token t):
    delta = softplus(delta_raw + delta_bias)
    h_t   = exp(delta A) h_{t-1} + delta B_t u_t
    y_t   = (sum_n C_t h_t + D u_t) * silu(z_t)
("State Space Models (SSMs) & Mamba", sections "State-Space Models (SSMs): A
Resurgent Paradigm" and "The Magic of Selective Scan"; "Mamba: How Selective
State Spaces Achieve 5x Faster Inference Than Transformers", section "The
selective mechanism: input-dependent SSM parameters".)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssmscan.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libssmscan.so is not built; run `python selective_state_space_123_b300/build.py`")

lib = ctypes.CDLL(LIB_PATH)

SSM_F32, SSM_BF16 = 0, 1
SSM_OK = 0
SSM_ERR_NULL, SSM_ERR_SHAPE, SSM_ERR_DTYPE, SSM_ERR_ALIGN = -1, -2, -3, -4
SSM_ERR_WORKSPACE, SSM_ERR_CUDA, SSM_ERR_TIMEOUT, SSM_ERR_UNSUPPORTED = -5, -6, -7, -8
SSM_ERR_SEQLENS = -9

# Every symbol include/ssm_scan.h declares.
EXPORTS = ("ssm_scan_workspace_bytes", "ssm_scan_fwd", "ssm_scan_fwd_conv", "ssm_scan_fwd_varlen",
           "ssm_scan_fwd_bidir", "ssm_scan_bwd", "ssm_scan_bwd_varlen", "ssm_scan_bwd_bidir",
           "ssm_scan_bwd_conv", "ssm_scan_step",
           "ssm_get_status", "ssm_strerror", "ssm_debug_expired_wait", "ssm_scan_fwd_noalloc")


class ssm_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("seqlen", ctypes.c_int64), ("in_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
lib.ssm_scan_workspace_bytes.argtypes = [ctypes.POINTER(ssm_shape), ctypes.c_int]
lib.ssm_scan_workspace_bytes.restype = ctypes.c_size_t
lib.ssm_scan_fwd.argtypes = [ctypes.POINTER(ssm_shape)] + [_P] * 12 + [ctypes.c_size_t, _P]
lib.ssm_scan_fwd.restype = ctypes.c_int
lib.ssm_scan_fwd_conv.argtypes = ([ctypes.POINTER(ssm_shape), _P, _P, _P, ctypes.c_int] + [_P] * 11
                                  + [ctypes.c_size_t, _P])
lib.ssm_scan_fwd_conv.restype = ctypes.c_int
lib.ssm_scan_fwd_varlen.argtypes = ([ctypes.POINTER(ssm_shape), _P, _P, ctypes.c_int, _P, _P,
                                     ctypes.c_int] + [_P] * 11 + [ctypes.c_size_t, _P])
lib.ssm_scan_fwd_varlen.restype = ctypes.c_int
lib.ssm_scan_fwd_bidir.argtypes = [ctypes.POINTER(ssm_shape)] + [_P] * 20 + [ctypes.c_size_t, _P]
lib.ssm_scan_fwd_bidir.restype = ctypes.c_int
lib.ssm_scan_bwd.argtypes = [ctypes.POINTER(ssm_shape)] + [_P] * 21 + [ctypes.c_size_t, _P]
lib.ssm_scan_bwd.restype = ctypes.c_int
lib.ssm_scan_bwd_varlen.argtypes = ([ctypes.POINTER(ssm_shape), _P, _P, ctypes.c_int] + [_P] * 20
                                    + [ctypes.c_size_t, _P])
lib.ssm_scan_bwd_varlen.restype = ctypes.c_int
lib.ssm_scan_bwd_bidir.argtypes = [ctypes.POINTER(ssm_shape)] + [_P] * 36 + [ctypes.c_size_t, _P]
lib.ssm_scan_bwd_bidir.restype = ctypes.c_int
lib.ssm_scan_bwd_conv.argtypes = ([ctypes.POINTER(ssm_shape), _P, _P, _P, ctypes.c_int] + [_P] * 22
                                  + [ctypes.c_size_t, _P])
lib.ssm_scan_bwd_conv.restype = ctypes.c_int
lib.ssm_scan_step.argtypes = [_I64, _I64, _I64, ctypes.c_int32, ctypes.c_int32] + [_P] * 12
lib.ssm_scan_step.restype = ctypes.c_int
lib.ssm_get_status.argtypes = [_P, _P]
lib.ssm_get_status.restype = ctypes.c_int
lib.ssm_strerror.argtypes = [ctypes.c_int]
lib.ssm_strerror.restype = ctypes.c_char_p
lib.ssm_debug_expired_wait.argtypes = [_P, ctypes.c_size_t, _I64, _P]
lib.ssm_debug_expired_wait.restype = ctypes.c_int
# scratch-free forward (no workspace argument; see include/ssm_scan.h)
lib.ssm_scan_fwd_noalloc.argtypes = [ctypes.POINTER(ssm_shape)] + [_P] * 12
lib.ssm_scan_fwd_noalloc.restype = ctypes.c_int
# SSM_NOALLOC_SCRATCH_BYTES of include/ssm_scan.h (a CPU test compares the two)
NOALLOC_SCRATCH_BYTES = 32 << 20


class SSMError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__("%s: %s (%d)" % (where, ssm_strerror(code), code))
        self.code = code


def ssm_strerror(code: int) -> str:
    return lib.ssm_strerror(int(code)).decode()


def _dt(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return SSM_BF16
    if t == torch.float32:
        return SSM_F32
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(t: Optional[torch.Tensor], name: str, shape, dtype=None, device=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def make_shape(batch, dim, dstate, seqlen, in_dtype, out_dtype) -> ssm_shape:
    return ssm_shape(int(batch), int(dim), int(dstate), int(seqlen), int(in_dtype),
                     int(out_dtype))


def ssm_scan_workspace_bytes(shape: ssm_shape, for_backward=False) -> int:
    """Workspace bytes: for_backward False/0 forward, True/1 backward, 2 the
    bidirectional forward."""
    return int(lib.ssm_scan_workspace_bytes(ctypes.byref(shape), int(for_backward)))


def _workspace(shape: ssm_shape, for_backward, device, workspace):
    need = ssm_scan_workspace_bytes(shape, for_backward)
    if need == 0:
        raise SSMError(SSM_ERR_SHAPE, "ssm_scan_workspace_bytes")
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace


def ssm_scan_fwd(u, delta_raw, A, B, C, D=None, z=None, delta_bias=None, h0=None, *,
                 out_dtype: Optional[torch.dtype] = None, y=None, hL=None,
                 return_final_state: bool = True, workspace=None,
                 stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Forward scan.  u, delta_raw, z: (Bt,D,L); B, C: (Bt,N,L) (all one dtype,
    fp32 or bf16); A: (D,N) fp32; D, delta_bias: (D,) fp32; h0: (Bt,D,N) fp32.
    Returns (y (Bt,D,L) in out_dtype [default: input dtype], hL (Bt,D,N) fp32 or None)."""
    Bt, Dm, L = u.shape
    N = A.shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_fwd runs on CUDA tensors only")
    tin = u.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    _check(u, "u", (Bt, Dm, L), tin, dev)
    _check(delta_raw, "delta_raw", (Bt, Dm, L), tin, dev)
    _check(z, "z", (Bt, Dm, L), tin, dev)
    _check(B, "B", (Bt, N, L), tin, dev)
    _check(C, "C", (Bt, N, L), tin, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _check(h0, "h0", (Bt, Dm, N), torch.float32, dev)
    if y is None:
        y = torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev)
    _check(y, "y", (Bt, Dm, L), out_dtype, dev)
    if hL is None and return_final_state:
        hL = torch.empty((Bt, Dm, N), dtype=torch.float32, device=dev)
    _check(hL, "hL", (Bt, Dm, N), torch.float32, dev)
    shape = make_shape(Bt, Dm, N, L, _dt(tin), _dt(out_dtype))
    workspace = _workspace(shape, False, dev, workspace)
    rc = lib.ssm_scan_fwd(ctypes.byref(shape), _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(B),
                          _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0), _ptr(y),
                          _ptr(hL), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_fwd")
    return y, hL


def ssm_scan_fwd_conv(x, conv_w, conv_b, delta_raw, A, B, C, D=None, z=None, delta_bias=None,
                      h0=None, *, out_dtype: Optional[torch.dtype] = None, y=None, hL=None,
                      return_final_state: bool = True, workspace=None,
                      stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Forward scan fed by the block's conv prologue: x (Bt,D,L) is the branch
    input, conv_w (D,K) fp32 with K <= 4, conv_b (D,) fp32 or None; the scan
    input is u = silu(causal depthwise conv of x), computed in the kernel.
    Other arguments and the result as ssm_scan_fwd."""
    Bt, Dm, L = x.shape
    N = A.shape[1]
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_fwd_conv runs on CUDA tensors only")
    tin = x.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    if conv_w is None or conv_w.dim() != 2:
        raise ValueError("conv_w must be a (D, K) tensor")
    K = conv_w.shape[1]
    _check(x, "x", (Bt, Dm, L), tin, dev)
    _check(conv_w, "conv_w", (Dm, K), torch.float32, dev)
    _check(conv_b, "conv_b", (Dm,), torch.float32, dev)
    _check(delta_raw, "delta_raw", (Bt, Dm, L), tin, dev)
    _check(z, "z", (Bt, Dm, L), tin, dev)
    _check(B, "B", (Bt, N, L), tin, dev)
    _check(C, "C", (Bt, N, L), tin, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _check(h0, "h0", (Bt, Dm, N), torch.float32, dev)
    if y is None:
        y = torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev)
    _check(y, "y", (Bt, Dm, L), out_dtype, dev)
    if hL is None and return_final_state:
        hL = torch.empty((Bt, Dm, N), dtype=torch.float32, device=dev)
    _check(hL, "hL", (Bt, Dm, N), torch.float32, dev)
    shape = make_shape(Bt, Dm, N, L, _dt(tin), _dt(out_dtype))
    workspace = _workspace(shape, False, dev, workspace)
    rc = lib.ssm_scan_fwd_conv(ctypes.byref(shape), _ptr(x), _ptr(conv_w), _ptr(conv_b), int(K),
                               _ptr(delta_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                               _ptr(delta_bias), _ptr(h0), _ptr(y), _ptr(hL), _ptr(workspace),
                               workspace.numel(), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_fwd_conv")
    return y, hL


def ssm_scan_fwd_varlen(u, cu_seqlens, delta_raw, A, B, C, D=None, z=None, delta_bias=None,
                        h0=None, *, conv_w=None, conv_b=None, out_dtype: Optional[torch.dtype] = None,
                        y=None, hL=None, return_final_state: bool = True, workspace=None,
                        stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Forward scan over packed sequences: every batch row holds nseq
    sequences, sequence s at tokens [cu_seqlens[s], cu_seqlens[s+1])
    (cu_seqlens: int32 (nseq+1,) on the device, 0 first, L last).  Each
    sequence starts from h0[s] (h0: (nseq,Bt,D,N) fp32, or zeros) and, with
    conv_w (D,K) given, u is the conv branch input x with the window
    restarting at every sequence start.  Returns (y (Bt,D,L), hL (nseq,Bt,D,N)
    fp32 or None); other arguments as ssm_scan_fwd."""
    Bt, Dm, L = u.shape
    N = A.shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_fwd_varlen runs on CUDA tensors only")
    if not isinstance(cu_seqlens, torch.Tensor) or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D tensor of nseq + 1 >= 2 offsets")
    nseq = cu_seqlens.numel() - 1
    tin = u.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    _check(cu_seqlens, "cu_seqlens", (nseq + 1,), torch.int32, dev)
    K = 0
    if conv_w is not None:
        if conv_w.dim() != 2:
            raise ValueError("conv_w must be a (D, K) tensor")
        K = conv_w.shape[1]
        _check(conv_w, "conv_w", (Dm, K), torch.float32, dev)
        _check(conv_b, "conv_b", (Dm,), torch.float32, dev)
    _check(u, "u", (Bt, Dm, L), tin, dev)
    _check(delta_raw, "delta_raw", (Bt, Dm, L), tin, dev)
    _check(z, "z", (Bt, Dm, L), tin, dev)
    _check(B, "B", (Bt, N, L), tin, dev)
    _check(C, "C", (Bt, N, L), tin, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _check(h0, "h0", (nseq, Bt, Dm, N), torch.float32, dev)
    if y is None:
        y = torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev)
    _check(y, "y", (Bt, Dm, L), out_dtype, dev)
    if hL is None and return_final_state:
        hL = torch.empty((nseq, Bt, Dm, N), dtype=torch.float32, device=dev)
    _check(hL, "hL", (nseq, Bt, Dm, N), torch.float32, dev)
    shape = make_shape(Bt, Dm, N, L, _dt(tin), _dt(out_dtype))
    workspace = _workspace(shape, False, dev, workspace)
    rc = lib.ssm_scan_fwd_varlen(ctypes.byref(shape), _ptr(u), _ptr(cu_seqlens), int(nseq),
                                 _ptr(conv_w), _ptr(conv_b if conv_w is not None else None), int(K),
                                 _ptr(delta_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                 _ptr(delta_bias), _ptr(h0), _ptr(y), _ptr(hL), _ptr(workspace),
                                 workspace.numel(), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_fwd_varlen")
    return y, hL


def ssm_scan_fwd_bidir(u, z, fwd: dict, rev: dict, *, out_dtype: Optional[torch.dtype] = None,
                       y=None, hL=None, hL_r=None, return_final_state: bool = True,
                       workspace=None, stream=None):
    """Bidirectional scan: the left-to-right scan with the parameters in
    `fwd` plus a right-to-left scan with those in `rev`, over the same u and
    gate z (nullable).  Each dict holds delta_raw, A, B, C and optional D,
    delta_bias, h0, shaped as for ssm_scan_fwd.  Returns (y, hL, hL_r): hL the
    left-to-right state after the last token, hL_r the right-to-left state
    after the first (fp32 (Bt,D,N) or None)."""
    Bt, Dm, L = u.shape
    N = fwd["A"].shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_fwd_bidir runs on CUDA tensors only")
    tin = u.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    _check(u, "u", (Bt, Dm, L), tin, dev)
    _check(z, "z", (Bt, Dm, L), tin, dev)
    for tag, d in (("fwd", fwd), ("rev", rev)):
        _check(d["delta_raw"], tag + ".delta_raw", (Bt, Dm, L), tin, dev)
        _check(d["B"], tag + ".B", (Bt, N, L), tin, dev)
        _check(d["C"], tag + ".C", (Bt, N, L), tin, dev)
        _check(d["A"], tag + ".A", (Dm, N), torch.float32, dev)
        _check(d.get("D"), tag + ".D", (Dm,), torch.float32, dev)
        _check(d.get("delta_bias"), tag + ".delta_bias", (Dm,), torch.float32, dev)
        _check(d.get("h0"), tag + ".h0", (Bt, Dm, N), torch.float32, dev)
    if y is None:
        y = torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev)
    _check(y, "y", (Bt, Dm, L), out_dtype, dev)
    if return_final_state:
        if hL is None:
            hL = torch.empty((Bt, Dm, N), dtype=torch.float32, device=dev)
        if hL_r is None:
            hL_r = torch.empty((Bt, Dm, N), dtype=torch.float32, device=dev)
    _check(hL, "hL", (Bt, Dm, N), torch.float32, dev)
    _check(hL_r, "hL_r", (Bt, Dm, N), torch.float32, dev)
    shape = make_shape(Bt, Dm, N, L, _dt(tin), _dt(out_dtype))
    workspace = _workspace(shape, 2, dev, workspace)
    f, r = fwd, rev
    rc = lib.ssm_scan_fwd_bidir(ctypes.byref(shape), _ptr(u), _ptr(z),
                                _ptr(f["delta_raw"]), _ptr(f["A"]), _ptr(f["B"]), _ptr(f["C"]),
                                _ptr(f.get("D")), _ptr(f.get("delta_bias")), _ptr(f.get("h0")),
                                _ptr(r["delta_raw"]), _ptr(r["A"]), _ptr(r["B"]), _ptr(r["C"]),
                                _ptr(r.get("D")), _ptr(r.get("delta_bias")), _ptr(r.get("h0")),
                                _ptr(y), _ptr(hL), _ptr(hL_r), _ptr(workspace), workspace.numel(),
                                _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_fwd_bidir")
    return y, hL, hL_r


def ssm_scan_bwd_bidir(u, z, fwd: dict, rev: dict, dy, dhL=None, dhL_r=None, *,
                       out_dtype: Optional[torch.dtype] = None, workspace=None,
                       stream=None) -> Tuple[dict, dict, dict]:
    """Reverse mode of ssm_scan_fwd_bidir.  `fwd` and `rev` hold each
    direction's delta_raw, A, B, C and optional D, delta_bias, h0 (as for
    ssm_scan_fwd_bidir); dhL, dhL_r the upstream gradients of the two final
    states (nullable).  Returns (shared, grads_fwd, grads_rev): shared = {du,
    dz} (out_dtype; dz None without z), each grads dict ddelta_raw (out_dtype),
    dA, dB, dC, dD, ddelta_bias, dh0 (fp32; dD, ddelta_bias, dh0 always
    returned)."""
    Bt, Dm, L = u.shape
    N = fwd["A"].shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_bwd_bidir runs on CUDA tensors only")
    tin = u.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    f32 = torch.float32
    _check(u, "u", (Bt, Dm, L), tin, dev)
    _check(z, "z", (Bt, Dm, L), tin, dev)
    _check(dy, "dy", (Bt, Dm, L), tin, dev)
    _check(dhL, "dhL", (Bt, Dm, N), f32, dev)
    _check(dhL_r, "dhL_r", (Bt, Dm, N), f32, dev)
    for tag, d in (("fwd", fwd), ("rev", rev)):
        _check(d["delta_raw"], tag + ".delta_raw", (Bt, Dm, L), tin, dev)
        _check(d["B"], tag + ".B", (Bt, N, L), tin, dev)
        _check(d["C"], tag + ".C", (Bt, N, L), tin, dev)
        _check(d["A"], tag + ".A", (Dm, N), f32, dev)
        _check(d.get("D"), tag + ".D", (Dm,), f32, dev)
        _check(d.get("delta_bias"), tag + ".delta_bias", (Dm,), f32, dev)
        _check(d.get("h0"), tag + ".h0", (Bt, Dm, N), f32, dev)
    emp = lambda shp, dt: torch.empty(shp, dtype=dt, device=dev)
    shared = {"du": emp((Bt, Dm, L), out_dtype), "dz": emp((Bt, Dm, L), out_dtype) if z is not None else None}

    def grads():
        return {"ddelta_raw": emp((Bt, Dm, L), out_dtype), "dA": emp((Dm, N), f32),
                "dB": emp((Bt, N, L), f32), "dC": emp((Bt, N, L), f32), "dD": emp((Dm,), f32),
                "ddelta_bias": emp((Dm,), f32), "dh0": emp((Bt, Dm, N), f32)}
    gf, gr = grads(), grads()
    shape = make_shape(Bt, Dm, N, L, _dt(tin), _dt(out_dtype))
    workspace = _workspace(shape, 3, dev, workspace)
    f, r = fwd, rev
    g_ptrs = lambda g: [_ptr(g[k]) for k in ("ddelta_raw", "dA", "dB", "dC", "dD", "ddelta_bias",
                                             "dh0")]
    rc = lib.ssm_scan_bwd_bidir(ctypes.byref(shape), _ptr(u), _ptr(z),
                                _ptr(f["delta_raw"]), _ptr(f["A"]), _ptr(f["B"]), _ptr(f["C"]),
                                _ptr(f.get("D")), _ptr(f.get("delta_bias")), _ptr(f.get("h0")),
                                _ptr(r["delta_raw"]), _ptr(r["A"]), _ptr(r["B"]), _ptr(r["C"]),
                                _ptr(r.get("D")), _ptr(r.get("delta_bias")), _ptr(r.get("h0")),
                                _ptr(dy), _ptr(dhL), _ptr(dhL_r), _ptr(shared["du"]),
                                _ptr(shared["dz"]), *g_ptrs(gf), *g_ptrs(gr),
                                _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_bwd_bidir")
    return shared, gf, gr


def ssm_scan_bwd(u, delta_raw, A, B, C, dy, D=None, z=None, delta_bias=None, h0=None,
                 dhL=None, *, out_dtype: Optional[torch.dtype] = None, workspace=None,
                 stream=None) -> dict:
    """Reverse mode of ssm_scan_fwd.  Returns a dict with du, ddelta_raw, dz
    (out_dtype, default input dtype), dA, dB, dC, dD, ddelta_bias, dh0 (fp32)."""
    Bt, Dm, L = u.shape
    N = A.shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_bwd runs on CUDA tensors only")
    tin = u.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    for t, n, s in ((u, "u", (Bt, Dm, L)), (delta_raw, "delta_raw", (Bt, Dm, L)),
                    (z, "z", (Bt, Dm, L)), (dy, "dy", (Bt, Dm, L)), (B, "B", (Bt, N, L)),
                    (C, "C", (Bt, N, L))):
        _check(t, n, s, tin, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _check(h0, "h0", (Bt, Dm, N), torch.float32, dev)
    _check(dhL, "dhL", (Bt, Dm, N), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = {
        "du": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev),
        "ddelta_raw": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev),
        "dz": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev) if z is not None else None,
        "dA": torch.empty((Dm, N), **f32), "dB": torch.empty((Bt, N, L), **f32),
        "dC": torch.empty((Bt, N, L), **f32), "dD": torch.empty((Dm,), **f32),
        "ddelta_bias": torch.empty((Dm,), **f32), "dh0": torch.empty((Bt, Dm, N), **f32),
    }
    shape = make_shape(Bt, Dm, N, L, _dt(tin), _dt(out_dtype))
    workspace = _workspace(shape, True, dev, workspace)
    rc = lib.ssm_scan_bwd(ctypes.byref(shape), _ptr(u), _ptr(delta_raw), _ptr(A), _ptr(B),
                          _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), _ptr(h0), _ptr(dy),
                          _ptr(dhL), _ptr(g["du"]), _ptr(g["ddelta_raw"]), _ptr(g["dA"]),
                          _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["dz"]),
                          _ptr(g["ddelta_bias"]), _ptr(g["dh0"]), _ptr(workspace),
                          workspace.numel(), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_bwd")
    return g


def ssm_scan_bwd_conv(x, conv_w, conv_b, delta_raw, A, B, C, dy, D=None, z=None,
                      delta_bias=None, h0=None, dhL=None, *, out_dtype: Optional[torch.dtype] = None,
                      workspace=None, stream=None) -> dict:
    """Reverse mode of ssm_scan_fwd_conv: x is the branch input, conv_w (D, K)
    fp32 with K <= 4, conv_b (D,) fp32 or None.  Returns the dict of
    ssm_scan_bwd with du replaced by dx (out_dtype) and dconv_w (D, K),
    dconv_b (D,) fp32 (None without conv_b)."""
    Bt, Dm, L = x.shape
    N = A.shape[1]
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_bwd_conv runs on CUDA tensors only")
    if conv_w.dim() != 2 or conv_w.shape[0] != Dm:
        raise ValueError("conv_w must be (D, K)")
    K = conv_w.shape[1]
    tin = x.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    for t, n, s in ((x, "x", (Bt, Dm, L)), (delta_raw, "delta_raw", (Bt, Dm, L)),
                    (z, "z", (Bt, Dm, L)), (dy, "dy", (Bt, Dm, L)), (B, "B", (Bt, N, L)),
                    (C, "C", (Bt, N, L))):
        _check(t, n, s, tin, dev)
    _check(conv_w, "conv_w", (Dm, K), torch.float32, dev)
    _check(conv_b, "conv_b", (Dm,), torch.float32, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _check(h0, "h0", (Bt, Dm, N), torch.float32, dev)
    _check(dhL, "dhL", (Bt, Dm, N), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = {
        "dx": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev),
        "ddelta_raw": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev),
        "dz": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev) if z is not None else None,
        "dA": torch.empty((Dm, N), **f32), "dB": torch.empty((Bt, N, L), **f32),
        "dC": torch.empty((Bt, N, L), **f32), "dD": torch.empty((Dm,), **f32),
        "ddelta_bias": torch.empty((Dm,), **f32), "dh0": torch.empty((Bt, Dm, N), **f32),
        "dconv_w": torch.empty((Dm, K), **f32),
        "dconv_b": torch.empty((Dm,), **f32) if conv_b is not None else None,
    }
    shape = make_shape(Bt, Dm, N, L, _dt(tin), _dt(out_dtype))
    workspace = _workspace(shape, 4, dev, workspace)
    rc = lib.ssm_scan_bwd_conv(ctypes.byref(shape), _ptr(x), _ptr(conv_w), _ptr(conv_b), K,
                               _ptr(delta_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                               _ptr(delta_bias), _ptr(h0), _ptr(dy), _ptr(dhL), _ptr(g["dx"]),
                               _ptr(g["ddelta_raw"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
                               _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]),
                               _ptr(g["dconv_w"]), _ptr(g["dconv_b"]), _ptr(workspace),
                               workspace.numel(), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_bwd_conv")
    return g


def ssm_scan_bwd_varlen(u, cu_seqlens, delta_raw, A, B, C, dy, D=None, z=None, delta_bias=None,
                        h0=None, dhL=None, *, out_dtype: Optional[torch.dtype] = None,
                        workspace=None, stream=None) -> dict:
    """Reverse mode of ssm_scan_fwd_varlen (no conv prologue): packed
    sequences at cu_seqlens (int32 CUDA tensor of nseq + 1 starts), h0, dhL
    (nseq, Bt, D, N) fp32 or None.  Returns the dict of ssm_scan_bwd with dh0
    (nseq, Bt, D, N)."""
    Bt, Dm, L = u.shape
    N = A.shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_bwd_varlen runs on CUDA tensors only")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor of nseq + 1 starts")
    _check(cu_seqlens, "cu_seqlens", tuple(cu_seqlens.shape), torch.int32, dev)
    nseq = cu_seqlens.numel() - 1
    tin = u.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    for t, n, s in ((u, "u", (Bt, Dm, L)), (delta_raw, "delta_raw", (Bt, Dm, L)),
                    (z, "z", (Bt, Dm, L)), (dy, "dy", (Bt, Dm, L)), (B, "B", (Bt, N, L)),
                    (C, "C", (Bt, N, L))):
        _check(t, n, s, tin, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _check(h0, "h0", (nseq, Bt, Dm, N), torch.float32, dev)
    _check(dhL, "dhL", (nseq, Bt, Dm, N), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = {
        "du": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev),
        "ddelta_raw": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev),
        "dz": torch.empty((Bt, Dm, L), dtype=out_dtype, device=dev) if z is not None else None,
        "dA": torch.empty((Dm, N), **f32), "dB": torch.empty((Bt, N, L), **f32),
        "dC": torch.empty((Bt, N, L), **f32), "dD": torch.empty((Dm,), **f32),
        "ddelta_bias": torch.empty((Dm,), **f32), "dh0": torch.empty((nseq, Bt, Dm, N), **f32),
    }
    shape = make_shape(Bt, Dm, N, L, _dt(tin), _dt(out_dtype))
    workspace = _workspace(shape, True, dev, workspace)
    rc = lib.ssm_scan_bwd_varlen(ctypes.byref(shape), _ptr(u), _ptr(cu_seqlens), nseq,
                                 _ptr(delta_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                 _ptr(delta_bias), _ptr(h0), _ptr(dy), _ptr(dhL), _ptr(g["du"]),
                                 _ptr(g["ddelta_raw"]), _ptr(g["dA"]), _ptr(g["dB"]),
                                 _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["dz"]),
                                 _ptr(g["ddelta_bias"]), _ptr(g["dh0"]), _ptr(workspace),
                                 workspace.numel(), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_bwd_varlen")
    return g


def ssm_scan_step(u, delta_raw, A, B, C, state, D=None, z=None, delta_bias=None, *,
                  out_dtype: Optional[torch.dtype] = None, y=None, status=None,
                  stream=None) -> torch.Tensor:
    """One decode step.  u, delta_raw, z: (Bt,D); B, C: (Bt,N); A: (D,N);
    state: (Bt,D,N) fp32, updated in place.  Returns y (Bt,D).  status: an
    optional int32 CUDA tensor whose first element receives SSM_ERR_TIMEOUT
    if a bounded wait in the kernel expires (read it with ssm_get_status)."""
    Bt, Dm = u.shape
    N = A.shape[1]
    dev = u.device
    if dev.type != "cuda":
        raise ValueError("ssm_scan_step runs on CUDA tensors only")
    tin = u.dtype
    out_dtype = tin if out_dtype is None else out_dtype
    for t, n, s in ((u, "u", (Bt, Dm)), (delta_raw, "delta_raw", (Bt, Dm)), (z, "z", (Bt, Dm)),
                    (B, "B", (Bt, N)), (C, "C", (Bt, N))):
        _check(t, n, s, tin, dev)
    _check(A, "A", (Dm, N), torch.float32, dev)
    _check(D, "D", (Dm,), torch.float32, dev)
    _check(delta_bias, "delta_bias", (Dm,), torch.float32, dev)
    _check(state, "state", (Bt, Dm, N), torch.float32, dev)
    if y is None:
        y = torch.empty((Bt, Dm), dtype=out_dtype, device=dev)
    _check(y, "y", (Bt, Dm), out_dtype, dev)
    if status is not None:
        if status.dtype != torch.int32 or status.device != dev or status.numel() < 1:
            raise ValueError("status must be an int32 tensor on %s" % dev)
    rc = lib.ssm_scan_step(Bt, Dm, N, _dt(tin), _dt(out_dtype), _ptr(u), _ptr(delta_raw),
                           _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                           _ptr(state), _ptr(y), _ptr(status), _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_scan_step")
    return y


def ssm_get_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return (and clear) the workspace status word."""
    return int(lib.ssm_get_status(_ptr(workspace), _stream_ptr(stream)))


def ssm_debug_expired_wait(workspace: torch.Tensor, spin_limit: int, stream=None) -> None:
    rc = lib.ssm_debug_expired_wait(_ptr(workspace), workspace.numel(), int(spin_limit),
                                    _stream_ptr(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_debug_expired_wait")
