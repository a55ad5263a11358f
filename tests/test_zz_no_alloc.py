"""ssm_scan_fwd_noalloc: the forward scan for callers that may not allocate
device memory (they are handed only their input and output buffers, e.g. a
plug-in inside an engine that owns all device memory, or a loop that must not
call the allocator after start-up).  It runs on a fixed scratch array inside
the library instead of a caller-allocated workspace.

Called through the C ABI and compared with the ordinary ssm_scan_fwd on two
calls in a row with different shapes and paths, so that whatever the first
call left in the shared scratch cannot leak into the second.  This file is
collected last on purpose.
"""
import ctypes

import pytest
import torch

from scan_inputs import make_inputs
from tests.gpu_util import device_args, load_ssm
from tests.parity import TOL, assert_close

pytestmark = pytest.mark.gpu


def _noalloc(ssm, a, x, out_dtype):
    Bt, D, L = x.u.shape
    N = x.A.shape[1]
    y = torch.empty((Bt, D, L), dtype=out_dtype, device="cuda")
    hL = torch.empty((Bt, D, N), dtype=torch.float32, device="cuda")
    tin = ssm.SSM_BF16 if x.in_dtype == "bf16" else ssm.SSM_F32
    tout = ssm.SSM_BF16 if out_dtype == torch.bfloat16 else ssm.SSM_F32
    shape = ssm.make_shape(Bt, D, N, L, tin, tout)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = ssm.lib.ssm_scan_fwd_noalloc(
        ctypes.byref(shape), P(a["u"]), P(a["delta_raw"]), P(a["A"]), P(a["B"]), P(a["C"]),
        P(a["D"]), P(a["z"]), P(a["delta_bias"]), P(a["h0"]), P(y), P(hL),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == ssm.SSM_OK, ssm.ssm_strerror(rc)
    torch.cuda.synchronize()
    return y, hL


def _reference(ssm, a, out_dtype):
    y, hL = ssm.ssm_scan_fwd(a["u"], a["delta_raw"], a["A"], a["B"], a["C"], a["D"], a["z"],
                             a["delta_bias"], a["h0"], out_dtype=out_dtype)
    torch.cuda.synchronize()
    return y, hL


def test_noalloc_matches_fwd_on_two_calls_in_a_row():
    ssm = load_ssm()
    calls = [
        # bf16 TMA path with an initial state and a ragged last tile
        (make_inputs(2, 96, 16, 600, seed=90, in_dtype="bf16", h0=True), torch.float32),
        # fp32 plain-load path (rows not 16-byte aligned), smaller scratch need
        (make_inputs(1, 70, 16, 77, seed=91, in_dtype="f32"), torch.float32),
    ]
    for x, out_dtype in calls:
        a = device_args(x)
        y, hL = _noalloc(ssm, a, x, out_dtype)
        y_ref, h_ref = _reference(ssm, a, out_dtype)
        tol = TOL[x.in_dtype]
        assert_close(y.float().cpu().numpy(), y_ref.float().cpu().numpy(), tol, "y")
        assert_close(hL.cpu().numpy(), h_ref.cpu().numpy(), tol, "hL")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    ssm = load_ssm()
    # a million tokens at 16 states needs a 128 MiB B/C copy: over the 32 MiB limit
    shape = ssm.make_shape(1, 1536, 16, 1 << 20, ssm.SSM_BF16, ssm.SSM_BF16)
    assert ssm.ssm_scan_workspace_bytes(shape) > ssm.NOALLOC_SCRATCH_BYTES
    V = ctypes.c_void_p
    rc = ssm.lib.ssm_scan_fwd_noalloc(ctypes.byref(shape), V(0x1000), V(0x2000), V(0x3000),
                                      V(0x4000), V(0x5000), None, None, None, None, V(0x6000),
                                      None, None)
    assert rc == ssm.SSM_ERR_WORKSPACE
    # an invalid shape reports the shape error
    bad = ssm.make_shape(1, 8, 0, 64, ssm.SSM_BF16, ssm.SSM_BF16)
    rc = ssm.lib.ssm_scan_fwd_noalloc(ctypes.byref(bad), V(0x1000), V(0x2000), V(0x3000),
                                      V(0x4000), V(0x5000), None, None, None, None, V(0x6000),
                                      None, None)
    assert rc == ssm.SSM_ERR_SHAPE
