"""Failure detection without a GPU fault: a device-side wait with a short poll
limit on a barrier nothing completes returns SSM_ERR_TIMEOUT through the
workspace status word; the context stays usable and the next call is clean."""
import pytest
import torch

from scan_inputs import make_inputs
from tests.gpu_util import device_args, load_ssm

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    ssm = load_ssm()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    ssm.ssm_debug_expired_wait(ws, spin_limit=2000)
    assert ssm.ssm_get_status(ws) == ssm.SSM_ERR_TIMEOUT
    # read-and-clear: the second read is clean
    assert ssm.ssm_get_status(ws) == ssm.SSM_OK
    # the context is still usable: a normal forward runs and reports ok
    x = make_inputs(1, 16, 16, 128, seed=30, in_dtype="bf16")
    a = device_args(x)
    shape = ssm.make_shape(1, 16, 16, 128, ssm.SSM_BF16, ssm.SSM_F32)
    need = ssm.ssm_scan_workspace_bytes(shape)
    ws2 = torch.empty(need, dtype=torch.uint8, device="cuda")
    ws2.fill_(0xAB)   # garbage status word: the call clears it
    y, hL = ssm.ssm_scan_fwd(a["u"], a["delta_raw"], a["A"], a["B"], a["C"], a["D"], a["z"],
                             a["delta_bias"], out_dtype=torch.float32, workspace=ws2)
    assert ssm.ssm_get_status(ws2) == ssm.SSM_OK
    assert torch.isfinite(y).all()
