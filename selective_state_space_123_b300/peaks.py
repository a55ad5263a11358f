"""Measured per-clock rates of the units that bound the scan (libssmpeaks.so).

The forward scan needs, per state update, one MUFU exponential and four FP32
operations, so its roofline is the slower of the MUFU ex2 rate and the FP32
rate, times the SM count and the SM clock.  `measure()` runs the
register-only probes of csrc/probe/ssm_peaks.cu (one CTA per SM, eight
independent chains per thread, cycles read from %clock64 inside each CTA)
and returns operations per SM clock cycle, which do not depend on the clock
the GPU happened to run at.
"""
from __future__ import annotations

import ctypes
import os
import statistics

_HERE = os.path.dirname(os.path.abspath(__file__))
PEAKS_LIB = os.path.join(_HERE, "libssmpeaks.so")

KINDS = {"ex2": 0, "fma": 1, "fma2": 2, "update_mix": 3, "lg2": 4, "rcp": 5}
_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(PEAKS_LIB):
            raise ImportError("libssmpeaks.so is not built; run "
                              "`python selective_state_space_123_b300/build.py`")
        lib = ctypes.CDLL(PEAKS_LIB)
        lib.ssm_peaks_launch.argtypes = [ctypes.c_int] * 4 + [ctypes.c_void_p] * 3
        lib.ssm_peaks_launch.restype = ctypes.c_longlong
        _LIB = lib
    return _LIB


def rate_per_clk_sm(kind: str, threads: int = 1024, iters: int = 2048, repeats: int = 3) -> float:
    """Median over CTAs (one per SM) of operations per clock cycle of one SM;
    the best of `repeats` launches."""
    import torch
    lib = _lib()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device="cuda")
    sink = torch.empty(sms * threads, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    best = 0.0
    for _ in range(repeats + 1):          # the first launch warms up
        ops = lib.ssm_peaks_launch(KINDS[kind], sms, threads, iters,
                                   ctypes.c_void_p(cycles.data_ptr()),
                                   ctypes.c_void_p(sink.data_ptr()), stream)
        if ops < 0:
            raise RuntimeError("ssm_peaks_launch failed (%s)" % kind)
        torch.cuda.synchronize()
        cyc = [int(c) for c in cycles.cpu().tolist()]
        rate = ops / statistics.median(cyc)
        best = max(best, rate)
    return best


def measure(threads: int = 1024) -> dict:
    """Per-clock, per-SM rates: MUFU ex2 results, FP32 lane operations
    (scalar FMA and packed f32x2 FMA), and state updates of the scan's
    update mix (delta*A, ex2, delta*u*B, state FMA, read-out FMA)."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return {
        "sms": sms,
        "threads_per_sm": threads,
        "ex2_per_clk_sm": rate_per_clk_sm("ex2", threads),
        "fp32_fma_lane_ops_per_clk_sm": rate_per_clk_sm("fma", threads),
        "fp32x2_fma_lane_ops_per_clk_sm": rate_per_clk_sm("fma2", threads),
        "update_mix_per_clk_sm": rate_per_clk_sm("update_mix", threads),
        "lg2_per_clk_sm": rate_per_clk_sm("lg2", threads),
        "rcp_per_clk_sm": rate_per_clk_sm("rcp", threads),
    }
