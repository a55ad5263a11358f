"""Benchmark of the selective scan on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Default workload (the headline): one forward selective scan -- softplus of
delta, discretisation, the recurrence, read-out, D skip, SiLU gate, final
state -- over one batch of the Mamba-1.4B layer shape: batch 4, D=4096
channels, N=16 states, L=4096 tokens, bf16 u/delta/z/B/C, fp32 A/D/bias,
fp32 arithmetic, bf16 y, fp32 final state.  Other workloads:
  mamba130m_fwd     forward, batch 8, D 1536, N 16, L 2048
  mamba2p8b_fwd     forward, batch 2, D 5120, N 16, L 8192
  mamba2p8b_fwdbwd  forward then backward (all gradients), same shape
  million_fwd       forward, batch 1, D 1536, N 16, L 1,048,576
  million_fwdbwd    forward then backward (all gradients), same shape (both segmented)
  mamba1p4b_conv_fwdbwd  the conv-prologue forward and its backward (dx, conv weight grads)
  decode_step       one recurrent step, batch 256, D 5120, N 16, state in place
Inputs are synthetic (seeded, drawn on the device) and resident in HBM before
the timed region; every workload's inputs exceed L2 (126 MB) except where the
JSON line says otherwise, in which case L2 is flushed between steps.

The JSON line (rank 0) reports B*D*L*N state updates per second for the whole
job (N GPUs run independent replicas: the channels of different sequences
never interact, so the work shards with no collective), the roofline of the
dominant kernel, clocks sampled during the timed region, the end-to-end rate
through the C ABI with host buffers (pinned host -> device copies of every
input and the device -> host read of every output inside the timed region),
and the fp64 CPU oracle timed on a bounded sample as the CPU baseline.
`--impl reference` times that oracle alone (this method has no runnable
reference implementation; the oracle is the reference arm).
"""
from __future__ import annotations

import argparse
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOADS = {
    "mamba1p4b_fwd": dict(mode="fwd", Bt=4, D=4096, N=16, L=4096, seed=2,
                          title="Mamba-1.4B layer forward"),
    "mamba130m_fwd": dict(mode="fwd", Bt=8, D=1536, N=16, L=2048, seed=1,
                          title="Mamba-130M layer forward"),
    "mamba2p8b_fwd": dict(mode="fwd", Bt=2, D=5120, N=16, L=8192, seed=3,
                          title="Mamba-2.8B layer forward"),
    "mamba2p8b_fwdbwd": dict(mode="fwdbwd", Bt=2, D=5120, N=16, L=8192, seed=3,
                             title="Mamba-2.8B layer forward + backward"),
    "million_fwd": dict(mode="fwd", Bt=1, D=1536, N=16, L=1 << 20, seed=4,
                        title="million-length forward"),
    # forward (B/C preparation, tail search, summary pass, carry, scan) +
    # segmented backward (B/C preparation, tail search, forward summary,
    # carry, head search, adjoint summary, carry, forward sweep, tangent
    # carry, reverse sweep)
    "million_fwdbwd": dict(mode="fwdbwd", Bt=1, D=1536, N=16, L=1 << 20, seed=4, launches=15,
                           title="million-length forward + backward"),
    "decode_step": dict(mode="step", Bt=256, D=5120, N=16, L=1, seed=4,
                        title="single-token decode step"),
    "mamba1p4b_conv_fwd": dict(mode="fwd", conv=4, Bt=4, D=4096, N=16, L=4096, seed=2,
                               title="Mamba-1.4B layer forward from the conv branch input "
                                     "(width-4 causal conv + SiLU fused)"),
    # 17 sequences of 256..16384 tokens (log-uniform) packed into one row;
    # the planner cuts the row into 4 segments at 148 SMs: B/C preparation,
    # sequence check, tail search, summary pass, carry, scan = 6 launches
    # two directions, each with its own delta/A/B/C/D/bias (B/C preparation
    # twice, right-to-left pass, left-to-right pass = 4 launches)
    # conv forward (B/C preparation, scan) + conv backward (B/C preparation,
    # forward sweep, reverse sweep, prologue's reverse mode)
    "mamba1p4b_conv_fwdbwd": dict(mode="fwdbwd", conv=4, Bt=4, D=4096, N=16, L=4096, seed=2,
                                  launches=6,
                                  title="Mamba-1.4B layer forward + backward from the conv branch "
                                        "input (width-4 causal conv + SiLU fused, and its "
                                        "reverse mode)"),
    "bidir_mamba1p4b_fwd": dict(mode="fwd", bidir=True, Bt=4, D=4096, N=16, L=4096, seed=6,
                                launches=4,
                                title="Mamba-1.4B layer bidirectional scan (left-to-right + "
                                      "right-to-left)"),
    "packed_mamba1p4b_fwd": dict(mode="fwd", varlen=True, Bt=1, D=4096, N=16, L=65536, seed=5,
                                 launches=6,
                                 title="Mamba-1.4B layer forward over packed sequences of mixed "
                                       "length"),
    # forward (6 launches as above) + packed backward (B/C preparation,
    # sequence check, forward sweep, reverse sweep)
    "packed_mamba1p4b_fwdbwd": dict(mode="fwdbwd", varlen=True, Bt=1, D=4096, N=16, L=65536,
                                    seed=5, launches=10,
                                    title="Mamba-1.4B layer forward + backward over packed "
                                          "sequences of mixed length"),
    # forward (4 launches) + backward of both directions: left-to-right
    # backward (3), status fold, 6 token reversals, right-to-left backward (3),
    # status fold, combine, 2 reversals of dB/dC
    "bidir_mamba1p4b_fwdbwd": dict(mode="fwdbwd", bidir=True, Bt=4, D=4096, N=16, L=4096, seed=6,
                                   launches=21,
                                   title="Mamba-1.4B layer bidirectional scan, forward + backward"),
}
WORKLOAD = WORKLOADS["mamba1p4b_fwd"]
METRIC = "selective scan: achieved HBM GB/s (% of roofline) and B*D*L*N state updates/s"
UNIT = "state updates/s"
# MUFU ex2 results per clock per SM, nominal for the B300; the roofline uses
# the rate the register-only probe (selective_state_space_123_b300/peaks.py)
# measures in the same process, and reports the nominal fraction beside it
SFU_EX2_PER_CLK_SM = 32
SMS = 148
L2_BYTES = 126 * 1024 * 1024


# dram traffic per launch of a kernel, from an ncu capture recorded in
# profiles/traffic.json together with a hash of the kernel's sources; it is
# reported only while those sources are unchanged
KERNEL_SOURCES = {
    "fwd_kernel": ["ssm_fwd.cuh", "ssm_fwd_launch.cuh", "ssm_fwd_np16.cu", "ssm_common.cuh",
                   "ssm_kernels.cuh"],
    "fwdbwd": ["ssm_fwd.cuh", "ssm_fwd_launch.cuh", "ssm_fwd_np16.cu", "ssm_bwd.cuh", "ssm_bwd_launch.cuh",
               "ssm_bwd_np16.cu", "ssm_common.cuh", "ssm_kernels.cuh"],
    "step_dec16_kernel": ["ssm_step.cu", "ssm_common.cuh", "ssm_kernels.cuh"],
}


def kernel_source_hash(kind):
    """Hash of the sources a kernel is built from, comments and blank space
    left out (a comment edit does not change the kernel)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "selective_state_space_123_b300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def rank_seed(seed, rank):
    """Each rank's replica draws its own inputs."""
    return seed + 1000 * rank


def max_over_ranks(x, world):
    """The largest of the ranks' values: the job is as slow as its slowest
    rank (NCCL on the GPUs, gloo on the host)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, updates_per_rank, ms_per_step):
    """Whole-job state updates per second: every rank runs one replica of
    the workload, so the job does world * updates_per_rank per step."""
    return world * updates_per_rank / (ms_per_step * 1e-3)


def recorded_traffic(kind, workload, seqlen=None):
    if seqlen is not None and seqlen != WORKLOADS.get(workload, {}).get("L"):
        return None     # the record is for the workload's own sequence length
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[kind + ":" + workload]
    except Exception:
        return None
    return rec["bytes_per_launch"] if rec.get("src_hash") == kernel_source_hash(kind) else None


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


def fwd_bytes(Bt, D, N, L, ein=2, eout=2):
    """Algorithmic bytes of one forward: read u, delta_raw, z (Bt,D,L), B, C
    (Bt,N,L), A (D,N), D and bias (D) once; write y (Bt,D,L) and h_L (Bt,D,N)."""
    return (3 * Bt * D * L * ein + 2 * Bt * N * L * ein + D * N * 4 + 2 * D * 4
            + Bt * D * L * eout + Bt * D * N * 4)


def bwd_bytes(Bt, D, N, L, ein=2, eout=2):
    """Algorithmic bytes of one backward: read u, delta_raw, z, dy (Bt,D,L), B,
    C (Bt,N,L), A, D, bias once; write du, ddelta_raw, dz (Bt,D,L), dB, dC
    (Bt,N,L) fp32, dA (D,N), dD, ddelta_bias (D), dh0 (Bt,D,N)."""
    return (4 * Bt * D * L * ein + 2 * Bt * N * L * ein + D * N * 4 + 2 * D * 4
            + 3 * Bt * D * L * eout + 2 * Bt * N * L * 4 + D * N * 4 + 2 * D * 4
            + Bt * D * N * 4)


def step_bytes(Bt, D, N, ein=2, eout=2):
    """Algorithmic bytes of one decode step: state read and written, u,
    delta_raw, z (Bt,D), B, C (Bt,N), A, D, bias read, y (Bt,D) written."""
    return 2 * Bt * D * N * 4 + 3 * Bt * D * ein + 2 * Bt * N * ein + D * N * 4 + 2 * D * 4 \
        + Bt * D * eout


# --------------------------------------------------------------- clocks ---
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def wait_first(self, limit_s=3.0):
        """Wait (bounded) until the sampler has produced its first line."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < limit_s:
            time.sleep(0.02)

    def stop(self, t_begin=None, t_end=None):
        """Summary of the samples taken between t_begin and t_end (wall
        clock; a sample lands up to one period after its reading), or of the
        nearest samples before and after when the region is shorter than the
        sampling period."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        lines = self.lines
        if t_begin is not None and t_end is not None:
            inside = [(t, ln) for t, ln in lines if t_begin <= t <= t_end + 0.15]
            if not inside:
                before = [(t, ln) for t, ln in lines if t < t_begin][-1:]
                after = [(t, ln) for t, ln in lines if t > t_end][:1]
                inside = before + after
            lines = inside
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------- CPU oracle ---
_INPUT_CACHE = {}


def _oracle_worker(args):
    """Run the oracle on a slice of channels; returns (updates, seconds of the
    oracle call alone -- drawing the inputs is not timed, and is cached)."""
    mode, seed, Bt, D, N, L, chans = args[:7]
    conv_k = args[7] if len(args) > 7 else 0
    varlen = args[8] if len(args) > 8 else False
    bidir = args[9] if len(args) > 9 else False
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import oracle
    from scan_inputs import make_inputs, make_step_inputs
    key = (mode, seed, Bt, D, N, L, tuple(chans), bidir)
    x = _INPUT_CACHE.get(key)
    if x is None:
        if len(_INPUT_CACHE) > 64:
            _INPUT_CACHE.clear()
        if mode == "step":
            x = make_step_inputs(Bt, D, N, seed=seed, in_dtype="bf16", channels=chans)
        else:
            x = make_inputs(Bt, D, N, L, seed=seed, in_dtype="bf16", channels=chans,
                            dy=(mode == "fwdbwd"))
            if bidir:
                x = (x, make_inputs(Bt, D, N, L, seed=seed + 1, in_dtype="bf16", channels=chans))
        _INPUT_CACHE[key] = x
    cw = cb = None
    if conv_k:
        import numpy as np
        g = np.random.default_rng(seed + 1000)
        cw = (0.5 * g.standard_normal((D, conv_k))).astype(np.float32)[chans]
        cb = (0.1 * g.standard_normal(D)).astype(np.float32)[chans]
    t0 = time.perf_counter()
    if bidir:
        xf, xr = x
        d = lambda v: dict(delta_raw=v.delta_raw, A=v.A, Bm=v.Bm, Cm=v.Cm, Dv=v.Dv,
                           delta_bias=v.delta_bias)
        oracle.scan_fwd_bidir(xf.u, xf.z, d(xf), d(xr))
        if mode == "fwdbwd":
            oracle.scan_bwd_bidir(xf.u, xf.z, d(xf), d(xr), xf.dy)
        return 2 * Bt * len(chans) * N * L, time.perf_counter() - t0
    if varlen:
        from scan_inputs import packed_seqlens
        cu = packed_seqlens(L, seed=seed)
        t0 = time.perf_counter()
        oracle.scan_fwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, cu, x.Dv, x.z, x.delta_bias)
        if mode == "fwdbwd":
            oracle.scan_bwd_varlen(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, cu, x.Dv, x.z,
                                   x.delta_bias)
    elif conv_k:
        oracle.scan_fwd_conv(x.u, cw, cb, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
        if mode == "fwdbwd":
            oracle.scan_bwd_conv(x.u, cw, cb, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z,
                                 x.delta_bias)
    elif mode == "fwd":
        oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
    elif mode == "fwdbwd":
        oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
        oracle.scan_bwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.dy, x.Dv, x.z, x.delta_bias,
                        x.h0, None)
    else:
        oracle.scan_step(x["u"], x["delta_raw"], x["A"], x["Bm"], x["Cm"], x["state"],
                         x["Dv"], x["z"], x["delta_bias"])
    return Bt * len(chans) * N * L, time.perf_counter() - t0


class OracleTimer:
    """The fp64 oracle as it stands, timed on disjoint channel subsets of the
    workload, one spawned process per host core (the pool is created with
    'spawn', so it is safe next to a CUDA context)."""

    def __init__(self, cores=None):
        import oracle
        oracle.build()
        self.cores = cores or os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.cores)
        w = WORKLOAD
        self.bt = w["Bt"] if w["mode"] == "step" else 1   # decode: all sequences of a channel
        warm_L = min(64, w["L"])
        self.conv_k = w.get("conv", 0)
        self.varlen = bool(w.get("varlen"))
        self.bidir = bool(w.get("bidir"))
        self.pool.map(_oracle_worker, [(w["mode"], w["seed"], self.bt, w["D"], w["N"], warm_L,
                                        [0], self.conv_k, self.varlen, self.bidir)] * self.cores)
        probe = 16 if w["mode"] == "step" else 1
        _, t = _oracle_worker((w["mode"], w["seed"], self.bt, w["D"], w["N"], w["L"],
                               list(range(probe)), self.conv_k, self.varlen, self.bidir))
        self.t_channel = t / probe
        self.next = 0

    def measure(self, seconds_per_core, fixed=False):
        """Oracle throughput on about `seconds_per_core` of work per process.
        fixed=True reuses the same channel sample every call (the reference
        arm's steps); otherwise the sample advances through the channels."""
        w = WORKLOAD
        per = max(1, min(w["D"], int(seconds_per_core / max(self.t_channel, 1e-7))))
        jobs = []
        start = 0 if fixed else self.next
        for i in range(self.cores):
            jobs.append((w["mode"], w["seed"], self.bt, w["D"], w["N"], w["L"],
                         [(start + i * per + j) % w["D"] for j in range(per)], self.conv_k,
                         self.varlen, self.bidir))
        if not fixed:
            self.next = (start + per * self.cores) % w["D"]
        res = self.pool.map(_oracle_worker, jobs)
        upd = sum(r[0] for r in res)
        busy = max(r[1] for r in res)
        what = {"fwd": "forward", "fwdbwd": "forward + backward", "step": "decode step"}[w["mode"]]
        if self.conv_k:
            what = "conv prologue + " + what
        if self.varlen:
            what = "packed-sequence " + what
        if self.bidir:
            what = "bidirectional scan " + what
        return {"value": upd / busy, "unit": UNIT, "cores": self.cores, "kind": "oracle",
                "sample": "%s of %d (channel, batch row) sequences x %d tokens x %d states of the "
                          "%s workload (channels taken in turn from its %d, batch row 0%s), one "
                          "spawned process per core (%d each); slowest process %.2f s"
                          % (what, per * self.cores * self.bt, w["L"], w["N"], w["name"], w["D"],
                             " .. %d" % (self.bt - 1) if self.bt > 1 else "", per * self.bt, busy)}

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_oracle_rate(target_seconds=12.0):
    t = OracleTimer()
    try:
        return t.measure(target_seconds)
    finally:
        t.close()


# ------------------------------------------------------------------ GPU ---
class Workload:
    """Device buffers and the step of one workload (inputs drawn on the device)."""

    def __init__(self, ssm, w, rank):
        import torch
        from scan_inputs import device_inputs
        self.ssm, self.w = ssm, w
        Bt, D, N, L = w["Bt"], w["D"], w["N"], w["L"]
        self.mode = w["mode"]
        # forward variants: conv prologue width, packed-sequence starts, two directions
        self.conv_k, self.cu, self.bidir = w.get("conv", 0), None, bool(w.get("bidir"))
        bf = torch.bfloat16
        if self.mode == "step":
            a = device_inputs(Bt, D, N, 1, seed=rank_seed(w["seed"], rank), in_dtype="bf16", h0=True)
            self.inp = {"u": a["u"][:, :, 0].contiguous(), "delta_raw": a["delta_raw"][:, :, 0].contiguous(),
                        "z": a["z"][:, :, 0].contiguous(), "Bm": a["Bm"][:, :, 0].contiguous(),
                        "Cm": a["Cm"][:, :, 0].contiguous(), "A": a["A"], "Dv": a["Dv"],
                        "delta_bias": a["delta_bias"]}
            self.state = a["h0"]
            # the step's working set (92 MB) fits in L2: successive steps
            # rotate through 4 copies of the state and the per-token inputs
            # (368 MB in all), so every step reads them from HBM
            self.rot = [(dict(self.inp), self.state)]
            for _ in range(3):
                self.rot.append(({k: (v.clone() if k in ("u", "delta_raw", "z", "Bm", "Cm") else v)
                                  for k, v in self.inp.items()}, self.state.clone()))
            self.rot_i = 0
            self.graphs = None
            self.y = torch.empty(Bt, D, dtype=bf, device="cuda")
            self.ws = None
            self.bytes = step_bytes(Bt, D, N)
            self.exps = Bt * D * N
            self.launches = 1
            self.outs = [self.y, self.state]
        else:
            a = device_inputs(Bt, D, N, L, seed=rank_seed(w["seed"], rank), in_dtype="bf16",
                              dy=(self.mode == "fwdbwd"))
            self.inp = {k: v for k, v in a.items() if v is not None}
            self.y = torch.empty(Bt, D, L, dtype=bf, device="cuda")
            self.hL = torch.empty(Bt, D, N, dtype=torch.float32, device="cuda")
            shape = ssm.make_shape(Bt, D, N, L, ssm.SSM_BF16, ssm.SSM_BF16)
            nb = ssm.ssm_scan_workspace_bytes(
                shape, (4 if self.conv_k else 1) if self.mode == "fwdbwd" else 0)
            nb = max(nb, ssm.ssm_scan_workspace_bytes(shape, False))
            self.ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
            self.bytes = fwd_bytes(Bt, D, N, L)
            self.exps = Bt * D * L * N
            if self.bidir:
                # the right-to-left direction's own parameters (u and z are shared)
                r = device_inputs(Bt, D, N, L, seed=rank_seed(w["seed"], rank) + 1, in_dtype="bf16")
                for k in ("delta_raw", "Bm", "Cm", "A", "Dv", "delta_bias"):
                    self.inp[k + "_r"] = r[k]
                del r
                self.hL_r = torch.empty(Bt, D, N, dtype=torch.float32, device="cuda")
                nb = ssm.ssm_scan_workspace_bytes(shape, 2)
                if self.mode == "fwdbwd":
                    nb = max(nb, ssm.ssm_scan_workspace_bytes(shape, 3))
                self.ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
                # second direction: delta_raw, B, C, A, D, bias read, final state written
                self.bytes += (Bt * D * L * 2 + 2 * Bt * N * L * 2 + D * N * 4 + 2 * D * 4
                               + Bt * D * N * 4)
                self.exps *= 2
            if w.get("varlen"):
                from scan_inputs import packed_seqlens
                self.cu = torch.tensor(packed_seqlens(L, seed=rank_seed(w["seed"], rank)),
                                       dtype=torch.int32, device="cuda")
                nseq = self.cu.numel() - 1
                # one final state per sequence, and the starts
                self.hL = torch.empty(nseq, Bt, D, N, dtype=torch.float32, device="cuda")
                self.bytes += (nseq - 1) * Bt * D * N * 4 + (nseq + 1) * 4
            if self.conv_k:
                # depthwise conv weights (D, K) and bias (D), read once
                g = torch.Generator(device="cuda")
                g.manual_seed(rank_seed(w["seed"], rank) + 1000)
                self.conv_w = 0.5 * torch.randn(D, self.conv_k, generator=g, device="cuda")
                self.conv_b = 0.1 * torch.randn(D, generator=g, device="cuda")
                self.bytes += D * (self.conv_k + 1) * 4
            # B/C preparation + scan; the million-length sequence takes the
            # segmented plan (preparation, tail search, summary pass, carry,
            # scan)
            self.launches = w.get("launches", 5 if L >= (1 << 18) and Bt * D <= 4096 else 2)
            self.outs = [self.y, self.hL]
            self.grads = None
            if self.mode == "fwdbwd":
                # the backward's algorithmic bytes, once per direction (each
                # reads its inputs and dy and writes its gradients)
                self.bytes += bwd_bytes(Bt, D, N, L) * (2 if self.bidir else 1)
                self.exps *= 3     # forward, and the backward's two sweeps
                if "launches" not in w:
                    self.launches += 3
        # state updates per step (the bidirectional scan runs two)
        self.updates = Bt * D * L * N * (2 if self.bidir else 1)
        if self.bidir:
            self.outs.append(self.hL_r)

    def capture_graphs(self):
        """Decode: one CUDA graph per rotating copy, each holding one
        ssm_scan_step call.  A decode step's kernel is shorter than the host
        work of one eager call (argument checks, ctypes, tensor-map encoding,
        launch), so eager steps would time the host; a serving loop replays
        graphs the same way."""
        import torch
        graphs = []
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(len(self.rot)):
                self.step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        for _ in range(len(self.rot)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step()
            graphs.append(g)
        torch.cuda.synchronize()
        self.graphs = graphs

    def step(self, inp=None):
        ssm, a = self.ssm, (inp or self.inp)
        import torch
        if self.mode == "step":
            state = self.state
            if inp is None:
                if self.graphs is not None:
                    self.graphs[self.rot_i].replay()
                    self.rot_i = (self.rot_i + 1) % len(self.rot)
                    return
                a, state = self.rot[self.rot_i]
                self.rot_i = (self.rot_i + 1) % len(self.rot)
            ssm.ssm_scan_step(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], state,
                              a["Dv"], a["z"], a["delta_bias"], out_dtype=torch.bfloat16, y=self.y)
            return
        if self.bidir:
            f = dict(delta_raw=a["delta_raw"], A=a["A"], B=a["Bm"], C=a["Cm"], D=a["Dv"],
                     delta_bias=a["delta_bias"])
            r = dict(delta_raw=a["delta_raw_r"], A=a["A_r"], B=a["Bm_r"], C=a["Cm_r"], D=a["Dv_r"],
                     delta_bias=a["delta_bias_r"])
            ssm.ssm_scan_fwd_bidir(a["u"], a["z"], f, r, out_dtype=torch.bfloat16, y=self.y,
                                   hL=self.hL, hL_r=self.hL_r, workspace=self.ws)
            if self.mode == "fwdbwd":
                self.grads = ssm.ssm_scan_bwd_bidir(a["u"], a["z"], f, r, a["dy"],
                                                    out_dtype=torch.bfloat16, workspace=self.ws)
            return
        if self.cu is not None:
            ssm.ssm_scan_fwd_varlen(a["u"], self.cu, a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["Dv"],
                                    a["z"], a["delta_bias"], None, out_dtype=torch.bfloat16, y=self.y,
                                    hL=self.hL, workspace=self.ws)
            if self.mode == "fwdbwd":
                self.grads = ssm.ssm_scan_bwd_varlen(a["u"], self.cu, a["delta_raw"], a["A"], a["Bm"],
                                                     a["Cm"], a["dy"], a["Dv"], a["z"], a["delta_bias"],
                                                     out_dtype=torch.bfloat16, workspace=self.ws)
            return
        if self.conv_k:
            # u holds the conv branch input x
            ssm.ssm_scan_fwd_conv(a["u"], self.conv_w, self.conv_b, a["delta_raw"], a["A"], a["Bm"],
                                  a["Cm"], a["Dv"], a["z"], a["delta_bias"], None,
                                  out_dtype=torch.bfloat16, y=self.y, hL=self.hL, workspace=self.ws)
            if self.mode == "fwdbwd":
                self.grads = ssm.ssm_scan_bwd_conv(a["u"], self.conv_w, self.conv_b, a["delta_raw"],
                                                   a["A"], a["Bm"], a["Cm"], a["dy"], a["Dv"], a["z"],
                                                   a["delta_bias"], None, None,
                                                   out_dtype=torch.bfloat16, workspace=self.ws)
            return
        ssm.ssm_scan_fwd(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["Dv"], a["z"],
                         a["delta_bias"], None, out_dtype=torch.bfloat16, y=self.y, hL=self.hL,
                         workspace=self.ws)
        if self.mode == "fwdbwd":
            self.grads = ssm.ssm_scan_bwd(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["dy"],
                                          a["Dv"], a["z"], a["delta_bias"], None, None,
                                          out_dtype=torch.bfloat16, workspace=self.ws)

    def results(self):
        outs = list(self.outs)
        if self.mode == "fwdbwd" and self.grads is not None:
            parts = self.grads if isinstance(self.grads, tuple) else (self.grads,)
            for g in parts:
                outs += [v for v in g.values() if v is not None]
        return outs


def pipelined_e2e(ssm, wl, host, dev, outs_host, state_host, ngroups=4):
    """End-to-end step through the public API with the host copies overlapped:
    the batch rows (or, for a single sequence, the channels) are split into
    `ngroups` groups that alternate between two streams; each group copies
    its inputs in, runs its own call (decode step, forward, conv-prologue
    forward, packed-sequence forward or bidirectional scan) and copies its
    outputs back, so one group's copies overlap another's scan and the two
    copy directions run at once.  Inputs shared by all groups are copied
    first; the conv weights stay resident like the other layer parameters of
    a serving loop do."""
    import torch
    bf = torch.bfloat16
    cur = torch.cuda.current_stream()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    Bt, D, N, L = wl.w["Bt"], wl.w["D"], wl.w["N"], wl.w["L"]
    by_batch = Bt > 1
    n = Bt if by_batch else D
    ngroups = max(1, min(ngroups, n))
    bounds = [(i * n // ngroups, (i + 1) * n // ngroups) for i in range(ngroups)]
    step = wl.mode == "step"
    # per group: which tensors are sliced (batch rows or channels)
    per_row = [k for k in ("u", "delta_raw", "z", "delta_raw_r") if k in host]
    per_b = [k for k in ("Bm", "Cm", "Bm_r", "Cm_r") if k in host]
    per_d = [k for k in ("A", "Dv", "delta_bias", "A_r", "Dv_r", "delta_bias_r") if k in host]
    state_dev = wl.state if step else None
    y_dev, y_host = wl.outs[0], outs_host[0]
    shared = (per_d if by_batch else per_b)
    varlen = wl.cu is not None
    nseq = wl.cu.numel() - 1 if varlen else 0

    def cut(t, lo, hi):
        return t[lo:hi] if by_batch else t[:, lo:hi]

    ws = hv = None
    if not step:
        gb = (bounds[0][1] - bounds[0][0]) if by_batch else Bt
        gd = D if by_batch else max(hi - lo for lo, hi in bounds)
        shape = ssm.make_shape(gb, gd, N, L, ssm.SSM_BF16, ssm.SSM_BF16)
        nb = ssm.ssm_scan_workspace_bytes(shape, 2 if wl.bidir else 0)
        ws = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in streams]
        if varlen:
            # packed final states (nseq, Bt, D, N): one contiguous block per
            # channel group, read back as such
            hv = [torch.empty(nseq, Bt, hi - lo, N, dtype=torch.float32, device="cuda")
                  for lo, hi in bounds]

    def one_step():
        for k in shared:
            dev[k].copy_(host[k], non_blocking=True)
        for s_ in streams:
            s_.wait_stream(cur)
        for gi, (lo, hi) in enumerate(bounds):
            s_ = streams[gi % 2]
            with torch.cuda.stream(s_):
                a = {}
                for k in per_row:
                    a[k] = cut(dev[k], lo, hi)
                    a[k].copy_(cut(host[k], lo, hi), non_blocking=True)
                for k in per_b:
                    if by_batch:
                        a[k] = dev[k][lo:hi]
                        a[k].copy_(host[k][lo:hi], non_blocking=True)
                    else:
                        a[k] = dev[k]
                for k in per_d:
                    if by_batch:
                        a[k] = dev[k]
                    else:
                        a[k] = dev[k][lo:hi]
                        a[k].copy_(host[k][lo:hi], non_blocking=True)
                yv = cut(y_dev, lo, hi)
                if step:
                    st = cut(state_dev, lo, hi)
                    st.copy_(cut(state_host, lo, hi), non_blocking=True)
                    ssm.ssm_scan_step(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], st, a["Dv"],
                                      a["z"], a["delta_bias"], out_dtype=bf, y=yv, stream=s_)
                    cut(y_host, lo, hi).copy_(yv, non_blocking=True)
                    cut(outs_host[1], lo, hi).copy_(st, non_blocking=True)
                    continue
                w_ = ws[gi % 2]
                if wl.bidir:
                    f = dict(delta_raw=a["delta_raw"], A=a["A"], B=a["Bm"], C=a["Cm"], D=a["Dv"],
                             delta_bias=a["delta_bias"])
                    r = dict(delta_raw=a["delta_raw_r"], A=a["A_r"], B=a["Bm_r"], C=a["Cm_r"],
                             D=a["Dv_r"], delta_bias=a["delta_bias_r"])
                    h1, h2 = cut(wl.outs[1], lo, hi), cut(wl.outs[2], lo, hi)
                    ssm.ssm_scan_fwd_bidir(a["u"], a["z"], f, r, out_dtype=bf, y=yv, hL=h1, hL_r=h2,
                                           workspace=w_, stream=s_)
                    outs = [(yv, cut(y_host, lo, hi)), (h1, cut(outs_host[1], lo, hi)),
                            (h2, cut(outs_host[2], lo, hi))]
                elif varlen:
                    ssm.ssm_scan_fwd_varlen(a["u"], wl.cu, a["delta_raw"], a["A"], a["Bm"], a["Cm"],
                                            a["Dv"], a["z"], a["delta_bias"], None, out_dtype=bf,
                                            y=yv, hL=hv[gi], workspace=w_, stream=s_)
                    hh = outs_host[1].view(-1)[nseq * Bt * lo * N:nseq * Bt * hi * N].view_as(hv[gi])
                    outs = [(yv, cut(y_host, lo, hi)), (hv[gi], hh)]
                else:
                    h1 = cut(wl.outs[1], lo, hi)
                    if wl.conv_k:
                        cw = wl.conv_w if by_batch else wl.conv_w[lo:hi]
                        cb = wl.conv_b if by_batch else wl.conv_b[lo:hi]
                        ssm.ssm_scan_fwd_conv(a["u"], cw, cb, a["delta_raw"], a["A"], a["Bm"],
                                              a["Cm"], a["Dv"], a["z"], a["delta_bias"], None,
                                              out_dtype=bf, y=yv, hL=h1, workspace=w_, stream=s_)
                    else:
                        ssm.ssm_scan_fwd(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["Dv"],
                                         a["z"], a["delta_bias"], None, out_dtype=bf, y=yv, hL=h1,
                                         workspace=w_, stream=s_)
                    outs = [(yv, cut(y_host, lo, hi)), (h1, cut(outs_host[1], lo, hi))]
                for d_, h_ in outs:
                    h_.copy_(d_, non_blocking=True)
        for s_ in streams:
            cur.wait_stream(s_)

    return one_step


def pipelined_e2e_fwdbwd(ssm, wl, host, dev, ngroups=4):
    """End-to-end forward + backward through the public API with the host
    copies overlapped: the batch rows (or, for a single row, the channels)
    are split into up to `ngroups` groups that alternate between two
    streams; each group copies its inputs in, runs the forward and the
    backward of its part (plain, conv prologue, packed sequences or
    bidirectional) and copies its outputs and gradients back, so one group's
    copies overlap another's kernels and the two copy directions run at once.
    Gradients that sum over the split dimension (per channel: dA, dD,
    ddelta_bias, the conv weights', when the batch rows are split; dB and dC
    when the channels are) are added over the groups on the device and copied
    back once.  Each output is copied into one pinned host buffer, group after
    group.  Returns (step, d2h bytes per step, groups, {key: host buffer})."""
    import torch
    bf = torch.bfloat16
    cur = torch.cuda.current_stream()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    Bt, D, N, L = wl.w["Bt"], wl.w["D"], wl.w["N"], wl.w["L"]
    by_batch = Bt > 1
    n = Bt if by_batch else D
    ngroups = max(1, min(ngroups, n))
    bounds = [(i * n // ngroups, (i + 1) * n // ngroups) for i in range(ngroups)]
    varlen = wl.cu is not None
    nseq = wl.cu.numel() - 1 if varlen else 0
    row_keys = [k for k in ("u", "delta_raw", "z", "dy", "delta_raw_r") if k in host]
    b_keys = [k for k in ("Bm", "Cm", "Bm_r", "Cm_r") if k in host]
    d_keys = [k for k in ("A", "Dv", "delta_bias", "A_r", "Dv_r", "delta_bias_r") if k in host]
    sliced = row_keys + (b_keys if by_batch else d_keys)
    shared = [k for k in host if k not in sliced]
    summed = ("dA", "dD", "ddelta_bias", "dconv_w", "dconv_b") if by_batch else ("dB", "dC")

    def cut(t, lo, hi):   # a (Bt, D, ...) tensor's part
        return t[lo:hi] if by_batch else t[:, lo:hi]

    def part(k, t, lo, hi):   # an input's part
        if k in row_keys:
            return cut(t, lo, hi)
        return t[lo:hi]

    gsize = max(hi - lo for lo, hi in bounds)
    shape = ssm.make_shape(gsize if by_batch else Bt, D if by_batch else gsize, N, L,
                           ssm.SSM_BF16, ssm.SSM_BF16)
    flag = 3 if wl.bidir else (4 if wl.conv_k else 1)
    nb = max(ssm.ssm_scan_workspace_bytes(shape, flag),
             ssm.ssm_scan_workspace_bytes(shape, 2 if wl.bidir else 0))
    ws = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in streams]
    hv = ([torch.empty(nseq, Bt, hi - lo, N, dtype=torch.float32, device="cuda")
           for lo, hi in bounds] if varlen else None)
    out_host = {}   # key -> flat pinned host buffer of the whole output

    def run_group(gi, a, p, lo, hi, s_):
        """Forward and backward of group gi on stream s_: returns the forward's
        outputs and the backward's gradient dicts."""
        w_ = ws[gi % 2]
        y = cut(wl.y, lo, hi)
        if wl.bidir:
            h1, h2 = cut(wl.hL, lo, hi), cut(wl.hL_r, lo, hi)
            f = dict(delta_raw=a["delta_raw"], A=p["A"], B=p["Bm"], C=p["Cm"], D=p["Dv"],
                     delta_bias=p["delta_bias"])
            r = dict(delta_raw=a["delta_raw_r"], A=p["A_r"], B=p["Bm_r"], C=p["Cm_r"],
                     D=p["Dv_r"], delta_bias=p["delta_bias_r"])
            ssm.ssm_scan_fwd_bidir(a["u"], a["z"], f, r, out_dtype=bf, y=y, hL=h1, hL_r=h2,
                                   workspace=w_, stream=s_)
            g = ssm.ssm_scan_bwd_bidir(a["u"], a["z"], f, r, a["dy"], out_dtype=bf,
                                       workspace=w_, stream=s_)
            return {"y": y, "hL": h1, "hL_r": h2}, g
        if varlen:
            h1 = hv[gi]
            ssm.ssm_scan_fwd_varlen(a["u"], wl.cu, a["delta_raw"], p["A"], p["Bm"], p["Cm"],
                                    p["Dv"], a["z"], p["delta_bias"], None, out_dtype=bf, y=y,
                                    hL=h1, workspace=w_, stream=s_)
            g = ssm.ssm_scan_bwd_varlen(a["u"], wl.cu, a["delta_raw"], p["A"], p["Bm"], p["Cm"],
                                        a["dy"], p["Dv"], a["z"], p["delta_bias"], out_dtype=bf,
                                        workspace=w_, stream=s_)
            return {"y": y, "hL": h1}, (g,)
        h1 = cut(wl.hL, lo, hi)
        if wl.conv_k:
            cw = wl.conv_w if by_batch else wl.conv_w[lo:hi]
            cb = wl.conv_b if by_batch else wl.conv_b[lo:hi]
            ssm.ssm_scan_fwd_conv(a["u"], cw, cb, a["delta_raw"], p["A"], p["Bm"], p["Cm"],
                                  p["Dv"], a["z"], p["delta_bias"], None, out_dtype=bf, y=y,
                                  hL=h1, workspace=w_, stream=s_)
            g = ssm.ssm_scan_bwd_conv(a["u"], cw, cb, a["delta_raw"], p["A"], p["Bm"], p["Cm"],
                                      a["dy"], p["Dv"], a["z"], p["delta_bias"], None, None,
                                      out_dtype=bf, workspace=w_, stream=s_)
            return {"y": y, "hL": h1}, (g,)
        ssm.ssm_scan_fwd(a["u"], a["delta_raw"], p["A"], p["Bm"], p["Cm"], p["Dv"], a["z"],
                         p["delta_bias"], None, out_dtype=bf, y=y, hL=h1, workspace=w_, stream=s_)
        g = ssm.ssm_scan_bwd(a["u"], a["delta_raw"], p["A"], p["Bm"], p["Cm"], a["dy"], p["Dv"],
                             a["z"], p["delta_bias"], None, None, out_dtype=bf, workspace=w_,
                             stream=s_)
        return {"y": y, "hL": h1}, (g,)

    sizes, dtypes = {}, {}   # key -> total elements and type, found by the first step

    def one_step():
        for k in shared:
            dev[k].copy_(host[k], non_blocking=True)
        for s_ in streams:
            s_.wait_stream(cur)
        offs = {}
        partial = []   # per group: {key: gradient summed over the groups}
        for gi, (lo, hi) in enumerate(bounds):
            s_ = streams[gi % 2]
            with torch.cuda.stream(s_):
                a, p = {}, dict(dev)
                for k in sliced:
                    t = part(k, dev[k], lo, hi)
                    t.copy_(part(k, host[k], lo, hi), non_blocking=True)
                    if k in row_keys:
                        a[k] = t
                    else:
                        p[k] = t
                a.setdefault("z", None)   # (a workload without a gate)
                outs, grads = run_group(gi, a, p, lo, hi, s_)
                items = list(outs.items())
                for pi, g in enumerate(grads):
                    items += [("%d.%s" % (pi, k), t) for k, t in g.items() if t is not None]
                mine = {}
                for key, t in items:
                    if key.split(".")[-1] in summed:
                        mine[key] = t
                        continue
                    if key not in out_host:
                        sizes[key] = sizes.get(key, 0) + t.numel()
                        dtypes[key] = t.dtype
                        continue
                    off = offs.get(key, 0)
                    out_host[key][off:off + t.numel()].view_as(t).copy_(t, non_blocking=True)
                    offs[key] = off + t.numel()
                partial.append(mine)
        for s_ in streams:
            cur.wait_stream(s_)
        for key, t in partial[0].items():
            tot = t
            for m in partial[1:]:
                tot = tot + m[key]
            if key not in out_host:
                sizes[key] = tot.numel()
                dtypes[key] = tot.dtype
                continue
            out_host[key].view_as(tot).copy_(tot, non_blocking=True)

    # a first step sizes the host buffers (nothing copied back), then the
    # buffers are allocated and every later step copies into them
    one_step()
    torch.cuda.synchronize()
    for key, nel in sizes.items():
        out_host[key] = torch.empty(nel, dtype=dtypes[key], pin_memory=True)
    one_step()
    torch.cuda.synchronize()
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())
    return one_step, d2h, ngroups, out_host


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)

    # the CPU baseline runs before the first GPU call of this process
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_rate(args.cpu_seconds)

    import selective_state_space_123_b300 as ssm
    from selective_state_space_123_b300 import peaks as ssm_peaks

    # the MUFU ex2 rate per SM clock, measured before the workload exists
    ex2_clk = ssm_peaks.rate_per_clk_sm("ex2")

    w = WORKLOAD
    wl = Workload(ssm, w, rank)
    Bt, D, N, L = w["Bt"], w["D"], w["N"], w["L"]
    stream = torch.cuda.current_stream()
    in_bytes = sum(v.numel() * v.element_size() for v in wl.inp.values())
    flush = None
    if in_bytes < 2 * L2_BYTES and wl.mode != "step":
        flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")

    flush_sink = torch.empty((), dtype=torch.float32, device="cuda")

    def do_flush():
        # read (not write) a buffer twice the size of L2: the lines left in L2
        # are clean, so the timed step pays no write-back of the flush
        torch.sum(flush, dim=0, out=flush_sink)

    def timed_step():
        if flush is not None:
            do_flush()
        wl.step()

    # clocks are sampled from before the warm-up, so that the timed region
    # follows the warm-up without an idle pause
    clocks = ClockSampler(local)
    clocks.start()
    clocks.wait_first()
    if wl.mode == "step":
        wl.capture_graphs()
    for _ in range(args.warmup):
        timed_step()
    torch.cuda.synchronize()
    if wl.ws is not None and ssm.ssm_get_status(wl.ws) != ssm.SSM_OK:
        raise RuntimeError("device status not ok after warm-up")

    # the flush (when needed) is timed separately and subtracted
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush_ms = 0.0
    if flush is not None:
        e0.record(stream)
        for _ in range(args.steps):
            do_flush()
        e1.record(stream)
        torch.cuda.synchronize()
        flush_ms = e0.elapsed_time(e1)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        timed_step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(t_begin, time.time())
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1) - flush_ms
    if wl.ws is not None and ssm.ssm_get_status(wl.ws) != ssm.SSM_OK:
        raise RuntimeError("device status not ok after the timed region")
    ms = max_over_ranks(ms, world)
    ms_step = ms / args.steps
    value = job_rate(world, wl.updates, ms_step)

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        host = {k: v.cpu().pin_memory() for k, v in wl.inp.items()}
        dev = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}
        if wl.mode == "step":
            state_host = wl.state.cpu().pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        if wl.mode == "step":
            h2d += state_host.numel() * 4
        if wl.mode == "fwdbwd":
            # (the pipelined step sizes and allocates its own host buffers)
            e2e_step, d2h, ng, _ = pipelined_e2e_fwdbwd(ssm, wl, host, dev)
            e2e_how = ("%d groups of %s on 2 streams: a group's copies overlap the other groups' "
                       "forward and backward; gradients summed over the split added on the device"
                       % (ng, "batch rows" if wl.w["Bt"] > 1 else "channels"))
        else:
            wl.step(dev)
            outs_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in wl.results()]
            d2h = sum(o.numel() * o.element_size() for o in outs_host)
        if wl.mode in ("fwd", "step"):
            e2e_step = pipelined_e2e(ssm, wl, host, dev, outs_host, state_host if wl.mode == "step" else None)
            e2e_how = ("4 groups of %s on 2 streams: a group's copies overlap the other groups' "
                       "scans and copies" % ("batch rows" if wl.w["Bt"] > 1 else "channels"))

        e2e_steps = max(3, min(args.steps // 20, 50))
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
        e2e_ms = max_over_ranks(e2e_ms, world)
        e2e = {"value": job_rate(world, wl.updates, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "how": e2e_how}

    # ---- roofline of the step: the slower of its algorithmic bytes at the
    # measured HBM bandwidth and its exps at the MUFU ex2 rate
    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs", 6400.0)
    hbm_basis = "MEASURED_PEAKS.json hbm_gbs (of measured)" if "hbm_gbs" in peaks else \
        "fallback 6400 GB/s (of fallback)"
    sm_mhz = clk.get("sm_mhz") or peaks.get("sm_max_mhz", 2032.0)
    sfu_peak = ex2_clk * SMS * sm_mhz * 1e6
    sfu_nominal = SFU_EX2_PER_CLK_SM * SMS * sm_mhz * 1e6
    t_s = ms_step * 1e-3
    gbs = wl.bytes / t_s / 1e9
    t_hbm = wl.bytes / (hbm_peak * 1e9)
    t_sfu = wl.exps / sfu_peak
    bound = "alu" if t_sfu >= t_hbm else "hbm"
    kernel = {"fwd": "fwd_kernel", "fwdbwd": "fwd_kernel + bwd_fwd_kernel + bwd_rev_kernel",
              "step": "step_dec16_kernel"}[wl.mode]
    roof = {
        "bound": bound,
        "kernel": kernel,
        "achieved": wl.exps / t_s / 1e12 if bound == "alu" else gbs,
        "peak": sfu_peak / 1e12 if bound == "alu" else hbm_peak,
        "unit": "Texp2/s" if bound == "alu" else "GB/s",
        "frac": (wl.exps / t_s / sfu_peak) if bound == "alu" else gbs / hbm_peak,
        "peak_basis": ("MUFU ex2 %.2f/clk/SM (measured in this process by the register-only "
                       "probe, selective_state_space_123_b300/peaks.py) x 148 SMs x median SM clock "
                       "%.0f MHz sampled in the timed region (of measured)" % (ex2_clk, sm_mhz))
                      if bound == "alu" else hbm_basis,
        "ex2_per_clk_sm_measured": ex2_clk,
        "frac_of_nominal_32_per_clk": (wl.exps / t_s / sfu_nominal) if bound == "alu" else None,
        "roofline_time_us": max(t_hbm, t_sfu) * 1e6,
        "frac_of_roofline_time": max(t_hbm, t_sfu) / t_s,
        "algorithmic_bytes": wl.bytes,
        "exps": wl.exps,
        "traffic": recorded_traffic({"fwd": "fwd_kernel", "fwdbwd": "fwdbwd", "step": "step_dec16_kernel"}[wl.mode],
                                    w["name"], w["L"]),
        "traffic_note": ("dram__bytes_read.sum + dram__bytes_write.sum of the forward and the two "
                         "backward sweeps of one step" if wl.mode == "fwdbwd" else
                         "dram__bytes_read.sum + dram__bytes_write.sum of the two passes (right to "
                         "left, left to right) of one step" if wl.bidir else
                         "dram__bytes_read.sum + dram__bytes_write.sum of one launch of the dominant "
                         "kernel") +
                        " (ncu, profiles/traffic.json); null when the kernels changed since",
        "fp32_ops_per_update": 4,
        "timing_note": ("achieved uses the whole step's CUDA-event time (one kernel per decode "
                        "step)" if wl.mode == "step" else
                        "achieved uses the whole step's CUDA-event time, which includes the small "
                        "B/C preparation kernel; 32 ex2/clk/SM equals the FP32 pipe's rate at the "
                        "4 FP32 operations an update needs, so the SFU bound is also the FP32 bound"),
    }
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "%s: %s, batch %d, D %d, N %d, L %d"
                               % (w["name"], w["title"], Bt, D, N, L),
                   "io_dtype": "bf16 u/delta/z/B/C/dy and outputs, fp32 A/D/bias/states",
                   "l2": ("flushed between steps (a 2x L2 buffer read, its time subtracted)" if flush is not None
                          else "4 rotating copies of state and inputs (368 MB > L2), no flush"
                          if wl.mode == "step" else "inputs larger than L2 (no flush)"),
                   "parallelism": "replicas",
                   "launch": ("one CUDA graph replay per step (a captured ssm_scan_step call)"
                              if wl.mode == "step" else "eager calls through the C ABI")},
        "hbm_gbs": gbs,
        "hbm_frac_of_measured": gbs / hbm_peak,
        "roofline": roof,
        "clocks": clk,
        "gpu_launches": wl.launches * args.steps,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # every step times the oracle on a bounded sample of the same workload;
    # the whole run is sized to about two minutes
    timer = OracleTimer()
    per_step = max(1e-3, 60.0 / max(1, args.steps + args.warmup))
    rates = []
    for i in range(args.warmup + args.steps):
        r = timer.measure(per_step, fixed=True)
        if i >= args.warmup:
            rates.append(r)
    timer.close()
    val = statistics.median(x["value"] for x in rates)
    w = WORKLOAD
    line = {
        "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": w["Bt"] * w["D"] * w["L"] * w["N"] / val * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": "%s: %s, batch %d, D %d, N %d, L %d"
                               % (w["name"], w["title"], w["Bt"], w["D"], w["N"], w["L"]),
                   "parallelism": "host cores"},
        "cpu_baseline": dict(rates[-1], value=val),
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def select_workload(name):
    global WORKLOAD
    WORKLOAD = dict(WORKLOADS.get(name, WORKLOADS["mamba1p4b_fwd"]), name=name)


def run_peaks(args):
    """The roofline's denominators measured on this GPU: MUFU ex2 results,
    FP32 lane operations (scalar and f32x2 FMA) and scan state updates per
    SM clock cycle, at several warp counts per SM, with the SM clock sampled
    meanwhile.  One JSON line."""
    import torch
    rank = int(os.environ.get("RANK", "0"))
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    from selective_state_space_123_b300 import peaks as ssm_peaks
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    clocks.wait_first()
    t0 = time.time()
    by_threads = {}
    for threads in (128, 256, 512, 1024):
        by_threads[threads] = {k: ssm_peaks.rate_per_clk_sm(k, threads)
                               for k in ("ex2", "fma", "fma2", "update_mix", "lg2", "rcp")}
    clk = clocks.stop(t0, time.time())
    best = {k: max(v[k] for v in by_threads.values())
            for k in ("ex2", "fma", "fma2", "update_mix", "lg2", "rcp")}
    sm_mhz = clk.get("sm_mhz") or 2032.0
    line = {
        "metric": "per-SM-clock peaks of the units that bound the scan",
        "unit": "operations per clock per SM",
        "ex2_per_clk_sm": best["ex2"],
        "fp32_fma_lane_ops_per_clk_sm": best["fma"],
        "fp32x2_fma_lane_ops_per_clk_sm": best["fma2"],
        "update_mix_per_clk_sm": best["update_mix"],
        "lg2_per_clk_sm": best["lg2"],
        "rcp_per_clk_sm": best["rcp"],
        "by_threads_per_sm": by_threads,
        "sms": SMS,
        "ex2_per_s_at_sampled_clock": best["ex2"] * SMS * sm_mhz * 1e6,
        "nominal_ex2_per_clk_sm": SFU_EX2_PER_CLK_SM,
        "method": "one CTA per SM, 8 independent register chains per thread, %clock64 per CTA, "
                  "best of 3 launches, median over CTAs",
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def _free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_entry(rank, world, port, target, args):
    """One spawned rank: the environment torchrun would give it, then the arm."""
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    select_workload(args.workload)   # a spawned process starts from a fresh import
    target(args)


def spawn_ranks(world, target, args):
    """`--gpus N` without an outside launcher: start N processes (spawned, one
    per GPU, ranks 0..N-1 on 127.0.0.1) that each run `target(args)`, as
    torchrun would; the arm then forms its process group from the
    environment.  Every rank runs an independent replica of the workload."""
    import torch.multiprocessing as tmp
    tmp.spawn(_rank_entry, args=(world, _free_port(), target, args), nprocs=world, join=True)


def main(argv=None, target=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end measurement (profiling runs)")
    ap.add_argument("--seqlen", type=int, default=0,
                    help="override the workload's sequence length (small profiler captures)")
    ap.add_argument("--workload", default="mamba1p4b_fwd", choices=sorted(WORKLOADS) + ["peaks"],
                    help="'peaks': the register-only MUFU / FP32 / update-mix rate probes")
    args = ap.parse_args(argv)
    select_workload(args.workload)
    if args.seqlen:
        # a shorter (or longer) sequence of the same layer, for profiler captures
        # that must stay small; the JSON line's config names the length used
        WORKLOAD["L"] = args.seqlen
        WORKLOAD["title"] += " (sequence length set by --seqlen)"
    if args.warmup < 3:
        args.warmup = 3
    if target is None:
        target = run_reference if args.impl == "reference" else \
            run_peaks if args.workload == "peaks" else run_ours
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        spawn_ranks(args.gpus, target, args)
    else:
        target(args)


if __name__ == "__main__":
    main()
