"""Benchmark of the selective scan on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one forward selective scan (softplus of delta, discretisation, the
recurrence, read-out, D skip, SiLU gate, final state) over one batch of the
Mamba-1.4B layer shape: batch 4, D=4096 channels, N=16 states, L=4096 tokens,
bf16 u/delta/z/B/C, fp32 A/D/bias, fp32 arithmetic, bf16 y, fp32 final state.
Inputs are synthetic (seeded, drawn on the device) and resident in HBM before
the timed region; they are larger than L2 (539 MB vs 126 MB), so no flush is
needed between steps.

The JSON line (rank 0) reports B*D*L*N state updates per second for the whole
job (N GPUs run independent replicas: the channels of different sequences
never interact, so the work shards with no collective), the roofline of the
dominant kernel, clocks sampled during the timed region, the end-to-end rate
through the C ABI with host buffers (pinned host -> device copies of every
input and the device -> host read of y and h_L inside the timed region), and
the fp64 CPU oracle timed on a bounded sample as the CPU baseline.
`--impl reference` times that oracle alone (this method has no runnable
reference implementation; the oracle is the reference arm).
"""
from __future__ import annotations

import argparse
import json
import math
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
    "mamba1p4b_fwd": dict(name="mamba1p4b_fwd", Bt=4, D=4096, N=16, L=4096, seed=2),
    "mamba130m_fwd": dict(name="mamba130m_fwd", Bt=8, D=1536, N=16, L=2048, seed=1),
    "mamba2p8b_fwd": dict(name="mamba2p8b_fwd", Bt=2, D=5120, N=16, L=8192, seed=3),
    "million_fwd": dict(name="million_fwd", Bt=1, D=1536, N=16, L=1 << 20, seed=4),
}
WORKLOAD = WORKLOADS["mamba1p4b_fwd"]
METRIC = "selective scan: achieved HBM GB/s (% of roofline) and B*D*L*N state updates/s"
UNIT = "state updates/s"
# measured on this machine's B300 with a register-only probe: MUFU ex2 results
# per clock per SM ("Rooflines")
SFU_EX2_PER_CLK_SM = 32
SMS = 148


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
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
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
    seed, Bt, D, N, L, chans = args
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import oracle
    from scan_inputs import make_inputs
    key = (seed, Bt, D, N, L, tuple(chans))
    x = _INPUT_CACHE.get(key)
    if x is None:
        if len(_INPUT_CACHE) > 64:
            _INPUT_CACHE.clear()
        x = _INPUT_CACHE[key] = make_inputs(Bt, D, N, L, seed=seed, in_dtype="bf16",
                                            channels=chans)
    t0 = time.perf_counter()
    oracle.scan_fwd(x.u, x.delta_raw, x.A, x.Bm, x.Cm, x.Dv, x.z, x.delta_bias, x.h0)
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
        self.pool.map(_oracle_worker, [(w["seed"], 1, w["D"], w["N"], 64, [0])] * self.cores)
        _, self.t_channel = _oracle_worker((w["seed"], 1, w["D"], w["N"], w["L"], [0]))
        self.next = 0

    def measure(self, seconds_per_core, fixed=False):
        """Oracle throughput on about `seconds_per_core` of work per process.
        fixed=True reuses the same channel sample every call (the reference
        arm's steps); otherwise the sample advances through the channels."""
        w = WORKLOAD
        per = max(1, int(seconds_per_core / max(self.t_channel, 1e-6)))
        jobs = []
        start = 0 if fixed else self.next
        for i in range(self.cores):
            jobs.append((w["seed"], 1, w["D"], w["N"], w["L"],
                         [(start + i * per + j) % w["D"] for j in range(per)]))
        if not fixed:
            self.next = (start + per * self.cores) % w["D"]
        res = self.pool.map(_oracle_worker, jobs)
        upd = sum(r[0] for r in res)
        busy = max(r[1] for r in res)
        return {"value": upd / busy, "unit": UNIT, "cores": self.cores, "kind": "oracle",
                "sample": "%d channels x %d tokens x %d states of the %s workload (batch row "
                          "0), one spawned process per core; slowest process %.2f s" %
                          (per * self.cores, w["L"], w["N"], w["name"], busy)}

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
    from scan_inputs import device_inputs

    w = WORKLOAD
    Bt, D, N, L = w["Bt"], w["D"], w["N"], w["L"]
    a = device_inputs(Bt, D, N, L, seed=w["seed"] + 1000 * rank, in_dtype="bf16")
    y = torch.empty(Bt, D, L, dtype=torch.bfloat16, device="cuda")
    hL = torch.empty(Bt, D, N, dtype=torch.float32, device="cuda")
    shape = ssm.make_shape(Bt, D, N, L, ssm.SSM_BF16, ssm.SSM_BF16)
    ws = torch.empty(ssm.ssm_scan_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        ssm.ssm_scan_fwd(a["u"], a["delta_raw"], a["A"], a["Bm"], a["Cm"], a["Dv"], a["z"],
                         a["delta_bias"], None, out_dtype=torch.bfloat16, y=y, hL=hL,
                         workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ssm.ssm_get_status(ws) != ssm.SSM_OK:
        raise RuntimeError("device status not ok after warm-up")

    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    if ssm.ssm_get_status(ws) != ssm.SSM_OK:
        raise RuntimeError("device status not ok after the timed region")
    if world > 1:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_step = ms / args.steps
    updates = Bt * D * L * N
    value = world * updates / (ms_step * 1e-3)

    # ---- end to end through the C ABI with host buffers
    host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in a.items()} \
        if not args.no_e2e else {}
    dev = {k: (torch.empty_like(v, device="cuda") if v is not None else None)
           for k, v in host.items()}
    y_host = torch.empty(Bt, D, L, dtype=torch.bfloat16, pin_memory=not args.no_e2e)
    h_host = torch.empty(Bt, D, N, dtype=torch.float32, pin_memory=not args.no_e2e)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = y_host.numel() * 2 + h_host.numel() * 4

    def e2e_step():
        for k, v in host.items():
            if v is not None:
                dev[k].copy_(v, non_blocking=True)
        ssm.ssm_scan_fwd(dev["u"], dev["delta_raw"], dev["A"], dev["Bm"], dev["Cm"], dev["Dv"],
                         dev["z"], dev["delta_bias"], None, out_dtype=torch.bfloat16, y=y,
                         hL=hL, workspace=ws)
        y_host.copy_(y, non_blocking=True)
        h_host.copy_(hL, non_blocking=True)

    e2e_steps = max(3, min(args.steps // 20, 50))
    e2e_ms = float("nan")
    if not args.no_e2e:
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if world > 1:
        t = torch.tensor([e2e_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())

    # ---- roofline of the dominant kernel (the forward scan kernel; the
    # call also runs the tiny B/C preparation kernel, included in the time)
    peaks = load_peaks()
    hbm_peak = peaks.get("hbm_gbs", 6400.0)
    sm_mhz = clk.get("sm_mhz") or peaks.get("sm_max_mhz", 2032.0)
    sfu_peak = SFU_EX2_PER_CLK_SM * SMS * sm_mhz * 1e6
    exps_per_s = updates / (ms_step * 1e-3)
    bytes_alg = fwd_bytes(Bt, D, N, L)
    gbs = bytes_alg / (ms_step * 1e-3) / 1e9
    t_hbm = bytes_alg / (hbm_peak * 1e9)
    t_sfu = updates / sfu_peak
    bound = "alu" if t_sfu >= t_hbm else "hbm"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "%s: batch %d, D %d, N %d, L %d (forward scan)"
                               % (w["name"], Bt, D, N, L),
                   "io_dtype": "bf16 u/delta/z/B/C/y, fp32 A/D/bias/h_L",
                   "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas"},
        "hbm_gbs": gbs,
        "hbm_frac_of_measured": gbs / hbm_peak,
        "roofline": {
            "bound": bound,
            "achieved": exps_per_s / 1e12 if bound == "alu" else gbs,
            "peak": sfu_peak / 1e12 if bound == "alu" else hbm_peak,
            "unit": "Texp2/s" if bound == "alu" else "GB/s",
            "frac": (exps_per_s / sfu_peak) if bound == "alu" else gbs / hbm_peak,
            "peak_basis": ("MUFU ex2 32/clk/SM x 148 SMs x median SM clock %.0f MHz "
                           "(probe-measured rate)" % sm_mhz) if bound == "alu" else
                          "MEASURED_PEAKS.json hbm_gbs",
            "roofline_time_us": max(t_hbm, t_sfu) * 1e6,
            "frac_of_roofline_time": max(t_hbm, t_sfu) / (ms_step * 1e-3),
            "traffic": None,
        },
        "clocks": clk,
        "e2e": {"value": world * updates / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if args.no_e2e:
        del line["e2e"]
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
        "config": {"workload": "%s: batch %d, D %d, N %d, L %d (Mamba-1.4B layer forward)"
                               % (w["name"], w["Bt"], w["D"], w["N"], w["L"]),
                   "parallelism": "host cores"},
        "cpu_baseline": dict(rates[-1], value=val),
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end measurement (profiling runs)")
    ap.add_argument("--workload", default="mamba1p4b_fwd", choices=sorted(WORKLOADS))
    args = ap.parse_args()
    global WORKLOAD
    WORKLOAD = WORKLOADS[args.workload]
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
