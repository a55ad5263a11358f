"""Host-side pieces of bench.py, without a GPU: the algorithmic byte counts
behind the roofline's "achieved", the kernel-source hash that keys recorded
DRAM traffic, and the traffic records themselves."""
import json
import os
import shutil

import pytest

import bench


def test_algorithmic_bytes_match_the_tensor_sizes():
    # Mamba-1.4B forward: u, delta_raw, z, y bf16 (4, 4096, 4096); B, C bf16
    # (4, 16, 4096); A fp32 (4096, 16); D, bias fp32 (4096); h_L fp32 (4, 4096, 16)
    Bt, D, N, L = 4, 4096, 16, 4096
    per_token = Bt * D * L * 2
    expect = 3 * per_token + 2 * Bt * N * L * 2 + D * N * 4 + 2 * D * 4 + per_token + Bt * D * N * 4
    assert bench.fwd_bytes(Bt, D, N, L) == expect == 539262976
    # decode (256, 5120, 16): the fp32 state is read and written
    assert bench.step_bytes(256, 5120, 16) == 2 * 256 * 5120 * 16 * 4 + 3 * 256 * 5120 * 2 \
        + 2 * 256 * 16 * 2 + 5120 * 16 * 4 + 2 * 5120 * 4 + 256 * 5120 * 2
    # the backward moves more than the forward at any shape
    assert bench.bwd_bytes(2, 5120, 16, 8192) > bench.fwd_bytes(2, 5120, 16, 8192)


def test_recorded_traffic_is_keyed_to_the_sources():
    """A record counts only while its kernels' sources are unchanged."""
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    assert rec, "no traffic records"
    for key, v in rec.items():
        kind, workload = key.split(":")
        assert v["bytes_per_launch"] > 0
        got = bench.recorded_traffic(kind, workload)
        if v["src_hash"] == bench.kernel_source_hash(kind):
            assert got == v["bytes_per_launch"], key
        else:
            assert got is None, key
    assert bench.recorded_traffic("fwd_kernel", "no_such_workload") is None
    # a run whose sequence length was overridden (--seqlen) gets no record
    assert bench.recorded_traffic("fwd_kernel", "mamba1p4b_fwd", 1024) is None


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = os.path.join(bench.ROOT, "selective_state_space_123_b300", "csrc")
    root = tmp_path / "r"
    shutil.copytree(csrc, root / "selective_state_space_123_b300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(root))
    base = bench.kernel_source_hash("step_dec16_kernel")
    f = root / "selective_state_space_123_b300" / "csrc" / "ssm_step.cu"
    text = f.read_text(encoding="utf-8")
    f.write_text(text + "\n// a comment\n/* another\n comment */\n", encoding="utf-8")
    assert bench.kernel_source_hash("step_dec16_kernel") == base
    f.write_text(text + "\nstatic int extra_symbol = 1;\n", encoding="utf-8")
    assert bench.kernel_source_hash("step_dec16_kernel") != base


@pytest.mark.parametrize("mode,variant,factor", [("fwd", (0, False, False), 1),
                                                 ("fwd", (4, False, False), 1),
                                                 ("fwd", (0, True, False), 1),
                                                 ("fwd", (0, False, True), 2),
                                                 ("fwdbwd", (0, False, False), 1),
                                                 ("fwdbwd", (0, True, False), 1),
                                                 ("fwdbwd", (0, False, True), 2)])
def test_oracle_worker_variants(mode, variant, factor):
    """The CPU baseline's worker runs every forward variant, and the
    backward of the plain, packed and bidirectional scans, and counts the
    state updates it did (two scans for the bidirectional one)."""
    conv_k, varlen, bidir = variant
    upd, secs = bench._oracle_worker((mode, 7, 1, 64, 16, 256, [0, 5], conv_k, varlen, bidir))
    assert upd == factor * 2 * 16 * 256
    assert secs >= 0.0


def _plan_lines(shape, kind):
    """The planner's choice for `shape`, printed by the library itself."""
    import subprocess
    import sys
    code = ("import selective_state_space_123_b300 as m\n"
            "m.ssm_scan_workspace_bytes(m.make_shape(%d, %d, %d, %d, 1, 1), %d)\n" % (shape + (kind,)))
    env = dict(os.environ, SSM_DEBUG_PLAN="1")
    for k in ("SSM_FWD_NT", "SSM_FWD_W", "SSM_FWD_NSEG", "SSM_FWD_CPS"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, "-c", code], cwd=bench.ROOT, env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return [ln for ln in r.stderr.splitlines() if ln.startswith("ssm fwd plan")]


def test_launch_counts_follow_the_plan():
    """The bench's launch claims for the packed and bidirectional workloads
    rest on the plan: 4 segments for the packed row (preparation, sequence
    check, tail search, summary, carry, scan); one segment per direction for
    the bidirectional workload's shape (preparation twice, two passes), while
    a few-channel long row is split in both directions."""
    from tests.buildlib import ensure_built
    ensure_built()
    w = bench.WORKLOADS["packed_mamba1p4b_fwd"]
    lines = _plan_lines((w["Bt"], w["D"], w["N"], w["L"]), 0)
    assert lines and "nseg=4 " in lines[-1] and w["launches"] == 6
    w = bench.WORKLOADS["bidir_mamba1p4b_fwd"]
    assert w["launches"] == 4
    lines = _plan_lines((w["Bt"], w["D"], w["N"], w["L"]), 2)
    assert lines and "nseg=1 " in lines[-1]
    lines = _plan_lines((1, 1536, 16, 1 << 20), 2)
    assert lines and "nseg=1 " not in lines[-1]
