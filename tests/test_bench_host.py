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
