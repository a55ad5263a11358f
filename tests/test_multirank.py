"""The bench's multi-rank host logic with two gloo ranks on the CPU: each rank
runs its own replica (distinct inputs), the job time is the slowest rank's,
and the job rate counts every rank's updates."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.5 + rank                       # rank 1 is the slower one
        job_ms = bench.max_over_ranks(ms, world)
        rate = bench.job_rate(world, 1000, job_ms)
        seed = bench.rank_seed(7, rank)
        seeds = [None] * world
        dist.all_gather_object(seeds, seed)
        out[rank] = (job_ms, rate, tuple(seeds))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        job_ms, rate, seeds = res[r]
        assert job_ms == pytest.approx(2.5)
        assert rate == pytest.approx(world * 1000 / 2.5e-3)
        assert len(set(seeds)) == world


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_rate(1, 500, 2.0) == pytest.approx(500 / 2e-3)


def _stub_arm(args):
    """Stands in for the GPU arm in a spawned rank: forms the process group
    from the environment the launcher set (gloo on the CPU), times nothing,
    and reports what the real arm reports about the job's shape."""
    import json
    import torch.distributed as dist
    import bench
    world = int(os.environ["WORLD_SIZE"])
    rank = int(os.environ["RANK"])
    assert os.environ["MASTER_ADDR"] == "127.0.0.1"
    assert os.environ["LOCAL_RANK"] == str(rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + rank, world)
        line = {"n_gpus": world, "rank": rank, "workload": bench.WORKLOAD["name"],
                "value": bench.job_rate(world, 100, ms)}
        with open(os.path.join(args.out_dir, "rank%d.json" % rank), "w") as f:
            json.dump(line, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_gpus_flag_spawns_ranks(tmp_path, monkeypatch):
    """`bench.py --gpus 2` without torchrun starts two ranks itself; each
    sees WORLD_SIZE 2 and its own RANK, and the chosen workload survives the
    spawn."""
    import json
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    parser_args = ["--gpus", "2", "--workload", "mamba130m_fwd"]
    real_parse = bench.argparse.ArgumentParser.parse_args

    def parse_with_out(self, argv=None, namespace=None):
        a = real_parse(self, argv, namespace)
        a.out_dir = str(tmp_path)
        return a

    monkeypatch.setattr(bench.argparse.ArgumentParser, "parse_args", parse_with_out)
    bench.main(parser_args, target=_stub_arm)
    lines = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    assert [ln["rank"] for ln in lines] == [0, 1]
    assert all(ln["n_gpus"] == 2 for ln in lines)
    assert all(ln["workload"] == "mamba130m_fwd" for ln in lines)
    assert lines[0]["value"] == pytest.approx(2 * 100 / 2e-3)
