"""The bench's multi-rank host logic on CPU with two gloo ranks.

Rows are independent, so N GPUs run N batches of the same shape (weak
scaling) with no collective on the data path.  The only cross-rank steps
are the timing barrier and the max-over-ranks reduction of the step time;
here two CPU processes check them: distinct per-rank batches, the slowest
rank's time on every rank, and the whole-job value from it.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    import workloads
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workloads.get("tiny")
        seeds = bench.rank_seeds(w, rank)
        local = 0.5 + rank            # rank 1 is the slow one
        dist.barrier()
        slowest = bench.max_over_ranks(local, "cpu", world)
        out[rank] = (seeds["q"], slowest, bench.job_value(world, w.n_raw, slowest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_only_timing():
    world, port = 2, _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    (q0, slow0, v0), (q1, slow1, v1) = out[0], out[1]
    assert q0 != q1                                 # each rank owns its own batch
    assert slow0 == slow1 == pytest.approx(1.5)     # max over ranks on both
    import workloads
    assert v0 == v1 == pytest.approx(2 * workloads.get("tiny").n_raw / 1.5)


def test_recorded_traffic_only_for_the_sources_it_was_taken_on(monkeypatch):
    import bench
    digest = bench.source_digest()
    monkeypatch.setattr(bench, "TRAFFIC", {"digest": digest, "fwd": 123, "bwd_dkdv": 456, "bwd_dq": None})
    assert bench.recorded_traffic("bwd_dkdv", bench.WORKLOAD) == 456
    assert bench.recorded_traffic("bwd_dq", bench.WORKLOAD) is None
    assert bench.recorded_traffic("fwd", "deep_small") is None          # another workload
    monkeypatch.setattr(bench, "TRAFFIC", {"digest": "0" * 64, "fwd": 123, "bwd_dkdv": 456, "bwd_dq": 7})
    assert bench.recorded_traffic("bwd_dkdv", bench.WORKLOAD) is None   # sources changed since


def test_source_digest_ignores_comments(tmp_path, monkeypatch):
    import shutil
    import bench
    root = tmp_path / "r"
    shutil.copytree(os.path.join(bench.ROOT, "prefix_tree_packed_dfs_gb300", "csrc"),
                    root / "prefix_tree_packed_dfs_gb300" / "csrc")
    shutil.copytree(os.path.join(bench.ROOT, "include"), root / "include")
    monkeypatch.setattr(bench, "ROOT", str(root))
    d0 = bench.source_digest()
    f = root / "prefix_tree_packed_dfs_gb300" / "csrc" / "scatter.cu"
    f.write_text("// a new comment line\n" + f.read_text().replace("{", "{ /* inline */", 1))
    assert bench.source_digest() == d0
    f.write_text(f.read_text().replace("kThreads = 256", "kThreads = 128"))
    assert bench.source_digest() != d0
