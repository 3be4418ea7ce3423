"""Multi-rank host logic on CPU with gloo ranks.

Rows are independent, so data-parallel ranks need no collective on the data
path.  bench.py runs N batches of the same shape (weak scaling); the only
cross-rank steps are the timing barrier and the max-over-ranks reduction of
the step time.  A single batch splits across ranks by whole rows
(tpk_plan_shard_rows, longest first to the least-loaded rank), each rank
planning its rows' sequences as a batch of its own that reproduces exactly
those rows.
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
    f = root / "prefix_tree_packed_dfs_gb300" / "csrc" / "attn_bwd.cu"
    f.write_text("// a new comment line\n" + f.read_text().replace("{", "{ /* inline */", 1))
    assert bench.source_digest() == d0
    f.write_text(f.read_text().replace("constexpr int kStat = 4;", "constexpr int kStat = 3;"))
    assert bench.source_digest() != d0
    # other kernels do not change what the attention kernels move
    d2 = bench.source_digest()
    g = root / "prefix_tree_packed_dfs_gb300" / "csrc" / "scatter.cu"
    g.write_text(g.read_text().replace("kThreads = 256", "kThreads = 128"))
    assert bench.source_digest() == d2
    # host-side API code does not change what the kernels move
    d1 = bench.source_digest()
    api = root / "prefix_tree_packed_dfs_gb300" / "csrc" / "api.cpp"
    api.write_text(api.read_text() + "\nint tpk_unused_probe() { return 0; }\n")
    assert bench.source_digest() == d1
    pl = root / "prefix_tree_packed_dfs_gb300" / "csrc" / "planner.cpp"
    pl.write_text(pl.read_text().replace("kOrderChunk = 128", "kOrderChunk = 64"))
    assert bench.source_digest() != d1          # the launch order does


# ---------------------------------------------------------------- rows across ranks
def _plan(name):
    import workloads
    from prefix_tree_packed_dfs_gb300 import ops
    w = workloads.get(name)
    return w, ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                      min_shared=w.min_shared)


def _row_pairs(plan):
    """Useful pairs per row from the exported layout: sum of depth + 1."""
    import numpy as np
    ex = plan.export()
    off, depth = ex["row_offsets"], ex["depth"].astype(np.int64)
    return np.array([int((depth[off[r]:off[r + 1]] + 1).sum()) for r in range(len(off) - 1)], np.int64)


@pytest.mark.parametrize("name", ["grpo", "agentic", "deep_small", "tiny"])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_shard_rows_is_a_balanced_partition(name, world):
    import numpy as np
    w, plan = _plan(name)
    pairs = _row_pairs(plan)
    rank_of_row, rank_pairs = plan.shard_rows(world)
    assert rank_of_row.min() >= 0 and rank_of_row.max() < world
    for k in range(world):
        assert rank_pairs[k] == pairs[rank_of_row == k].sum()
    assert rank_pairs.sum() == plan.info["useful_pairs"]
    # greedy least-loaded assignment: no rank ends more than one row above the lightest
    assert rank_pairs.max() - rank_pairs.min() <= pairs.max()
    if world >= len(pairs):
        assert np.bincount(rank_of_row, minlength=world).max() == 1
    again, _ = plan.shard_rows(world)
    assert np.array_equal(again, rank_of_row)          # reproducible
    # every sequence belongs to exactly one rank
    seqs = [plan.sequences_of_rank(rank_of_row, k) for k in range(world)]
    allseq = np.sort(np.concatenate(seqs))
    assert np.array_equal(allseq, np.arange(len(w.sequences)))


def test_shard_rows_within_grahams_bound_of_the_optimum():
    """Longest-processing-time-first list scheduling is within
    4/3 - 1/(3m) of the best makespan (Graham 1969); the optimum here is by
    brute force over every assignment of the GRPO batch's 7 rows."""
    import itertools
    w, plan = _plan("grpo")
    pairs = _row_pairs(plan)
    for m in (2, 3):
        best = min(max(sum(int(pairs[r]) for r in range(len(pairs)) if a[r] == k) for k in range(m))
                   for a in itertools.product(range(m), repeat=len(pairs)))
        _, rank_pairs = plan.shard_rows(m)
        assert best <= rank_pairs.max() <= (4 / 3 - 1 / (3 * m)) * best


def test_shard_rows_rejects_bad_arguments():
    from prefix_tree_packed_dfs_gb300 import binding
    lib = binding.load()
    import ctypes
    assert lib.tpk_plan_shard_rows(None, 2, ctypes.c_void_p(16), None) == -1
    _, plan = _plan("tiny")
    assert lib.tpk_plan_shard_rows(plan.handle, 0, ctypes.c_void_p(16), None) == -1
    assert lib.tpk_plan_shard_rows(plan.handle, 2, None, None) == -1


def _shard_worker(rank, world, port, out):
    import numpy as np
    import torch.distributed as dist
    import workloads
    from prefix_tree_packed_dfs_gb300 import ops
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank plans the whole batch on its host, takes its rows' sequences
        # and plans them as its own batch: nothing but this listing crosses ranks
        w = workloads.get("grpo")
        full = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                       min_shared=w.min_shared)
        rank_of_row, rank_pairs = full.shard_rows(world)
        sub, mine = full.rank_plan(w.sequences, rank_of_row, rank, w.row_capacity, w.min_shared)
        # the rank's plan is its rows of the whole batch's plan, row for row
        ex_full, ex_sub = full.export(), sub.export()
        rows = np.flatnonzero(rank_of_row == rank)
        same = [np.array_equal(ex_full[k][ex_full["row_offsets"][r]:ex_full["row_offsets"][r + 1]],
                               ex_sub[k][ex_sub["row_offsets"][j]:ex_sub["row_offsets"][j + 1]])
                for j, r in enumerate(rows) for k in ("fwd_token", "depth")]
        got = [None] * world
        dist.all_gather_object(got, (mine.tolist(), sub.info["n_raw"], sub.info["useful_pairs"]))
        out[rank] = (got, int(rank_pairs[rank]), full.info["n_raw"], len(w.sequences), all(same),
                     sub.info["n_rows"] == len(rows))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_one_batch_by_rows():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_shard_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    got0, pairs0, n_raw, n_seq, same0, nrows0 = out[0]
    got1, pairs1, _, _, same1, nrows1 = out[1]
    assert got0 == got1                                   # both ranks see the same split
    seqs = sorted(got0[0][0] + got0[1][0])
    assert seqs == list(range(n_seq))                     # each sequence on exactly one rank
    assert got0[0][1] + got0[1][1] == n_raw               # raw tokens add up
    # each rank's plan holds exactly its rows: same tokens and depths, same work
    assert same0 and same1 and nrows0 and nrows1
    assert got0[0][2] == pairs0 and got0[1][2] == pairs1
