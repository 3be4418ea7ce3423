#!/usr/bin/env python
"""Benchmark of the prefix-tree-packed DFS attention hot path on GB300.

One step = the whole path over one batch of the deep-tree workload (root of
4096 tokens, branching factor 1-3 every 256-1024 tokens down to depth 24000,
128 leaves, rows of 65536 forwarded tokens, 32 query / 8 KV heads, head_dim
128, bf16):
    RoPE at depth (Q, K, in place)  ->  tree attention forward (O, LSE)
    ->  scatter to raw-token order (O, LSE)  ->  raw-order dO summed into the
    packed layout (the scatter's transpose)  ->  tree attention backward
    (prep, dK/dV pass, dQ pass; the inverse RoPE of dQ, dK inside the
    passes' epilogues).
The same step is also timed in the precise mode (P and dS as hi + lo bf16
pairs, the forward's O residual), and the forward alone on the other
workloads (tiny, GRPO, agentic, the packing-ratio sweep with its
sequence-packing twins) under ``configs``.
The plan (host) is built once for ``value``; the ``e2e`` leg rebuilds it
every step and moves inputs from pinned host memory and the raw-order LSE
back, through the same public API, preparing step i+1 (plan build, uploads)
while the GPU runs step i.

Metric: raw tokens/s (whole job), with useful TFLOP/s and % of the measured
dense bf16 peak alongside.  Useful FLOPs count visible (query, key) pairs
only: 4*d*Hq*pairs forward + 10*d*Hq*pairs backward, pairs = sum(depth+1).

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload instead (rank 0 only).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOAD = "deep"
WORKLOAD_DESC = ("deep random tree: root 4096, branching {1,2,3} every 256-1024 tokens to depth 24000, "
                 "128 leaves, rows 65536, Hq 32 / Hkv 8 / d 128, fwd+bwd")
METRIC = "tree-attn raw tokens/s, useful TFLOP/s and % of GB300 bf16 dense peak"
LAUNCHES_PER_STEP = 8   # rope, fwd, scatter rows, scatter lse, dO sum, bwd prep, bwd dK/dV, bwd dQ

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# attention kernels on the deep-tree workload, from one ncu capture of
#   bench.py --steps 1 --warmup 1 --e2e-steps 0 --no-cpu-baseline
# (first launch of each kernel; the summary is in profiles/), tagged with a
# digest of the kernel and planner sources they were built from.  Once those
# differ the figure no longer describes the kernel and is reported as null.
TRAFFIC = {"digest": "100edcac35ca9338fcb582255699e5ceff033039501fb48da7ae28a266c0c8d8",
           "fwd": 175401812480, "bwd_dkdv": 478771346944, "bwd_dq": 274274299136}


# the sources that decide the recorded kernels' memory traffic: the attention
# kernels, the device headers they include, and the planner that orders their
# work (csrc/planner.*, plan_handle.h)
TRAFFIC_SOURCES = ("attn_fwd.cu", "attn_bwd.cu", "ptx.cuh", "common.cuh", "planner.cpp", "planner.h",
                   "plan_handle.h")


def source_digest():
    """sha256 over TRAFFIC_SOURCES, in name order, with comments and
    whitespace removed: edits to comments, to host-side API code or to other
    kernels leave it alone."""
    import hashlib
    import re
    h = hashlib.sha256()
    dirs = [os.path.join(ROOT, "prefix_tree_packed_dfs_gb300", "csrc")]
    for d in dirs:
        for name in sorted(os.listdir(d)):
            if name in TRAFFIC_SOURCES:
                with open(os.path.join(d, name)) as f:
                    code = f.read()
                code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
                code = re.sub(r"//[^\n]*", " ", code)
                h.update(name.encode())
                h.update(" ".join(code.split()).encode())
    return h.hexdigest()


def recorded_traffic(kernel, workload):
    if workload != WORKLOAD or TRAFFIC.get(kernel) is None or TRAFFIC["digest"] != source_digest():
        return None
    return TRAFFIC[kernel]


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--shard-rows", action="store_true",
                    help="with several ranks: split one batch across them by whole rows (strong scaling) "
                         "instead of one batch of the same shape per rank")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="bound on the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-precise", action="store_true", help="skip the precise-mode step")
    ap.add_argument("--no-configs", action="store_true", help="skip the forward on the other workloads")
    ap.add_argument("--no-gdn", action="store_true", help="skip the GDN tree path sub-bench")
    ap.add_argument("--gdn", action="store_true", help="the GDN tree path alone on --workload; one line")
    ap.add_argument("--planner", action="store_true",
                    help="host planner of the library vs the oracle's planner on every workload (no GPU)")
    ap.add_argument("--layout", action="store_true",
                    help="raw order <-> packed layout kernels (materialisation gather, sum of raw-order rows) "
                         "on --workload; one line")
    ap.add_argument("--sweep", action="store_true",
                    help="packing-ratio sweep (32,768-token rows): forward time against forwarded and raw "
                         "tokens, tree layout vs sequence packing of the same raw tokens; one line per point")
    return ap.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class Clocks:
    """nvidia-smi sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seeds(w, rank):
    """Seeds of this rank's batch.  Weak scaling: every rank owns one batch of
    the same shape (rows are independent, nothing crosses ranks on the data
    path), drawn with seeds shifted by 1000 per rank."""
    return {k: v + 1000 * rank for k, v in w.seeds.items()}


def max_over_ranks(x, device, world):
    """The slowest rank's value (step time): the only cross-rank reduction."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, raw_tokens_per_rank, seconds):
    """Whole-job raw tokens/s: every rank's tokens over the slowest rank's time."""
    return world * raw_tokens_per_rank / seconds


def _cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


class OracleSampler:
    """The fp64 oracle on a bounded sample of the workload: for raw tokens
    drawn uniformly from two of its sequences, the forward row and the dQ row
    (``oracle.attention.forward_rows`` / ``backward_rows_q``).  The input rows
    of those two sequences are regenerated once, before any timing."""

    def __init__(self, w, plan_ref, seed=0):
        import torch
        from workloads import rng as wrng
        self.w, self.ref = w, plan_ref
        rng = np.random.Generator(np.random.PCG64(seed))
        off = plan_ref["seq_offsets"]
        ti = plan_ref["token_index"]
        self.seqs = rng.choice(len(off) - 1, size=2, replace=False)
        rows = np.unique(np.concatenate([ti[off[x]:off[x + 1]] for x in self.seqs]))
        self.pos = np.full(plan_ref["n_fwd"], -1, dtype=np.int64)
        self.pos[rows] = np.arange(len(rows))
        self.vals = {}
        for key, heads in (("q", w.n_heads_q), ("k", w.n_heads_kv), ("v", w.n_heads_kv), ("do", w.n_heads_q)):
            v = wrng.rows_bf16(w.seeds[key], rows, heads * w.head_dim).to(torch.float64).numpy()
            self.vals[key] = v.reshape(len(rows), heads, w.head_dim)

    def getter(self, key):
        vals, pos = self.vals[key], self.pos
        return lambda idx: vals[pos[np.asarray(idx, dtype=np.int64)]]

    def run(self, budget_s, seed=0):
        from oracle import attention as oa
        rng = np.random.Generator(np.random.PCG64(1000 + seed))
        off = self.ref["seq_offsets"]
        Qr, Kr, Vr, dOr = (self.getter(k) for k in ("q", "k", "v", "do"))
        done, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < budget_s:
            x = int(rng.choice(self.seqs))
            r = int(off[x] + rng.integers(0, off[x + 1] - off[x]))
            oa.forward_rows(self.ref, Qr, Kr, Vr, [r], self.w.rope_base)
            oa.backward_rows_q(self.ref, Qr, Kr, Vr, dOr, [r], self.w.rope_base)
            done += 1
        return done, time.perf_counter() - t0


def run_reference(a):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import workloads
    from oracle import planner as op
    w = workloads.get(a.workload)
    ref = op.plan(w.sequences, group_ids=w.group_ids, min_shared=w.min_shared, row_capacity=w.row_capacity)
    per_step = max(1.0, min(a.cpu_seconds, 120.0 / max(1, a.steps + a.warmup)))
    sampler = OracleSampler(w, ref)
    for i in range(a.warmup):
        sampler.run(per_step / 4, seed=100 + i)
    n_tot, t_tot = 0, 0.0
    for i in range(a.steps):
        n, dt = sampler.run(per_step, seed=i)
        n_tot += n
        t_tot += dt
    value = n_tot / t_tot
    cores = _cpu_threads()
    sample = ("fp64 oracle forward row + dQ row for %d raw tokens drawn uniformly from 2 of the 128 "
              "24000-token sequences (%d steps of ~%.0f s); dK/dV rows not included" % (n_tot, a.steps, per_step))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "raw tokens/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * t_tot / a.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "raw_tokens": ref["n_raw"], "forwarded_tokens": ref["n_fwd"]},
        "cpu_baseline": {"value": value, "unit": "raw tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "raw tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def _time_launches(fn, flush, min_s=0.5, min_n=10, warmup=3):
    """Median CUDA-event time (ms) of fn() on the current stream, L2 flushed
    (a write larger than L2) before each launch; repeated until ``min_s`` of
    device time and ``min_n`` launches, so a clock sample spans it."""
    import torch
    for _ in range(warmup):
        fn()
    times = []
    while len(times) < min_n or sum(times) < 1e3 * min_s:
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
        if len(times) >= 2000:
            break
    return statistics.median(times), len(times)


CONFIG_WORKLOADS = (["tiny", "grpo", "agentic"] + ["sweep_%.2f" % r for r in (1.00, 1.45, 2.0, 2.8, 3.56)]
                    + ["sweep_%.2f_seqpack" % r for r in (1.45, 2.0, 2.8, 3.56)])


def run_configs(peaks, local, warmup):
    """Forward on every other workload: one launch timed at a time (L2
    flushed before each, median), with its own clock sample."""
    import torch
    import workloads
    from prefix_tree_packed_dfs_gb300 import ops
    from workloads import rng as wrng
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = {}
    for name in CONFIG_WORKLOADS:
        w = workloads.get(name)
        plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                       min_shared=w.min_shared)
        dp = plan.to_device()
        info = plan.info
        F, Hq, Hkv, d = info["n_fwd"], w.n_heads_q, w.n_heads_kv, w.head_dim
        q = wrng.normal_bf16(w.seeds["q"], (F, Hq, d), "cuda")
        k = wrng.normal_bf16(w.seeds["k"], (F, Hkv, d), "cuda")
        v = wrng.normal_bf16(w.seeds["v"], (F, Hkv, d), "cuda")
        ops.rope_by_depth(q, k, dp.depth, w.rope_base)
        o = torch.empty_like(q)
        lse = torch.empty((Hq, F), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        clocks = Clocks(local)
        torch.cuda.synchronize()
        clocks.start()
        ms, n = _time_launches(lambda: ops.tree_attn_fwd(dp, q, k, v, out=o, lse=lse, dev_err=err), flush,
                               warmup=max(3, warmup))
        clk = clocks.stop()
        if int(err.item()) != 0:
            raise SystemExit("device wait timed out (TPK_E_TIMEOUT) on %s" % name)
        flops = 4.0 * d * Hq * info["useful_pairs"]
        tfl = flops / ms / 1e9
        out[name] = {"raw_tokens": info["n_raw"], "forwarded_tokens": F, "rows": info["n_rows"],
                     "packing_ratio": info["packing_ratio"], "useful_pairs": info["useful_pairs"],
                     "Hq": Hq, "Hkv": Hkv, "head_dim": d, "ms": ms, "launches_timed": n,
                     "raw_tokens_per_s": info["n_raw"] / ms * 1e3, "forwarded_tokens_per_s": F / ms * 1e3,
                     "useful_tflops": tfl, "frac_of_burst_peak": tfl / peaks["bf16_tflops"], "clocks": clk}
        del q, k, v, o, lse, dp, plan
        torch.cuda.empty_cache()
    for rho in (1.45, 2.0, 2.8, 3.56):
        tree, seq = out["sweep_%.2f" % rho], out["sweep_%.2f_seqpack" % rho]
        tree["speedup_vs_sequence_packing"] = seq["ms"] / tree["ms"]
    return {"what": "forward only, one launch timed at a time: L2 flushed (256 MiB write) before each, median "
                    "of >= 10 launches and >= 0.5 s; frac against the burst bf16 peak (%s); "
                    "sweep_<rho>_seqpack = the same raw tokens without sharing" % peaks["source"],
            "peak_tflops": peaks["bf16_tflops"], "workloads": out}


GDN_WORKLOADS = ("grpo", "deep")
GDN_SHAPE = {"H": 16, "dk": 128, "dv": 128, "W": 4}


def fp32_peak_tflops(sm_mhz=None):
    """Dense fp32 FMA peak of this GPU: SMs x 128 fp32 lanes x 2 FLOP per FMA
    x the SM clock (the maximum clock unless one is given)."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = sm_mhz or 2070.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12, sms


def run_gdn(peaks, local, warmup, names=GDN_WORKLOADS):
    """The GDN tree path (causal conv + gated delta rule, H 16, dk = dv 128,
    conv width 4) on the tree batches: each call timed alone with L2 flushed
    before it, median, with its own clock sample."""
    import torch
    import workloads
    from prefix_tree_packed_dfs_gb300 import ops
    from workloads import rng as wrng
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    H, dk, dv, W = GDN_SHAPE["H"], GDN_SHAPE["dk"], GDN_SHAPE["dv"], GDN_SHAPE["W"]
    C = H * (2 * dk + dv)
    out = {}
    for name in names:
        w = workloads.get(name)
        plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                       min_shared=w.min_shared)
        dp = plan.to_device()
        info = plan.info
        F = info["n_fwd"]
        x, wc, g, b = wrng.gdn_inputs(w.seed_base + 50, F, C, H, W, "cuda")
        y = torch.empty_like(x)
        o = torch.empty((F, H, dv), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(max(int(ops.B.load().tpk_gdn_workspace_bytes(plan.handle, H, dk, dv)), 256),
                         dtype=torch.uint8, device="cuda")
        q, k, v = (y[:, :H * dk].unflatten(1, (H, dk)), y[:, H * dk:2 * H * dk].unflatten(1, (H, dk)),
                   y[:, 2 * H * dk:].unflatten(1, (H, dv)))
        clocks = Clocks(local)
        torch.cuda.synchronize()
        clocks.start()
        ms_conv, n_conv = _time_launches(lambda: ops.gdn_conv(dp, x, wc, y=y), flush, min_s=0.3, warmup=warmup)
        ms_delta, n_delta = _time_launches(lambda: ops.gdn_delta_rule(dp, q, k, v, g, b, out=o, workspace=ws),
                                           flush, min_s=0.5, min_n=5, warmup=warmup)
        # backward: the delta rule's gradients as column slices of one dy,
        # which the convolution's backward reads
        dO = wrng.normal_bf16(w.seed_base + 51, (F, H, dv), "cuda")
        dy, dx = torch.empty_like(x), torch.empty_like(x)
        dw = torch.empty_like(wc)
        dq, dkk, dvv = (dy[:, :H * dk].unflatten(1, (H, dk)), dy[:, H * dk:2 * H * dk].unflatten(1, (H, dk)),
                        dy[:, 2 * H * dk:].unflatten(1, (H, dv)))
        dg = torch.empty((F, H), dtype=torch.float32, device="cuda")
        db = torch.empty_like(dg)
        lib = ops.B.load()
        wsb = torch.empty(max(int(lib.tpk_gdn_bwd_workspace_bytes(plan.handle, H, dk, dv)), 256), dtype=torch.uint8,
                          device="cuda")
        wsc = torch.empty(max(int(lib.tpk_gdn_conv_bwd_workspace_bytes(plan.handle, C, W)), 256), dtype=torch.uint8,
                          device="cuda")
        ms_dbwd, n_dbwd = _time_launches(
            lambda: ops.gdn_delta_rule_bwd(dp, q, k, v, g, b, dO, ws, dq=dq, dk=dkk, dv=dvv, dg=dg, dbeta=db,
                                           workspace=wsb), flush, min_s=0.5, min_n=3, warmup=warmup)
        ms_cbwd, n_cbwd = _time_launches(lambda: ops.gdn_conv_bwd(dp, x, wc, dy, dx=dx, dw=dw, workspace=wsc), flush,
                                         min_s=0.3, warmup=warmup)
        clk = clocks.stop()
        conv_bytes = 2 * F * C * 2 + 4 * F + 4 * C * W          # x read, y written, parent, weights
        # x and dy read, dx written; parent, depth, subtree_end; dw partials
        # written and read back
        conv_bwd_bytes = 3 * F * C * 2 + 12 * F + 2 * (wsc.numel() // 4 * 4)
        delta_flop = 6.0 * dk * dv * F * H                      # S k, the update, S q per token and head
        # executed: the recomputed forward (6) and, walking back, the output
        # term, D k, S^T do, D^T u, the reversal (3), S^T y, the D update (3)
        delta_bwd_flop = 22.0 * dk * dv * F * H
        peak32, sms = fp32_peak_tflops(clk.get("sm_mhz"))
        out[name] = {"forwarded_tokens": F, "raw_tokens": info["n_raw"], "segment_instances": info["n_seg_instances"],
                     "levels": info["n_seg_levels"], "conv_ms": ms_conv, "conv_gbs": conv_bytes / ms_conv / 1e6,
                     "conv_frac_of_copy_peak": conv_bytes / ms_conv / 1e6 / peaks["hbm_gbs"],
                     "delta_ms": ms_delta, "delta_tflops": delta_flop / ms_delta / 1e9,
                     "delta_frac_of_fp32_peak": delta_flop / ms_delta / 1e9 / peak32,
                     "fp32_peak_tflops": peak32, "forwarded_tokens_per_s": F / (ms_conv + ms_delta) * 1e3,
                     "raw_tokens_per_s": info["n_raw"] / (ms_conv + ms_delta) * 1e3,
                     "delta_bwd_ms": ms_dbwd, "delta_bwd_tflops": delta_bwd_flop / ms_dbwd / 1e9,
                     "delta_bwd_frac_of_fp32_peak": delta_bwd_flop / ms_dbwd / 1e9 / peak32,
                     "conv_bwd_ms": ms_cbwd, "conv_bwd_gbs": conv_bwd_bytes / ms_cbwd / 1e6,
                     "conv_bwd_frac_of_copy_peak": conv_bwd_bytes / ms_cbwd / 1e6 / peaks["hbm_gbs"],
                     "fwd_bwd_raw_tokens_per_s": info["n_raw"] / (ms_conv + ms_delta + ms_dbwd + ms_cbwd) * 1e3,
                     "launches_timed": [n_conv, n_delta, n_dbwd, n_cbwd], "clocks": clk}
        del x, y, o, ws, q, k, v, dO, dy, dx, dw, dq, dkk, dvv, dg, db, wsb, wsc, dp, plan
        torch.cuda.empty_cache()
    return {"what": "GDN tree path, H %d, dk = dv = %d, conv width %d: conv and its backward (HBM-bound: against "
                    "the copy peak) and gated delta rule forward and backward (one launch per tree level, fp32 "
                    "state: against the fp32 FMA peak = SMs x 128 lanes x 2 x the median SM clock; the backward's "
                    "executed FLOP include its recomputed forward); L2 flushed before every timed call"
                    % (H, dk, W), "workloads": out}


def run_ours(a):
    import torch
    import workloads
    from prefix_tree_packed_dfs_gb300 import ops
    from workloads import rng as wrng

    world, rank, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (no CPU path exists)")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    peaks = _peaks()
    w = workloads.get(a.workload)
    # rows are independent, so no data crosses ranks.  Weak scaling (default):
    # every rank owns one batch of the same shape.  --shard-rows: one batch,
    # its rows dealt to the ranks longest first; each rank plans its rows'
    # sequences with their row as the group, which rebuilds exactly those rows.
    sharded = a.shard_rows and world > 1
    t0 = time.perf_counter()
    full = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                   min_shared=w.min_shared)
    if sharded:
        rank_of_row, _ = full.shard_rows(world)
        plan, my_seqs = full.rank_plan(w.sequences, rank_of_row, rank, w.row_capacity, w.min_shared)
        my_groups = full.export()["row_of_seq"][my_seqs]
    else:
        plan, my_seqs, my_groups = full, np.arange(len(w.sequences)), w.group_ids
    plan_s = time.perf_counter() - t0
    info = plan.info
    # raw / forwarded tokens per second of the whole job
    job_rate = ((lambda n_rank, n_full, secs: n_full / secs) if sharded
                else (lambda n_rank, n_full, secs: job_value(world, n_rank, secs)))
    F, R, d, Hq, Hkv = info["n_fwd"], info["n_raw"], w.head_dim, w.n_heads_q, w.n_heads_kv
    pairs = info["useful_pairs"]
    dp = plan.to_device()
    dev = torch.device("cuda", local)
    s = rank_seeds(w, rank)
    Q = wrng.normal_bf16(s["q"], (F, Hq, d), dev)
    K = wrng.normal_bf16(s["k"], (F, Hkv, d), dev)
    V = wrng.normal_bf16(s["v"], (F, Hkv, d), dev)
    # the output gradient arrives in raw order, one row per raw token, and is
    # summed into the packed layout inside the step (transpose of the scatter)
    dO_raw = wrng.normal_bf16(s["do"], (R, Hq, d), dev)
    dO = torch.empty((F, Hq, d), dtype=torch.bfloat16, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty((Hq, F), dtype=torch.float32, device=dev)
    O_raw = torch.empty((R, Hq, d), dtype=torch.bfloat16, device=dev)
    LSE_raw = torch.empty((Hq, R), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    ws = torch.empty(max(ops.attn_workspace_bytes(dp, Hq, Hkv, d, True), 256), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    names = ["rope", "fwd", "scatter", "dO_sum", "bwd_prep", "bwd_dkdv", "bwd_dq"]

    def step(dplan, ev=None, ready=None, sig=None, qkv=None, precise=False, o_lo=None):
        """One pass of the path.  Q and K are rotated in place; the backward
        returns dQ, dK w.r.t. the un-rotated inputs (inverse RoPE in its
        epilogues).  End to end only: ``qkv`` replaces (Q, K, V) (double-
        buffered inputs); ``ready`` holds events of the input uploads, each
        waited for right before the first kernel that reads that input ("qk",
        "v", "do"), and "lse_free" (the previous step's raw-order LSE has been
        read back) before the scatter; ``sig`` receives events recorded once
        the raw-order outputs are final ("out"), the raw dO has been summed
        ("dosum") and the step is complete ("done")."""
        Qt, Kt, Vt = (Q, K, V) if qkv is None else qkv
        mark = (lambda i: ev[i].record()) if ev is not None else (lambda i: None)
        wait = ((lambda k: torch.cuda.current_stream().wait_event(ready[k]) if k in ready else None)
                if ready else (lambda k: None))
        note = (lambda k: sig[k].record()) if sig is not None else (lambda k: None)
        mark(0)
        wait("qk")
        ops.rope_by_depth(Qt, Kt, dplan.depth, w.rope_base)
        mark(1)
        wait("v")
        ops.tree_attn_fwd(dplan, Qt, Kt, Vt, out=O, lse=LSE, dev_err=err, precise=precise, o_lo=o_lo)
        mark(2)
        wait("lse_free")
        ops.scatter_token_index(dplan.token_index, O, LSE, dst=O_raw, lse_dst=LSE_raw)
        note("out")
        mark(3)
        wait("do")
        ops.sum_to_forwarded(dplan, dO_raw, dst=dO)
        note("dosum")
        mark(4)
        for ph in (0, 1, 2):
            ops.tree_attn_bwd(dplan, Qt, Kt, Vt, O, LSE, dO, dq=dq, dk=dk, dv=dv, workspace=ws, dev_err=err,
                              phases=(ph,), precise=precise, o_lo=o_lo, rope_base=w.rope_base)
            mark(5 + ph)
        note("done")

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def timed(n_steps, **kw):
        """n_steps steps between a barrier + synchronize on both sides, with
        a clock sample; returns (ms per step, per-kernel mean ms, clocks)."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(n_steps)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = Clocks(local)
        barrier()
        torch.cuda.synchronize()
        clocks.start()
        start.record()
        for i in range(n_steps):
            step(dp, evs[i], **kw)
        stop.record()
        torch.cuda.synchronize()
        barrier()
        clk = clocks.stop()
        per = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_steps))
               for j, n in enumerate(names)}
        if int(err.item()) != 0:
            raise SystemExit("device wait timed out (TPK_E_TIMEOUT)")
        return start.elapsed_time(stop) / n_steps, per, clk

    for _ in range(a.warmup):
        step(dp)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit("device wait timed out (TPK_E_TIMEOUT)")
    ms, per, clk = timed(a.steps)
    ms = max_over_ranks(ms, dev, world)

    # ---- the same step in the precise mode ---------------------------------
    fwd_flop = 4.0 * d * Hq * pairs
    bwd_flop = 10.0 * d * Hq * pairs
    precise = None
    if not a.no_precise:
        O_lo = torch.empty_like(Q)
        n_p = max(2, min(a.steps, 3))
        for _ in range(max(1, min(a.warmup, 2))):
            step(dp, precise=True, o_lo=O_lo)
        ms_p, per_p, clk_p = timed(n_p, precise=True, o_lo=O_lo)
        ms_p = max_over_ranks(ms_p, dev, world)
        del O_lo
        torch.cuda.empty_cache()
        t_bwd = (per_p["bwd_prep"] + per_p["bwd_dkdv"] + per_p["bwd_dq"]) / 1e3
        precise = {"what": "same step with P and dS as hi + lo bf16 pairs (one more product each for PV, dV, dK, "
                           "dQ) and D from O before its rounding; gradients within the stated max-abs 1e-2",
                   "value": job_rate(R, full.info["n_raw"], ms_p / 1e3), "unit": "raw tokens/s",
                   "ms_per_step": ms_p, "steps": n_p, "useful_tflops": (fwd_flop + bwd_flop) / (ms_p / 1e3) / 1e12,
                   "fwd_tflops": fwd_flop / (per_p["fwd"] / 1e3) / 1e12, "bwd_tflops": bwd_flop / t_bwd / 1e12,
                   "kernels_ms": per_p, "clocks": clk_p, "slowdown_vs_fast": ms_p / ms}

    # ---- end to end through the public API, host buffers -----------------
    e2e = None
    if a.e2e_steps > 0:
        tokens = np.concatenate([w.sequences[i] for i in my_seqs]).astype(np.int32)
        offs = np.zeros(len(my_seqs) + 1, np.int64)
        offs[1:] = np.cumsum([len(w.sequences[i]) for i in my_seqs])
        hQ, hK, hV, hdO = (torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (Q, K, V, dO_raw))
        for h, x in zip((hQ, hK, hV, hdO), (Q, K, V, dO_raw)):
            h.copy_(x)
        hLSE = torch.empty((Hq, R), dtype=torch.float32).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in (hQ, hK, hV, hdO)) + plan.device_bytes()
        d2h = hLSE.numel() * hLSE.element_size()

        # Q, K (rotated in place) and V are read until the end of the
        # backward, so step i+1's inputs go to a second set of buffers, as a
        # prefetching data loader fills them; the raw dO is free once summed
        sets = ((Q, K, V), (torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)))
        copy_stream = torch.cuda.Stream(dev)

        def build_plan():
            return ops.Plan(tokens, offs, group_ids=my_groups, row_capacity=w.row_capacity,
                            min_shared=w.min_shared, placement="groups" if sharded else "bfd")

        def events(*keys, timing=False):
            return {k: torch.cuda.Event(enable_timing=timing) for k in keys}

        def upload(j, make_plan, prev, prev2):
            """Step j's inputs on the copy stream into buffer set j % 2, behind
            the kernel of step j-2 (``prev2``) that last read that set and,
            for the raw dO and the LSE read-back, behind step j-1 (``prev``),
            in the order the GPU reaches them.  The host builds step j's plan
            (``make_plan``) while Q and K go up.  Returns (device plan, events
            step j waits for)."""
            ready = events("q", "k", "qk", "v", "do", "lse_free", timing=True)
            qj, kj, vj = sets[j % 2]
            with torch.cuda.stream(copy_stream):
                if prev2:
                    copy_stream.wait_event(prev2["done"])   # step j-2 read this set
                qj.copy_(hQ, non_blocking=True)
                ready["q"].record()
                kj.copy_(hK, non_blocking=True)
                ready["k"].record()
                t_host = [time.perf_counter()]
                p2 = make_plan()
                t_host.append(time.perf_counter())
                d2 = p2.to_device(dev)   # the plan image right behind Q, K
                t_host.append(time.perf_counter())
                ready["qk"].record()
                ready["host_s"] = t_host
                vj.copy_(hV, non_blocking=True)
                ready["v"].record()
                if prev:
                    copy_stream.wait_event(prev["out"])
                    hLSE.copy_(LSE_raw, non_blocking=True)
                ready["lse_free"].record()
                if prev:
                    copy_stream.wait_event(prev["dosum"])
                dO_raw.copy_(hdO, non_blocking=True)
                ready["do"].record()
            return d2, ready

        def run_e2e(n):
            """n steps through the public API from host buffers, as a training
            loop with a prefetching data loader runs them: while the GPU
            executes step i, the host builds step i+1's plan and the copy
            stream uploads step i+1's inputs.  Every step's uploads, plan
            build and LSE read-back happen inside the timed region; the first
            step's uploads are not hidden behind anything.  Returns (seconds,
            per-step GPU intervals in ms, the first step's milestones in ms)."""
            torch.cuda.synchronize()
            barrier()
            t0 = time.perf_counter()
            origin = torch.cuda.Event(enable_timing=True)
            origin.record(copy_stream)
            d_cur, ready = upload(0, build_plan, None, None)
            ready0 = ready
            live = [None, d_cur]          # device plans of steps i-1, i
            sigs = []
            for i in range(n):
                sig = events("out", "dosum", "done", timing=True)
                step(live[-1], ready=ready, sig=sig, qkv=sets[i % 2])
                sigs.append(sig)
                if i + 1 < n:
                    d_nxt, ready = upload(i + 1, build_plan, sig, sigs[-2] if i > 0 else None)
                else:
                    with torch.cuda.stream(copy_stream):
                        copy_stream.wait_event(sig["out"])
                        hLSE.copy_(LSE_raw, non_blocking=True)
                    d_nxt = None
                if i > 0:
                    sigs[-2]["done"].synchronize()   # step i-1 has finished with its plan
                live = [live[-1], d_nxt]
            torch.cuda.synchronize()
            dt = time.perf_counter() - t0
            barrier()
            gaps = [sigs[i - 1]["done"].elapsed_time(sigs[i]["done"]) for i in range(1, n)]
            first = {k: round(origin.elapsed_time(e), 1) for k, e in
                     (("q_ready", ready0["q"]), ("k_ready", ready0["k"]), ("qk_plan_ready", ready0["qk"]),
                      ("v_ready", ready0["v"]), ("do_ready", ready0["do"]),
                      ("step_out", sigs[0]["out"]), ("step_done", sigs[0]["done"]))}
            hs = ready0["host_s"]
            first["host_plan_build"] = round(1e3 * (hs[1] - hs[0]), 1)
            first["host_plan_upload_call"] = round(1e3 * (hs[2] - hs[1]), 1)
            first["host_start_to_plan_built"] = round(1e3 * (hs[1] - t0), 1)
            return dt, gaps, first

        run_e2e(2)                        # warm-up: allocations, page-locked staging
        dt, gaps, first = run_e2e(a.e2e_steps)
        dt = max_over_ranks(dt / a.e2e_steps, dev, world)
        e2e = {"value": job_rate(R, full.info["n_raw"], dt), "unit": "raw tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": 1e3 * dt, "steps": a.e2e_steps,
               "ms_between_step_ends": [round(x, 1) for x in gaps], "first_step_ms": first,
               "statistic": "wall time of all steps / steps",
               "includes": "one plan build on the host per step, plan image + Q/K/V + raw-order dO "
                           "host->device and the raw-order LSE device->host every step; step i+1's "
                           "plan is built and its inputs uploaded while the GPU runs step i (Q, K, V "
                           "double-buffered); the first step's uploads are not overlapped"}
        del hQ, hK, hV, hdO, sets

    # ---- CPU baseline (oracle), rank 0 only ----------------------------------
    cpu = None
    if rank == 0 and not a.no_cpu_baseline and a.cpu_seconds > 0:
        from oracle import planner as op
        ref = op.plan(w.sequences, group_ids=w.group_ids, min_shared=w.min_shared, row_capacity=w.row_capacity)
        n, dt = OracleSampler(w, ref).run(a.cpu_seconds)
        cpu = {"value": n / dt, "unit": "raw tokens/s", "cores": _cpu_threads(), "kind": "oracle",
               "sample": "fp64 oracle forward row + dQ row for %d raw tokens drawn uniformly from 2 of the 128 "
                         "24000-token sequences (%.1f s); dK/dV rows not included" % (n, dt)}

    # ---- roofline of the dominant kernel ------------------------------------
    algo = {   # algorithmic FLOPs (tensor kernels) or bytes (HBM kernels) per launch
        "fwd": ("tensor", fwd_flop),
        "bwd_dkdv": ("tensor", 8.0 * d * Hq * pairs),     # S^T, dP^T, dV, dK products
        "bwd_dq": ("tensor", 2.0 * d * Hq * pairs),       # dQ product (S, dP recomputed on top)
        "rope": ("hbm", F * (Hq + Hkv) * d * 2 * 2 + 4 * F),
        "scatter": ("hbm", R * Hq * (2 * d + 4) * 2 + 4 * R),
        "dO_sum": ("hbm", (R + F) * Hq * d * 2 + 4 * (F + 1) + 4 * R),
        "bwd_prep": ("hbm", F * Hq * d * 2 * 2 + 4 * F * Hq),
    }
    dom = max(per, key=per.get)
    bound, amount = algo[dom]
    secs = per[dom] / 1e3
    if bound == "tensor":
        peak = peaks["bf16_tflops_sustained"]
        roof = {"kernel": dom, "bound": "tensor", "achieved": amount / secs / 1e12, "peak": peak,
                "unit": "TFLOP/s", "frac": amount / secs / 1e12 / peak, "traffic": recorded_traffic(dom, a.workload),
                "peak_kind": "sustained bf16 (%s)" % peaks["source"],
                "frac_of_burst": amount / secs / 1e12 / peaks["bf16_tflops"]}
    else:
        peak = peaks["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": amount / secs / 1e9, "peak": peak, "unit": "GB/s",
                "frac": amount / secs / 1e9 / peak, "traffic": recorded_traffic(dom, a.workload), "peak_kind": "copy bandwidth (%s)" % peaks["source"]}
    kernels = {}
    for n in names:
        b, amt = algo[n]
        t_s = per[n] / 1e3
        kernels[n] = {"ms": per[n], ("tflops" if b == "tensor" else "gbs"):
                      amt / t_s / (1e12 if b == "tensor" else 1e9)}

    # ---- forward on the other workloads (after the deep tree's buffers go) --
    configs = gdn = None
    if (not a.no_configs or not a.no_gdn) and rank == 0:
        del Q, K, V, dO_raw, dO, O, LSE, O_raw, LSE_raw, dq, dk, dv, ws
        torch.cuda.empty_cache()
    if not a.no_configs and rank == 0:
        configs = run_configs(peaks, local, a.warmup)
    if not a.no_gdn and rank == 0:
        gdn = run_gdn(peaks, local, max(1, min(a.warmup, 3)))

    useful_tflops = (fwd_flop + bwd_flop) / (ms / 1e3) / 1e12
    out = {
        "metric": METRIC, "value": job_rate(R, full.info["n_raw"], ms / 1e3), "unit": "raw tokens/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if sharded else "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC, "raw_tokens": R, "forwarded_tokens": F, "rows": info["n_rows"],
                   "packing_ratio": info["packing_ratio"], "useful_pairs": pairs,
                   "visited_pairs_fwd": info["visited_pairs"], "Hq": Hq, "Hkv": Hkv, "head_dim": d,
                   "row_capacity": w.row_capacity, "precision": "fast (bf16 P and dS operands)",
                   "l2": "inputs larger than L2 (Q alone %.1f GB)" % (F * Hq * d * 2 / 1e9),
                   "parallelism": ("one batch, whole rows per rank (longest first), no collective" if sharded
                                   else "one batch per rank, no collective" if world > 1 else "single GPU")},
        "useful_tflops": useful_tflops,
        "pct_of_peak": 100.0 * useful_tflops / peaks["bf16_tflops_sustained"],
        "pct_of_burst_peak": 100.0 * useful_tflops / peaks["bf16_tflops"],
        "forwarded_tokens_per_s": job_rate(F, full.info["n_fwd"], ms / 1e3),
        "fwd_tflops": fwd_flop / (per["fwd"] / 1e3) / 1e12,
        "bwd_tflops": bwd_flop / ((per["bwd_prep"] + per["bwd_dkdv"] + per["bwd_dq"]) / 1e3) / 1e12,
        "kernels": kernels,
        "plan_ms": plan_s * 1e3,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "precise": precise,
        "configs": configs,
        "gdn": gdn,
        "gpu_launches": LAUNCHES_PER_STEP * a.steps,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_sweep(a):
    """Forward attention over one 32,768-forwarded-token row at packing ratios
    1.00 .. 3.56, and over the same raw tokens laid out without sharing
    (sequence packing: min shared length above every run).  L2 is flushed
    (a 256 MiB write) before every timed launch; CUDA events bracket the
    attention kernel alone on the current stream; each point carries its own
    nvidia-smi clock sample."""
    import torch
    import workloads
    from prefix_tree_packed_dfs_gb300 import ops
    from workloads import rng as wrng
    peaks = _peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def time_fwd(name):
        w = workloads.get(name)
        plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                       min_shared=w.min_shared)
        dp = plan.to_device()
        info = plan.info
        F, Hq, Hkv, d = info["n_fwd"], w.n_heads_q, w.n_heads_kv, w.head_dim
        q = wrng.normal_bf16(w.seeds["q"], (F, Hq, d), "cuda")
        k = wrng.normal_bf16(w.seeds["k"], (F, Hkv, d), "cuda")
        v = wrng.normal_bf16(w.seeds["v"], (F, Hkv, d), "cuda")
        ops.rope_by_depth(q, k, dp.depth, w.rope_base)
        o = torch.empty_like(q)
        lse = torch.empty((Hq, F), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        clocks = Clocks(0)
        torch.cuda.synchronize()
        clocks.start()
        ms, n = _time_launches(lambda: ops.tree_attn_fwd(dp, q, k, v, out=o, lse=lse, dev_err=err), flush,
                               min_n=max(a.steps, 10), warmup=max(a.warmup, 3))
        clk = clocks.stop()
        if int(err.item()) != 0:
            raise SystemExit("device wait timed out (TPK_E_TIMEOUT)")
        flops = 4.0 * d * Hq * info["useful_pairs"]
        return {"raw_tokens": info["n_raw"], "forwarded_tokens": F, "rows": info["n_rows"],
                "useful_pairs": info["useful_pairs"], "visited_pairs": info["visited_pairs"], "ms": ms,
                "launches_timed": n, "useful_tflops": flops / ms / 1e9, "raw_tokens_per_s": info["n_raw"] / ms * 1e3,
                "forwarded_tokens_per_s": F / ms * 1e3, "clocks": clk}

    for rho in workloads.SWEEP_RHOS:
        tree = time_fwd("sweep_%.2f" % rho)
        seq = time_fwd("sweep_%.2f_seqpack" % rho)
        tree["pct_of_peak"] = 100.0 * tree["useful_tflops"] / peaks["bf16_tflops"]
        print(json.dumps({
            "mode": "sweep", "metric": METRIC, "packing_ratio": tree["raw_tokens"] / tree["forwarded_tokens"],
            "tree": tree, "sequence_packing": seq, "speedup_vs_sequence_packing": seq["ms"] / tree["ms"],
            "peak_tflops": peaks["bf16_tflops"], "peak_kind": "burst bf16 (%s): kernel timed alone" % peaks["source"],
            "config": {"workload": "one row of 32768 forwarded tokens from 4 rollouts sharing a prefix; Hq 16 / Hkv 8 "
                                   "/ d 128; sequence packing = the same raw tokens with no sharing, rows of 32768",
                       "l2": "flushed (256 MiB write) before every timed launch"},
        }), flush=True)


def run_layout(a):
    """Raw order <-> packed layout kernels on one workload (default: the deep
    tree): materialisation of a per-token payload by owner (int32 token ids,
    and rows of Hq*d bf16) and the sum of raw-order rows into the packed
    layout.  L2 flushed before every timed launch; one JSON line."""
    import torch
    import workloads
    from prefix_tree_packed_dfs_gb300 import ops
    from workloads import rng as wrng
    peaks = _peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    w = workloads.get(a.workload)
    plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                   min_shared=w.min_shared)
    dp = plan.to_device()
    F, R, Hq, d = plan.info["n_fwd"], plan.info["n_raw"], w.n_heads_q, w.head_dim
    tokens = torch.from_numpy(np.concatenate(w.sequences).astype(np.int32)).cuda()
    rows = wrng.normal_bf16(w.seeds["do"], (R, Hq, d), "cuda")
    tok_f = torch.empty(F, dtype=torch.int32, device="cuda")
    rows_f = torch.empty((F, Hq, d), dtype=torch.bfloat16, device="cuda")

    def timed(fn):
        for _ in range(a.warmup):
            fn()
        times = []
        for _ in range(max(a.steps, 3)):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    idx = 4 * (F + 1) + 4 * F   # CSR begin + one raw index per position
    out = {}
    for name, fn, nbytes in (
            ("gather_token_ids", lambda: ops.gather_to_forwarded(dp, tokens, dst=tok_f), 8 * F + idx),
            ("gather_rows_bf16", lambda: ops.gather_to_forwarded(dp, rows, dst=rows_f), 2 * F * Hq * d * 2 + idx),
            ("sum_rows_bf16", lambda: ops.sum_to_forwarded(dp, rows, dst=rows_f), (R + F) * Hq * d * 2 + 4 * (F + 1 + R))):
        ms = timed(fn)
        out[name] = {"ms": ms, "gbs": nbytes / ms / 1e6, "frac_of_copy_peak": nbytes / ms / 1e6 / peaks["hbm_gbs"],
                     "algorithmic_bytes": nbytes}
    print(json.dumps({"mode": "layout", "workload": a.workload, "raw_tokens": R, "forwarded_tokens": F,
                      "row_bytes": Hq * d * 2, "kernels": out, "peak_gbs": peaks["hbm_gbs"],
                      "peak_kind": "copy bandwidth (%s)" % peaks["source"],
                      "l2": "flushed (256 MiB write) before every timed launch"}), flush=True)


def _time_library_planner(ops, w):
    """(first build ms, median of three further builds ms, last plan).  Each
    plan is destroyed before the next build, as a loop that plans one batch
    per step does, so later builds reuse the previous plan's storage."""
    def build():
        t0 = time.perf_counter()
        plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                       min_shared=w.min_shared)
        return plan, time.perf_counter() - t0
    plan, first = build()
    times = []
    for _ in range(3):
        plan.close()
        plan, dt = build()
        times.append(dt)
    return 1e3 * first, 1e3 * statistics.median(times), plan


def _planner_threads():
    env = os.environ.get("TPK_PLANNER_THREADS", "")
    if env.isdigit() and int(env) >= 1:
        return min(int(env), 16)
    return min(os.cpu_count() or 1, 16)


def run_planner(a):
    """Host planner of the library against the oracle's planner, every
    workload: the library's first build and the median of three more, one
    oracle build.  No GPU."""
    import workloads
    from oracle import planner as op
    from prefix_tree_packed_dfs_gb300 import ops
    cores = _cpu_threads()
    for name in workloads.ALL:
        w = workloads.get(name)
        first_ms, ms, plan = _time_library_planner(ops, w)
        t0 = time.perf_counter()
        op.plan(w.sequences, group_ids=w.group_ids, min_shared=w.min_shared, row_capacity=w.row_capacity)
        t_or = time.perf_counter() - t0
        info = plan.info
        print(json.dumps({"mode": "planner", "workload": name, "raw_tokens": info["n_raw"],
                          "forwarded_tokens": info["n_fwd"], "rows": info["n_rows"],
                          "library_ms": ms, "library_first_ms": first_ms, "oracle_ms": 1e3 * t_or,
                          "oracle_over_library": t_or * 1e3 / ms,
                          "library_raw_tokens_per_s": info["n_raw"] / ms * 1e3, "host_threads": cores,
                          "library_threads": _planner_threads(), "oracle_threads": 1}), flush=True)
    # scaling with the number of leaves, on stand-ins for the multi-task
    # batches of "Prefix Tree Packing in ART" (section "Bin packing, with a
    # twist"), whose table gives tree walk / bin packing ms and rows for the
    # same group and completion counts (another machine, another language:
    # context only)
    pages = {12: (0.9, 1.4, 15), 48: (9.6, 4.2, 61), 192: (42.0, 48.7, 227), 768: (291.2, 743.5, 918)}
    for g, n_comp in workloads.CURRICULUM.items():
        w = workloads.get("curriculum_%d" % g)
        first_ms, ms, plan = _time_library_planner(ops, w)
        t0 = time.perf_counter()
        op.plan(w.sequences, group_ids=w.group_ids, min_shared=w.min_shared, row_capacity=w.row_capacity)
        t_or = time.perf_counter() - t0
        info = plan.info
        walk, pack, rows = pages[g]
        print(json.dumps({"mode": "planner_scaling", "workload": w.name, "groups": g, "completions": n_comp,
                          "raw_tokens": info["n_raw"], "forwarded_tokens": info["n_fwd"], "rows": info["n_rows"],
                          "library_ms": ms, "library_first_ms": first_ms, "oracle_ms": 1e3 * t_or,
                          "host_threads": cores, "library_threads": _planner_threads(), "oracle_threads": 1,
                          "pages_context": {"tree_walk_ms": walk, "bin_packing_ms": pack, "rows": rows,
                                            "batch_shape": "not given on the page"}}), flush=True)


def main():
    a = _args()
    if a.planner:
        run_planner(a)
    elif a.sweep:
        run_sweep(a)
    elif a.layout:
        run_layout(a)
    elif a.gdn:
        import torch
        print(json.dumps({"mode": "gdn", **run_gdn(_peaks(), 0, max(a.warmup, 1), names=(a.workload,))}), flush=True)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
