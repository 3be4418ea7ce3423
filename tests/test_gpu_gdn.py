"""GPU parity of the GDN tree path (tpk_gdn_conv, tpk_gdn_delta_rule) against
the fp64 oracle of oracle/gdn.py, which runs every root-to-leaf sequence
unpacked from zero state.

Acceptance: the outputs are bf16, so as for the attention output O:
relative L2 <= 5e-3 and |got - ref| <= 1e-2 * max(1, |ref|); the convolution
(one fp32 sum, one bf16 rounding) is held to one bf16 step: |got - ref| <=
2^-7 |ref| + 1e-5.  Small trees are compared in full; the full-size batch in
the bench's launch configuration on sampled raw tokens (each one's sequence
prefix run by the oracle from zero).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import gdn as og
from oracle import planner as op
from oracle.bf16 import round_to_bf16
from workloads import rng as wrng

from tests.test_gpu_kernels import SMALL, assert_close, f64, record

pytestmark = pytest.mark.gpu

W = 4


@pytest.fixture(scope="module")
def ops():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from prefix_tree_packed_dfs_gb300 import ops as _ops
    _ops.B.load()
    return _ops


def _plans(ops, w):
    plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                   min_shared=w.min_shared)
    ref = op.plan(w.sequences, group_ids=w.group_ids, min_shared=w.min_shared, row_capacity=w.row_capacity)
    return plan, plan.to_device(), ref


def _split(y, H, dk, dv):
    """q, k, v views of the convolution's output [F, H*(2dk+dv)]."""
    q = y[:, :H * dk].unflatten(1, (H, dk))
    k = y[:, H * dk:2 * H * dk].unflatten(1, (H, dk))
    v = y[:, 2 * H * dk:].unflatten(1, (H, dv))
    return q, k, v


CASES = [("tiny_fit", 2, 64), ("deep_small", 2, 128), ("ragged_d128_h1", 3, 128), ("ragged_d64_gqa2", 2, 64),
         ("ragged_d64_h1", 1, 64)]


@pytest.mark.parametrize("name,H,d", CASES)
def test_gdn_full_parity(ops, name, H, d):
    """Convolution and delta rule, each against the oracle on the same inputs,
    and the two chained through strided views of the convolution's output."""
    w = SMALL[name]()
    plan, dp, ref = _plans(ops, w)
    F = plan.info["n_fwd"]
    C = H * 3 * d
    x, wc, g, b = wrng.gdn_inputs(w.seed_base + 50, F, C, H, W)
    # the GPU generates the same bits
    xg, wg, gg, bg = wrng.gdn_inputs(w.seed_base + 50, F, C, H, W, "cuda")
    assert torch.equal(xg.cpu(), x) and torch.equal(wg.cpu(), wc) and torch.equal(gg.cpu(), g) \
        and torch.equal(bg.cpu(), b)
    y = ops.gdn_conv(dp, xg, wg)
    torch.cuda.synchronize()
    yr = og.conv(ref, x.double().numpy(), wc.double().numpy())
    got = f64(y)
    err = np.abs(got - yr)
    record("%s gdn conv" % name, max_abs=float(err.max()), rel_l2=float(np.linalg.norm(got - yr) / np.linalg.norm(yr)))
    assert np.all(err <= 2.0 ** -7 * np.abs(yr) + 1e-5)
    # delta rule on the GPU's own (bf16) convolution output, through strided views
    q, k, v = _split(y, H, d, d)
    o = ops.gdn_delta_rule(dp, q, k, v, gg, bg)
    torch.cuda.synchronize()
    qn, kn, vn = (f64(t) for t in _split(y, H, d, d))
    ro = og.delta_rule(ref, qn, kn, vn, g.double().numpy(), b.double().numpy())
    assert_close(f64(o), ro, "%s gdn delta rule" % name)
    # end to end against the oracle's own chain (its fp64 convolution rounded
    # to bf16, as the library stores it)
    yq, yk, yv = (round_to_bf16(a) for a in (yr[:, :H * d], yr[:, H * d:2 * H * d], yr[:, 2 * H * d:]))
    ro2 = og.delta_rule(ref, yq.reshape(F, H, d), yk.reshape(F, H, d), yv.reshape(F, H, d), g.double().numpy(),
                        b.double().numpy())
    assert_close(f64(o), ro2, "%s gdn conv + delta rule" % name)


def test_gdn_contiguous_inputs_and_repeated_calls(ops):
    """Separate contiguous q, k, v give the same output as strided views, and
    two calls in a row give identical bits (deterministic, no hidden state)."""
    w = SMALL["ragged_d128_gqa4"]()
    plan, dp, ref = _plans(ops, w)
    F, H, d = plan.info["n_fwd"], 2, 128
    x, wc, g, b = wrng.gdn_inputs(4242, F, H * 3 * d, H, W, "cuda")
    y = ops.gdn_conv(dp, x, wc)
    q, k, v = _split(y, H, d, d)
    o1 = ops.gdn_delta_rule(dp, q, k, v, g, b)
    o2 = ops.gdn_delta_rule(dp, q.contiguous(), k.contiguous(), v.contiguous(), g, b)
    o3 = ops.gdn_delta_rule(dp, q, k, v, g, b)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(o1, o3)


GDN_FULL = [("grpo", 16, 128), ("agentic", 16, 128)]


@pytest.mark.parametrize("name,H,d", GDN_FULL)
def test_gdn_full_size_sampled(ops, name, H, d):
    """The full batch on the GPU in the bench's configuration; the oracle runs
    the sequence prefix of sampled raw tokens from zero state."""
    w = workloads.get(name)
    plan, dp, ref = _plans(ops, w)
    F = plan.info["n_fwd"]
    C = H * 3 * d
    seed = w.seed_base + 50
    x, wc, g, b = wrng.gdn_inputs(seed, F, C, H, W, "cuda")
    y = ops.gdn_conv(dp, x, wc)
    q, k, v = _split(y, H, d, d)
    o = ops.gdn_delta_rule(dp, q, k, v, g, b)
    torch.cuda.synchronize()
    rng = np.random.Generator(np.random.PCG64(11))
    off = ref["seq_offsets"]
    seqs = rng.choice(len(off) - 1, size=3, replace=False)
    raw = sorted({int(off[s] + rng.integers(0, off[s + 1] - off[s])) for s in seqs} | {int(off[seqs[0] + 1]) - 1})
    # the oracle's inputs: the GPU's convolution output rows (bf16) and the
    # regenerated g, beta rows
    yc = y.cpu()
    wcpu = wc.cpu().double().numpy()

    def rows(key, idx):
        idx = np.asarray(idx, dtype=np.int64)
        if key in ("g", "b"):
            _, gr, br = wrng.gdn_rows(seed, idx, C, H)
            return (gr if key == "g" else br).double().numpy()
        part = {"q": (0, H * d), "k": (H * d, 2 * H * d), "v": (2 * H * d, C)}[key]
        return yc[idx, part[0]:part[1]].double().numpy().reshape(len(idx), H, d)
    ro = og.delta_rule_rows(ref, rows, raw)
    ti = torch.tensor(ref["token_index"][raw], device="cuda")
    assert_close(f64(o[ti]), ro, "%s gdn delta rule samples" % name)
    # the convolution at the same rows, from the regenerated inputs
    path_rows = []
    for r in raw:
        s = int(np.searchsorted(off, r, side="right") - 1)
        path_rows.append(ref["token_index"][max(off[s], r - W + 1):r + 1])
    for r, pr in zip(raw, path_rows):
        xr, _, _ = wrng.gdn_rows(seed, pr, C, H)
        xs = xr.double().numpy()
        acc = sum(wcpu[:, W - len(pr) + i] * xs[i] for i in range(len(pr)))
        want = acc / (1 + np.exp(-acc))
        got = f64(y[int(ref["token_index"][r])])
        assert np.all(np.abs(got - want) <= 2.0 ** -7 * np.abs(want) + 1e-5)


# ---------------------------------------------------------------- backward
BWD_CASES = [("tiny_fit", 2, 64), ("ragged_d128_h1", 3, 128), ("ragged_d64_gqa2", 2, 64), ("ragged_d64_h1", 1, 64)]


def test_gdn_segment_arrays_on_device(ops):
    """The plan image's level table (start, length, parent, level-local
    offset) equals the oracle's, on a tree with six levels."""
    w = SMALL["deep_small"]()
    plan, dp, ref = _plans(ops, w)
    for name in ("seg_start", "seg_len", "seg_parent", "seg_off"):
        assert np.array_equal(getattr(dp, name).cpu().numpy(), ref[name]), name


def _bwd_layer(ops, dp, y, gg, bg, H, d, dO, state=None):
    """Delta rule forward and backward on views of the convolution output;
    the gradients land as column slices of one [F, C] dy."""
    q, k, v = _split(y, H, d, d)
    ws = ops.gdn_workspace(dp, H, d, d) if state is None else state
    o = ops.gdn_delta_rule(dp, q, k, v, gg, bg, workspace=ws)
    dy = torch.empty_like(y)
    dq, dk, dv = _split(dy, H, d, d)
    _, _, _, dg, db = ops.gdn_delta_rule_bwd(dp, q, k, v, gg, bg, dO, ws, dq=dq, dk=dk, dv=dv)
    return o, dy, dg, db


@pytest.mark.parametrize("name,H,d", BWD_CASES)
def test_gdn_bwd_full_parity(ops, name, H, d):
    """Gradients of the delta rule (dq, dk, dv, dg, dbeta) and of the
    convolution (dx, dw) against the oracle's fp64 autograd over the unpacked
    sequences, on the same (bf16) inputs; the delta rule's gradients are
    written as column slices of one dy, which feeds the convolution's
    backward."""
    w = SMALL[name]()
    plan, dp, ref = _plans(ops, w)
    F = plan.info["n_fwd"]
    C = H * 3 * d
    x, wc, g, b = wrng.gdn_inputs(w.seed_base + 60, F, C, H, W, "cuda")
    dO = wrng.normal_bf16(w.seed_base + 61, (F, H, d), "cuda")
    y = ops.gdn_conv(dp, x, wc)
    o, dy, dg, db = _bwd_layer(ops, dp, y, g, b, H, d, dO)
    torch.cuda.synchronize()
    qn, kn, vn = (f64(t) for t in _split(y, H, d, d))
    grads = og.delta_rule_bwd(ref, qn, kn, vn, f64(g), f64(b), f64(dO))
    dq, dk, dv = _split(dy, H, d, d)
    for got, want, n in zip((dq, dk, dv, dg, db), grads, ("dq", "dk", "dv", "dg", "dbeta")):
        assert_close(f64(got), want, "%s gdn bwd %s" % (name, n))
    dx, dw = ops.gdn_conv_bwd(dp, x, wc, dy)
    torch.cuda.synchronize()
    rdx, rdw = og.conv_bwd(ref, f64(x), f64(wc), f64(dy))
    assert_close(f64(dx), rdx, "%s gdn conv bwd dx" % name)
    assert_close(f64(dw), rdw, "%s gdn conv bwd dw" % name)


def test_gdn_bwd_strong_decay_and_repeat(ops):
    """Decay strong enough that walking the state backwards would lose it
    (log decay -60 on one token in five, -3 on others): those steps are
    replayed from a checkpoint; the gradients still match the oracle, and a
    second call gives identical bits."""
    w = SMALL["ragged_d64_h1"]()
    plan, dp, ref = _plans(ops, w)
    F, H, d = plan.info["n_fwd"], 2, 64
    x, wc, g, b = wrng.gdn_inputs(w.seed_base + 70, F, H * 3 * d, H, W, "cuda")
    sel = torch.arange(F, device="cuda") % 5 == 0
    g = torch.where(sel[:, None], torch.full_like(g, -60.0), g - 3.0 * (torch.arange(F, device="cuda") % 7 == 1)[:, None])
    dO = wrng.normal_bf16(w.seed_base + 71, (F, H, d), "cuda")
    y = ops.gdn_conv(dp, x, wc)
    o, dy, dg, db = _bwd_layer(ops, dp, y, g, b, H, d, dO)
    o2, dy2, dg2, db2 = _bwd_layer(ops, dp, y, g, b, H, d, dO)
    torch.cuda.synchronize()
    assert torch.equal(dy, dy2) and torch.equal(dg, dg2) and torch.equal(db, db2)
    qn, kn, vn = (f64(t) for t in _split(y, H, d, d))
    grads = og.delta_rule_bwd(ref, qn, kn, vn, f64(g), f64(b), f64(dO))
    dq, dk, dv = _split(dy, H, d, d)
    for got, want, n in zip((dq, dk, dv, dg, db), grads, ("dq", "dk", "dv", "dg", "dbeta")):
        assert_close(f64(got), want, "strong decay gdn bwd %s" % n)


def _sparse_bwd(ops, name, H, d, n_picks, max_prefix, seed, last=False):
    """The full batch's backward on the GPU with an output gradient that is
    zero except at a few raw tokens' positions (each at most ``max_prefix``
    tokens into its sequence, or with ``last`` each sequence's final token);
    the oracle differentiates those outputs over their own prefixes.  Every
    other row's gradient must be exactly zero."""
    w = workloads.get(name) if name in ("grpo", "agentic") else SMALL[name]()
    plan, dp, ref = _plans(ops, w)
    F = plan.info["n_fwd"]
    C = H * 3 * d
    x, wc, g, b = wrng.gdn_inputs(seed, F, C, H, W, "cuda")
    y = ops.gdn_conv(dp, x, wc)
    rng = np.random.Generator(np.random.PCG64(seed))
    off, ti = ref["seq_offsets"], ref["token_index"]
    picks, seen = [], set()
    while len(picks) < n_picks:
        s = int(rng.integers(0, len(off) - 1))
        r = int(off[s + 1] - 1) if last else int(off[s] + rng.integers(0, min(max_prefix, off[s + 1] - off[s])))
        if int(ti[r]) in seen:
            continue
        seen.add(int(ti[r]))
        picks.append((r, rng.standard_normal((H, d)).astype(np.float32)))
    dO = torch.zeros((F, H, d), dtype=torch.bfloat16, device="cuda")
    for r, dd in picks:
        dO[int(ti[r])] = torch.from_numpy(dd).to("cuda", torch.bfloat16)
    o, dy, dg, db = _bwd_layer(ops, dp, y, g, b, H, d, dO)
    torch.cuda.synchronize()
    yc = y.cpu()
    gc, bc = g.cpu().double().numpy(), b.cpu().double().numpy()

    def rows(key, idx):
        if key == "g":
            return gc[idx]
        if key == "b":
            return bc[idx]
        part = {"q": (0, H * d), "k": (H * d, 2 * H * d), "v": (2 * H * d, C)}[key]
        return yc[idx, part[0]:part[1]].double().numpy().reshape(len(idx), H, d)
    picks64 = [(r, np.asarray(f64(dO[int(ti[r])]))) for r, _ in picks]
    pos, want = og.delta_rule_bwd_rows(ref, rows, picks64)
    dq, dk, dv = _split(dy, H, d, d)
    pt = torch.as_tensor(pos, device="cuda")
    for got, wnt, n in zip((dq, dk, dv, dg, db), want, ("dq", "dk", "dv", "dg", "dbeta")):
        assert_close(f64(got[pt]), wnt, "%s gdn bwd %s (sampled)" % (name, n))
        rest = torch.ones(F, dtype=torch.bool, device="cuda")
        rest[pt] = False
        assert not bool(got[rest].any()), "%s: nonzero gradient off the picked paths" % n
    return plan, dp, ref, x, wc, picks


def test_gdn_bwd_deep_small_sampled(ops):
    """Six levels of forks: the final tokens of three sequences, so each
    picked output's gradient crosses several instance boundaries, handed
    from child to parent."""
    plan, _, ref, _, _, picks = _sparse_bwd(ops, "deep_small", 2, 128, 3, 0, 77, last=True)
    starts, lens, ti = ref["seg_start"], ref["seg_len"], ref["token_index"]

    def level_of(pos):
        i = int(np.nonzero((starts <= pos) & (pos < starts + lens))[0][0])
        return int(np.searchsorted(ref["seg_level_begin"], i, side="right") - 1)
    assert min(level_of(int(ti[r])) for r, _ in picks) >= 2


def test_gdn_bwd_full_size_sampled(ops):
    """The GRPO batch at the bench's shape (16 heads, d = 128), full
    backward launch; two picked outputs checked over their prefixes."""
    _sparse_bwd(ops, "grpo", 16, 128, 2, 1200, 78)


def test_gdn_conv_bwd_full_size_sampled(ops):
    """The convolution's backward on the GRPO batch with dy nonzero at a few
    positions: dx at their windows and dw against the oracle."""
    w = workloads.get("grpo")
    plan, dp, ref = _plans(ops, w)
    F, H, d = plan.info["n_fwd"], 16, 128
    C = H * 3 * d
    x, wc, _, _ = wrng.gdn_inputs(w.seed_base + 80, F, C, H, W, "cuda")
    rng = np.random.Generator(np.random.PCG64(80))
    ti = ref["token_index"]
    raw = sorted({int(r) for r in rng.integers(0, plan.info["n_raw"], size=4)})
    raw = [r for i, r in enumerate(raw) if int(ti[r]) not in {int(ti[q]) for q in raw[:i]}]
    dy = torch.zeros((F, C), dtype=torch.bfloat16, device="cuda")
    picks = []
    for r in raw:
        dd = wrng.normal_bf16(w.seed_base + 81 + r, (C,))
        dy[int(ti[r])] = dd.to("cuda")
        picks.append((r, dd.double().numpy()))
    dx, dw = ops.gdn_conv_bwd(dp, x, wc, dy)
    torch.cuda.synchronize()
    xc = x.cpu()
    pos, rdx, rdw = og.conv_bwd_rows(ref, lambda idx: xc[idx].double().numpy(), f64(wc), picks)
    pt = torch.as_tensor(pos, device="cuda")
    assert_close(f64(dx[pt]), rdx, "grpo gdn conv bwd dx (sampled)")
    assert_close(f64(dw), rdw, "grpo gdn conv bwd dw (sampled)")
    rest = torch.ones(F, dtype=torch.bool, device="cuda")
    rest[pt] = False
    assert not bool(dx[rest].any())


@pytest.mark.parametrize("width", [1, 2, 3, 5, 8])
def test_gdn_conv_widths(ops, width):
    """Every compiled window width other than 4: the convolution and its
    backward against the oracle on a ragged tree with forks (a fork within
    W - 1 steps below a position sends its dx through the general walk)."""
    w = SMALL["ragged_d64_gqa2"]()
    plan, dp, ref = _plans(ops, w)
    F, C = plan.info["n_fwd"], 3 * 2 * 64
    x, wc, _, _ = wrng.gdn_inputs(w.seed_base + 90 + width, F, C, 2, width, "cuda")
    dy = wrng.normal_bf16(w.seed_base + 95 + width, (F, C), "cuda")
    y = ops.gdn_conv(dp, x, wc)
    dx, dw = ops.gdn_conv_bwd(dp, x, wc, dy)
    torch.cuda.synchronize()
    yr = og.conv(ref, f64(x), f64(wc))
    err = np.abs(f64(y) - yr)
    record("W=%d gdn conv" % width, max_abs=float(err.max()))
    assert np.all(err <= 2.0 ** -7 * np.abs(yr) + 1e-5)
    rdx, rdw = og.conv_bwd(ref, f64(x), f64(wc), f64(dy))
    assert_close(f64(dx), rdx, "W=%d gdn conv bwd dx" % width)
    assert_close(f64(dw), rdw, "W=%d gdn conv bwd dw" % width)


def _edge_tree():
    """Sequences over one 80-token base, cut at 1, 2, 16, 31, 32, 33, 47 and
    64 tokens (segment boundaries on either side of the kernels' 16-token
    rounds and 32-token checkpoints), then tails of 1 to 40 tokens; four
    sequences share the 32-token cut (a position with four children), and
    two are one token long."""
    rng = np.random.Generator(np.random.PCG64(4321))
    base = rng.integers(0, 50, size=80)
    seqs = [base[:1].copy(), base[:1].copy()]
    for cut, tail in [(2, 1), (16, 5), (31, 33), (32, 1), (32, 16), (32, 40), (32, 2), (33, 31), (47, 17), (64, 3),
                      (80, 0)]:
        t = rng.integers(50, 100, size=tail)
        seqs.append(np.concatenate([base[:cut], t]).astype(np.int32))
    return [np.asarray(s, dtype=np.int32) for s in seqs]


def test_gdn_edge_segments(ops):
    """Forward and backward on the crafted tree (minimum shared run 1), with
    a width-4 convolution: every boundary case of the level schedule and of
    the backward's rounds and checkpoints against the oracle."""
    seqs = _edge_tree()
    plan = ops.Plan.from_sequences(seqs, row_capacity=4096, min_shared=1)
    dp = plan.to_device()
    ref = op.plan(seqs, min_shared=1, row_capacity=4096)
    assert plan.info["n_fwd"] == ref["n_fwd"]
    F, H, d = plan.info["n_fwd"], 2, 64
    lens = np.asarray(ref["seg_len"])
    assert lens.min() == 1 and plan.info["n_seg_levels"] >= 3
    x, wc, g, b = wrng.gdn_inputs(777, F, 3 * H * d, H, W, "cuda")
    dO = wrng.normal_bf16(778, (F, H, d), "cuda")
    y = ops.gdn_conv(dp, x, wc)
    o, dy, dg, db = _bwd_layer(ops, dp, y, g, b, H, d, dO)
    dx, dw = ops.gdn_conv_bwd(dp, x, wc, dy)
    torch.cuda.synchronize()
    qn, kn, vn = (f64(t) for t in _split(y, H, d, d))
    assert_close(f64(o), og.delta_rule(ref, qn, kn, vn, f64(g), f64(b)), "edge gdn delta rule")
    grads = og.delta_rule_bwd(ref, qn, kn, vn, f64(g), f64(b), f64(dO))
    dq, dk, dv = _split(dy, H, d, d)
    for got, want, n in zip((dq, dk, dv, dg, db), grads, ("dq", "dk", "dv", "dg", "dbeta")):
        assert_close(f64(got), want, "edge gdn bwd %s" % n)
    rdx, rdw = og.conv_bwd(ref, f64(x), f64(wc), f64(dy))
    assert_close(f64(dx), rdx, "edge gdn conv bwd dx")
    assert_close(f64(dw), rdw, "edge gdn conv bwd dw")
