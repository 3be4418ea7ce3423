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
