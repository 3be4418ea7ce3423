"""Parity of the raw-order <-> packed-layout kernels with the oracle.

tpk_gather_to_forwarded (materialisation by owner) must match the oracle bit
for bit for any row width; tpk_sum_to_forwarded (transpose of the raw-order
scatter) sums in fp32 over a position's raw tokens in ascending order and
rounds to bf16 once, so it must match the oracle's fp64 sum rounded to bf16
within one bf16 unit (the fp32 sum can sit on the other side of a rounding
boundary), and exactly where a position has a single raw token.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import layout as ol
from oracle import planner as op
from oracle.bf16 import round_to_bf16
from workloads import rng as wrng

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    assert torch.cuda.is_available()
    from prefix_tree_packed_dfs_gb300 import ops as o
    return o


def _plans(ops, name):
    w = workloads.get(name)
    ref = op.plan(w.sequences, group_ids=w.group_ids, min_shared=w.min_shared, row_capacity=w.row_capacity)
    plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                   min_shared=w.min_shared)
    return w, ref, plan.to_device()


def _f64(t):
    return t.float().double().cpu().numpy() if t.dtype == torch.bfloat16 else t.double().cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "grpo", "deep_small", "sweep_1.00"])
def test_gather_to_forwarded_bit_exact(ops, name):
    w, ref, dp = _plans(ops, name)
    R = ref["n_raw"]
    g = torch.Generator().manual_seed(5)
    tokens = torch.from_numpy(np.concatenate(w.sequences).astype(np.int32))
    payloads = [
        tokens,                                                            # 4-byte rows
        torch.randn(R, 3, generator=g),                                    # 12-byte rows
        torch.randint(0, 256, (R, 5), generator=g, dtype=torch.uint8),     # 5-byte rows
        torch.randn(R, 2, 64, generator=g).to(torch.bfloat16),             # 256-byte rows (16-byte path)
    ]
    for x in payloads:
        got = ops.gather_to_forwarded(dp, x.cuda())
        exp = ol.gather_to_forwarded(ref, x.numpy() if x.dtype != torch.bfloat16 else x.view(torch.int16).numpy())
        got_np = got.cpu().numpy() if x.dtype != torch.bfloat16 else got.cpu().view(torch.int16).numpy()
        assert np.array_equal(got_np, exp), (name, x.dtype, tuple(x.shape))
    # token ids land as the planner's forwarded tokens
    assert np.array_equal(ops.gather_to_forwarded(dp, tokens.cuda()).cpu().numpy(), np.asarray(ref["fwd_token"]))


def _check_sum(got, src64, ref, rows=None):
    """got: bf16 [n, ...] sums for forwarded ``rows`` (all if None)."""
    exp = ol.sum_to_forwarded(ref, src64)
    if rows is not None:
        exp = exp[rows]
    g = _f64(got)
    ulp = np.abs(round_to_bf16(exp)) * 2.0 ** -8
    assert np.all(np.abs(g - round_to_bf16(exp)) <= ulp + 1e-30)
    return exp


@pytest.mark.parametrize("name", ["tiny", "grpo", "deep_small", "sweep_1.00"])
def test_sum_to_forwarded_matches_oracle(ops, name):
    w, ref, dp = _plans(ops, name)
    R, F = ref["n_raw"], ref["n_fwd"]
    H, d = (2, 64) if name == "tiny" else (4, 128)
    x = wrng.normal_bf16(91, (R, H, d), "cpu")
    lse = torch.randn(H, R, generator=torch.Generator().manual_seed(6)) * 4
    got, got_lse = ops.sum_to_forwarded(dp, x.cuda(), lse.cuda())
    _check_sum(got, _f64(x), ref)
    # a position with one raw token is a plain copy, bit for bit
    counts = np.bincount(np.asarray(ref["token_index"]), minlength=F)
    single = np.flatnonzero(counts == 1)
    src_rows = np.asarray(ref["fwd_src"])[single]
    assert torch.equal(got.cpu()[torch.from_numpy(single)], x[torch.from_numpy(src_rows)])
    # fp32 sums: within fp32 rounding of the sum of magnitudes
    exp_lse = ol.sum_to_forwarded(ref, lse.double().numpy().T).T
    mag = ol.sum_to_forwarded(ref, np.abs(lse.double().numpy().T)).T
    assert np.all(np.abs(got_lse.double().cpu().numpy() - exp_lse) <= 2.0 ** -22 * mag * counts.max() + 1e-30)
    if name == "grpo":
        # the system prompt is laid out once per row and shared by every
        # sequence placed in that row (about ten of the 64)
        assert counts.max() >= 8
    if name == "sweep_1.00":
        assert counts.max() == 1     # no sharing: the sum is a permutation


@pytest.mark.parametrize("name", ["deep", "agentic"])
def test_layout_kernels_full_size_sampled(ops, name):
    w, ref, dp = _plans(ops, name)
    R, F = ref["n_raw"], ref["n_fwd"]
    H, d = w.n_heads_q, w.head_dim
    x = wrng.normal_bf16(93, (R, H, d), "cuda")
    got, _ = ops.sum_to_forwarded(dp, x)
    rng = np.random.Generator(np.random.PCG64(8))
    counts = np.bincount(np.asarray(ref["token_index"]), minlength=F)
    rows = np.unique(np.concatenate([rng.integers(0, F, 24), np.argsort(counts)[-8:], [0, F - 1]]))
    # the oracle sum restricted to the sampled positions
    ti = np.asarray(ref["token_index"])
    sel = np.isin(ti, rows)
    sub = {"n_fwd": F, "token_index": ti[sel]}
    xs = _f64(x[torch.from_numpy(np.flatnonzero(sel)).cuda()])
    _check_sum(got[torch.from_numpy(rows).cuda()], xs, sub, rows)
    # gather by owner at full size: every sampled position holds its owner's row
    gat = ops.gather_to_forwarded(dp, x)
    own = np.asarray(ref["fwd_src"])[rows]
    assert torch.equal(gat[torch.from_numpy(rows).cuda()], x[torch.from_numpy(own).cuda()])
