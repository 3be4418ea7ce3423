"""Pins of the oracle against what the pages and the mathematics fix.

Every oracle function is checked against something other than itself: values
the pages print (tests/golden/*.json), library routines (torch SDPA and
autograd in fp64, torch's float32->bf16 conversion, NumPy complex arithmetic),
closed forms, invariants and brute force on tiny inputs.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import planner as op
from oracle.bf16 import round_to_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- planner pins
def test_docs_example_ten_raw_eight_forwarded():
    g = golden("docs_example.json")
    p = op.plan(g["sequences"], min_shared=g["min_shared"], row_capacity=g["row_capacity"])
    assert p["n_raw"] == g["expected"]["n_raw"]
    assert p["n_fwd"] == g["expected"]["n_fwd"]
    # the duplicated join token is what makes it 8 and not 7: untrained
    # prompt positions (no target in the key) merge the last prompt token
    flags = [[0, 0, 0, 1, 1], [0, 0, 0, 1, 1]]
    p7 = op.plan(g["sequences"], trained=flags, min_shared=1, row_capacity=16)
    assert p7["n_fwd"] == g["expected"]["n_fwd_without_join_duplication"]


def _art_example():
    g = golden("art_32_rollouts.json")["construction"]
    rng = np.random.Generator(np.random.PCG64(7))
    used = set()

    def fresh(n):
        t = rng.integers(0, 32000, size=n)
        while int(t[0]) in used:
            t[0] = rng.integers(0, 32000)
        used.add(int(t[0]))
        return t
    root = rng.integers(0, 32000, size=g["root_tokens"])
    seqs, flags, groups, labels = [], [], [], []
    for gi, (label, comp_len) in enumerate(g["groups_in_arrival_order"]):
        prefix = fresh(g["group_prefix_tokens"])
        for _ in range(g["rollouts_per_group"]):
            comp = fresh(comp_len)
            s = np.concatenate([root, prefix, comp])
            f = np.zeros(len(s), dtype=np.int64)
            n_prompt = len(root) + len(prefix)
            f[n_prompt - 1:] = 1
            seqs.append(s)
            flags.append(f)
            groups.append(gi)
            labels.append(label)
    return g, seqs, flags, np.asarray(groups), labels


def _row_contents(p, labels):
    rows = []
    for r in range(p["n_rows"]):
        c = {}
        for s in np.flatnonzero(p["row_of_seq"] == r):
            c[labels[s]] = c.get(labels[s], 0) + 1
        rows.append(c)
    return rows


def test_art_example_best_fit_decreasing_rows():
    g, seqs, flags, groups, labels = _art_example()
    exp = golden("art_32_rollouts.json")["expected"]
    p = op.plan(seqs, trained=flags, group_ids=groups, min_shared=g["min_shared"],
                row_capacity=g["row_capacity"], placement="bfd")
    assert p["row_loads"] == exp["best_fit_decreasing_row_loads"]
    assert _row_contents(p, labels) == exp["best_fit_decreasing_rows"]
    assert p["n_rows"] * g["row_capacity"] == exp["allocated_tokens_bfd"]
    assert list(np.diff(p["row_offsets"])) == exp["best_fit_decreasing_row_loads"]


def test_art_example_in_order_rows():
    g, seqs, flags, groups, labels = _art_example()
    exp = golden("art_32_rollouts.json")["expected"]
    p = op.plan(seqs, trained=flags, group_ids=groups, min_shared=g["min_shared"],
                row_capacity=g["row_capacity"], placement="next_fit")
    assert p["row_loads"] == exp["in_order_row_loads"]
    assert _row_contents(p, labels) == exp["in_order_rows"]
    assert p["n_rows"] * g["row_capacity"] == exp["allocated_tokens_in_order"]


def test_art_example_accounting():
    # 4,096 root + 11,999 shared group prefix + (completion + 1) per rollout
    g, seqs, flags, groups, labels = _art_example()
    p = op.plan(seqs, trained=flags, group_ids=groups, min_shared=64, row_capacity=10**7)
    lens = [2000, 2000, 12000, 7000]
    assert p["n_fwd"] == 4096 + sum(11999 + 8 * (c + 1) for c in lens)


def test_mask_figure():
    g = golden("mask_figure.json")
    p = op.plan(g["sequences"], trained=g["trained"], min_shared=1, row_capacity=64)
    assert p["n_fwd"] == g["expected"]["n_fwd"]
    assert op.visible_by_parent_walk(p["parent"], 7) == g["expected"]["visible_to_query_7"]
    assert op.visible_by_parent_walk(p["parent"], 4) == g["expected"]["visible_to_query_4"]
    # the interval form of the same mask: j visible to i iff j <= i < subtree_end[j]
    se = p["subtree_end"]
    for i in range(9):
        vis = [j for j in range(9) if j <= i < se[j]]
        assert vis == op.visible_by_parent_walk(p["parent"], i)


def test_toy_ratio():
    g = golden("toy_ratio.json")["expected"]
    rng = np.random.Generator(np.random.PCG64(11))
    hist = rng.integers(0, 32000, size=20000)
    comps = []
    used = set()
    for _ in range(8):
        c = rng.integers(0, 32000, size=2000)
        while int(c[0]) in used:
            c[0] = rng.integers(0, 32000)
        used.add(int(c[0]))
        comps.append(c)
    seqs = [np.concatenate([hist, c]) for c in comps]
    p = op.plan(seqs, min_shared=64, row_capacity=10**6)
    assert p["n_raw"] == g["n_raw"]
    assert p["n_fwd"] == g["n_fwd_all_trained"]
    assert round(p["packing_ratio"], 1) == g["ratio_printed_1dp"]
    flags = [np.concatenate([np.zeros(20000, np.int64), np.ones(2000, np.int64)]) for _ in seqs]
    p2 = op.plan(seqs, trained=flags, min_shared=64, row_capacity=10**6)
    assert p2["n_fwd"] == g["n_fwd_printed"]


def _textbook_bfd(sizes, cap):
    """Classical best-fit decreasing on fixed sizes (independent restatement)."""
    loads, assign = [], {}
    for i in sorted(range(len(sizes)), key=lambda i: -sizes[i]):
        fits = [b for b in range(len(loads)) if loads[b] + sizes[i] <= cap]
        if fits:
            b = min(fits, key=lambda b: (cap - loads[b] - sizes[i], b))
        else:
            loads.append(0)
            b = len(loads) - 1
        loads[b] += sizes[i]
        assign[i] = b
    return loads, assign


@pytest.mark.parametrize("seed", range(6))
def test_private_segments_reduce_to_classical_bfd(seed):
    # appendix "Still NP-hard": with every segment private, the marginal cost is
    # the plain item size and the placement is ordinary best-fit decreasing
    rng = np.random.Generator(np.random.PCG64(100 + seed))
    n = 40
    sizes = [int(x) for x in rng.integers(5, 60, size=n)]
    firsts = rng.permutation(32000)[:n]
    seqs = [np.concatenate([[firsts[i]], rng.integers(0, 32000, size=sizes[i] - 1)]) for i in range(n)]
    cap = 100
    p = op.plan(seqs, group_ids=np.arange(n), min_shared=1, row_capacity=cap)
    loads, assign = _textbook_bfd(sizes, cap)
    assert p["row_loads"] == loads
    assert [assign[i] for i in range(n)] == list(p["row_of_seq"])


def _distinct_keys(seqs, flags):
    """Brute force: the set of distinct position keys (p, symbols 0..p)."""
    keys = set()
    for s, f in zip(seqs, flags):
        L = len(s)
        for p in range(L):
            prefix = tuple((int(s[i]), int(f[i])) for i in range(p + 1))
            if f[p] or p == L - 1:
                tgt = int(s[p + 1]) if p + 1 < L else -1
            else:
                tgt = None
            keys.add((prefix, tgt))
    return keys


@pytest.mark.parametrize("seed", range(30))
def test_minimality_against_brute_force(seed):
    rng = np.random.Generator(np.random.PCG64(200 + seed))
    n = int(rng.integers(1, 7))
    seqs = [rng.integers(0, 3, size=int(rng.integers(1, 9))) for _ in range(n)]
    flags = [rng.integers(0, 2, size=len(s)) for s in seqs] if seed % 2 else [np.ones(len(s), np.int64) for s in seqs]
    p = op.plan(seqs, trained=flags, min_shared=1, row_capacity=10**6)
    assert p["n_fwd"] == len(_distinct_keys(seqs, flags))
    _check_layout_invariants(p, seqs)


def _check_layout_invariants(p, seqs):
    ti, depth, parent, tok = p["token_index"], p["depth"], p["parent"], p["fwd_token"]
    off = p["seq_offsets"]
    for s, seq in enumerate(seqs):
        path = ti[off[s]:off[s + 1]]
        assert list(tok[path]) == list(seq)                 # tokens survive the layout
        assert list(depth[path]) == list(range(len(seq)))   # positions = depth
        assert parent[path[0]] == -1
        assert list(parent[path[1:]]) == list(path[:-1])    # the path is a parent chain
        row = p["row_of_seq"][s]
        lo, hi = p["row_offsets"][row], p["row_offsets"][row + 1]
        assert np.all((path >= lo) & (path < hi))
    # depth-first: a parent precedes its children; subtrees are contiguous
    F = len(depth)
    for f in range(F):
        if parent[f] >= 0:
            assert parent[f] < f and depth[f] == depth[parent[f]] + 1
    se = p["subtree_end"]
    for f in range(F):
        inside = [g for g in range(F) if f in op.visible_by_parent_walk(parent, g)]
        assert inside == list(range(f, se[f]))
    assert np.all(ti[p["fwd_src"]] == np.arange(F))


@pytest.mark.parametrize("seed", range(10))
def test_min_shared_dissolves_short_runs(seed):
    rng = np.random.Generator(np.random.PCG64(300 + seed))
    n = int(rng.integers(2, 7))
    base = rng.integers(0, 4, size=12)
    seqs = []
    for _ in range(n):
        cut = int(rng.integers(0, 12))
        seqs.append(np.concatenate([base[:cut], rng.integers(0, 4, size=int(rng.integers(1, 6)))]))
    for m in (1, 2, 3, 5, 100):
        p = op.plan(seqs, min_shared=m, row_capacity=10**6)
        _check_layout_invariants(p, seqs)
        for seg in p["segments"]:
            if not seg.is_leaf:
                assert seg.end - seg.start >= m
        if m == 100:   # nothing shared: forwarded == raw, rows = concatenated sequences
            assert p["n_fwd"] == p["n_raw"] - _dup_raw(seqs)


# Hand-counted forwarded totals for the minimum shared-segment length
# ("Prefix Tree Packing in ART", section "The tree": a shared run shorter than
# the minimum is not shared; the walk splits there and recurses from the same
# start, so the children's runs include the positions above them).  Every
# position is trained, so position p of a sequence is shared with another
# sequence iff their tokens 0..p+1 agree (the target is part of the key).
#
#   P = [1, 2, 3]; X = [10..19]; Y = [20..29]   (10 tokens each)
#   s0 = P + X + [100, 101]     s1 = P + X + [200, 201]
#   s2 = P + Y + [300, 301]     s3 = P + Y + [400, 401]    (R = 4 * 15 = 60)
#
# All four agree on tokens 0..2 and split at token 3 (X[0] vs Y[0]), so the
# run shared by all four is positions 0, 1 (position 2's key holds token 3):
# length 2.  s0, s1 agree on tokens 0..12 and split at token 13, so they share
# positions 2..11 (10 positions); likewise s2, s3.  Each sequence keeps
# positions 12..14 (3) to itself: the join token X[9] / Y[9] at position 12
# appears once per branch.
#   m <= 2:  root 2 + two runs of 10 + 4 leaves of 3            F = 34
#   m = 3:   the root run (2 < 3) is copied into both children, whose runs
#            become positions 0..11 (12 >= 3, kept):  12 + 12 + 4 * 3 = 36
#   m = 11, 12: the children's runs count their carried positions: 12 >= m,
#            kept (counting only their own 10 positions would dissolve them
#            at m = 11 and give 60)                               F = 36
#   m = 13:  12 < 13, dissolved as well: nothing is shared        F = 60
MIN_SHARED_CASE = {1: 34, 2: 34, 3: 36, 11: 36, 12: 36, 13: 60}


def _min_shared_case():
    P, X, Y = [1, 2, 3], list(range(10, 20)), list(range(20, 30))
    return [np.array(P + X + [100, 101]), np.array(P + X + [200, 201]),
            np.array(P + Y + [300, 301]), np.array(P + Y + [400, 401])]


@pytest.mark.parametrize("m", sorted(MIN_SHARED_CASE))
def test_min_shared_carry_down_hand_counted(m):
    seqs = _min_shared_case()
    p = op.plan(seqs, min_shared=m, row_capacity=1000)
    assert p["n_raw"] == 60
    assert p["n_fwd"] == MIN_SHARED_CASE[m]
    _check_layout_invariants(p, seqs)
    # the shared segments' lengths, as counted above
    shared = sorted(seg.end - seg.start for seg in p["segments"] if not seg.is_leaf)
    want = {34: [2, 10, 10], 36: [12, 12], 60: []}[MIN_SHARED_CASE[m]]
    assert shared == want


def test_min_shared_tiny_workload_hand_counted():
    # the tiny workload: 4 sequences share 128 tokens; sequences 1 and 2 share
    # 64 more; tails of 64..128 own tokens.  Position 127's key holds token
    # 128, which is the first token of a tail for sequences 0, 3 and of the
    # 64-token run for 1, 2: all four share positions 0..126 (127), sequences
    # 1, 2 share 127..190 (64), and each sequence keeps its last
    # tail + 1 positions (the join token repeated per branch).  Both shared
    # runs are >= 16, so min_shared = 16 keeps them:
    #   F = 127 + 64 + sum(tail_i + 1) = 195 + sum(tails) = R - 445.
    import workloads
    w = workloads.get("tiny")
    L = [len(x) for x in w.sequences]
    tails = [L[0] - 128, L[1] - 192, L[2] - 192, L[3] - 128]
    assert all(64 <= t <= 128 for t in tails)
    p = op.plan(w.sequences, group_ids=w.group_ids, min_shared=16, row_capacity=10**6)
    assert p["n_fwd"] == 195 + sum(tails)
    assert p["n_raw"] - p["n_fwd"] == 3 * 127 + 64
    # min_shared = 65 drops the 64-token run (carried into the two tails)
    p65 = op.plan(w.sequences, group_ids=w.group_ids, min_shared=65, row_capacity=10**6)
    assert p65["n_fwd"] == 127 + sum(t + 1 for t in tails) + 2 * 64


def _dup_raw(seqs):
    seen, extra = set(), 0
    for s in seqs:
        key = tuple(int(x) for x in s)
        if key in seen:
            extra += len(s)
        seen.add(key)
    return extra


# -------------------------------------------------------------------- bf16 pin
def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.Generator(np.random.PCG64(1))
    x32 = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                          (rng.standard_normal(1000) * 1e-30).astype(np.float32)])
    ours = round_to_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_rounding_is_nearest_on_float64_values():
    rng = np.random.Generator(np.random.PCG64(2))
    x = rng.standard_normal(20000) * 3
    r = round_to_bf16(x)
    # brute force: neighbours on the bf16 grid of x's binade
    e = np.floor(np.log2(np.abs(x)))
    ulp = 2.0 ** (e - 7)
    lo = np.floor(x / ulp) * ulp
    hi = lo + ulp
    best = np.where(np.abs(x - lo) <= np.abs(hi - x), lo, hi)
    tie = np.isclose(np.abs(x - lo), np.abs(hi - x), rtol=0, atol=0)
    assert np.array_equal(r[~tie], best[~tie])


# -------------------------------------------------------------------- RoPE pins
def test_rope_matches_complex_rotation_and_inverts():
    rng = np.random.Generator(np.random.PCG64(3))
    L, H, d = 17, 3, 64
    x = rng.standard_normal((L, H, d))
    pos = rng.integers(0, 30000, size=L)
    y = oa.rope(x, pos, 1e6)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    ang = np.outer(pos, 1e6 ** (-np.arange(d // 2) * 2.0 / d))
    w = z * np.exp(1j * ang)[:, None, :]
    assert np.allclose(y[..., : d // 2], w.real, atol=1e-12)
    assert np.allclose(y[..., d // 2:], w.imag, atol=1e-12)
    assert np.allclose(oa.rope(y, pos, 1e6, inverse=True), x, atol=1e-12)


def test_rope_scores_depend_only_on_depth_difference():
    # "DAG packing", section "Positions": every parent->child edge has
    # relative distance 1 wherever it sits in the row
    rng = np.random.Generator(np.random.PCG64(4))
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    s = [float(np.sum(oa.rope(q, [p + 1], 1e4) * oa.rope(k, [p], 1e4))) for p in (0, 5, 777, 12345)]
    assert np.allclose(s, s[0], rtol=1e-9)


# ----------------------------------------------------------------- attention pins
def _sdpa(q, k, v):
    """fp64 causal attention by torch's library routine (GQA by head repeat)."""
    hq, hkv = q.shape[1], k.shape[1]
    rep = hq // hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(rep, 0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(rep, 0)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    return o.permute(1, 0, 2).numpy()


def test_causal_attention_matches_sdpa():
    rng = np.random.Generator(np.random.PCG64(5))
    L, hq, hkv, d = 70, 4, 2, 32
    q, k, v = rng.standard_normal((L, hq, d)), rng.standard_normal((L, hkv, d)), rng.standard_normal((L, hkv, d))
    o, lse = oa.causal_attention(q, k, v, 1 / np.sqrt(d), chunk=16)
    assert np.allclose(o, _sdpa(q, k, v), atol=1e-12)
    # closed form at position 0: a single visible key
    assert np.allclose(lse[:, 0], [q[0, h] @ k[0, h // 2] / np.sqrt(d) for h in range(hq)])


def test_lse_against_one_hot_values():
    # with V = identity rows, O[p] is the softmax row itself: O[p, j] = exp(s_pj - LSE_p)
    rng = np.random.Generator(np.random.PCG64(6))
    L, d = 24, 32
    q, k = rng.standard_normal((L, 1, d)), rng.standard_normal((L, 1, d))
    v = np.eye(L, d)[:, None, :]
    o, lse = oa.causal_attention(q, k, v, 0.3)
    s = (q[:, 0] @ k[:, 0].T) * 0.3
    for p in range(L):
        assert np.allclose(o[p, 0, : p + 1], np.exp(s[p, : p + 1] - lse[0, p]), atol=1e-13)
        assert lse[0, p] >= s[p, p]
        assert np.isclose(o[p, 0].sum(), 1.0)


def _tiny_tree(seed, hq=2, hkv=1, d=16):
    rng = np.random.Generator(np.random.PCG64(400 + seed))
    seqs = []
    base = rng.integers(0, 50, size=30)
    for _ in range(5):
        cut = int(rng.integers(3, 25))
        seqs.append(np.concatenate([base[:cut], rng.integers(0, 50, size=int(rng.integers(1, 12)))]))
    p = op.plan(seqs, min_shared=3, row_capacity=45)
    F = p["n_fwd"]
    Q = round_to_bf16(rng.standard_normal((F, hq, d)))
    K = round_to_bf16(rng.standard_normal((F, hkv, d)))
    V = round_to_bf16(rng.standard_normal((F, hkv, d)))
    return seqs, p, Q, K, V


@pytest.mark.parametrize("seed", range(5))
def test_packed_dense_mask_equals_unpacked(seed):
    # brute force on the packed layout: dense mask from parent walks, RoPE at depth
    seqs, p, Q, K, V = _tiny_tree(seed)
    F, hq, d = Q.shape
    base = 1e4
    o_fwd, lse_fwd, o_raw, _ = oa.forward(p, Q, K, V, base)
    qr = round_to_bf16(oa.rope(Q, p["depth"], base))
    kr = round_to_bf16(oa.rope(K, p["depth"], base))
    mask = np.full((F, F), -np.inf)
    for i in range(F):
        mask[i, op.visible_by_parent_walk(p["parent"], i)] = 0.0
    for h in range(hq):
        s = qr[:, h] @ kr[:, h // 2 if K.shape[1] > 1 else 0].T / np.sqrt(d) + mask
        m = s.max(1, keepdims=True)
        w = np.exp(s - m)
        ref = (w / w.sum(1, keepdims=True)) @ V[:, 0 if K.shape[1] == 1 else h // 2]
        assert np.allclose(o_fwd[:, h], ref, atol=1e-12)
        assert np.allclose(lse_fwd[h], (m + np.log(w.sum(1, keepdims=True)))[:, 0], atol=1e-12)
    assert np.allclose(o_raw, o_fwd[p["token_index"]], atol=0)


def test_no_sharing_is_block_diagonal_varlen_causal():
    # "DAG packing", intro: with nothing shared, the row is plain document
    # packing with a block-diagonal causal mask
    rng = np.random.Generator(np.random.PCG64(8))
    firsts = rng.permutation(1000)[:4]
    seqs = [np.concatenate([[firsts[i]], rng.integers(0, 1000, size=int(rng.integers(5, 40)))]) for i in range(4)]
    p = op.plan(seqs, min_shared=1000, row_capacity=1000)
    assert p["n_fwd"] == p["n_raw"] and p["n_rows"] == 1
    order = np.argsort([s[0] for s in seqs], kind="stable")  # layout order: by first token
    starts = np.cumsum([0] + [len(seqs[i]) for i in order])
    for j, s in enumerate(order):
        assert list(p["token_index"][p["seq_offsets"][s]:p["seq_offsets"][s + 1]]) == list(range(starts[j], starts[j + 1]))
    F, d = p["n_fwd"], 32
    Q = round_to_bf16(rng.standard_normal((F, 2, d)))
    K = round_to_bf16(rng.standard_normal((F, 2, d)))
    V = round_to_bf16(rng.standard_normal((F, 2, d)))
    o_fwd, _, _, _ = oa.forward(p, Q, K, V, 1e4)
    for j in range(4):
        lo, hi = starts[j], starts[j + 1]
        pos = np.arange(hi - lo)
        q = round_to_bf16(oa.rope(Q[lo:hi], pos, 1e4))
        k = round_to_bf16(oa.rope(K[lo:hi], pos, 1e4))
        assert np.allclose(o_fwd[lo:hi], _sdpa(q, k, V[lo:hi]), atol=1e-12)


def test_forward_rows_matches_full_forward():
    seqs, p, Q, K, V = _tiny_tree(1)
    _, _, o_raw, lse_raw = oa.forward(p, Q, K, V, 1e4)
    raw = [0, 5, p["n_raw"] // 2, p["n_raw"] - 1]
    o, lse = oa.forward_rows(p, lambda i: Q[i], lambda i: K[i], lambda i: V[i], raw, 1e4)
    assert np.allclose(o, o_raw[raw], atol=1e-12)
    assert np.allclose(lse, lse_raw[:, raw], atol=1e-12)


def test_causal_backward_matches_torch_autograd():
    rng = np.random.Generator(np.random.PCG64(9))
    L, hq, hkv, d = 33, 4, 2, 16
    q, k, v = rng.standard_normal((L, hq, d)), rng.standard_normal((L, hkv, d)), rng.standard_normal((L, hkv, d))
    do = rng.standard_normal((L, hq, d))
    o, _ = oa.causal_attention(q, k, v, 1 / np.sqrt(d))
    dq, dk, dv = oa.causal_attention_backward(q, k, v, o, do, 1 / np.sqrt(d))
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    qt = tq.permute(1, 0, 2)
    kt = tk.permute(1, 0, 2).repeat_interleave(2, 0)
    vt = tv.permute(1, 0, 2).repeat_interleave(2, 0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    (out * torch.from_numpy(do).permute(1, 0, 2)).sum().backward()
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_packed_backward_matches_finite_differences():
    seqs, p, Q, K, V = _tiny_tree(2, hq=2, hkv=1, d=8)
    rng = np.random.Generator(np.random.PCG64(10))
    dO = rng.standard_normal(Q.shape)
    base = 1e4
    dQ, dK, dV = oa.backward(p, Q, K, V, dO, base, round_rotated=False)

    def loss(Qx, Kx, Vx):
        o_fwd, _, _, _ = oa.forward(p, Qx, Kx, Vx, base, round_rotated=False)
        return float(np.sum(o_fwd * dO))
    eps = 1e-6
    F = Q.shape[0]
    for f in sorted({0, 1, F // 3, F // 2, F - 1}):
        for (T, G) in ((Q, dQ), (K, dK), (V, dV)):
            for h in range(T.shape[1]):
                for i in (0, 3, T.shape[2] - 1):
                    Tp, Tm = T.copy(), T.copy()
                    Tp[f, h, i] += eps
                    Tm[f, h, i] -= eps
                    args_p = [Tp if X is T else X for X in (Q, K, V)]
                    args_m = [Tm if X is T else X for X in (Q, K, V)]
                    fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                    assert abs(fd - G[f, h, i]) < 1e-6 * max(1.0, abs(fd)), (f, h, i)


def test_backward_rows_match_full_backward():
    seqs, p, Q, K, V = _tiny_tree(3, hq=2, hkv=1, d=8)
    rng = np.random.Generator(np.random.PCG64(12))
    dO = rng.standard_normal(Q.shape)
    dQ, dK, dV = oa.backward(p, Q, K, V, dO, 1e4)
    rows = lambda X: (lambda i: X[i])
    raw = [0, 3, p["n_raw"] // 2, p["n_raw"] - 1]
    dq = oa.backward_rows_q(p, rows(Q), rows(K), rows(V), rows(dO), raw, 1e4)
    assert np.allclose(dq, dQ[p["token_index"][raw]], atol=1e-12)
    fw = [0, 1, p["n_fwd"] // 2, p["n_fwd"] - 1]
    dk, dv = oa.backward_rows_kv(p, rows(Q), rows(K), rows(V), rows(dO), fw, 1e4)
    assert np.allclose(dk, dK[fw], atol=1e-12)
    assert np.allclose(dv, dV[fw], atol=1e-12)
    # the batched per-key form (queries of one sequence as one product, in
    # chunks smaller than a sequence) gives the same gradients at every key
    every = list(range(p["n_fwd"]))
    dk, dv = oa.backward_keys(p, rows(Q), rows(K), rows(V), rows(dO), every, 1e4, chunk=3)
    assert np.allclose(dk, dK, atol=1e-12)
    assert np.allclose(dv, dV, atol=1e-12)


def test_backward_dv_sums_to_do_per_kv_head():
    # every softmax row sums to one, so over all keys dV adds up to dO summed
    # over all queries and the query heads that share the KV head; a wrong
    # head grouping, a transposed P or a missing normalisation breaks it
    seqs, p, Q, K, V = _tiny_tree(4, hq=4, hkv=2, d=8)
    rng = np.random.Generator(np.random.PCG64(13))
    dO = rng.standard_normal(Q.shape)
    _, _, dV = oa.backward(p, Q, K, V, dO, 1e4)
    G = Q.shape[1] // K.shape[1]
    for g in range(K.shape[1]):
        lhs = dV[:, g, :].sum(axis=0)
        rhs = dO[:, g * G:(g + 1) * G, :].sum(axis=(0, 1))
        assert np.allclose(lhs, rhs, rtol=1e-12, atol=1e-10)


# ------------------------------------------------- raw order <-> packed layout
@pytest.mark.parametrize("seed", range(6))
def test_sum_to_forwarded_is_the_transpose_of_the_scatter(seed):
    # <scatter(x), y> over raw tokens equals <x, sum_to_forwarded(y)> over
    # forwarded positions for every x, y: the defining property of a transpose
    from oracle import layout as ol
    rng = np.random.Generator(np.random.PCG64(400 + seed))
    seqs = [rng.integers(0, 3, size=int(rng.integers(1, 40))) for _ in range(int(rng.integers(2, 9)))]
    p = op.plan(seqs, min_shared=int(rng.choice([1, 4])), row_capacity=400)
    F, R = p["n_fwd"], p["n_raw"]
    x = rng.standard_normal((F, 3, 4))
    y = rng.standard_normal((R, 3, 4))
    lhs = np.sum(ol.scatter_to_raw(p, x) * y)
    rhs = np.sum(x * ol.sum_to_forwarded(p, y))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))
    # unit vectors: a raw token's weight lands on its own position only
    e = np.zeros((R, 1))
    r = int(rng.integers(0, R))
    e[r] = 1.0
    s = ol.sum_to_forwarded(p, e)
    assert s[p["token_index"][r], 0] == 1.0 and s.sum() == 1.0


def test_gather_to_forwarded_reproduces_the_packed_tokens():
    # token ids gathered by owner are the planner's forwarded tokens, and
    # every raw token of a position carries that position's token
    from oracle import layout as ol
    seqs, p, _, _, _ = _tiny_tree(5, hq=1, hkv=1, d=8)
    tokens = np.concatenate(seqs).astype(np.int32)
    g = ol.gather_to_forwarded(p, tokens)
    assert np.array_equal(g, np.asarray(p["fwd_token"]))
    assert np.array_equal(g[p["token_index"]], tokens)
