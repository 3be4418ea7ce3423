"""C++ planner (through the C ABI) against the oracle planner: bit-exact.

Host-only: the planner needs no GPU.  Also checks the kernels' work lists
against visibility computed independently by the oracle (parent walks).
"""
import numpy as np
import pytest

import workloads
from oracle import planner as op

LAYOUT_KEYS = ["row_offsets", "row_of_seq", "fwd_token", "fwd_src", "parent", "depth", "token_index",
               "subtree_end"]


def _cpp_plan(seqs, trained=None, groups=None, min_shared=64, cap=65536, placement="bfd"):
    from prefix_tree_packed_dfs_gb300 import ops
    return ops.Plan.from_sequences(seqs, trained=trained, group_ids=groups, row_capacity=cap,
                                   min_shared=min_shared, placement=placement)


def _compare(seqs, trained=None, groups=None, min_shared=64, cap=65536, placement="bfd"):
    ref = op.plan(seqs, trained=trained, group_ids=groups, min_shared=min_shared, row_capacity=cap,
                  placement=placement)
    got = _cpp_plan(seqs, trained, groups, min_shared, cap, placement)
    ex = got.export()
    for k in LAYOUT_KEYS:
        assert np.array_equal(np.asarray(ex[k], np.int64), np.asarray(ref[k], np.int64)), k
    assert list(ex["row_loads"]) == ref["row_loads"]
    info = got.info
    assert info["n_rows"] == ref["n_rows"] and info["n_fwd"] == ref["n_fwd"] and info["n_raw"] == ref["n_raw"]
    assert info["n_segments"] == ref["n_segments"]
    assert info["useful_pairs"] == ref["useful_pairs"]
    assert info["packing_ratio"] == ref["packing_ratio"]
    assert info["row_fill_frac"] == ref["row_fill_frac"]
    assert info["fork_frac"] == ref["fork_frac"]
    # segment instances by tree level (the recurrent layers' schedule)
    lb, start, length, par = got.segments()
    for mine, key in ((lb, "seg_level_begin"), (start, "seg_start"), (length, "seg_len"), (par, "seg_parent")):
        assert np.array_equal(np.asarray(mine, np.int64), np.asarray(ref[key], np.int64)), key
    return ref, got


@pytest.mark.parametrize("name", [n for n in workloads.ALL if n != "deep"])
def test_workloads_bit_exact(lib, name):
    w = workloads.get(name)
    _compare(w.sequences, None, w.group_ids, w.min_shared, w.row_capacity)


@pytest.mark.parametrize("name", ["curriculum_12", "curriculum_48"])
def test_curriculum_batches_bit_exact(lib, name):
    """The planner-scaling stand-ins (many groups under shared task prompts)."""
    w = workloads.get(name)
    ref, got = _compare(w.sequences, None, w.group_ids, w.min_shared, w.row_capacity)
    assert got.info["n_leaves"] == workloads.CURRICULUM[int(name.split("_")[1])]


@pytest.mark.slow
def test_deep_workload_bit_exact(lib):
    w = workloads.get("deep")
    _compare(w.sequences, None, w.group_ids, w.min_shared, w.row_capacity)


@pytest.mark.parametrize("placement", ["bfd", "next_fit"])
def test_art_example_rows(lib, placement):
    from tests.test_oracle_pins import _art_example, golden
    g, seqs, flags, groups, labels = _art_example()
    exp = golden("art_32_rollouts.json")["expected"]
    _, got = _compare(seqs, flags, groups, g["min_shared"], g["row_capacity"], placement)
    key = "best_fit_decreasing_row_loads" if placement == "bfd" else "in_order_row_loads"
    assert list(got.export()["row_loads"]) == exp[key]


def _random_case(rng, alphabet, n_max, len_max):
    n = int(rng.integers(1, n_max + 1))
    base = rng.integers(0, alphabet, size=len_max)
    seqs = []
    for _ in range(n):
        cut = int(rng.integers(0, len_max))
        tail = rng.integers(0, alphabet, size=int(rng.integers(1, max(2, len_max // 2))))
        seqs.append(np.concatenate([base[:cut], tail]))
    if rng.random() < 0.3 and n > 1:   # exact duplicates
        seqs[-1] = seqs[0].copy()
    return seqs


@pytest.mark.parametrize("seed", range(60))
def test_random_small_bit_exact(lib, seed):
    rng = np.random.Generator(np.random.PCG64(1000 + seed))
    seqs = _random_case(rng, int(rng.integers(2, 6)), 12, 24)
    trained = [rng.integers(0, 2, size=len(s)) for s in seqs] if seed % 3 == 0 else None
    groups = rng.integers(0, 3, size=len(seqs)) if seed % 2 else None
    m = int(rng.choice([0, 1, 2, 3, 5, 8, 100]))
    cap = int(max(len(s) for s in seqs) + rng.integers(0, 40))
    placement = "next_fit" if seed % 4 == 1 else "bfd"
    _compare(seqs, trained, groups, m, cap, placement)


def test_errors(lib):
    from prefix_tree_packed_dfs_gb300 import binding as B, ops
    with pytest.raises(B.TpkError) as e:
        ops.Plan(np.array([1, 2, 3], np.int32), np.array([0, 3], np.int64), row_capacity=2)
    assert e.value.status == -2
    with pytest.raises(B.TpkError) as e:
        ops.Plan(np.array([1, 2, 3], np.int32), np.array([0, 2, 2, 3], np.int64))
    assert e.value.status == -1
    with pytest.raises(B.TpkError) as e:
        ops.Plan(np.array([1, -2, 3], np.int32), np.array([0, 3], np.int64))
    assert e.value.status == -1
    with pytest.raises(B.TpkError) as e:
        ops.Plan(np.array([1, 2, 3], np.int32), np.array([1, 3], np.int64))
    assert e.value.status == -1


def _visible(parent, F):
    vis = np.zeros((F, F), dtype=bool)
    for i in range(F):
        for j in op.visible_by_parent_walk(parent, i):
            vis[i, j] = True
    return vis


@pytest.mark.parametrize("seed", range(12))
def test_worklists_cover_exactly_the_tree_mask(lib, seed):
    rng = np.random.Generator(np.random.PCG64(2000 + seed))
    seqs = _random_case(rng, 3, 8, 300)
    m = int(rng.choice([1, 16, 64]))
    cap = int(max(len(s) for s in seqs) + rng.integers(0, 400))
    ref = op.plan(seqs, min_shared=m, row_capacity=cap)
    got = _cpp_plan(seqs, min_shared=m, cap=cap)
    wl = got.worklists()
    F = ref["n_fwd"]
    vis = _visible(ref["parent"], F)
    kb = wl["kb"].reshape(-1, 2)
    covered = np.zeros((F, F), dtype=bool)
    assert sorted(wl["qt_order"]) == list(range(len(wl["qt_q0"])))
    for t in range(len(wl["qt_q0"])):
        q0, nq = wl["qt_q0"][t], wl["qt_nq"][t]
        assert 1 <= nq <= 128
        keys = []
        for b in range(wl["qt_kb_begin"][t], wl["qt_kb_begin"][t + 1]):
            k0, meta = kb[b]
            nk, full = meta & 0xFFFF, meta >> 16
            assert 1 <= nk <= 128
            keys.extend(range(k0, k0 + nk))
            sub = vis[q0:q0 + nq, k0:k0 + nk]
            if full:   # the kernel skips the mask for all 128 columns it loads
                assert nk == 128 and sub.all()
            covered[q0:q0 + nq, k0:k0 + nk] = True
        assert len(keys) == len(set(keys))           # no key visited twice
        assert (keys == sorted(keys))
    assert np.all(covered[vis])                      # every visible pair visited
    # backward: key tiles' query blocks
    qb = wl["qb"].reshape(-1, 2)
    covered[:] = False
    for u in range(len(wl["kt_k0"])):
        k0, nk = wl["kt_k0"][u], wl["kt_nk"][u]
        for c in range(wl["kt_qb_begin"][u], wl["kt_qb_begin"][u + 1]):
            qs, meta = qb[c]
            nq, full = meta & 0xFFFF, meta >> 16
            assert 1 <= nq <= 128
            if full:
                assert nq == 128 and vis[qs:qs + nq, k0:k0 + nk].all()
            covered[qs:qs + nq, k0:k0 + nk] = True
    assert np.all(covered[vis])
    # tiles stay inside rows
    ro = ref["row_offsets"]
    for t in range(len(wl["qt_q0"])):
        r = np.searchsorted(ro, wl["qt_q0"][t], side="right") - 1
        assert wl["qt_q0"][t] + wl["qt_nq"][t] <= ro[r + 1]


def test_worklists_visit_only_the_ancestor_chain(lib):
    # work follows forwarded tokens: in the rho=3.56 sweep row the visited key
    # columns are close to the useful pairs
    w = workloads.get("sweep_3.56")
    got = _cpp_plan(w.sequences, groups=w.group_ids, min_shared=w.min_shared, cap=w.row_capacity)
    info = got.info
    assert info["visited_pairs"] < 1.1 * info["useful_pairs"] * 2  # diagonal blocks count full squares
    assert info["visited_pairs"] >= info["useful_pairs"]


def _check_launch_order(order, begin, run=128):
    work = np.diff(begin)
    n = len(work)
    assert sorted(order) == list(range(n))
    runs = [order[i:i + min(run, n - i)] for i in range(0, n, run)]
    # the order is a sequence of whole runs of consecutive tiles ...
    pos, run_work = 0, []
    seen = set()
    while pos < n:
        r = order[pos] // run
        assert r not in seen
        seen.add(r)
        size = min(run, n - r * run)
        chunk = order[pos:pos + size]
        assert sorted(chunk) == list(range(r * run, r * run + size))
        # ... longest first inside a run ...
        assert all(work[a] >= work[b] for a, b in zip(chunk, chunk[1:]))
        run_work.append(int(work[chunk].sum()))
        pos += size
    # ... and runs by decreasing total work
    assert all(a >= b for a, b in zip(run_work, run_work[1:]))
    assert len(runs) == len(seen)


@pytest.mark.parametrize("name", ["deep_small", "grpo", "sweep_2.00"])
def test_launch_order_runs_longest_first(lib, name):
    w = workloads.get(name)
    got = _cpp_plan(w.sequences, groups=w.group_ids, min_shared=w.min_shared, cap=w.row_capacity)
    wl = got.worklists()
    _check_launch_order(list(wl["qt_order"]), wl["qt_kb_begin"])
    _check_launch_order(list(wl["kt_order"]), wl["kt_qb_begin"])


@pytest.mark.parametrize("name", ["tiny", "grpo", "deep_small", "sweep_1.00"])
def test_raw_of_forwarded_is_token_index_inverted(lib, name):
    # the CSR of raw tokens per forwarded position, built from the oracle's
    # token_index: stable order of raw tokens by position, first = owner
    w = workloads.get(name)
    ref = op.plan(w.sequences, group_ids=w.group_ids, min_shared=w.min_shared, row_capacity=w.row_capacity)
    got = _cpp_plan(w.sequences, groups=w.group_ids, min_shared=w.min_shared, cap=w.row_capacity)
    begin, raw = got.raw_of_forwarded()
    ti = np.asarray(ref["token_index"])
    exp_begin = np.concatenate([[0], np.cumsum(np.bincount(ti, minlength=ref["n_fwd"]))]).astype(np.int32)
    exp_raw = np.argsort(ti, kind="stable").astype(np.int32)
    assert np.array_equal(begin, exp_begin)
    assert np.array_equal(raw, exp_raw)
    assert np.array_equal(raw[begin[:-1]], np.asarray(ref["fwd_src"]))


@pytest.mark.parametrize("seed", range(10))
def test_one_row_per_group_bit_exact(lib, seed):
    """Placement "groups": one row per group id, rows in increasing id --
    library and oracle agree bit for bit, and every row holds exactly one
    group's sequences."""
    rng = np.random.Generator(np.random.PCG64(500 + seed))
    seqs = _random_case(rng, int(rng.integers(2, 6)), 12, 24)
    groups = (rng.integers(0, 4, size=len(seqs)) * 3 + 7).astype(np.int32)     # sparse, unordered ids
    _, got = _compare(seqs, None, groups, int(rng.choice([0, 2, 5])), 1 << 20, "groups")
    # identical sequences are one leaf, placed with the group of the lowest-index copy
    first = {}
    eff = np.array([groups[first.setdefault(tuple(x.tolist()), i)] for i, x in enumerate(seqs)])
    ids = sorted(set(eff.tolist()))
    assert got.info["n_rows"] == len(ids)
    assert np.array_equal(got.export()["row_of_seq"], np.searchsorted(ids, eff))


def test_one_row_per_group_rebuilds_the_rows_of_a_plan(lib):
    """A BFD plan's rows, planned again with each sequence's row as its group,
    come back identical (the per-rank plan of a row-sharded batch)."""
    w = workloads.get("grpo")
    full = _cpp_plan(w.sequences, None, w.group_ids, w.min_shared, w.row_capacity)
    rows = full.export()["row_of_seq"]
    _, again = _compare(w.sequences, None, rows, w.min_shared, w.row_capacity, "groups")
    a, b = full.export(), again.export()
    for k in ("row_offsets", "fwd_token", "depth", "parent", "subtree_end", "token_index", "row_of_seq"):
        assert np.array_equal(a[k], b[k]), k


def test_one_row_per_group_rejects_an_oversized_group(lib):
    from prefix_tree_packed_dfs_gb300 import binding as B
    seqs = [np.arange(40, dtype=np.int32) + 100 * i for i in range(3)]
    with pytest.raises(B.TpkError):
        _cpp_plan(seqs, None, np.zeros(3, np.int32), 4, 100, "groups")
    with pytest.raises(op.PlanError):
        op.plan(seqs, group_ids=np.zeros(3, np.int32), row_capacity=100, min_shared=4, placement="groups")


@pytest.mark.parametrize("name", ["curriculum_48", "curriculum_192", "deep_small", "grpo", "agentic"])
def test_plan_does_not_depend_on_the_thread_count(lib, monkeypatch, name):
    """The planner's parallel passes (symbols per sequence, sort in chunks,
    layout / work lists / raw-token lists per row, image in pieces) give the
    same plan on 1, 3 and 16 host threads."""
    w = workloads.get(name)
    outs = []
    for threads in ("1", "3", "16"):
        monkeypatch.setenv("TPK_PLANNER_THREADS", threads)
        p = _cpp_plan(w.sequences, None, w.group_ids, w.min_shared, w.row_capacity)
        outs.append((p.export(), p.worklists(), p.raw_of_forwarded(), dict(p.info), p.device_bytes()))
        p.close()
    e0, w0, r0, i0, d0 = outs[0]
    for e, wl, r, i, d in outs[1:]:
        assert all(np.array_equal(e0[k], e[k]) for k in e0)
        assert all(np.array_equal(w0[k], wl[k]) for k in w0)
        assert all(np.array_equal(a, b) for a, b in zip(r0, r))
        assert i == i0 and d == d0


@pytest.mark.parametrize("m", [1, 2, 3, 11, 12, 13])
def test_min_shared_carry_down_hand_counted(lib, m):
    """The library on the hand-counted carry-down case of the oracle pins:
    forwarded totals 34 / 36 / 60 as derived there, and bit-exact layouts."""
    from tests.test_oracle_pins import MIN_SHARED_CASE, _min_shared_case
    seqs = _min_shared_case()
    ref, got = _compare(seqs, min_shared=m, cap=1000)
    assert got.info["n_fwd"] == MIN_SHARED_CASE[m]


def test_shape_checks_before_any_launch(lib, monkeypatch):
    """The torch wrappers check every tensor's shape against the plan (and
    each other) before calling the library: a mismatched tensor would make
    the kernels read or write outside its allocation."""
    import types
    import torch
    from prefix_tree_packed_dfs_gb300 import binding as B
    from prefix_tree_packed_dfs_gb300 import ops

    class NoKernels:
        """The real library, with its GPU entry points replaced by a trap."""
        def __getattr__(self, name):
            if name.startswith("tpk_tree_attn_") and name != "tpk_tree_attn_workspace_bytes":
                raise AssertionError("%s reached despite a bad argument" % name)
            return getattr(lib, name)
    monkeypatch.setattr(B, "load", lambda *a, **k: NoKernels())
    w = workloads.get("tiny_fit")
    plan = _cpp_plan(w.sequences, min_shared=w.min_shared, cap=w.row_capacity)
    F = plan.info["n_fwd"]
    dp = types.SimpleNamespace(plan=plan, n_fwd=F, image=torch.empty(256, dtype=torch.uint8))
    Hq, Hkv, d = 4, 2, 64
    bf = dict(dtype=torch.bfloat16)
    q, k, v = torch.zeros(F, Hq, d, **bf), torch.zeros(F, Hkv, d, **bf), torch.zeros(F, Hkv, d, **bf)
    o, do, lse = torch.zeros(F, Hq, d, **bf), torch.zeros(F, Hq, d, **bf), torch.zeros(Hq, F)

    def raises(fn, what):
        with pytest.raises(ValueError, match=what):
            fn()
    # forward: rows against the plan, k/v against q, caller-supplied outputs
    raises(lambda: ops.tree_attn_fwd(dp, q[:-1], k[:-1], v[:-1]), "forwarded positions")
    raises(lambda: ops.tree_attn_fwd(dp, q, k, v[:, :1].contiguous()), "v must have shape")
    raises(lambda: ops.tree_attn_fwd(dp, q, k[:, :, :32].contiguous(), v), "k must have shape")
    raises(lambda: ops.tree_attn_fwd(dp, q, k, v, out=o[:-1]), "out must have shape")
    raises(lambda: ops.tree_attn_fwd(dp, q, k, v, lse=lse[:-1]), "lse must have shape")
    raises(lambda: ops.tree_attn_fwd(dp, q, k, v, precise=True, o_lo=o[:, :2].contiguous()), "o_lo must have shape")
    # backward: o, do, lse, every caller-supplied gradient, o_lo, workspace
    bwd = lambda **kw: ops.tree_attn_bwd(dp, kw.get("q", q), k, v, kw.get("o", o), kw.get("lse", lse),
                                         kw.get("do", do), dq=kw.get("dq"), dk=kw.get("dk"), dv=kw.get("dv"),
                                         o_lo=kw.get("o_lo"), workspace=kw.get("ws"))
    raises(lambda: bwd(o=o[:-1]), "o must have shape")
    raises(lambda: bwd(do=do[:, :1].contiguous()), "do must have shape")
    raises(lambda: bwd(lse=lse[:1].contiguous()), "lse must have shape")
    raises(lambda: bwd(dq=torch.zeros(F, Hkv, d, **bf)), "dq must have shape")
    raises(lambda: bwd(dk=torch.zeros(F, Hq, d, **bf)), "dk must have shape")
    raises(lambda: bwd(dv=torch.zeros(F + 1, Hkv, d, **bf)), "dv must have shape")
    raises(lambda: bwd(o_lo=o[:-2]), "o_lo must have shape")
    raises(lambda: bwd(ws=torch.empty(16, dtype=torch.uint8)), "workspace has 16 bytes")
    # right shapes, host tensors: refused as such (there is no CPU path)
    raises(lambda: ops.tree_attn_fwd(dp, q, k, v), "must be a CUDA tensor")
    raises(lambda: bwd(), "must be a CUDA tensor")


def test_gdn_shape_checks_before_any_launch(lib, monkeypatch):
    """The GDN wrappers (forward and backward) check every tensor against
    the plan and each other before calling the library."""
    import types
    import torch
    from prefix_tree_packed_dfs_gb300 import binding as B
    from prefix_tree_packed_dfs_gb300 import ops

    class NoKernels:
        """The real library, with its GDN entry points (not the size queries) replaced by a trap."""
        def __getattr__(self, name):
            if name.startswith("tpk_gdn_") and not name.endswith("_bytes"):
                raise AssertionError("%s reached despite a bad argument" % name)
            return getattr(lib, name)
    monkeypatch.setattr(B, "load", lambda *a, **k: NoKernels())
    w = workloads.get("tiny_fit")
    plan = _cpp_plan(w.sequences, min_shared=w.min_shared, cap=w.row_capacity)
    F = plan.info["n_fwd"]
    dp = types.SimpleNamespace(plan=plan, n_fwd=F, image=torch.empty(256, dtype=torch.uint8))
    H, d, W = 2, 64, 4
    C = 3 * H * d
    bf = dict(dtype=torch.bfloat16)
    x, dy = torch.zeros(F, C, **bf), torch.zeros(F, C, **bf)
    wc = torch.zeros(C, W)
    y = torch.zeros(F, C, **bf)
    q, k, v = (y[:, i * H * d:(i + 1) * H * d].unflatten(1, (H, d)) for i in range(3))
    g, b = torch.zeros(F, H), torch.zeros(F, H)
    do = torch.zeros(F, H, d, **bf)
    state = torch.empty(int(lib.tpk_gdn_workspace_bytes(plan.handle, H, d, d)) + 256, dtype=torch.uint8)

    def raises(fn, what, exc=ValueError):
        with pytest.raises(exc, match=what):
            fn()
    # convolution backward
    raises(lambda: ops.gdn_conv_bwd(dp, x[:-1], wc, dy[:-1]), "forwarded positions")
    raises(lambda: ops.gdn_conv_bwd(dp, x, wc[:-1].contiguous(), dy), "w must have shape")
    raises(lambda: ops.gdn_conv_bwd(dp, x, wc, dy[:, :8].contiguous()), "dy must have shape")
    raises(lambda: ops.gdn_conv_bwd(dp, x, wc, dy, dx=dy[:-1]), "dx must have shape")
    raises(lambda: ops.gdn_conv_bwd(dp, x, wc, dy, dw=wc[:, :1].contiguous()), "dw must have shape")
    raises(lambda: ops.gdn_conv_bwd(dp, x, wc, dy, workspace=torch.empty(16, dtype=torch.uint8)),
           "workspace has 16 bytes")
    raises(lambda: ops.gdn_conv_bwd(dp, x, wc, dy), "must be a CUDA tensor")
    # delta rule backward
    bwd = lambda **kw: ops.gdn_delta_rule_bwd(dp, kw.get("q", q), k, v, kw.get("g", g), b, kw.get("do", do),
                                              kw.get("state", state), dq=kw.get("dq"), dk=kw.get("dk"),
                                              dv=kw.get("dv"), dg=kw.get("dg"), workspace=kw.get("ws"))
    raises(lambda: bwd(q=q[:-1]), "forwarded positions")
    raises(lambda: bwd(g=g[:, :1].contiguous()), "g must have shape")
    raises(lambda: bwd(do=do[:-1]), "dout must have shape")
    raises(lambda: bwd(dq=torch.zeros(F, H, d + 8, **bf)), "dq must have shape")
    raises(lambda: bwd(dv=torch.zeros(F, H + 1, d, **bf)), "dv must have shape")
    raises(lambda: bwd(dk=torch.zeros(F, H, d // 2, **bf)), "dk must have shape")
    raises(lambda: bwd(dg=torch.zeros(F, H + 1)), "dg must have shape")
    raises(lambda: bwd(state=torch.empty(16, dtype=torch.uint8)), "state has 16 bytes")
    raises(lambda: bwd(ws=torch.empty(16, dtype=torch.uint8)), "workspace has 16 bytes")
    raises(lambda: bwd(), "must be a CUDA tensor")
