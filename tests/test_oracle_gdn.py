"""Pins of the GDN oracle (oracle/gdn.py) against what fixes it from outside:
library routines, closed forms of the recurrence, an independently derived
chunked form, and the unpacked sequences themselves.  CPU only."""
import numpy as np
import pytest

from oracle import gdn as og
from oracle import planner as op


def _chain_plan(L):
    return op.plan([np.arange(L) + 1], min_shared=1, row_capacity=10 ** 6)


def _rand(rng, F, H, dk, dv, g_scale=0.3):
    Q = rng.standard_normal((F, H, dk))
    K = rng.standard_normal((F, H, dk))
    V = rng.standard_normal((F, H, dv))
    G = -g_scale * rng.random((F, H))          # log decay <= 0
    B = rng.uniform(0.05, 0.95, (F, H))
    return Q, K, V, G, B


def _tree(seed, n=6):
    rng = np.random.Generator(np.random.PCG64(600 + seed))
    base = rng.integers(0, 5, size=25)
    seqs = []
    for _ in range(n):
        cut = int(rng.integers(2, 20))
        seqs.append(np.concatenate([base[:cut], rng.integers(0, 5, size=int(rng.integers(1, 9)))]))
    return op.plan(seqs, min_shared=int(rng.choice([1, 3])), row_capacity=int(rng.choice([40, 400])))


# ------------------------------------------------------------------ conv
@pytest.mark.parametrize("W", [1, 2, 4])
def test_conv_is_numpy_convolve_on_a_chain(W):
    # a chain is one sequence: channel c is numpy's full convolution of x_c
    # with the reversed kernel, cut to the sequence, through SiLU
    rng = np.random.Generator(np.random.PCG64(W))
    L, C = 17, 5
    p = _chain_plan(L)
    X = rng.standard_normal((L, C))
    w = rng.standard_normal((C, W))
    y = og.conv(p, X, w)
    for c in range(C):
        ref = np.convolve(X[:, c], w[c, ::-1])[:L]
        assert np.allclose(y[:, c], ref / (1 + np.exp(-ref)), rtol=1e-13, atol=1e-13)


def test_conv_width_one_is_silu_and_branches_see_only_their_path():
    p = _tree(0)
    rng = np.random.Generator(np.random.PCG64(9))
    X = rng.standard_normal((p["n_fwd"], 3))
    y = og.conv(p, X, np.ones((3, 1)))
    assert np.allclose(y, X / (1 + np.exp(-X)), rtol=1e-14)
    # width 3 on the tree: position f mixes f, parent(f), parent(parent(f))
    w = rng.standard_normal((3, 3))
    y = og.conv(p, X, w)
    par = p["parent"]
    for f in range(p["n_fwd"]):
        a1 = par[f]
        a2 = par[a1] if a1 >= 0 else -1
        acc = w[:, 2] * X[f] + (w[:, 1] * X[a1] if a1 >= 0 else 0) + (w[:, 0] * X[a2] if a2 >= 0 else 0)
        assert np.allclose(y[f], acc / (1 + np.exp(-acc)), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------ delta rule
def test_zero_beta_writes_nothing():
    rng = np.random.Generator(np.random.PCG64(1))
    p = _chain_plan(9)
    Q, K, V, G, B = _rand(rng, 9, 2, 4, 3)
    assert np.all(og.delta_rule(p, Q, K, V, G, np.zeros_like(B)) == 0)


def test_full_decay_keeps_only_the_current_token():
    # alpha = exp(-60) ~ 1e-26: S_t = beta_t v_t k_t^T, so
    # o_t = beta_t scale (k_t . q_t) v_t with k, q normalised
    rng = np.random.Generator(np.random.PCG64(2))
    p = _chain_plan(12)
    Q, K, V, G, B = _rand(rng, 12, 3, 8, 5)
    G[:] = -60.0
    o = og.delta_rule(p, Q, K, V, G, B, scale=0.5)
    kn = K / np.linalg.norm(K, axis=-1, keepdims=True)
    qn = Q / np.linalg.norm(Q, axis=-1, keepdims=True)
    ref = (B * 0.5 * np.sum(kn * qn, axis=-1))[..., None] * V
    assert np.allclose(o, ref, rtol=1e-12, atol=1e-14)


def test_orthonormal_keys_are_stored_exactly():
    # alpha = 1, beta = 1 and one-hot keys: the delta rule stores v_s under
    # key e_{j(s)} exactly, so querying with e_{j(s)} at any later t returns
    # scale * v_s
    L, dk, dv = 6, 8, 3
    rng = np.random.Generator(np.random.PCG64(3))
    p = _chain_plan(L)
    slots = rng.permutation(dk)[:L]
    K = np.zeros((L, 1, dk))
    K[np.arange(L), 0, slots] = rng.uniform(0.5, 2.0, L)     # positive multiples of e_j
    V = rng.standard_normal((L, 1, dv))
    look = [int(rng.integers(0, t + 1)) for t in range(L)]    # an earlier (or the same) token
    Q = np.zeros((L, 1, dk))
    Q[np.arange(L), 0, slots[look]] = 3.0
    o = og.delta_rule(p, Q, K, V, np.zeros((L, 1)), np.ones((L, 1)), scale=0.25)
    assert np.allclose(o[:, 0], 0.25 * V[look, 0], rtol=1e-13, atol=1e-13)


def test_repeated_key_is_overwritten():
    # alpha = 1, beta = 1, the same key every step: S_t k = v_t (the delta
    # rule replaces the value stored under k), so q = k reads the latest v
    L, dk, dv = 7, 4, 2
    rng = np.random.Generator(np.random.PCG64(4))
    p = _chain_plan(L)
    k = rng.standard_normal(dk)
    K = np.tile(k, (L, 1, 1))
    V = rng.standard_normal((L, 1, dv))
    o = og.delta_rule(p, K.copy(), K, V, np.zeros((L, 1)), np.ones((L, 1)), scale=1.0)
    assert np.allclose(o[:, 0], V[:, 0], rtol=1e-12, atol=1e-13)


def test_scalar_state_closed_form():
    # dk = dv = 1: k_t / |k_t| = s_t in {-1, 1}, so
    # S_t = alpha_t (1 - beta_t) S_{t-1} + beta_t v_t s_t and
    # S_t = sum_{u <= t} beta_u v_u s_u prod_{r = u+1..t} alpha_r (1 - beta_r)
    L = 15
    rng = np.random.Generator(np.random.PCG64(5))
    p = _chain_plan(L)
    Q, K, V, G, B = _rand(rng, L, 1, 1, 1)
    o = og.delta_rule(p, Q, K, V, G, B, scale=0.7)[:, 0, 0]
    s, a, b, v, sq = np.sign(K[:, 0, 0]), np.exp(G[:, 0]), B[:, 0], V[:, 0, 0], np.sign(Q[:, 0, 0])
    for t in range(L):
        St = sum(b[u] * v[u] * s[u] * np.prod([a[r] * (1 - b[r]) for r in range(u + 1, t + 1)]) for u in range(t + 1))
        assert np.isclose(o[t], 0.7 * sq[t] * St, rtol=1e-12, atol=1e-14)


def _chunked(Q, K, V, G, B, scale, C):
    """The recurrence in chunks of C tokens, derived independently of the
    step-by-step form: within a chunk with cumulative decay Gamma_i (product
    of alpha_1..alpha_i from the chunk start) and S0 the state entering it,
    the written values u_i = beta_i (v_i - alpha_i S_{i-1} k_i) solve the
    lower-triangular system
        u_i + beta_i sum_{j<i} (Gamma_i/Gamma_j)(k_i.k_j) u_j = beta_i (v_i - Gamma_i S0 k_i),
    then o_i = Gamma_i S0 q_i + sum_{j<=i} (Gamma_i/Gamma_j)(q_i.k_j) u_j and
    the chunk's final state is Gamma_C S0 + sum_j (Gamma_C/Gamma_j) u_j k_j^T."""
    L, dk = K.shape
    K = K / np.linalg.norm(K, axis=-1, keepdims=True)
    Q = scale * Q / np.linalg.norm(Q, axis=-1, keepdims=True)
    S = np.zeros((V.shape[1], dk))
    out = np.zeros((L, V.shape[1]))
    for c0 in range(0, L, C):
        k, q, v, g, b = K[c0:c0 + C], Q[c0:c0 + C], V[c0:c0 + C], G[c0:c0 + C], B[c0:c0 + C]
        n = len(k)
        cum = np.cumsum(g)
        ratio = np.exp(cum[:, None] - cum[None, :])               # Gamma_i / Gamma_j
        A = np.tril(ratio * (k @ k.T), -1)
        rhs = b[:, None] * (v - np.exp(cum)[:, None] * (k @ S.T))
        u = np.linalg.solve(np.eye(n) + b[:, None] * A, rhs)
        out[c0:c0 + n] = np.exp(cum)[:, None] * (q @ S.T) + (np.tril(ratio) * (q @ k.T)) @ u
        S = np.exp(cum[-1]) * S + (np.exp(cum[-1] - cum)[:, None] * u).T @ k
    return out


@pytest.mark.parametrize("C", [1, 3, 8, 64])
def test_recurrence_equals_the_chunked_form(C):
    rng = np.random.Generator(np.random.PCG64(10 + C))
    L, dk, dv = 40, 6, 5
    p = _chain_plan(L)
    Q, K, V, G, B = _rand(rng, L, 1, dk, dv)
    o = og.delta_rule(p, Q, K, V, G, B, scale=0.4)[:, 0]
    ref = _chunked(Q[:, 0], K[:, 0], V[:, 0], G[:, 0], B[:, 0], 0.4, C)
    assert np.allclose(o, ref, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("seed", range(6))
def test_level_schedule_equals_unpacked_sequences(seed):
    # the pages' schedule (segment instances level by level, each from its
    # parent's final state) reproduces every sequence run alone from zero
    p = _tree(seed)
    rng = np.random.Generator(np.random.PCG64(700 + seed))
    Q, K, V, G, B = _rand(rng, p["n_fwd"], 2, 4, 3)
    assert np.allclose(og.delta_rule_tree(p, Q, K, V, G, B), og.delta_rule(p, Q, K, V, G, B), rtol=1e-12,
                       atol=1e-13)
    # the level table covers every position once; parents lie one level up
    begin, start, length, par = (p[k] for k in ("seg_level_begin", "seg_start", "seg_len", "seg_parent"))
    cover = np.zeros(p["n_fwd"], int)
    for s, n in zip(start, length):
        cover[s:s + n] += 1
    assert np.all(cover == 1)
    # level-local offsets: the lengths of the earlier instances of the level
    for lv in range(len(begin) - 1):
        i0, i1 = begin[lv], begin[lv + 1]
        assert list(p["seg_off"][i0:i1]) == [int(np.sum(length[i0:i])) for i in range(i0, i1)]
        assert np.all(np.diff(start[i0:i1]) > 0)   # ascending starts within a level
    for lv in range(len(begin) - 1):
        for i in range(begin[lv], begin[lv + 1]):
            if lv == 0:
                assert par[i] == -1 and p["parent"][start[i]] == -1
            else:
                assert begin[lv - 1] <= par[i] < begin[lv]
                assert p["parent"][start[i]] == start[par[i]] + length[par[i]] - 1


def test_sampled_rows_match_the_full_run():
    p = _tree(3)
    rng = np.random.Generator(np.random.PCG64(800))
    X = _rand(rng, p["n_fwd"], 2, 4, 3)
    full = og.delta_rule(p, *X)
    keys = dict(zip(("q", "k", "v", "g", "b"), X))
    raw = [0, 5, p["n_raw"] // 2, p["n_raw"] - 1]
    got = og.delta_rule_rows(p, lambda key, idx: keys[key][idx], raw)
    assert np.allclose(got, full[p["token_index"][raw]], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- gradients
def _fd(f, arrays, i, h=1e-6):
    """Central differences of the scalar f(*arrays) w.r.t. every entry of
    arrays[i]."""
    base = [np.array(a, dtype=np.float64) for a in arrays]
    x = base[i]
    out = np.zeros_like(x)
    for j in np.ndindex(x.shape):
        old = x[j]
        x[j] = old + h
        up = f(*base)
        x[j] = old - h
        dn = f(*base)
        x[j] = old
        out[j] = (up - dn) / (2 * h)
    return out


def test_conv_bwd_matches_central_differences():
    # a small tree with branch points, width 3: dX sums over every
    # descendant within two steps on every branch, dw over all positions
    p = _tree(1, n=4)
    rng = np.random.Generator(np.random.PCG64(31))
    F, C, W = p["n_fwd"], 2, 3
    X = rng.standard_normal((F, C))
    w = rng.standard_normal((C, W))
    dY = rng.standard_normal((F, C))
    dX, dw = og.conv_bwd(p, X, w, dY)
    loss = lambda X_, w_: float(np.sum(dY * og.conv(p, X_, w_)))
    assert np.allclose(dX, _fd(loss, [X, w], 0), rtol=1e-7, atol=1e-8)
    assert np.allclose(dw, _fd(loss, [X, w], 1), rtol=1e-7, atol=1e-8)
    # the tree has a branch point, so some dX row gathers from two children
    assert np.any(np.bincount(p["parent"][p["parent"] >= 0]) >= 2)


def test_conv_bwd_width_one_closed_form():
    # W = 1: y = silu(w x) per channel, so dX = dY silu'(w x) w and
    # dw = sum_f dY silu'(w x) x, with silu'(a) = s(a) (1 + a (1 - s(a)))
    p = _tree(2)
    rng = np.random.Generator(np.random.PCG64(32))
    F, C = p["n_fwd"], 4
    X, dY = rng.standard_normal((F, C)), rng.standard_normal((F, C))
    w = rng.standard_normal((C, 1))
    a = X * w[:, 0]
    s = 1 / (1 + np.exp(-a))
    ds = s * (1 + a * (1 - s))
    dX, dw = og.conv_bwd(p, X, w, dY)
    assert np.allclose(dX, dY * ds * w[:, 0], rtol=1e-12, atol=1e-14)
    assert np.allclose(dw[:, 0], np.sum(dY * ds * X, axis=0), rtol=1e-12, atol=1e-12)


def test_delta_bwd_matches_central_differences():
    # every input, on a tree whose sequences fork: gradients of the forked
    # states are summed over the children
    p = _tree(4, n=4)
    rng = np.random.Generator(np.random.PCG64(33))
    F, H, dk, dv = p["n_fwd"], 2, 3, 2
    Q, K, V, G, B = _rand(rng, F, H, dk, dv)
    dO = rng.standard_normal((F, H, dv))
    grads = og.delta_rule_bwd(p, Q, K, V, G, B, dO, scale=0.6)
    loss = lambda *a: float(np.sum(dO * og.delta_rule(p, *a, scale=0.6)))
    for i, gr in enumerate(grads):
        assert np.allclose(gr, _fd(loss, [Q, K, V, G, B], i), rtol=1e-6, atol=1e-8), "input %d" % i
    assert np.any(np.bincount(p["parent"][p["parent"] >= 0]) >= 2)


def test_delta_bwd_zero_beta_closed_form():
    # beta = 0 writes nothing (S = 0), so dq, dk, dv and dg vanish, and to
    # first order in beta, o_s = sum_{t <= s} beta_t Gamma(s, t) (k_t . q_s) v_t
    # with Gamma(s, t) = prod_{t < r <= s} alpha_r: on a chain,
    # dbeta_t = sum_{s >= t} Gamma(s, t) (k_t . q_s) (v_t . dO_s)
    L, H, dk, dv = 11, 2, 5, 3
    p = _chain_plan(L)
    rng = np.random.Generator(np.random.PCG64(34))
    Q, K, V, G, B = _rand(rng, L, H, dk, dv)
    dO = rng.standard_normal((L, H, dv))
    dQ, dK, dV, dG, dB = og.delta_rule_bwd(p, Q, K, V, G, np.zeros_like(B), dO, scale=0.3)
    for z in (dQ, dK, dV, dG):
        assert np.all(z == 0)
    kn = K / np.linalg.norm(K, axis=-1, keepdims=True)
    qn = 0.3 * Q / np.linalg.norm(Q, axis=-1, keepdims=True)
    want = np.zeros((L, H))
    for t in range(L):
        for s in range(t, L):
            gam = np.exp(np.sum(G[t + 1:s + 1], axis=0))
            want[t] += gam * np.sum(kn[t] * qn[s], axis=-1) * np.sum(V[t] * dO[s], axis=-1)
    assert np.allclose(dB, want, rtol=1e-12, atol=1e-13)


def test_bwd_rows_match_the_dense_gradients():
    # an output gradient at three positions only: the sampled form (each
    # pick's prefix run alone) equals the dense one, which is zero elsewhere
    p = _tree(5)
    rng = np.random.Generator(np.random.PCG64(35))
    F, H, dk, dv, C, W = p["n_fwd"], 2, 4, 3, 5, 3
    X = _rand(rng, F, H, dk, dv)
    ti = p["token_index"]
    raw = [3, p["n_raw"] // 2, p["n_raw"] - 1]
    assert len({int(ti[r]) for r in raw}) == 3
    dO = np.zeros((F, H, dv))
    picks = []
    for r in raw:
        d = rng.standard_normal((H, dv))
        dO[ti[r]] = d
        picks.append((r, d))
    dense = og.delta_rule_bwd(p, *X, dO)
    keys = dict(zip(("q", "k", "v", "g", "b"), X))
    pos, rows = og.delta_rule_bwd_rows(p, lambda key, idx: keys[key][idx], picks)
    for a, b in zip(dense, rows):
        assert np.allclose(a[pos], b, rtol=1e-10, atol=1e-12)
        rest = np.ones(F, dtype=bool)
        rest[pos] = False
        assert np.all(a[rest] == 0)
    xc, wc = rng.standard_normal((F, C)), rng.standard_normal((C, W))
    dY = np.zeros((F, C))
    cp = []
    for r in raw:
        d = rng.standard_normal(C)
        dY[ti[r]] = d
        cp.append((r, d))
    dX, dw = og.conv_bwd(p, xc, wc, dY)
    pos, dXr, dwr = og.conv_bwd_rows(p, lambda idx: xc[idx], wc, cp)
    assert np.allclose(dX[pos], dXr, rtol=1e-10, atol=1e-12) and np.allclose(dw, dwr, rtol=1e-10, atol=1e-12)
    rest = np.ones(F, dtype=bool)
    rest[pos] = False
    assert np.all(dX[rest] == 0)
