"""Oracle of the GDN (Gated DeltaNet) token mixer over a packed prefix tree, fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"Prefix Tree Packing in ART", section "Token-mixing layers": packing is valid
for a layer only if a token mixes with its own ancestor chain and nothing
else.  For attention that is a mask; GDN is recurrent instead -- a running
state threaded token by token, forked once per branch point and reset at
every tree root -- and it runs as a short causal convolution followed by the
gated delta rule.  What the packed computation must reproduce is therefore
the plain recurrence over every root-to-leaf sequence, unpacked, from a zero
state and a zero convolution history: that is what this module computes,
sequence by sequence (``conv``, ``delta_rule``).  ``delta_rule_tree`` is the
pages' schedule instead (one pass per tree level, a child segment starting
from its parent's final state); it is here only to be checked against the
unpacked form, which pins the planner's level table.

The pages name the layer but do not define it.  The reading taken is the
published Gated DeltaNet layer: per head, with k and q L2-normalised,
alpha_t = exp(g_t) and 0 < beta_t < 1,
    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T   (S: dv x dk, S_0 = 0)
    o_t = S_t (scale q_t),
and before it a depthwise causal convolution of width W with SiLU on every
channel of the q, k, v projections.
"""
import numpy as np


def _silu(x):
    return x / (1.0 + np.exp(-x))


def _paths(plan):
    off = plan["seq_offsets"]
    ti = plan["token_index"]
    return [ti[off[s]:off[s + 1]] for s in range(len(off) - 1)]


def _assign(out, path, vals, seen):
    """Write one sequence's rows into the forwarded layout; positions shared
    with an earlier sequence must agree (a causal layer cannot see past the
    shared prefix), to 1e-12 relative."""
    old = seen[path]
    if old.any():
        ref = out[path[old]]
        assert np.max(np.abs(ref - vals[old])) <= 1e-12 * max(1.0, float(np.max(np.abs(ref))))
    out[path] = vals
    seen[path] = True


def conv(plan, X, w):
    """Depthwise causal convolution + SiLU along every sequence.

    X [F, C] in forwarded layout, w [C, W]: for position p of a sequence,
    y_p[c] = silu(sum_j w[c, j] x_{p-W+1+j}[c]) with x before the sequence's
    first token taken as 0.  Returns y [F, C]."""
    X = np.asarray(X, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    F, C = X.shape
    W = w.shape[1]
    out = np.zeros((F, C))
    seen = np.zeros(F, dtype=bool)
    for path in _paths(plan):
        xs = np.concatenate([np.zeros((W - 1, C)), X[path]], axis=0)
        acc = np.zeros((len(path), C))
        for j in range(W):
            acc += w[:, j][None, :] * xs[j:j + len(path)]
        _assign(out, path, _silu(acc), seen)
    return out


def _l2n(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _step(S, q, k, v, g, b, scale):
    """One token for every head: S [H, dv, dk]; q, k [H, dk]; v [H, dv];
    g, b [H].  Returns (new S, o [H, dv])."""
    k = _l2n(k)
    q = _l2n(q)
    alpha = np.exp(g)[:, None, None]
    Sk = np.einsum("hec,hc->he", S, k)
    S = alpha * (S - b[:, None, None] * np.einsum("he,hc->hec", Sk, k)) \
        + b[:, None, None] * np.einsum("he,hc->hec", v, k)
    return S, np.einsum("hec,hc->he", S, scale * q)


def delta_rule(plan, Q, K, V, G, B, scale=None):
    """The gated delta rule along every sequence from S = 0.

    Q, K [F, H, dk], V [F, H, dv], G (log decay, <= 0), B (beta) [F, H] in
    forwarded layout.  Returns O [F, H, dv]."""
    Q, K, V, G, B = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, G, B))
    F, H, dk = Q.shape
    dv = V.shape[2]
    scale = 1.0 / np.sqrt(dk) if scale is None else scale
    out = np.zeros((F, H, dv))
    seen = np.zeros(F, dtype=bool)
    for path in _paths(plan):
        S = np.zeros((H, dv, dk))
        o = np.zeros((len(path), H, dv))
        for p, f in enumerate(path):
            S, o[p] = _step(S, Q[f], K[f], V[f], G[f], B[f], scale)
        _assign(out, path, o, seen)
    return out


def delta_rule_rows(plan, rows, raw, scale=None):
    """O at the forwarded positions of raw tokens ``raw`` only: each one's
    sequence prefix is run from S = 0.  ``rows(key, idx)`` returns rows
    ``idx`` of the forwarded input ``key`` in ("q", "k", "v", "g", "b")."""
    off = plan["seq_offsets"]
    ti = plan["token_index"]
    out = []
    for r in raw:
        s = int(np.searchsorted(off, r, side="right") - 1)
        path = ti[off[s]:r + 1]
        Q, K, V, G, B = (np.asarray(rows(key, path), dtype=np.float64) for key in ("q", "k", "v", "g", "b"))
        H, dk = Q.shape[1], Q.shape[2]
        sc = 1.0 / np.sqrt(dk) if scale is None else scale
        S = np.zeros((H, V.shape[2], dk))
        for p in range(len(path)):
            S, o = _step(S, Q[p], K[p], V[p], G[p], B[p], sc)
        out.append(o)
    return np.stack(out)


def delta_rule_tree(plan, Q, K, V, G, B, scale=None):
    """The pages' schedule: segment instances level by level (the plan's
    seg_level_begin / seg_start / seg_len / seg_parent), each starting from
    its parent instance's final state (zero at a root).  Equal to
    ``delta_rule`` if the level table is right."""
    Q, K, V, G, B = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, G, B))
    F, H, dk = Q.shape
    dv = V.shape[2]
    scale = 1.0 / np.sqrt(dk) if scale is None else scale
    out = np.full((F, H, dv), np.nan)
    begin, start, length, par = (plan[k] for k in ("seg_level_begin", "seg_start", "seg_len", "seg_parent"))
    final = {}
    for lv in range(len(begin) - 1):
        for i in range(begin[lv], begin[lv + 1]):
            assert par[i] < begin[lv], "a parent lies on an earlier level"
            S = final[par[i]] if par[i] >= 0 else np.zeros((H, dv, dk))
            for f in range(start[i], start[i] + length[i]):
                S, out[f] = _step(S, Q[f], K[f], V[f], G[f], B[f], scale)
            final[i] = S
    return out
