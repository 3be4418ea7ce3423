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


# ---------------------------------------------------------------- gradients
# The packed layer is a function of the packed inputs, and its output at a
# position f is the output of any sequence through f (they agree: a causal
# layer sees only f's own path).  Its vector-Jacobian product with dO is
# therefore the sum over f of the gradient of <dO[f], out(f)> taken through
# ONE sequence containing f (the first, as ``_assign`` keeps), with that
# sequence's inputs read out of the packed arrays -- so the gradients of a
# shared position's inputs, and of a forked state, are summed over every
# branch below it, as the pages have autograd do for the broadcast initial
# state of each child ("Prefix Tree Packing in ART", section "Token-mixing
# layers").  The per-sequence forwards below restate ``conv`` and ``_step``
# in torch fp64 so that autograd can differentiate them; the tests pin the
# gradients to central differences of the NumPy forwards above.

def _torch():
    import torch
    return torch


def _conv_seq_t(x, w):
    """``conv`` for one sequence in torch: x [L, C], w [C, W] -> y [L, C]."""
    torch = _torch()
    L, C = x.shape
    W = w.shape[1]
    xs = torch.cat([torch.zeros((W - 1, C), dtype=x.dtype), x], dim=0)
    acc = sum(w[:, j] * xs[j:j + L] for j in range(W))
    return acc * torch.sigmoid(acc)


def _delta_seq_t(q, k, v, g, b, scale):
    """``delta_rule`` for one sequence in torch from S = 0: q, k [L, H, dk],
    v [L, H, dv], g, b [L, H] -> o [L, H, dv]."""
    torch = _torch()
    k = k / torch.linalg.norm(k, dim=-1, keepdim=True)
    q = scale * q / torch.linalg.norm(q, dim=-1, keepdim=True)
    L, H, dk = k.shape
    S = torch.zeros((H, v.shape[2], dk), dtype=k.dtype)
    out = []
    for t in range(L):
        a = torch.exp(g[t])[:, None, None]
        bt = b[t][:, None, None]
        Sk = torch.einsum("hec,hc->he", S, k[t])
        S = a * (S - bt * torch.einsum("he,hc->hec", Sk, k[t])) + bt * torch.einsum("he,hc->hec", v[t], k[t])
        out.append(torch.einsum("hec,hc->he", S, q[t]))
    return torch.stack(out)


def _vjp(plan, per_pos, params, dout, fn):
    """Gradients of sum_f <dout[f], out[f]> w.r.t. ``per_pos`` (packed arrays
    [F, ...]) and ``params`` (shared by every position); ``fn(*rows,
    *params)`` is one sequence's forward on its gathered rows."""
    torch = _torch()
    dout = np.asarray(dout, dtype=np.float64)
    leaves = [torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True) for a in per_pos]
    pleaves = [torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True) for a in params]
    dO = torch.tensor(dout)
    seen = np.zeros(plan["n_fwd"], dtype=bool)
    loss = torch.zeros((), dtype=torch.float64)
    for path in _paths(plan):
        own = np.nonzero(~seen[path])[0]
        seen[path] = True
        if len(own) == 0:
            continue
        pt = torch.as_tensor(np.asarray(path, dtype=np.int64))
        out = fn(*[l[pt] for l in leaves], *pleaves)
        loss = loss + (out[torch.as_tensor(own)] * dO[torch.as_tensor(np.asarray(path[own], dtype=np.int64))]).sum()
    loss.backward()
    return [np.zeros(l.shape) if l.grad is None else l.grad.numpy() for l in leaves + pleaves]


def conv_bwd(plan, X, w, dY):
    """Gradients of ``conv``: returns (dX [F, C], dw [C, W]) for the output
    gradient dY [F, C]."""
    dX, dw = _vjp(plan, [X], [w], dY, _conv_seq_t)
    return dX, dw


def delta_rule_bwd(plan, Q, K, V, G, B, dO, scale=None):
    """Gradients of ``delta_rule`` (w.r.t. the un-normalised q, k; v; the log
    decay g; beta) for the output gradient dO [F, H, dv]: returns
    (dQ, dK, dV, dG, dB)."""
    dk = np.asarray(Q).shape[2]
    scale = 1.0 / np.sqrt(dk) if scale is None else scale
    return tuple(_vjp(plan, [Q, K, V, G, B], [], dO, lambda q, k, v, g, b: _delta_seq_t(q, k, v, g, b, scale)))


def _prefix(plan, r):
    off = plan["seq_offsets"]
    s = int(np.searchsorted(off, r, side="right") - 1)
    return plan["token_index"][off[s]:r + 1]


def delta_rule_bwd_rows(plan, rows, picks, scale=None):
    """The gradients for an output gradient that is zero except at the
    forwarded positions of a few raw tokens: ``picks`` is a list of (raw
    token r, dO row [H, dv]) with distinct forwarded positions; ``rows(key,
    idx)`` returns rows ``idx`` of input ``key`` in ("q", "k", "v", "g",
    "b").  Each pick's sequence prefix is run from S = 0.  Returns (pos,
    (dQ, dK, dV, dG, dB)) with the gradient rows at the sorted forwarded
    positions ``pos`` (every other row's gradient is zero)."""
    torch = _torch()
    ti = plan["token_index"]
    assert len({int(ti[r]) for r, _ in picks}) == len(picks), "picks share a forwarded position"
    paths = [_prefix(plan, r) for r, _ in picks]
    pos = np.unique(np.concatenate(paths))
    leaves = [torch.tensor(np.asarray(rows(key, pos), dtype=np.float64), requires_grad=True)
              for key in ("q", "k", "v", "g", "b")]
    dk = leaves[0].shape[2]
    sc = 1.0 / np.sqrt(dk) if scale is None else scale
    loss = torch.zeros((), dtype=torch.float64)
    for path, (_, d) in zip(paths, picks):
        at = torch.as_tensor(np.searchsorted(pos, path))
        o = _delta_seq_t(*[l[at] for l in leaves], sc)
        loss = loss + (o[-1] * torch.tensor(np.asarray(d, dtype=np.float64))).sum()
    loss.backward()
    return pos, tuple(l.grad.numpy() for l in leaves)


def conv_bwd_rows(plan, rows, w, picks):
    """``conv_bwd`` for an output gradient that is zero except at the
    forwarded positions of a few raw tokens: ``picks`` is a list of (raw
    token r, dY row [C]) with distinct forwarded positions; ``rows(idx)``
    returns rows ``idx`` of x.  Returns (pos, dX rows at pos, dw)."""
    torch = _torch()
    ti = plan["token_index"]
    assert len({int(ti[r]) for r, _ in picks}) == len(picks), "picks share a forwarded position"
    W = np.asarray(w).shape[1]
    paths = [_prefix(plan, r)[-W:] for r, _ in picks]
    pos = np.unique(np.concatenate(paths))
    x = torch.tensor(np.asarray(rows(pos), dtype=np.float64), requires_grad=True)
    wt = torch.tensor(np.asarray(w, dtype=np.float64), requires_grad=True)
    loss = torch.zeros((), dtype=torch.float64)
    for path, (r, d) in zip(paths, picks):
        # the window of the last position: its own path, zero above a root
        # (a prefix shorter than W starts at the root)
        y = _conv_seq_t(x[torch.as_tensor(np.searchsorted(pos, path))], wt)
        loss = loss + (y[-1] * torch.tensor(np.asarray(d, dtype=np.float64))).sum()
    loss.backward()
    return pos, x.grad.numpy(), wt.grad.numpy()
