"""Oracle attention: every root-to-leaf sequence unpacked, fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The packed computation must reproduce, for every raw token, ordinary causal
attention over its own sequence with position ids 0..L-1: a token attends to
itself and its ancestors and to nothing else ("DAG packing", section "The
mask"; "Prefix Tree Packing in ART", section "Token-mixing layers": prefix
sharing is only valid because the layers are causal), with position ids equal
to tree depth, i.e. the token's index in its own sequence ("DAG packing",
section "Positions").  So the oracle does exactly that, sequence by sequence,
with no packing at all:

* gather the sequence's rows of the forwarded Q/K/V through ``token_index``
  (the map from raw tokens to forwarded positions, "TRL Tree Packing for
  AsyncGRPO", section "How tree packing works");
* RoPE in fp64 at positions 0..L-1 (half-split "rotate_half" pairing,
  angle p * base**(-2i/d)), then round the rotated Q, K to bfloat16 (the
  packed path stores its RoPE output in bf16);
* causal softmax attention in fp64 with scale 1/sqrt(d); natural-log LSE;
  grouped-query heads: query head h uses key/value head h // (Hq/Hkv).

Backward: the loss is sum over forwarded f and heads h of <dO[f,h], O[f,h]>.
Each forwarded position is owned by exactly one raw token (the lowest raw
index mapping to it), so each sequence runs the ordinary causal backward with
dO present only at the positions it owns, and the per-sequence gradients are
summed into forwarded positions (over the heads of a group for dK, dV).  The
gradient of the bf16 rounding is taken as identity; dQ and dK are given with
respect to the un-rotated inputs (inverse rotation applied).
"""
import numpy as np

from .bf16 import round_to_bf16


def rope(x, positions, base, inverse=False):
    """Rotate x [L, H, d] (fp64) by angle positions[l] * base**(-2i/d).

    Pair i < d/2 is (x_i, x_{i+d/2}): (a, b) -> (a cos t - b sin t, a sin t + b cos t);
    ``inverse`` rotates by -t.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = float(base) ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    theta = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    if inverse:
        theta = -theta
    c = np.cos(theta)[:, None, :]
    s = np.sin(theta)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def _kv_head(h, hq, hkv):
    return h // (hq // hkv)


def causal_attention(q, k, v, scale, chunk=512):
    """Causal attention over one sequence.  q [L,Hq,d], k/v [L,Hkv,d] fp64.

    Returns O [L, Hq, d] and LSE [Hq, L]."""
    L, hq, d = q.shape
    hkv = k.shape[1]
    out = np.zeros((L, hq, d))
    lse = np.zeros((hq, L))
    for h in range(hq):
        g = _kv_head(h, hq, hkv)
        for lo in range(0, L, chunk):
            hi = min(L, lo + chunk)
            s = (q[lo:hi, h, :] @ k[:hi, g, :].T) * scale           # [c, hi]
            mask = np.arange(hi)[None, :] > np.arange(lo, hi)[:, None]
            s[mask] = -np.inf
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            z = p.sum(axis=1, keepdims=True)
            out[lo:hi, h, :] = (p / z) @ v[:hi, g, :]
            lse[h, lo:hi] = (m + np.log(z))[:, 0]
    return out, lse


def causal_attention_backward(q, k, v, o, do, scale):
    """Gradients of sum(<do, O>) for one sequence, fp64, w.r.t. the (rotated) q, k and v."""
    L, hq, d = q.shape
    hkv = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    causal = np.tril(np.ones((L, L), dtype=bool))
    for h in range(hq):
        g = _kv_head(h, hq, hkv)
        s = (q[:, h, :] @ k[:, g, :].T) * scale
        s[~causal] = -np.inf
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        dv[:, g, :] += p.T @ do[:, h, :]
        dp = do[:, h, :] @ v[:, g, :].T
        rowdot = np.sum(do[:, h, :] * o[:, h, :], axis=1, keepdims=True)
        ds = p * (dp - rowdot)
        dq[:, h, :] = (ds @ k[:, g, :]) * scale
        dk[:, g, :] += (ds.T @ q[:, h, :]) * scale
    return dq, dk, dv


def _sequence_paths(plan):
    off = plan["seq_offsets"]
    ti = plan["token_index"]
    return [ti[off[s]:off[s + 1]] for s in range(len(off) - 1)]


def _rotated(x, path, base, round_rotated=True):
    y = rope(x[path], np.arange(len(path)), base)
    return round_to_bf16(y) if round_rotated else y


def forward(plan, Q, K, V, base, scale=None, round_rotated=True):
    """Packed-layout outputs computed from unpacked sequences.

    Q [F,Hq,d], K/V [F,Hkv,d] (any float dtype; bf16 values).  Returns
    (O_fwd [F,Hq,d], LSE_fwd [Hq,F], O_raw [R,Hq,d], LSE_raw [Hq,R]).
    Every forwarded position is computed once per sequence through it; the
    copies must agree (checked to 1e-12 relative), which is the statement that
    sharing a prefix changes nothing for a causal layer.
    """
    Q, K, V = (np.asarray(t, dtype=np.float64) for t in (Q, K, V))
    F, hq, d = Q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    R = int(plan["seq_offsets"][-1])
    o_fwd = np.full((F, hq, d), np.nan)
    lse_fwd = np.full((hq, F), np.nan)
    o_raw = np.zeros((R, hq, d))
    lse_raw = np.zeros((hq, R))
    off = plan["seq_offsets"]
    for s, path in enumerate(_sequence_paths(plan)):
        o, lse = causal_attention(_rotated(Q, path, base, round_rotated),
                                  _rotated(K, path, base, round_rotated), V[path], scale)
        o_raw[off[s]:off[s + 1]] = o
        lse_raw[:, off[s]:off[s + 1]] = lse
        seen = ~np.isnan(lse_fwd[0, path])
        if seen.any():
            ref = o_fwd[path[seen]]
            assert np.max(np.abs(ref - o[seen])) <= 1e-12 * max(1.0, np.max(np.abs(ref)))
        o_fwd[path] = o
        lse_fwd[:, path] = lse
    return o_fwd, lse_fwd, o_raw, lse_raw


def forward_rows(plan, Q_rows, K_rows, V_rows, raw, base, scale=None):
    """Outputs for selected raw tokens only (full-size sampling).

    ``raw``: raw token indices.  ``Q_rows(idx)``, ``K_rows(idx)``,
    ``V_rows(idx)`` return the [len(idx), H, d] rows of the forwarded tensors.
    Returns (O [n, Hq, d], LSE [Hq, n]) for the tokens in ``raw``."""
    off = plan["seq_offsets"]
    ti = plan["token_index"]
    outs, lses = [], []
    for r in raw:
        s = int(np.searchsorted(off, r, side="right") - 1)
        p = int(r - off[s])
        path = ti[off[s]:off[s] + p + 1]
        q = round_to_bf16(rope(Q_rows(path[-1:]), [p], base))
        k = round_to_bf16(rope(K_rows(path), np.arange(p + 1), base))
        v = np.asarray(V_rows(path), dtype=np.float64)
        hq, d = q.shape[1], q.shape[2]
        hkv = k.shape[1]
        sc = 1.0 / np.sqrt(d) if scale is None else scale
        o = np.zeros((hq, d))
        lse = np.zeros(hq)
        for h in range(hq):
            g = _kv_head(h, hq, hkv)
            sv = (k[:, g, :] @ q[0, h, :]) * sc
            m = sv.max()
            w = np.exp(sv - m)
            z = w.sum()
            o[h] = (w / z) @ v[:, g, :]
            lse[h] = m + np.log(z)
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses, axis=1)


def backward(plan, Q, K, V, dO, base, scale=None, round_rotated=True):
    """Gradients (dQ, dK, dV) in forwarded layout of sum <dO, O_fwd>.

    dQ, dK are with respect to the un-rotated Q, K.  ``round_rotated=False``
    skips the bf16 rounding of the rotated Q, K (used to check the gradients
    against finite differences of ``forward``, which rounding would break)."""
    Q, K, V, dO = (np.asarray(t, dtype=np.float64) for t in (Q, K, V, dO))
    F, hq, d = Q.shape
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    off = plan["seq_offsets"]
    src = plan["fwd_src"]
    for s, path in enumerate(_sequence_paths(plan)):
        L = len(path)
        pos = np.arange(L)
        q = _rotated(Q, path, base, round_rotated)
        k = _rotated(K, path, base, round_rotated)
        v = V[path]
        o, _ = causal_attention(q, k, v, scale)
        owned = src[path] == off[s] + pos
        do = np.where(owned[:, None, None], dO[path], 0.0)
        dq, dk, dv = causal_attention_backward(q, k, v, o, do, scale)
        np.add.at(dQ, path, rope(dq, pos, base, inverse=True))
        np.add.at(dK, path, rope(dk, pos, base, inverse=True))
        np.add.at(dV, path, dv)
    return dQ, dK, dV


def _path_rows(plan, r):
    off = plan["seq_offsets"]
    s = int(np.searchsorted(off, r, side="right") - 1)
    p = int(r - off[s])
    return s, p, plan["token_index"][off[s]:off[s] + p + 1]


def backward_rows_q(plan, Q_rows, K_rows, V_rows, dO_rows, raw, base, scale=None):
    """dQ (w.r.t. un-rotated Q) at the forwarded positions of the raw tokens
    ``raw``.  A query's own row is the only place its Q enters the loss, so
    dQ[f] needs only f's own softmax row: P_j, dP_j = dO_f.v_j, D = dO_f.O_f,
    dS_j = P_j (dP_j - D), dQ_rot = scale sum_j dS_j k_j, then the inverse
    rotation at f's position.  Returns [n, Hq, d]."""
    out = []
    for r in raw:
        _, p, path = _path_rows(plan, r)
        q = round_to_bf16(rope(Q_rows(path[-1:]), [p], base))
        k = round_to_bf16(rope(K_rows(path), np.arange(p + 1), base))
        v = np.asarray(V_rows(path), dtype=np.float64)
        do = np.asarray(dO_rows(path[-1:]), dtype=np.float64)[0]
        hq, d = q.shape[1], q.shape[2]
        hkv = k.shape[1]
        sc = 1.0 / np.sqrt(d) if scale is None else scale
        dq = np.zeros((1, hq, d))
        for h in range(hq):
            g = _kv_head(h, hq, hkv)
            s = (k[:, g, :] @ q[0, h, :]) * sc
            w = np.exp(s - s.max())
            pr = w / w.sum()
            o = pr @ v[:, g, :]
            dp = v[:, g, :] @ do[h]
            ds = pr * (dp - do[h] @ o)
            dq[0, h] = sc * (ds @ k[:, g, :])
        out.append(rope(dq, [p], base, inverse=True)[0])
    return np.stack(out)


def backward_rows_kv(plan, Q_rows, K_rows, V_rows, dO_rows, fwd, base, scale=None):
    """dK (w.r.t. un-rotated K) and dV at forwarded key positions ``fwd``.

    Key j receives gradient from every forwarded query that sees it (the
    positions of its subtree).  Each such query i is taken once, through the
    sequence owning it (its lowest raw index), with its full softmax row over
    that sequence's prefix.  Returns ([n, Hkv, d], [n, Hkv, d])."""
    off = plan["seq_offsets"]
    ti = plan["token_index"]
    src = plan["fwd_src"]
    se = plan["subtree_end"]
    dks, dvs = [], []
    for j in fwd:
        pj = int(plan["depth"][j])
        dk_acc = None
        dv_acc = None
        for i in range(int(j), int(se[j])):
            r = int(src[i])
            s, p, path = _path_rows(plan, r)
            if pj > p or path[pj] != j:
                continue   # j is not on i's path (a later subtree of the row)
            q = round_to_bf16(rope(Q_rows(path[-1:]), [p], base))
            k = round_to_bf16(rope(K_rows(path), np.arange(p + 1), base))
            v = np.asarray(V_rows(path), dtype=np.float64)
            do = np.asarray(dO_rows(path[-1:]), dtype=np.float64)[0]
            hq, d = q.shape[1], q.shape[2]
            hkv = k.shape[1]
            sc = 1.0 / np.sqrt(d) if scale is None else scale
            if dk_acc is None:
                dk_acc = np.zeros((hkv, d))
                dv_acc = np.zeros((hkv, d))
            for h in range(hq):
                g = _kv_head(h, hq, hkv)
                sv = (k[:, g, :] @ q[0, h, :]) * sc
                w = np.exp(sv - sv.max())
                pr = w / w.sum()
                o = pr @ v[:, g, :]
                dp = v[:, g, :] @ do[h]
                ds = pr * (dp - do[h] @ o)
                dv_acc[g] += pr[pj] * do[h]
                dk_acc[g] += sc * ds[pj] * q[0, h]
        dks.append(rope(dk_acc[None], [pj], base, inverse=True)[0])
        dvs.append(dv_acc)
    return np.stack(dks), np.stack(dvs)


def backward_keys(plan, Q_rows, K_rows, V_rows, dO_rows, fwd, base, scale=None, chunk=256):
    """dK (w.r.t. un-rotated K) and dV at forwarded key positions ``fwd``, the
    same quantities as ``backward_rows_kv`` for keys with long subtrees.

    The queries that see key j are the positions of its subtree [j,
    subtree_end[j]); each is taken through the sequence that owns it, with its
    full softmax row over that sequence's prefix.  The queries one sequence
    owns inside the subtree are positions of that sequence, so they are taken
    together: the sequence's prefix is rotated once and each head's scores of
    those queries are one matrix product (``chunk`` query rows at a time,
    keys after a query's own position masked).  Returns ([n, Hkv, d],
    [n, Hkv, d])."""
    off = plan["seq_offsets"]
    ti = plan["token_index"]
    src = plan["fwd_src"]
    se = plan["subtree_end"]
    depth = plan["depth"]
    dks, dvs = [], []
    for j in fwd:
        j = int(j)
        pj = int(depth[j])
        qs = np.arange(j, int(se[j]))
        seq_of = np.searchsorted(off, src[qs], side="right") - 1
        dk_acc = dv_acc = None
        for s in np.unique(seq_of):
            mine = qs[seq_of == s]
            pos = depth[mine].astype(np.int64)        # positions of those queries in sequence s
            path = ti[off[s]:off[s] + int(pos.max()) + 1]
            if path[pj] != j:
                continue
            q = round_to_bf16(rope(Q_rows(path[pos]), pos, base))
            k = round_to_bf16(rope(K_rows(path), np.arange(len(path)), base))
            v = np.asarray(V_rows(path), dtype=np.float64)
            do = np.asarray(dO_rows(path[pos]), dtype=np.float64)
            hq, d = q.shape[1], q.shape[2]
            hkv = k.shape[1]
            sc = 1.0 / np.sqrt(d) if scale is None else scale
            if dk_acc is None:
                dk_acc = np.zeros((hkv, d))
                dv_acc = np.zeros((hkv, d))
            for lo in range(0, len(pos), chunk):
                hi = min(len(pos), lo + chunk)
                masked = np.arange(len(path))[None, :] > pos[lo:hi, None]
                for h in range(hq):
                    g = _kv_head(h, hq, hkv)
                    sv = (q[lo:hi, h, :] @ k[:, g, :].T) * sc
                    sv[masked] = -np.inf
                    w = np.exp(sv - sv.max(axis=1, keepdims=True))
                    pr = w / w.sum(axis=1, keepdims=True)
                    o = pr @ v[:, g, :]
                    dp_j = do[lo:hi, h, :] @ v[pj, g, :]
                    ds_j = pr[:, pj] * (dp_j - np.sum(do[lo:hi, h, :] * o, axis=1))
                    dv_acc[g] += pr[:, pj] @ do[lo:hi, h, :]
                    dk_acc[g] += sc * (ds_j @ q[lo:hi, h, :])
        dks.append(rope(dk_acc[None], [pj], base, inverse=True)[0])
        dvs.append(dv_acc)
    return np.stack(dks), np.stack(dvs)
