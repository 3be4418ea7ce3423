"""Oracle packing plan: prefix tree, row placement and depth-first layout.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Plain Python with
NumPy used only to compare token runs.  Each step follows a passage of the
pages; where the pages are silent, the reading taken is stated at the step
it affects.

Steps and the passages they follow
----------------------------------
1. ``position_symbols``   -- what makes two positions the same forwarded
   position.  A position is merged with another only if the model would face
   the same input *and* the same target there: the last common token before a
   fork is therefore kept once per branch ("Prefix Tree Packing in ART",
   section "The tree", the off-by-one note on the duplicated join token;
   "DAG packing", section "The walk": the last common node is copied once per
   child because each copy predicts a different next token).  Positions whose
   prediction carries no loss (untrained) are merged without regard to the
   target, which is ART's accounting of its 32-rollout example ("Prefix Tree
   Packing in ART", section "Does it actually help?": the 4,096-token root is
   paid once per row, the final prompt token stays on each rollout leaf).
2. ``build_tree``         -- the recursive walk of "Prefix Tree Packing in
   ART", section "The tree": take the longest run every active sequence
   agrees on, emit it once, split the rest by the next symbol and recurse;
   plus the minimum shared-segment length of the same section.
3. ``place_best_fit_decreasing`` / ``place_next_fit`` -- "Prefix Tree Packing
   in ART", section "Bin packing, with a twist" (marginal cost of a leaf =
   length of the path segments the row does not hold yet; groups ordered by
   their most expensive leaf; each leaf to the row it leaves least room in),
   and the in-order fill of sections "One tree, not one per group" and "Does
   it actually help?".  ``place_one_row_per_group`` has no counterpart on the
   pages: one row per placement group, rows in increasing group id (how a
   data-parallel rank rebuilds the rows it owns of a larger batch); pinned by
   replanning a best-fit-decreasing plan with each sequence's row as its group,
   which must give back the same rows.
4. ``layout_rows``        -- depth-first layout ("DAG packing", section "The
   walk"; "TRL Tree Packing for AsyncGRPO", section "How tree packing
   works"), positions = tree depth ("DAG packing", section "Positions"),
   token_index mapping every raw token to its forwarded position (TRL page,
   same section).
"""
import sys
from dataclasses import dataclass, field
from functools import cmp_to_key

import numpy as np

NONE = -2   # target field of an untrained position: no target in the key
EOS = -1    # target of the last position of a sequence


# --------------------------------------------------------------------------
# 1. position symbols
# --------------------------------------------------------------------------
def position_symbols(tokens, trained=None):
    """Per-position symbols (token, trained flag, target) of one sequence.

    Two sequences' positions p are merged iff the symbols at 0..p agree.  The
    target of position p is the next token (EOS at the end) when p carries a
    loss; for an untrained position it is NONE, except at the last position,
    where EOS is kept so that every sequence ends in a leaf of its own.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    L = len(tokens)
    flags = np.ones(L, dtype=np.int64) if trained is None else np.asarray(trained, dtype=np.int64)
    nxt = np.empty(L, dtype=np.int64)
    nxt[:-1] = tokens[1:]
    nxt[-1] = EOS
    target = np.where(flags != 0, nxt, NONE)
    target[-1] = EOS
    return np.stack([tokens, flags, target], axis=0)  # [3, L]


def _first_difference(a, b, start):
    """Smallest p >= start where symbol columns of a and b differ (or None)."""
    n = min(a.shape[1], b.shape[1])
    if start >= n:
        return None if a.shape[1] == b.shape[1] else n
    neq = np.any(a[:, start:n] != b[:, start:n], axis=0)
    hit = np.flatnonzero(neq)
    if len(hit):
        return start + int(hit[0])
    return None if a.shape[1] == b.shape[1] else n


def compare_symbol_sequences(a, b):
    """Lexicographic order of two symbol sequences (token, flag, target)."""
    p = _first_difference(a, b, 0)
    if p is None:
        return 0
    if p >= a.shape[1]:
        return -1
    if p >= b.shape[1]:
        return 1
    ta, tb = tuple(a[:, p]), tuple(b[:, p])
    return -1 if ta < tb else 1


# --------------------------------------------------------------------------
# 2. the tree
# --------------------------------------------------------------------------
@dataclass
class Segment:
    id: int
    parent: int          # -1 for a root
    start: int           # depth of the first position
    end: int             # one past the depth of the last position
    is_leaf: bool
    children: list = field(default_factory=list)


@dataclass
class Leaf:
    id: int
    members: list        # indices of the (identical) sequences ending here
    path: list           # [(segment id, length)] from the root to this leaf

    @property
    def representative(self):
        return min(self.members)

    @property
    def standalone_cost(self):
        # cost of the leaf in an empty row: its full, unshared length
        return sum(length for _, length in self.path)


def build_tree(symbols, min_shared):
    """Segments and leaves of the prefix tree over ``symbols`` (list of [3, L]).

    The walk keeps, for a set of sequences that agree on everything before
    ``seg_start``, the depth where the pending (not yet emitted) run began.
    It finds the first depth ``end`` where the set disagrees.  A run of at
    least ``min_shared`` positions is emitted once as a shared segment; a
    shorter one is not shared: it is carried down and becomes the head of each
    child's segment.  The set is then split by the symbol at ``end`` (children
    in increasing symbol order) and each part is walked again.  A set of
    identical sequences is a leaf and is always emitted, whatever its length.
    """
    segments, leaves = [], []
    min_len = max(int(min_shared), 1)
    sys.setrecursionlimit(max(sys.getrecursionlimit(), 4 * len(symbols) + 1000))

    def emit(parent, start, end, is_leaf):
        seg = Segment(len(segments), parent, start, end, is_leaf)
        segments.append(seg)
        if parent >= 0:
            segments[parent].children.append(seg.id)
        return seg.id

    def path_to(seg_id):
        out = []
        while seg_id >= 0:
            s = segments[seg_id]
            out.append((s.id, s.end - s.start))
            seg_id = s.parent
        return out[::-1]

    def walk(active, seg_start, run_start, parent):
        first = symbols[active[0]]
        end = None
        for other in active[1:]:
            p = _first_difference(first, symbols[other], run_start)
            if p is not None and (end is None or p < end):
                end = p
        if end is None:  # all identical: a leaf
            sid = emit(parent, seg_start, first.shape[1], True)
            leaves.append(Leaf(len(leaves), sorted(active), path_to(sid)))
            return
        if end > seg_start and end - seg_start >= min_len:
            parent = emit(parent, seg_start, end, False)
            seg_start = end
        parts = {}
        for i in active:
            parts.setdefault(tuple(int(v) for v in symbols[i][:, end]), []).append(i)
        for key in sorted(parts):
            walk(parts[key], seg_start, end, parent)

    # one walk over all sequences: roots are the first split (a forest)
    walk(list(range(len(symbols))), 0, 0, -1)
    return segments, leaves


# --------------------------------------------------------------------------
# 3. placement
# --------------------------------------------------------------------------
class _Row:
    """One fixed-capacity row: the set of tree segments it already holds."""

    def __init__(self):
        self.segments = set()
        self.load = 0
        self.leaves = []

    def marginal_cost(self, leaf):
        return sum(length for seg, length in leaf.path if seg not in self.segments)

    def take(self, leaf):
        self.load += self.marginal_cost(leaf)
        self.segments.update(seg for seg, _ in leaf.path)
        self.leaves.append(leaf)


def place_best_fit_decreasing(groups, capacity):
    """Best-fit decreasing over marginal cost.

    ``groups``: list of lists of leaves, in first-appearance order.  Groups are
    visited by decreasing standalone cost of their most expensive leaf (a
    stable sort, so equal groups keep their order); each leaf goes to the
    existing row whose load after taking it leaves the least room, earliest row
    on ties; a new row is opened when none fits.
    """
    order = sorted(range(len(groups)),
                   key=lambda g: max(leaf.standalone_cost for leaf in groups[g]),
                   reverse=True)
    rows = []
    for g in order:
        for leaf in groups[g]:
            best, best_room = None, None
            for row in rows:
                load = row.load + row.marginal_cost(leaf)
                if load <= capacity and (best_room is None or capacity - load < best_room):
                    best, best_room = row, capacity - load
            if best is None:
                best = _Row()
                rows.append(best)
            best.take(leaf)
    return rows


def place_next_fit(groups, capacity):
    """In-order filling: one open row; a new one whenever the next leaf does not fit."""
    rows = []
    for group in groups:
        for leaf in group:
            if not rows or rows[-1].load + rows[-1].marginal_cost(leaf) > capacity:
                rows.append(_Row())
            rows[-1].take(leaf)
    return rows


def place_one_row_per_group(groups, keys, capacity):
    """One row per placement group, rows in increasing group id (no
    counterpart on the pages: it lets a data-parallel rank that owns some
    rows of a larger batch plan its sequences with their global row index as
    the group and get exactly those rows back).  A group that does not fit in
    one row is an error."""
    rows = []
    for g in sorted(range(len(groups)), key=lambda g: keys[g]):
        row = _Row()
        for leaf in groups[g]:
            row.take(leaf)
        if row.load > capacity:
            raise PlanError("group larger than a row")
        rows.append(row)
    return rows


# --------------------------------------------------------------------------
# 4. layout
# --------------------------------------------------------------------------
class PlanError(ValueError):
    pass


def plan(sequences, trained=None, group_ids=None, min_shared=64,
         row_capacity=65536, placement="bfd"):
    """Full oracle plan.  ``sequences``: list of int token arrays (ids >= 0).

    Returns a dict of NumPy arrays and scalars:
      row_offsets [n_rows+1], row_of_seq [n], fwd_token [F], fwd_src [F],
      parent [F], depth [F], token_index [R], subtree_end [F], row_loads,
      seq_offsets [n+1], plus the tree (segments, leaves) for inspection.
    """
    n = len(sequences)
    if n == 0:
        raise PlanError("no sequences")
    seqs = [np.asarray(s, dtype=np.int64) for s in sequences]
    if any(len(s) == 0 for s in seqs):
        raise PlanError("empty sequence")
    flags = [None] * n if trained is None else [np.asarray(t) for t in trained]
    symbols = [position_symbols(s, f) for s, f in zip(seqs, flags)]
    segments, leaves = build_tree(symbols, min_shared)

    # groups: explicit ids, else the tree family (root segment) of each leaf
    def group_of(leaf):
        if group_ids is not None:
            return int(group_ids[leaf.representative])
        return leaf.path[0][0]
    leaves_in_input_order = sorted(leaves, key=lambda lf: lf.representative)
    groups, index, keys = [], {}, []
    for leaf in leaves_in_input_order:
        g = group_of(leaf)
        if g not in index:
            index[g] = len(groups)
            groups.append([])
            keys.append(g)
        groups[index[g]].append(leaf)

    for leaf in leaves:
        if leaf.standalone_cost > row_capacity:
            raise PlanError("sequence longer than the row capacity")
    if placement == "bfd":
        rows = place_best_fit_decreasing(groups, row_capacity)
    elif placement == "next_fit":
        rows = place_next_fit(groups, row_capacity)
    elif placement == "groups":
        rows = place_one_row_per_group(groups, keys, row_capacity)
    else:
        raise PlanError("unknown placement")

    seq_offsets = np.zeros(n + 1, dtype=np.int64)
    seq_offsets[1:] = np.cumsum([len(s) for s in seqs])
    R = int(seq_offsets[-1])

    fwd_token, depth, parent = [], [], []
    token_index = np.full(R, -1, dtype=np.int64)
    row_of_seq = np.full(n, -1, dtype=np.int64)
    row_offsets = [0]
    order_key = cmp_to_key(lambda a, b: compare_symbol_sequences(symbols[a.representative],
                                                                 symbols[b.representative]))
    instances = []                       # (first position, length, parent instance) in placement order
    for r, row in enumerate(rows):
        placed = {}                      # segment id -> forwarded index of its first position
        placed_inst = {}                 # segment id -> its instance (the segment placed in this row)
        for leaf in sorted(row.leaves, key=order_key):
            rep = seqs[leaf.representative]
            prev_seg = -1
            for seg_id, _ in leaf.path:
                seg = segments[seg_id]
                if seg_id not in placed:
                    f0 = len(depth)
                    placed[seg_id] = f0
                    placed_inst[seg_id] = len(instances)
                    instances.append((f0, seg.end - seg.start, placed_inst[prev_seg] if prev_seg >= 0 else -1))
                    depth.extend(range(seg.start, seg.end))
                    fwd_token.extend(int(t) for t in rep[seg.start:seg.end])
                    if prev_seg >= 0:
                        ps = segments[prev_seg]
                        parent.append(placed[prev_seg] + (ps.end - 1 - ps.start))
                    else:
                        parent.append(-1)
                    parent.extend(range(f0, f0 + seg.end - seg.start - 1))
                prev_seg = seg_id
            for s in leaf.members:
                row_of_seq[s] = r
                for seg_id, _ in leaf.path:
                    seg = segments[seg_id]
                    lo = seq_offsets[s] + seg.start
                    token_index[lo:lo + seg.end - seg.start] = placed[seg_id] + np.arange(seg.end - seg.start)
        row_offsets.append(len(depth))

    F = len(depth)
    # lowest raw index of each forwarded position: scanning raw indices from
    # the top, the last write to each position is its lowest raw index
    fwd_src = np.full(F, R, dtype=np.int64)
    fwd_src[token_index[::-1]] = np.arange(R - 1, -1, -1)
    parent = np.asarray(parent, dtype=np.int64)
    subtree_end = np.arange(1, F + 1, dtype=np.int64)
    for f in range(F - 1, -1, -1):
        if parent[f] >= 0 and subtree_end[f] > subtree_end[parent[f]]:
            subtree_end[parent[f]] = subtree_end[f]
    depth = np.asarray(depth, dtype=np.int64)
    rows_arr = np.asarray(row_offsets, dtype=np.int64)
    seg_levels = segment_levels(instances)
    forks = sum(1 for s in segments if len(s.children) >= 2)
    return {
        "row_offsets": rows_arr,
        "row_of_seq": row_of_seq,
        "fwd_token": np.asarray(fwd_token, dtype=np.int64),
        "fwd_src": fwd_src,
        "parent": parent,
        "depth": depth,
        "token_index": token_index,
        "subtree_end": subtree_end,
        "row_loads": [row.load for row in rows],
        "seq_offsets": seq_offsets,
        "n_rows": len(rows),
        "n_fwd": F,
        "n_raw": R,
        "n_segments": len(segments),
        "packing_ratio": R / F,
        "row_fill_frac": F / (len(rows) * row_capacity),
        "fork_frac": forks / len(segments),
        "useful_pairs": int(np.sum(depth + 1)),
        "segments": segments,
        "leaves": leaves,
        **seg_levels,
    }


def segment_levels(instances):
    """Segment instances (a segment placed in one row) grouped by tree level,
    the order in which a recurrent layer threads its state through the tree
    ("Prefix Tree Packing in ART", section "Token-mixing layers": the GDN
    planner walks the tree depth by depth, every segment of a depth across
    all rows in one pass; a child starts from its parent's final state, a
    root from zero).  ``instances``: (first position, length, parent
    instance or -1) in placement order, parents before children.  Level = the
    number of ancestor instances; within a level, placement order.  Returns
    level_begin [n_levels+1] and seg_start / seg_len / seg_parent [n] in that
    order, parents given as indices into it, and seg_off [n]: the summed
    length of the instances before it on its level."""
    n = len(instances)
    level = [0] * n
    for i, (_, _, par) in enumerate(instances):
        level[i] = 0 if par < 0 else level[par] + 1
    order = sorted(range(n), key=lambda i: (level[i], i))
    new_index = {old: new for new, old in enumerate(order)}
    n_levels = (max(level) + 1) if n else 0
    begin = [0] * (n_levels + 1)
    for lv in level:
        begin[lv + 1] += 1
    for lv in range(n_levels):
        begin[lv + 1] += begin[lv]
    off = [0] * n
    for lv in range(n_levels):
        acc = 0
        for j in range(begin[lv], begin[lv + 1]):
            off[j] = acc
            acc += instances[order[j]][1]
    return {
        "seg_off": np.asarray(off, dtype=np.int64),
        "seg_level_begin": np.asarray(begin, dtype=np.int64),
        "seg_start": np.asarray([instances[i][0] for i in order], dtype=np.int64),
        "seg_len": np.asarray([instances[i][1] for i in order], dtype=np.int64),
        "seg_parent": np.asarray([new_index[instances[i][2]] if instances[i][2] >= 0 else -1 for i in order],
                                 dtype=np.int64),
    }


def visible_by_parent_walk(parent, i):
    """Keys visible to query i: i itself and every ancestor reached through parent.

    The mask of "DAG packing", section "The mask": a token attends to itself
    and the positions on its own root-to-leaf path, nothing else.
    """
    out = []
    while i >= 0:
        out.append(i)
        i = parent[i]
    return sorted(out)
