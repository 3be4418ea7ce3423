"""Seeded synthetic workloads shaped like the pages' batches.

Shared by the tests (oracle side and library side alike) and by ``bench.py``.
It holds no arithmetic of the method: it only draws token sequences with an
explicit sharing structure and names the attention shapes.  Token ids are
uniform in [0, 32000) from NumPy's PCG64 seeded with ``1000*c`` for workload
c.  Shared parts are literally the same token arrays; at every fork the
children's first tokens are redrawn until distinct (and unrelated groups'
first tokens are distinct), so the realised tree is exactly the one described.
Q/K/V/dO values come from ``workloads.rng`` (counter-based) with seeds
``1000*c + 1..4``.

Workloads (names used by tests and bench):
  tiny         4 sequences sharing a 128-token prefix, sequences 1-2 sharing a
               further 64-token run, tails of 64-128 tokens; min shared 16;
               rows of 512; 1 head, head_dim 64; RoPE base 1e4.
  tiny_fit     the same sequences in rows of 1024 (one row).
  grpo         512-token system prompt shared by 64 sequences, 8 prompts of
               1024 tokens, 8 completions each of 256-2048 tokens; groups =
               prompt; min shared 64; rows of 16384; Hq 16 / Hkv 8 / d 128;
               RoPE base 1e6.
  agentic      4 groups: 20000-token shared history, 8 rollouts of 4 turns of
               500 tokens, pairs of rollouts sharing turns 1-2; rows of
               32768; 16/8/128.
  sweep_<rho>  one row of exactly 32768 forwarded tokens from 4 rollouts of T
               raw tokens sharing a P-token prefix (4T - 3P + 3 = 32768, the
               join token counted once per branch); rho = 4T/32768 in
               {1.00, 1.45, 2.0, 2.8, 3.56}; rho 1.00 = 4 unrelated rollouts
               of 8192.  ``sweep_<rho>_seqpack``: the same raw tokens with no
               sharing (min shared larger than any run).
  deep         root of 4096 tokens, then segments of 256-1024 tokens with a
               branching factor drawn from {1,2,3} at every segment end, down
               to depth 24000, exactly 128 leaves; one group; min shared 64;
               rows of 65536; Hq 32 / Hkv 8 / d 128; forward and backward.
  deep_small   the same construction scaled down (root 512, segments
               96-384, depth 3000, 16 leaves, rows of 8192, Hq 8 / Hkv 2).
"""
from dataclasses import dataclass
from typing import List, Optional

import numpy as np

VOCAB = 32000
SWEEP_RHOS = (1.00, 1.45, 2.0, 2.8, 3.56)


@dataclass
class Workload:
    name: str
    sequences: List[np.ndarray]
    group_ids: Optional[np.ndarray]
    trained: Optional[List[np.ndarray]]
    min_shared: int
    row_capacity: int
    n_heads_q: int
    n_heads_kv: int
    head_dim: int
    rope_base: float
    seed_base: int
    backward: bool = False
    placement: str = "bfd"

    @property
    def n_raw(self):
        return int(sum(len(s) for s in self.sequences))

    def flat_tokens(self):
        return np.concatenate(self.sequences).astype(np.int32)

    def seq_offsets(self):
        off = np.zeros(len(self.sequences) + 1, dtype=np.int64)
        off[1:] = np.cumsum([len(s) for s in self.sequences])
        return off

    @property
    def seeds(self):
        b = self.seed_base
        return {"q": b + 1, "k": b + 2, "v": b + 3, "do": b + 4}


class _Tokens:
    def __init__(self, seed):
        self.rng = np.random.Generator(np.random.PCG64(seed))

    def draw(self, n, avoid_first=()):
        t = self.rng.integers(0, VOCAB, size=n, dtype=np.int64)
        while n and int(t[0]) in avoid_first:
            t[0] = self.rng.integers(0, VOCAB)
        return t

    def siblings(self, lengths, avoid_first=()):
        """Token arrays for sibling runs whose first tokens are all distinct."""
        used = set(avoid_first)
        out = []
        for n in lengths:
            t = self.draw(n, used)
            used.add(int(t[0]))
            out.append(t)
        return out


def tiny(capacity=512):
    tk = _Tokens(1000)
    shared = tk.draw(128)
    tails = [int(x) for x in tk.rng.integers(64, 129, size=4)]
    t0, run12, t3 = tk.siblings([tails[0], 64, tails[3]])
    t1, t2 = tk.siblings([tails[1], tails[2]])
    seqs = [np.concatenate(p) for p in ([shared, t0], [shared, run12, t1],
                                         [shared, run12, t2], [shared, t3])]
    return Workload("tiny" if capacity == 512 else "tiny_fit", seqs, np.zeros(4, np.int32), None,
                    16, capacity, 1, 1, 64, 1e4, 1000)


def grpo():
    tk = _Tokens(2000)
    system = tk.draw(512)
    prompts = tk.siblings([1024] * 8)
    seqs, groups = [], []
    for g, prompt in enumerate(prompts):
        lens = [int(x) for x in tk.rng.integers(256, 2049, size=8)]
        for comp in tk.siblings(lens):
            seqs.append(np.concatenate([system, prompt, comp]))
            groups.append(g)
    return Workload("grpo", seqs, np.asarray(groups, np.int32), None, 64, 16384, 16, 8, 128, 1e6, 2000)


def agentic():
    tk = _Tokens(3000)
    histories = tk.siblings([20000] * 4)
    seqs, groups = [], []
    for g, hist in enumerate(histories):
        for turns12 in tk.siblings([1000] * 4):
            for turns34 in tk.siblings([1000] * 2):
                seqs.append(np.concatenate([hist, turns12, turns34]))
                groups.append(g)
    return Workload("agentic", seqs, np.asarray(groups, np.int32), None, 64, 32768, 16, 8, 128, 1e6, 3000)


def sweep_lengths(rho, row=32768):
    """(T, P): rollout length and shared prefix with 4T - 3P + 3 == row."""
    if rho == 1.0:
        return row // 4, 0
    target = row * rho / 4
    best = None
    for T in range(int(target) - 3, int(target) + 4):
        if (4 * T + 3 - row) % 3 == 0:
            if best is None or abs(T - target) < abs(best - target):
                best = T
    return best, (4 * best + 3 - row) // 3


def sweep(rho, seqpack=False):
    tk = _Tokens(4000 + int(round(rho * 100)))
    T, P = sweep_lengths(rho)
    if P == 0:
        seqs = tk.siblings([T] * 4)
    else:
        prefix = tk.draw(P)
        seqs = [np.concatenate([prefix, tail]) for tail in tk.siblings([T - P] * 4)]
    name = "sweep_%.2f" % rho + ("_seqpack" if seqpack else "")
    min_shared = T + 1 if seqpack else 64
    return Workload(name, seqs, np.zeros(4, np.int32), None, min_shared, 32768, 16, 8, 128, 1e6, 4000)


def _branching_tree(tk, root_len, seg_lo, seg_hi, depth, n_leaves):
    """Random tree of token runs; returns the root-to-leaf token sequences in
    left-to-right order.  Every tip below ``depth`` forks into b in {1,2,3}
    children (b clamped so the tips never exceed ``n_leaves``)."""
    nodes = [{"tokens": tk.draw(root_len), "end": root_len, "children": []}]
    tips = [0]
    count = 1
    while any(nodes[t]["end"] < depth for t in tips):
        new_tips = []
        for t in tips:
            node = nodes[t]
            if node["end"] >= depth:
                new_tips.append(t)
                continue
            b = min(int(tk.rng.integers(1, 4)), 1 + n_leaves - count)
            count += b - 1
            lens = []
            for _ in range(b):
                n = int(tk.rng.integers(seg_lo, seg_hi + 1))
                lens.append(min(n, depth - node["end"]))
            for run in tk.siblings(lens):
                nodes.append({"tokens": run, "end": node["end"] + len(run), "children": []})
                node["children"].append(len(nodes) - 1)
                new_tips.append(len(nodes) - 1)
        tips = new_tips
    seqs = []

    def dfs(i, prefix):
        cur = prefix + [nodes[i]["tokens"]]
        if not nodes[i]["children"]:
            seqs.append(np.concatenate(cur))
        for c in nodes[i]["children"]:
            dfs(c, cur)
    dfs(0, [])
    assert len(seqs) == n_leaves, len(seqs)
    assert all(len(s) == depth for s in seqs)
    return seqs


def deep():
    tk = _Tokens(5000)
    seqs = _branching_tree(tk, 4096, 256, 1024, 24000, 128)
    return Workload("deep", seqs, np.zeros(len(seqs), np.int32), None, 64, 65536, 32, 8, 128, 1e6,
                    5000, backward=True)


def deep_small():
    tk = _Tokens(6000)
    seqs = _branching_tree(tk, 512, 96, 384, 3000, 16)
    return Workload("deep_small", seqs, np.zeros(len(seqs), np.int32), None, 64, 8192, 8, 2, 128, 1e6,
                    6000, backward=True)


# Planner-scaling batches.  "Prefix Tree Packing in ART" (section "Bin
# packing, with a twist") times its tree walk and bin packing on a
# "multi-task curriculum" batch of 12 / 48 / 192 / 768 groups with 105 / 450 /
# 1,668 / 6,686 completions, without giving the batch's shape.  These stand
# in for it with the same counts: tasks whose system prompt is shared by
# several groups (so one tree spans groups), a prompt per group, completions
# of 256-3072 tokens, rows of 16,384.
CURRICULUM = {12: 105, 48: 450, 192: 1668, 768: 6686}


def curriculum(n_groups):
    n_comp = CURRICULUM[n_groups]
    tk = _Tokens(7000 + n_groups)
    n_tasks = max(2, n_groups // 6)
    systems = tk.siblings([int(x) for x in tk.rng.integers(200, 801, size=n_tasks)])
    base, extra = divmod(n_comp, n_groups)
    counts = [base + (1 if g < extra else 0) for g in range(n_groups)]
    first_of_prompts = [set() for _ in range(n_tasks)]   # a task's prompts are siblings
    seqs, groups = [], []
    for g in range(n_groups):
        t = g % n_tasks
        prompt = tk.draw(int(tk.rng.integers(100, 501)), avoid_first=first_of_prompts[t])
        first_of_prompts[t].add(int(prompt[0]))
        for comp in tk.siblings([int(x) for x in tk.rng.integers(256, 3073, size=counts[g])]):
            seqs.append(np.concatenate([systems[t], prompt, comp]))
            groups.append(g)
    return Workload("curriculum_%d" % n_groups, seqs, np.asarray(groups, np.int32), None, 64, 16384,
                    16, 8, 128, 1e6, 7000 + n_groups)


def get(name):
    if name == "tiny":
        return tiny(512)
    if name == "tiny_fit":
        return tiny(1024)
    if name == "grpo":
        return grpo()
    if name == "agentic":
        return agentic()
    if name == "deep":
        return deep()
    if name == "deep_small":
        return deep_small()
    if name.startswith("curriculum_"):
        return curriculum(int(name.split("_")[1]))
    if name.startswith("sweep_"):
        parts = name.split("_")
        return sweep(float(parts[1]), seqpack=len(parts) > 2 and parts[2] == "seqpack")
    raise KeyError(name)


ALL = ["tiny", "tiny_fit", "grpo", "agentic"] + ["sweep_%.2f" % r for r in SWEEP_RHOS] + ["deep", "deep_small"]
