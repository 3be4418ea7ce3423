"""Plain CPU oracle for prefix-tree-packed DFS attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the C++/CUDA library (``prefix_tree_packed_dfs_gb300``) and never
imports it.

Contents
--------
``planner``    the packing plan, following the pages' own steps:
               the recursive longest-shared-run walk ("Prefix Tree Packing in
               ART", section "The tree"), the minimum shared-segment length and
               the duplicated join token (same section; "DAG packing", section
               "The walk"), best-fit-decreasing over marginal cost ("Prefix Tree
               Packing in ART", section "Bin packing, with a twist"), the
               in-order fill ("Prefix Tree Packing in ART", sections "One tree,
               not one per group" and "Does it actually help?"), one row per
               placement group (no counterpart on the pages) and the
               depth-first layout with depth positions and token_index ("DAG
               packing", sections "The walk" and "Positions"; "TRL Tree Packing
               for AsyncGRPO", section "How tree packing works").
``attention``  the plain definition the packed computation must reproduce:
               every root-to-leaf sequence unpacked, RoPE at positions
               0..L-1, ordinary causal softmax attention in fp64 ("DAG
               packing", section "The mask"; "Prefix Tree Packing in ART",
               section "Token-mixing layers"), and its backward.
``layout``     per-token data between raw order and the packed layout: the
               materialisation gather by owner ("Prefix Tree Packing in ART",
               section "Metadata space first"), the raw-order scatter through
               token_index and its transpose, the sum over a position's raw
               tokens ("TRL Tree Packing for AsyncGRPO", section "How tree
               packing works").
``gdn``        the GDN token mixer (causal convolution + gated delta rule)
               along every unpacked root-to-leaf sequence, its gradients by
               fp64 autograd over the unpacked sequences, and the pages'
               level-by-level schedule ("Prefix Tree Packing in ART", section
               "Token-mixing layers").
``bf16``       round-to-nearest-even rounding of fp64 values to bfloat16.

Every function is pinned by a ``-m "not gpu"`` test against values the pages
print, closed forms, library routines or brute force (see ``tests/``).
"""
