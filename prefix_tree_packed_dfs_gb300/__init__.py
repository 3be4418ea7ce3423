"""Prefix-tree-packed DFS attention for one GB300 GPU (sm_103a).

The library (``libtpk.so``, C ABI in ``include/tpk.h``) holds the host
planner and the CUDA kernels; this package is its thin Python binding:

    from prefix_tree_packed_dfs_gb300 import ops
    plan = ops.Plan.from_sequences(seqs, row_capacity=32768, min_shared=64)
    dplan = plan.to_device()
    ops.rope_by_depth(q, k, dplan.depth, base=1e6)
    o, lse = ops.tree_attn_fwd(dplan, q, k, v)
    o_raw, lse_raw = ops.scatter_token_index(dplan.token_index, o, lse)

Importing the package does not load the library; ``ops``/``binding`` build
and load it on first use and raise if it cannot be built or loaded (there is
no CPU fallback).
"""
__all__ = ["ops", "binding", "build"]
