"""Oracle for moving per-token data between raw order and the packed layout.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* Materialisation ("Prefix Tree Packing in ART", section "Metadata space
  first"): after planning, one pass slices per-token payloads (token ids,
  logprobs, advantages, ...) into the packed tensors.  A forwarded position
  stands for every raw token that maps to it; it takes the row of its owner,
  the lowest such raw token (``fwd_src`` of the oracle planner).
* The raw-order scatter ("TRL Tree Packing for AsyncGRPO", section "How tree
  packing works": ``token_index`` maps every raw token to its forwarded
  position) reads O_raw[r] = O[token_index[r]].  Its transpose sums: a
  forwarded position receives the sum of the rows of all its raw tokens.
  Written here as that plain definition, in fp64.
"""
import numpy as np


def gather_to_forwarded(plan, src):
    """dst[f] = src[fwd_src[f]] for a per-raw-token array ``src`` [R, ...]."""
    src = np.asarray(src)
    return src[np.asarray(plan["fwd_src"])].copy()


def scatter_to_raw(plan, src):
    """O_raw[r] = O[token_index[r]] for a forwarded array ``src`` [F, ...]."""
    return np.asarray(src)[np.asarray(plan["token_index"])].copy()


def sum_to_forwarded(plan, src):
    """dst[f] = sum of src[r] over the raw tokens r with token_index[r] = f (fp64)."""
    src = np.asarray(src, dtype=np.float64)
    dst = np.zeros((plan["n_fwd"],) + src.shape[1:], dtype=np.float64)
    ti = np.asarray(plan["token_index"])
    for r in range(len(ti)):
        dst[ti[r]] += src[r]
    return dst
