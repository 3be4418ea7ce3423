"""The backward entry point that allocates nothing, against the regular one.

``tpk_tree_attn_bwd_noalloc`` exists for callers that cannot allocate device
memory when they call the library -- hosts that own all device memory and
give plugins none at call time, code that must not call cudaMalloc/cudaFree
because those can synchronise the device, C runtimes without a device
allocator.  Its scratch is a fixed array inside the library instead of a
caller-provided workspace.  These tests call it through the C ABI twice in a
row and compare each result with ``tpk_tree_attn_bwd`` (given a torch
workspace): both run the same deterministic kernels (no atomics) on the same
inputs, so the gradients must be bit-identical.  They also check that a
problem too large for the fixed array is refused.  The file is named so that
pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from workloads import rng as wrng

pytestmark = pytest.mark.gpu

TPK_E_SCRATCH_LIMIT = -8


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_backward_matches_workspace_backward():
    assert torch.cuda.is_available()
    from prefix_tree_packed_dfs_gb300 import binding, ops
    lib = binding.load()
    w = workloads.get("deep_small")
    plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                   min_shared=w.min_shared)
    dp = plan.to_device()
    F, Hq, Hkv, d = plan.info["n_fwd"], w.n_heads_q, w.n_heads_kv, w.head_dim
    s = w.seeds
    q = wrng.normal_bf16(s["q"], (F, Hq, d), "cuda")
    k = wrng.normal_bf16(s["k"], (F, Hkv, d), "cuda")
    v = wrng.normal_bf16(s["v"], (F, Hkv, d), "cuda")
    do = wrng.normal_bf16(s["do"], (F, Hq, d), "cuda")
    ops.rope_by_depth(q, k, dp.depth, w.rope_base)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = ops.tree_attn_fwd(dp, q, k, v, dev_err=err)
    ref = ops.tree_attn_bwd(dp, q, k, v, o, lse, do, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    scale = 1.0 / np.sqrt(d)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        st = lib.tpk_tree_attn_bwd_noalloc(plan.handle, _ptr(dp.image), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                           _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), Hq, Hkv, d, scale,
                                           _ptr(err), stream)
        assert st == 0, binding.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for got, want, name in zip((dq, dk, dv), ref, ("dQ", "dK", "dV")):
            assert torch.isfinite(got).all(), "call %d %s" % (call, name)
            assert torch.equal(got, want), "call %d %s differs from the workspace backward" % (call, name)


def test_noalloc_backward_refuses_problems_beyond_its_scratch():
    from prefix_tree_packed_dfs_gb300 import binding, ops
    lib = binding.load()
    w = workloads.get("deep_small")
    plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                   min_shared=w.min_shared)
    F = plan.info["n_fwd"]
    hq = (8388608 // F + 1)          # Hq * F just above the 8,388,608 limit
    hq += (-hq) % 2
    st = lib.tpk_tree_attn_bwd_noalloc(plan.handle, None, None, None, None, None, None, None, None, None, None,
                                       hq, 2, 128, 0.1, None, None)
    assert st == TPK_E_SCRATCH_LIMIT
    assert b"static scratch" in lib.tpk_status_string(st)
