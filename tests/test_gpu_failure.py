"""Device-side failure detection without a GPU fault.

Every wait in the attention kernels is bounded; a wait that runs out sets an
abort flag, the CTA leaves its loops and the launch reports TPK_E_TIMEOUT
through the caller's device status word.  Here a self-test kernel makes that
wait run out on a barrier nothing arrives at (a one-tenth-second limit), and
the test checks the status and that the context still runs the attention
path afterwards.  Host-side failures (bad offsets, over-long sequences,
missing workspace) are status codes covered by the CPU tests.
"""
import ctypes
import time

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

TPK_E_TIMEOUT = -6


def test_bounded_wait_reports_timeout_and_context_survives():
    assert torch.cuda.is_available()
    from prefix_tree_packed_dfs_gb300 import binding, ops
    lib = binding.load()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    t0 = time.perf_counter()
    st = lib.tpk_selftest_wait_timeout(100_000_000, ctypes.c_void_p(err.data_ptr()), stream)
    assert st == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) == TPK_E_TIMEOUT
    assert 0.05 < elapsed < 5.0
    # the context is intact: a full forward still runs and reports no error
    w = workloads.get("tiny_fit")
    plan = ops.Plan.from_sequences(w.sequences, group_ids=w.group_ids, row_capacity=w.row_capacity,
                                   min_shared=w.min_shared)
    dp = plan.to_device()
    F = plan.info["n_fwd"]
    q = torch.randn(F, 1, 64, device="cuda").to(torch.bfloat16)
    k = torch.randn(F, 1, 64, device="cuda").to(torch.bfloat16)
    v = torch.randn(F, 1, 64, device="cuda").to(torch.bfloat16)
    err.zero_()
    o, lse = ops.tree_attn_fwd(dp, q, k, v, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_selftest_rejects_bad_arguments():
    from prefix_tree_packed_dfs_gb300 import binding
    lib = binding.load()
    assert lib.tpk_selftest_wait_timeout(0, None, None) == -1
    assert lib.tpk_selftest_wait_timeout(10 ** 10, ctypes.c_void_p(16), None) == -1
