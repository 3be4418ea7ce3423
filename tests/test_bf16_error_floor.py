"""Where the backward's max-abs tolerances come from (CPU only).

The attention kernels multiply bf16 operands on the tensor cores.  This test
runs each precision mode's arithmetic with everything else exact (fp64, dense
masks from the plan) and measures its error against the oracle's exact
gradients, in units of max(1, |ref|) as the GPU parity tests count it:

* fast: the probabilities P (for dV, and for O in the forward) and
  dS = P * (dP - D) (for dK and dQ) are rounded to bf16 before their
  products, as every bf16 flash-attention backward does, and D = dO . O takes
  the bf16-rounded O.  On these inputs that reaches about 1.3% -- above the
  stated flat 1e-2 -- while its relative L2 error stays near 2.5e-3.  The GPU
  tests hold the fast mode to relative L2 5e-3 (as stated) and max-abs 2e-2
  (the floor with a 1.5x margin).
* precise: P and dS enter as a bf16 pair hi + lo (hi = bf16(x), lo =
  bf16(x - hi)), in the forward's PV product too, and D is taken from O
  before its rounding (O + O_lo).  What is left is the bf16 rounding of the
  gradients themselves (at most 2^-8 of max(1, |ref|)), well inside the stated
  1e-2, which the GPU tests apply to this mode.
"""
import numpy as np
import pytest

from oracle import attention as oa
from oracle import planner as op
from oracle.bf16 import round_to_bf16 as rb
from workloads import rng as wrng

GRAD_MAX_ABS_FAST = 2e-2   # in units of max(1, |ref|)
GRAD_MAX_ABS = 1e-2
REL_L2 = 5e-3


def _hilo(x):
    hi = rb(x)
    return hi + rb(x - hi)


def emulated_backward(ref, Q, K, V, dO, base, precise):
    """Gradients with the kernels' operand roundings, everything else fp64."""
    F, hq, d = Q.shape
    hkv = K.shape[1]
    sc = 1 / np.sqrt(d)
    op_round = _hilo if precise else rb
    qr = rb(oa.rope(Q, ref["depth"], base))
    kr = rb(oa.rope(K, ref["depth"], base))
    se = ref["subtree_end"]
    vis = np.zeros((F, F), bool)
    for j in range(F):
        vis[j:se[j], j] = True
    dq, dk, dv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for h in range(hq):
        g = h // (hq // hkv)
        s = qr[:, h] @ kr[:, g].T * sc
        s[~vis] = -np.inf
        p = np.exp(s - s.max(1, keepdims=True))
        l_sum = p.sum(1, keepdims=True)
        P = p / l_sum
        # the forward's O: unnormalised P through its PV operand, then / l
        o32 = (op_round(p) @ V[:, g]) / l_sum
        o = o32 if precise else rb(o32)          # precise: O + O_lo
        D = np.sum(dO[:, h] * o, 1, keepdims=True)
        dS = op_round(P * (dO[:, h] @ V[:, g].T - D))
        dv[:, g] += op_round(P).T @ dO[:, h]
        dk[:, g] += sc * dS.T @ qr[:, h]
        dq[:, h] = sc * dS @ kr[:, g]
    dq = oa.rope(dq, ref["depth"], base, inverse=True)
    dk = oa.rope(dk, ref["depth"], base, inverse=True)
    return rb(dq), rb(dk), rb(dv)


@pytest.fixture(scope="module")
def case():
    from tests.test_gpu_kernels import _ragged
    w = _ragged(3, 8, 2, 128, cap=1024)
    ref = op.plan(w.sequences, group_ids=w.group_ids, min_shared=w.min_shared, row_capacity=w.row_capacity)
    F, s = ref["n_fwd"], w.seeds
    X = [wrng.normal_bf16(s[k], (F, h, w.head_dim)).double().numpy()
         for k, h in (("q", w.n_heads_q), ("k", w.n_heads_kv), ("v", w.n_heads_kv), ("do", w.n_heads_q))]
    return w, ref, X, oa.backward(ref, *X, w.rope_base)


def _worst(approx, exact):
    worst = 0.0
    for a, b in zip(approx, exact):
        worst = max(worst, float(np.max(np.abs(a - b) / np.maximum(1.0, np.abs(b)))))
        assert np.linalg.norm(a - b) / np.linalg.norm(b) < REL_L2
    return worst


def test_fast_mode_error_floor(case):
    w, ref, X, exact = case
    worst = _worst(emulated_backward(ref, *X, w.rope_base, precise=False), exact)
    # the floor sits above the flat 1e-2 and below the bound the GPU tests use
    assert 1e-2 < worst < GRAD_MAX_ABS_FAST / 1.4


def test_precise_mode_meets_the_stated_bound(case):
    w, ref, X, exact = case
    worst = _worst(emulated_backward(ref, *X, w.rope_base, precise=True), exact)
    # only the gradients' own bf16 rounding is left: 2^-8 of max(1, |ref|) at most
    assert worst <= 2.0 ** -8 * 1.01
    assert worst < GRAD_MAX_ABS / 2
