"""The C-ABI library loads and exports every symbol include/tpk.h declares.

No GPU calls here: only loading, symbol lookup, status strings and the
host-side argument checks that return before touching the device.
"""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "tpk.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tpk_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_calls():
    names = _declared()
    for n in ("tpk_plan_build", "tpk_rope_by_depth", "tpk_tree_attn_fwd", "tpk_tree_attn_bwd",
              "tpk_scatter_token_index"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from prefix_tree_packed_dfs_gb300 import build
    raw = ctypes.CDLL(build.LIB)
    missing = [n for n in _declared() if not hasattr(raw, n)]
    assert not missing, missing


def test_binding_export_list_matches_header():
    from prefix_tree_packed_dfs_gb300 import binding
    assert sorted(binding.EXPORTS) == _declared()


def test_status_strings(lib):
    for code in range(-9, 1):
        assert lib.tpk_status_string(code)
    assert b"sm_103a" in lib.tpk_version()


def test_gpu_entry_points_reject_bad_arguments_before_any_device_call(lib):
    # NULL plan / pointers are rejected on the host with TPK_E_ARG
    assert lib.tpk_tree_attn_fwd(None, None, None, None, None, None, None, 1, 1, 128, 0.1, None, 0, None,
                                 None) == -1
    assert lib.tpk_tree_attn_bwd(None, None, None, None, None, None, None, None, None, None, None, 1, 1, 128,
                                 0.1, None, 0, None, None) == -1
    assert lib.tpk_rope_by_depth(None, None, None, None, None, 10, 1, 1, 96, 1e4, 0, None) == -1
    assert lib.tpk_tree_attn_bwd_phase(7, None, None, None, None, None, None, None, None, None, None, None, 1, 1,
                                       128, 0.1, None, 0, None, None) == -1
    assert lib.tpk_scatter_token_index(None, 1, 1, None, None, None, None, 1, 64, None) == -1
    # empty work is a no-op that never touches the device
    assert lib.tpk_scatter_token_index(ctypes.c_void_p(16), 0, 0, None, None, None, None, 1, 64, None) == 0
    # materialisation gather and its transpose: NULL pointers, negative or
    # inconsistent sizes and misaligned rows are host-side errors
    P = ctypes.c_void_p
    assert lib.tpk_gather_to_forwarded(None, P(16), 1, 1, P(16), P(16), 4, None) == -1
    assert lib.tpk_gather_to_forwarded(P(16), P(16), 2, 1, P(16), P(16), 4, None) == -1     # F > R
    assert lib.tpk_gather_to_forwarded(P(16), P(16), 1, 1, P(16), P(16), 0, None) == -1     # empty rows
    assert lib.tpk_gather_to_forwarded(P(16), P(16), 0, 0, P(16), P(16), 4, None) == 0      # no work
    assert lib.tpk_sum_to_forwarded(P(16), P(16), 1, 1, P(16), None, None, None, 1, 64, None) == -1
    assert lib.tpk_sum_to_forwarded(P(16), P(16), 1, 1, P(16), P(16), None, None, 1, 60, None) == -1  # H*d*2 % 16
    assert lib.tpk_sum_to_forwarded(P(16), P(16), 1, 1, P(8), P(16), None, None, 1, 64, None) == -1   # alignment
    assert lib.tpk_sum_to_forwarded(P(16), P(16), 0, 0, None, None, P(16), P(16), 1, 8, None) == 0
