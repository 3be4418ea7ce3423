"""ctypes binding of ``libtpk.so`` (the C ABI in ``include/tpk.h``).

Argument marshalling only: every step of the computation runs in the library.
There is no fallback: if the library is missing or a call fails, an exception
is raised.
"""
import ctypes
import os

from . import build as _build

TPK_OK = 0
STATUS = {
    0: "TPK_OK", -1: "TPK_E_ARG", -2: "TPK_E_SEQ_TOO_LONG", -3: "TPK_E_OVERFLOW",
    -4: "TPK_E_UNSUPPORTED", -5: "TPK_E_CUDA", -6: "TPK_E_TIMEOUT", -7: "TPK_E_WORKSPACE",
    -8: "TPK_E_SCRATCH_LIMIT", -9: "TPK_E_HOST",
}
BWD_ALL, BWD_PREP, BWD_DKDV, BWD_DQ = -1, 0, 1, 2
PREC_FAST, PREC_PRECISE = 0, 1
PLACE_BFD = 0
PLACE_NEXT_FIT = 1
PLACE_GROUPS = 2
FIELD_DEPTH, FIELD_TOKEN_INDEX, FIELD_SUBTREE_END, FIELD_PARENT = 0, 1, 2, 3
FIELD_FWD_RAW_BEGIN, FIELD_FWD_RAW = 4, 5
FIELD_SEG_START, FIELD_SEG_LEN, FIELD_SEG_PARENT, FIELD_SEG_OFF = 6, 7, 8, 9

# every symbol include/tpk.h declares
EXPORTS = [
    "tpk_plan_build", "tpk_plan_info_get", "tpk_plan_export", "tpk_plan_worklists", "tpk_plan_raw_of_forwarded",
    "tpk_plan_shard_rows", "tpk_plan_segments",
    "tpk_plan_device_bytes", "tpk_plan_field_offset", "tpk_plan_upload", "tpk_plan_destroy",
    "tpk_rope_by_depth", "tpk_attn_workspace_bytes", "tpk_tree_attn_fwd", "tpk_tree_attn_fwd_ex",
    "tpk_tree_attn_bwd", "tpk_tree_attn_bwd_ex", "tpk_tree_attn_bwd_phase", "tpk_tree_attn_bwd_noalloc", "tpk_selftest_wait_timeout",
    "tpk_scatter_token_index", "tpk_gather_to_forwarded", "tpk_sum_to_forwarded", "tpk_gdn_conv",
    "tpk_gdn_workspace_bytes", "tpk_gdn_delta_rule", "tpk_gdn_conv_bwd_workspace_bytes", "tpk_gdn_conv_bwd",
    "tpk_gdn_bwd_workspace_bytes", "tpk_gdn_delta_rule_bwd", "tpk_status_string",
    "tpk_version",
]


class TpkError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (what, STATUS.get(status, status), _LIB.tpk_status_string(status).decode() if _LIB else ""))


class PlanOpts(ctypes.Structure):
    _fields_ = [("row_capacity", ctypes.c_int64), ("min_shared", ctypes.c_int32), ("placement", ctypes.c_int32)]


class AttnOpts(ctypes.Structure):
    """tpk_attn_opts: precision, inverse RoPE base (backward), O's rounding residual."""
    _fields_ = [("precision", ctypes.c_int32), ("reserved", ctypes.c_int32), ("rope_base", ctypes.c_double),
                ("o_lo", ctypes.c_void_p)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "n_seqs", "n_rows", "n_fwd", "n_raw", "n_segments", "n_leaves", "n_qtiles", "n_kblocks",
        "n_ktiles", "n_qblocks", "useful_pairs", "visited_pairs", "max_depth")] + \
        [(n, ctypes.c_double) for n in ("packing_ratio", "row_fill_frac", "fork_frac")] + \
        [(n, ctypes.c_int64) for n in ("n_seg_instances", "n_seg_levels")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_LIB = None
P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
SZ = ctypes.c_size_t


def _sig(lib):
    lib.tpk_plan_build.argtypes = [P, P, I32, P, P, ctypes.POINTER(PlanOpts), ctypes.POINTER(P)]
    lib.tpk_plan_info_get.argtypes = [P, ctypes.POINTER(PlanInfo)]
    lib.tpk_plan_export.argtypes = [P] * 10
    lib.tpk_plan_worklists.argtypes = [P] * 11
    lib.tpk_plan_raw_of_forwarded.argtypes = [P, P, P]
    lib.tpk_plan_device_bytes.argtypes = [P]
    lib.tpk_plan_device_bytes.restype = SZ
    lib.tpk_plan_shard_rows.argtypes = [P, I32, P, P]
    lib.tpk_plan_segments.argtypes = [P, P, P, P, P]
    lib.tpk_plan_field_offset.argtypes = [P, I32, ctypes.POINTER(SZ)]
    lib.tpk_plan_upload.argtypes = [P, P, P]
    lib.tpk_plan_destroy.argtypes = [P]
    lib.tpk_plan_destroy.restype = None
    lib.tpk_rope_by_depth.argtypes = [P, P, P, P, P, I64, I32, I32, I32, ctypes.c_double, I32, P]
    lib.tpk_attn_workspace_bytes.argtypes = [P, I32, I32, I32, I32]
    lib.tpk_attn_workspace_bytes.restype = SZ
    lib.tpk_tree_attn_fwd.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, ctypes.c_float, P, SZ, P, P]
    lib.tpk_tree_attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I32, I32, I32, ctypes.c_float, P, SZ, P, P]
    lib.tpk_tree_attn_bwd_phase.argtypes = [I32] + lib.tpk_tree_attn_bwd.argtypes
    lib.tpk_tree_attn_fwd_ex.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, ctypes.c_float,
                                         ctypes.POINTER(AttnOpts), P, P]
    lib.tpk_tree_attn_bwd_ex.argtypes = [I32, P, P, P, P, P, P, P, P, P, P, P, I32, I32, I32, ctypes.c_float,
                                         ctypes.POINTER(AttnOpts), P, SZ, P, P]
    lib.tpk_tree_attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, P, P, I32, I32, I32, ctypes.c_float, P, P]
    lib.tpk_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P, P]
    lib.tpk_scatter_token_index.argtypes = [P, I64, I64, P, P, P, P, I32, I32, P]
    lib.tpk_gather_to_forwarded.argtypes = [P, P, I64, I64, P, P, I64, P]
    lib.tpk_sum_to_forwarded.argtypes = [P, P, I64, I64, P, P, P, P, I32, I32, P]
    lib.tpk_gdn_conv.argtypes = [P, P, P, P, P, I32, I32, P]
    lib.tpk_gdn_workspace_bytes.argtypes = [P, I32, I32, I32]
    lib.tpk_gdn_workspace_bytes.restype = SZ
    lib.tpk_gdn_delta_rule.argtypes = [P, P, P, P, P, I64, I64, P, P, P, I32, I32, I32, ctypes.c_float, P, SZ, P]
    lib.tpk_gdn_conv_bwd_workspace_bytes.argtypes = [P, I32, I32]
    lib.tpk_gdn_conv_bwd_workspace_bytes.restype = SZ
    lib.tpk_gdn_conv_bwd.argtypes = [P, P, P, P, P, P, P, I32, I32, P, SZ, P]
    lib.tpk_gdn_bwd_workspace_bytes.argtypes = [P, I32, I32, I32]
    lib.tpk_gdn_bwd_workspace_bytes.restype = SZ
    lib.tpk_gdn_delta_rule_bwd.argtypes = [P, P, P, P, P, I64, I64, P, P, P, P, P, P, I64, I64, P, P, I32, I32, I32,
                                           ctypes.c_float, P, SZ, P, SZ, P]
    lib.tpk_status_string.argtypes = [ctypes.c_int]
    lib.tpk_status_string.restype = ctypes.c_char_p
    lib.tpk_version.argtypes = []
    lib.tpk_version.restype = ctypes.c_char_p
    for name in EXPORTS:
        f = getattr(lib, name)
        if f.restype is ctypes.c_int and name not in ("tpk_status_string",):
            f.restype = ctypes.c_int
    return lib


def load(build_if_missing=True):
    """Load libtpk.so (building it in-tree first if needed) and return it."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if build_if_missing:
        path = _build.build_library(quiet=True)
    if not os.path.exists(path):
        raise RuntimeError("libtpk.so is not built (%s); run prefix_tree_packed_dfs_gb300/build.py" % path)
    _LIB = _sig(ctypes.CDLL(path))
    return _LIB


def check(status, what):
    if status != TPK_OK:
        raise TpkError(status, what)
