"""Torch-facing wrappers over the C ABI (same names as ``include/tpk.h``).

PyTorch only provides device memory and the current stream; the wrappers check
dtypes/shapes/contiguity, allocate outputs with torch and pass raw pointers.
"""
import ctypes
import math

import numpy as np
import torch

from . import binding as B


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, dtype, name, ndim=None, cuda=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if cuda and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (no CPU path exists)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))


class Plan:
    """Host packing plan (``tpk_plan_build``)."""

    def __init__(self, tokens, seq_offsets, trained=None, group_ids=None, row_capacity=65536,
                 min_shared=64, placement="bfd"):
        lib = B.load()
        self._lib = lib
        self._h = None
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        offs = np.ascontiguousarray(seq_offsets, dtype=np.int64)
        n = len(offs) - 1
        tr = None if trained is None else np.ascontiguousarray(trained, dtype=np.uint8)
        gr = None if group_ids is None else np.ascontiguousarray(group_ids, dtype=np.int32)
        if tr is not None and len(tr) != len(tokens):
            raise ValueError("trained must have one flag per token")
        if gr is not None and len(gr) != n:
            raise ValueError("group_ids must have one id per sequence")
        opts = B.PlanOpts(int(row_capacity), int(min_shared),
                          {"bfd": B.PLACE_BFD, "next_fit": B.PLACE_NEXT_FIT, "groups": B.PLACE_GROUPS}[placement])
        h = ctypes.c_void_p()
        st = lib.tpk_plan_build(tokens.ctypes.data, offs.ctypes.data, n,
                                None if tr is None else tr.ctypes.data,
                                None if gr is None else gr.ctypes.data,
                                ctypes.byref(opts), ctypes.byref(h))
        B.check(st, "tpk_plan_build")
        self._h = h
        info = B.PlanInfo()
        B.check(lib.tpk_plan_info_get(h, ctypes.byref(info)), "tpk_plan_info_get")
        self.info = info.as_dict()

    @classmethod
    def from_sequences(cls, sequences, trained=None, **kw):
        seqs = [np.asarray(s) for s in sequences]
        offs = np.zeros(len(seqs) + 1, dtype=np.int64)
        offs[1:] = np.cumsum([len(s) for s in seqs])
        tr = None if trained is None else np.concatenate([np.asarray(t) for t in trained])
        return cls(np.concatenate(seqs), offs, trained=tr, **kw)

    @property
    def handle(self):
        return self._h

    def __getattr__(self, name):
        info = self.__dict__.get("info")
        if info is not None and name in info:
            return info[name]
        raise AttributeError(name)

    def export(self):
        i = self.info
        F, R, n, rows = i["n_fwd"], i["n_raw"], i["n_seqs"], i["n_rows"]
        out = {
            "row_offsets": np.zeros(rows + 1, np.int64), "row_loads": np.zeros(rows, np.int64),
            "row_of_seq": np.zeros(n, np.int32), "fwd_token": np.zeros(F, np.int32),
            "fwd_src": np.zeros(F, np.int32), "parent": np.zeros(F, np.int32), "depth": np.zeros(F, np.int32),
            "token_index": np.zeros(R, np.int32), "subtree_end": np.zeros(F, np.int32),
        }
        order = ["row_offsets", "row_loads", "row_of_seq", "fwd_token", "fwd_src", "parent", "depth",
                 "token_index", "subtree_end"]
        B.check(self._lib.tpk_plan_export(self._h, *[out[k].ctypes.data for k in order]), "tpk_plan_export")
        return out

    def worklists(self):
        i = self.info
        T, NB, KT, NQB = i["n_qtiles"], i["n_kblocks"], i["n_ktiles"], i["n_qblocks"]
        out = {
            "qt_q0": np.zeros(T, np.int32), "qt_nq": np.zeros(T, np.int32), "qt_kb_begin": np.zeros(T + 1, np.int32),
            "kb": np.zeros(2 * NB, np.int32), "qt_order": np.zeros(T, np.int32),
            "kt_k0": np.zeros(KT, np.int32), "kt_nk": np.zeros(KT, np.int32),
            "kt_qb_begin": np.zeros(KT + 1, np.int32), "qb": np.zeros(2 * NQB, np.int32),
            "kt_order": np.zeros(KT, np.int32),
        }
        order = ["qt_q0", "qt_nq", "qt_kb_begin", "kb", "qt_order", "kt_k0", "kt_nk", "kt_qb_begin", "qb",
                 "kt_order"]
        B.check(self._lib.tpk_plan_worklists(self._h, *[out[k].ctypes.data for k in order]), "tpk_plan_worklists")
        return out

    def raw_of_forwarded(self):
        """(fwd_raw_begin [F+1], fwd_raw [R]): the raw tokens of each forwarded position, ascending."""
        F, R = self.info["n_fwd"], self.info["n_raw"]
        begin, raw = np.zeros(F + 1, np.int32), np.zeros(R, np.int32)
        B.check(self._lib.tpk_plan_raw_of_forwarded(self._h, begin.ctypes.data, raw.ctypes.data),
                "tpk_plan_raw_of_forwarded")
        return begin, raw

    def segments(self):
        """Segment instances by tree level: (level_begin [n_levels+1],
        seg_start, seg_len, seg_parent [n_instances]), int32."""
        n, L = self.info["n_seg_instances"], self.info["n_seg_levels"]
        out = (np.zeros(L + 1, np.int32), np.zeros(n, np.int32), np.zeros(n, np.int32), np.zeros(n, np.int32))
        B.check(self._lib.tpk_plan_segments(self._h, *[a.ctypes.data for a in out]), "tpk_plan_segments")
        return out

    def shard_rows(self, world):
        """Whole rows to `world` data-parallel ranks, heaviest row first to the
        least-loaded rank (work = useful pairs).  Returns (rank_of_row int32
        [n_rows], rank_pairs int64 [world])."""
        rows = self.info["n_rows"]
        rank_of_row, rank_pairs = np.zeros(rows, np.int32), np.zeros(world, np.int64)
        B.check(self._lib.tpk_plan_shard_rows(self._h, int(world), rank_of_row.ctypes.data, rank_pairs.ctypes.data),
                "tpk_plan_shard_rows")
        return rank_of_row, rank_pairs

    def sequences_of_rank(self, rank_of_row, rank):
        """Indices (input order) of the sequences whose row `rank` owns."""
        return np.flatnonzero(np.asarray(rank_of_row)[self.export()["row_of_seq"]] == rank)

    def rank_plan(self, sequences, rank_of_row, rank, row_capacity, min_shared=64, trained=None):
        """The plan of rank `rank`'s rows (``shard_rows``): its sequences,
        planned with their row in this plan as the group and one row per
        group, i.e. exactly those rows.  Returns (plan, sequence indices);
        ``sequences`` / ``trained`` are the inputs this plan was built from."""
        idx = self.sequences_of_rank(rank_of_row, rank)
        rows = self.export()["row_of_seq"][idx]
        sub = Plan.from_sequences([sequences[i] for i in idx],
                                  trained=None if trained is None else [trained[i] for i in idx],
                                  group_ids=rows, row_capacity=row_capacity, min_shared=min_shared,
                                  placement="groups")
        return sub, idx

    def device_bytes(self):
        return int(self._lib.tpk_plan_device_bytes(self._h))

    def field_offset(self, field):
        off = ctypes.c_size_t()
        B.check(self._lib.tpk_plan_field_offset(self._h, field, ctypes.byref(off)), "tpk_plan_field_offset")
        return off.value

    def to_device(self, device="cuda"):
        return DevicePlan(self, device)

    def close(self):
        if self._h is not None:
            self._lib.tpk_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DevicePlan:
    """A plan plus its device image (one torch uint8 buffer)."""

    def __init__(self, plan, device="cuda"):
        self.plan = plan
        nbytes = max(plan.device_bytes(), 256)
        self.image = torch.empty(nbytes, dtype=torch.uint8, device=device)
        if self.image.data_ptr() % 256:
            raise RuntimeError("device image not 256-byte aligned")
        B.check(plan._lib.tpk_plan_upload(plan.handle, _ptr(self.image), _stream()), "tpk_plan_upload")
        F, R = plan.info["n_fwd"], plan.info["n_raw"]
        self.depth = self._field(B.FIELD_DEPTH, F)
        self.token_index = self._field(B.FIELD_TOKEN_INDEX, R)
        self.subtree_end = self._field(B.FIELD_SUBTREE_END, F)
        self.parent = self._field(B.FIELD_PARENT, F)
        self.fwd_raw_begin = self._field(B.FIELD_FWD_RAW_BEGIN, F + 1)
        self.fwd_raw = self._field(B.FIELD_FWD_RAW, R)
        n_inst = plan.info["n_seg_instances"]
        self.seg_start = self._field(B.FIELD_SEG_START, n_inst)
        self.seg_len = self._field(B.FIELD_SEG_LEN, n_inst)
        self.seg_parent = self._field(B.FIELD_SEG_PARENT, n_inst)
        self.seg_off = self._field(B.FIELD_SEG_OFF, n_inst)

    def _field(self, field, n):
        off = self.plan.field_offset(field)
        return self.image[off:off + 4 * n].view(torch.int32)

    @property
    def n_fwd(self):
        return self.plan.info["n_fwd"]

    @property
    def n_raw(self):
        return self.plan.info["n_raw"]


def rope_by_depth(q, k, depth, base, inverse=False, q_out=None, k_out=None):
    """RoPE of q [F,Hq,d] and/or k [F,Hkv,d] at ``depth`` (int32 [F]).

    In place unless ``q_out`` / ``k_out`` are given.  Returns (q_out, k_out)."""
    lib = B.load()
    ref = q if q is not None else k
    F, _, d = ref.shape
    if q is not None:
        _need(q, torch.bfloat16, "q", 3)
        q_out = q if q_out is None else q_out
        _need(q_out, torch.bfloat16, "q_out", 3)
    if k is not None:
        _need(k, torch.bfloat16, "k", 3)
        k_out = k if k_out is None else k_out
        _need(k_out, torch.bfloat16, "k_out", 3)
    _need(depth, torch.int32, "depth", 1)
    if depth.numel() != F or (q is not None and k is not None and k.shape[0] != F):
        raise ValueError("shape mismatch")
    Hq = q.shape[1] if q is not None else 0
    Hkv = k.shape[1] if k is not None else 0
    B.check(lib.tpk_rope_by_depth(_ptr(q), _ptr(k), _ptr(q_out) if q is not None else None,
                                  _ptr(k_out) if k is not None else None, _ptr(depth), F, Hq, Hkv, d,
                                  float(base), 1 if inverse else 0, _stream()), "tpk_rope_by_depth")
    return q_out, k_out


def _shape(t, shape, name):
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _on_device(ref, *named):
    """Every tensor (None skipped) a CUDA tensor on ref's device.  Checked after
    the shapes, so a wrong shape is reported as such wherever the tensors live."""
    for t, n in ((ref, "q"),) + named:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor (no CPU path exists)" % n)
        if t.device != ref.device:
            raise ValueError("%s is on %s, expected %s" % (n, t.device, ref.device))


def _attn_shapes(dplan, q, k, v):
    """(F, Hq, Hkv, d) of q [F,Hq,d], k/v [F,Hkv,d], checked against the plan."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n, 3, cuda=False)
    F, Hq, d = q.shape
    Hkv = k.shape[1]
    if F != dplan.n_fwd:
        raise ValueError("q has %d rows, the plan has %d forwarded positions" % (F, dplan.n_fwd))
    _shape(k, (F, Hkv, d), "k")
    _shape(v, (F, Hkv, d), "v")
    return F, Hq, Hkv, d


def _opts(precise, rope_base=None, o_lo=None):
    return B.AttnOpts(B.PREC_PRECISE if precise else B.PREC_FAST, 0,
                      0.0 if rope_base is None else float(rope_base), None if o_lo is None else o_lo.data_ptr())


def tree_attn_fwd(dplan, q, k, v, scale=None, out=None, lse=None, dev_err=None, precise=False, o_lo=None):
    """Forward tree attention; returns (O [F,Hq,d] bf16, LSE [Hq,F] fp32).

    ``precise``: P enters the PV product as a hi + lo bf16 pair, and O's bf16
    rounding residual is written to ``o_lo`` (allocated if None); the return
    value is then (O, LSE, O_lo)."""
    lib = B.load()
    F, Hq, Hkv, d = _attn_shapes(dplan, q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, F), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out", 3, cuda=False)
    _shape(out, (F, Hq, d), "out")
    _need(lse, torch.float32, "lse", 2, cuda=False)
    _shape(lse, (Hq, F), "lse")
    if precise:
        o_lo = torch.empty_like(q) if o_lo is None else o_lo
        _need(o_lo, torch.bfloat16, "o_lo", 3, cuda=False)
        _shape(o_lo, (F, Hq, d), "o_lo")
    if dev_err is not None:
        _need(dev_err, torch.int32, "dev_err", cuda=False)
    _on_device(q, (k, "k"), (v, "v"), (dplan.image, "the plan image"), (out, "out"), (lse, "lse"),
               (o_lo if precise else None, "o_lo"), (dev_err, "dev_err"))
    opts = _opts(precise, None, o_lo if precise else None)
    st = lib.tpk_tree_attn_fwd_ex(dplan.plan.handle, _ptr(dplan.image), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                  _ptr(lse), Hq, Hkv, d, scale, ctypes.byref(opts), _ptr(dev_err), _stream())
    B.check(st, "tpk_tree_attn_fwd_ex")
    return (out, lse, o_lo) if precise else (out, lse)


def attn_workspace_bytes(dplan, Hq, Hkv, d, backward):
    lib = B.load()
    return int(lib.tpk_attn_workspace_bytes(dplan.plan.handle, Hq, Hkv, d, 1 if backward else 0))


def tree_attn_bwd(dplan, q, k, v, o, lse, do, scale=None, dq=None, dk=None, dv=None, workspace=None,
                  dev_err=None, phases=(0, 1, 2), precise=False, o_lo=None, rope_base=None):
    """Backward tree attention; returns (dQ, dK, dV).

    Gradients are w.r.t. the rotated q, k unless ``rope_base`` is given, in
    which case the inverse RoPE at depth is applied inside the kernels and
    dQ, dK are w.r.t. the un-rotated inputs.  ``precise`` selects the hi + lo
    bf16 products (and uses the forward's ``o_lo`` for dO . O when given).
    ``phases`` selects the launches (0 prep, 1 dK/dV pass, 2 dQ pass); the
    default runs all three in order."""
    lib = B.load()
    F, Hq, Hkv, d = _attn_shapes(dplan, q, k, v)
    for t, n in ((o, "o"), (do, "do")):
        _need(t, torch.bfloat16, n, 3, cuda=False)
        _shape(t, (F, Hq, d), n)
    _need(lse, torch.float32, "lse", 2, cuda=False)
    _shape(lse, (Hq, F), "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n, shp in ((dq, "dq", (F, Hq, d)), (dk, "dk", (F, Hkv, d)), (dv, "dv", (F, Hkv, d))):
        _need(t, torch.bfloat16, n, 3, cuda=False)
        _shape(t, shp, n)
    if o_lo is not None:
        _need(o_lo, torch.bfloat16, "o_lo", 3, cuda=False)
        _shape(o_lo, (F, Hq, d), "o_lo")
    need = attn_workspace_bytes(dplan, Hq, Hkv, d, True)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor")
    ws_bytes = workspace.numel() * workspace.element_size()
    if ws_bytes < need:
        raise ValueError("workspace has %d bytes, the backward needs %d" % (ws_bytes, need))
    if dev_err is not None:
        _need(dev_err, torch.int32, "dev_err", cuda=False)
    _on_device(q, (k, "k"), (v, "v"), (dplan.image, "the plan image"), (o, "o"), (do, "do"), (lse, "lse"),
               (dq, "dq"), (dk, "dk"), (dv, "dv"), (o_lo, "o_lo"), (workspace, "workspace"), (dev_err, "dev_err"))
    opts = _opts(precise, rope_base, o_lo)
    args = (dplan.plan.handle, _ptr(dplan.image), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
            _ptr(dq), _ptr(dk), _ptr(dv), Hq, Hkv, d, scale, ctypes.byref(opts), _ptr(workspace), ws_bytes,
            _ptr(dev_err), _stream())
    if tuple(phases) == (0, 1, 2):
        B.check(lib.tpk_tree_attn_bwd_ex(B.BWD_ALL, *args), "tpk_tree_attn_bwd_ex")
    else:
        for ph in phases:
            B.check(lib.tpk_tree_attn_bwd_ex(int(ph), *args), "tpk_tree_attn_bwd_ex")
    return dq, dk, dv


def scatter_token_index(token_index, src=None, lse_src=None, dst=None, lse_dst=None):
    """Raw-order copies: dst[r] = src[token_index[r]], lse_dst[:, r] = lse_src[:, token_index[r]]."""
    lib = B.load()
    _need(token_index, torch.int32, "token_index", 1)
    R = token_index.numel()
    if src is not None:
        _need(src, torch.bfloat16, "src", 3)
        F, H, d = src.shape
        if dst is None:
            dst = torch.empty((R, H, d), dtype=src.dtype, device=src.device)
    if lse_src is not None:
        _need(lse_src, torch.float32, "lse_src", 2)
        H, F = lse_src.shape
        if lse_dst is None:
            lse_dst = torch.empty((H, R), dtype=torch.float32, device=lse_src.device)
    if src is None and lse_src is None:
        return None, None
    d = src.shape[2] if src is not None else 8
    B.check(lib.tpk_scatter_token_index(_ptr(token_index), R, F, _ptr(src), _ptr(dst), _ptr(lse_src),
                                        _ptr(lse_dst), H, d, _stream()), "tpk_scatter_token_index")
    return dst, lse_dst


def gather_to_forwarded(dplan, src, dst=None):
    """Packed-layout copy of a per-raw-token payload: dst[f] = src[owner of f].

    ``src`` is any contiguous device tensor whose first dimension is the raw
    token (R); every forwarded position takes its owner's row (the lowest
    raw token mapping to it)."""
    lib = B.load()
    R, F = dplan.n_raw, dplan.n_fwd
    if not src.is_cuda or not src.is_contiguous() or src.shape[0] != R:
        raise ValueError("src must be a contiguous device tensor with %d rows" % R)
    if dst is None:
        dst = torch.empty((F,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    if dst.dtype != src.dtype or tuple(dst.shape) != (F,) + tuple(src.shape[1:]) or not dst.is_contiguous():
        raise ValueError("dst must be a contiguous %s tensor of shape %s" % (src.dtype, (F,) + tuple(src.shape[1:])))
    row_bytes = src[0].numel() * src.element_size() if R else 1
    B.check(lib.tpk_gather_to_forwarded(_ptr(dplan.fwd_raw_begin), _ptr(dplan.fwd_raw), F, R, _ptr(src), _ptr(dst),
                                        row_bytes, _stream()), "tpk_gather_to_forwarded")
    return dst


def sum_to_forwarded(dplan, src=None, lse_src=None, dst=None, lse_dst=None):
    """Adjoint of the raw-order scatter: dst[f] = sum of src[r] over the raw tokens r of f.

    ``src`` [R, H, d] bf16 -> [F, H, d] bf16; ``lse_src`` [H, R] fp32 -> [H, F]
    (a per-token fp32 weight is the case H = 1).  fp32 sums in ascending raw
    order."""
    lib = B.load()
    R, F = dplan.n_raw, dplan.n_fwd
    H, d = 1, 8
    if src is not None:
        _need(src, torch.bfloat16, "src", 3)
        if src.shape[0] != R:
            raise ValueError("src must have %d rows" % R)
        _, H, d = src.shape
        if dst is None:
            dst = torch.empty((F, H, d), dtype=src.dtype, device=src.device)
    if lse_src is not None:
        _need(lse_src, torch.float32, "lse_src", 2)
        if lse_src.shape[1] != R or (src is not None and lse_src.shape[0] != H):
            raise ValueError("lse_src must be [H, %d]" % R)
        H = lse_src.shape[0]
        if lse_dst is None:
            lse_dst = torch.empty((H, F), dtype=torch.float32, device=lse_src.device)
    if src is None and lse_src is None:
        return None, None
    B.check(lib.tpk_sum_to_forwarded(_ptr(dplan.fwd_raw_begin), _ptr(dplan.fwd_raw), F, R, _ptr(src), _ptr(dst),
                                     _ptr(lse_src), _ptr(lse_dst), H, d, _stream()), "tpk_sum_to_forwarded")
    return dst, lse_dst


def gdn_conv(dplan, x, w, y=None):
    """Causal depthwise convolution + SiLU along each position's path
    (``tpk_gdn_conv``): x [F, C] bf16, w [C, W] fp32 -> y [F, C] bf16."""
    lib = B.load()
    _need(x, torch.bfloat16, "x", 2, cuda=False)
    _need(w, torch.float32, "w", 2, cuda=False)
    F, C = x.shape
    if F != dplan.n_fwd:
        raise ValueError("x has %d rows, the plan has %d forwarded positions" % (F, dplan.n_fwd))
    if w.shape[0] != C:
        raise ValueError("w must have shape (%d, W)" % C)
    y = torch.empty_like(x) if y is None else y
    _need(y, torch.bfloat16, "y", 2, cuda=False)
    _shape(y, (F, C), "y")
    _on_device(x, (w, "w"), (y, "y"), (dplan.image, "the plan image"))
    B.check(lib.tpk_gdn_conv(dplan.plan.handle, _ptr(dplan.image), _ptr(x), _ptr(w), _ptr(y), C, w.shape[1],
                             _stream()), "tpk_gdn_conv")
    return y


def gdn_delta_rule(dplan, q, k, v, g, beta, scale=None, out=None, workspace=None):
    """Gated delta rule along every root-to-leaf path (``tpk_gdn_delta_rule``).

    q, k [F, H, dk] and v [F, H, dv] bf16 -- views whose rows may be strided
    (e.g. column slices of the convolution's output), unit stride inside a
    row; g (log decay), beta [F, H] fp32.  Returns o [F, H, dv] bf16."""
    lib = B.load()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 3:
            raise TypeError("%s must be a 3-d bf16 tensor" % n)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError("%s: heads and elements must be contiguous inside a row" % n)
    F, H, dk = q.shape
    dv = v.shape[2]
    if F != dplan.n_fwd:
        raise ValueError("q has %d rows, the plan has %d forwarded positions" % (F, dplan.n_fwd))
    _shape(k, (F, H, dk), "k")
    _shape(v, (F, H, dv), "v")
    if q.stride(0) != k.stride(0):
        raise ValueError("q and k must share one row stride")
    for t, n in ((g, "g"), (beta, "beta")):
        _need(t, torch.float32, n, 2, cuda=False)
        _shape(t, (F, H), n)
    scale = 1.0 / math.sqrt(dk) if scale is None else float(scale)
    out = torch.empty((F, H, dv), dtype=torch.bfloat16, device=q.device) if out is None else out
    _need(out, torch.bfloat16, "out", 3, cuda=False)
    _shape(out, (F, H, dv), "out")
    need = int(lib.tpk_gdn_workspace_bytes(dplan.plan.handle, H, dk, dv))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if ws_bytes < need:
        raise ValueError("workspace has %d bytes, the delta rule needs %d" % (ws_bytes, need))
    _on_device(q, (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (out, "out"), (workspace, "workspace"),
               (dplan.image, "the plan image"))
    B.check(lib.tpk_gdn_delta_rule(dplan.plan.handle, _ptr(dplan.image), _ptr(q), _ptr(k), _ptr(v), q.stride(0),
                                   v.stride(0), _ptr(g), _ptr(beta), _ptr(out), H, dk, dv, scale, _ptr(workspace),
                                   ws_bytes, _stream()), "tpk_gdn_delta_rule")
    return out


def gdn_workspace(dplan, H, dk, dv):
    """A workspace for ``gdn_delta_rule`` (its saved per-instance final
    states); keep it for ``gdn_delta_rule_bwd``."""
    lib = B.load()
    need = int(lib.tpk_gdn_workspace_bytes(dplan.plan.handle, H, dk, dv))
    return torch.empty(max(need, 256), dtype=torch.uint8, device=dplan.image.device)


def _rows3(t, name, shape=None):
    """A 3-d bf16 view whose rows may be strided, contiguous inside a row."""
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or t.dim() != 3:
        raise TypeError("%s must be a 3-d bf16 tensor" % name)
    if shape is not None:
        _shape(t, shape, name)
    if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError("%s: heads and elements must be contiguous inside a row" % name)


def gdn_conv_bwd(dplan, x, w, dy, dx=None, dw=None, workspace=None):
    """Gradients of ``gdn_conv`` (``tpk_gdn_conv_bwd``): x, dy [F, C] bf16,
    w [C, W] fp32 -> (dx [F, C] bf16, dw [C, W] fp32)."""
    lib = B.load()
    _need(x, torch.bfloat16, "x", 2, cuda=False)
    _need(w, torch.float32, "w", 2, cuda=False)
    _need(dy, torch.bfloat16, "dy", 2, cuda=False)
    F, C = x.shape
    W = w.shape[1]
    if F != dplan.n_fwd:
        raise ValueError("x has %d rows, the plan has %d forwarded positions" % (F, dplan.n_fwd))
    if w.shape[0] != C:
        raise ValueError("w must have shape (%d, W)" % C)
    _shape(dy, (F, C), "dy")
    dx = torch.empty_like(x) if dx is None else dx
    dw = torch.empty_like(w) if dw is None else dw
    _need(dx, torch.bfloat16, "dx", 2, cuda=False)
    _shape(dx, (F, C), "dx")
    _need(dw, torch.float32, "dw", 2, cuda=False)
    _shape(dw, (C, W), "dw")
    need = int(lib.tpk_gdn_conv_bwd_workspace_bytes(dplan.plan.handle, C, W))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if ws_bytes < need:
        raise ValueError("workspace has %d bytes, the convolution's backward needs %d" % (ws_bytes, need))
    _on_device(x, (w, "w"), (dy, "dy"), (dx, "dx"), (dw, "dw"), (workspace, "workspace"),
               (dplan.image, "the plan image"))
    B.check(lib.tpk_gdn_conv_bwd(dplan.plan.handle, _ptr(dplan.image), _ptr(x), _ptr(w), _ptr(dy), _ptr(dx), _ptr(dw),
                                 C, W, _ptr(workspace), ws_bytes, _stream()), "tpk_gdn_conv_bwd")
    return dx, dw


def gdn_delta_rule_bwd(dplan, q, k, v, g, beta, dout, state, scale=None, dq=None, dk=None, dv=None, dg=None,
                       dbeta=None, workspace=None):
    """Gradients of ``gdn_delta_rule`` (``tpk_gdn_delta_rule_bwd``).

    q, k, v, g, beta as given to the forward; ``state`` the workspace the
    forward filled; dout [F, H, dv] bf16.  dq, dk (sharing one row stride)
    and dv may be strided views, e.g. column slices of one [F, C] gradient.
    Returns (dq, dk, dv, dg, dbeta)."""
    lib = B.load()
    _rows3(q, "q")
    F, H, dkk = q.shape
    dvv = v.shape[2]
    if F != dplan.n_fwd:
        raise ValueError("q has %d rows, the plan has %d forwarded positions" % (F, dplan.n_fwd))
    _rows3(k, "k", (F, H, dkk))
    _rows3(v, "v", (F, H, dvv))
    if q.stride(0) != k.stride(0):
        raise ValueError("q and k must share one row stride")
    for t, n in ((g, "g"), (beta, "beta")):
        _need(t, torch.float32, n, 2, cuda=False)
        _shape(t, (F, H), n)
    _need(dout, torch.bfloat16, "dout", 3, cuda=False)
    _shape(dout, (F, H, dvv), "dout")
    dev = q.device
    dq = torch.empty((F, H, dkk), dtype=torch.bfloat16, device=dev) if dq is None else dq
    dk = torch.empty((F, H, dkk), dtype=torch.bfloat16, device=dev) if dk is None else dk
    dv = torch.empty((F, H, dvv), dtype=torch.bfloat16, device=dev) if dv is None else dv
    _rows3(dq, "dq", (F, H, dkk))
    _rows3(dk, "dk", (F, H, dkk))
    _rows3(dv, "dv", (F, H, dvv))
    if dq.stride(0) != dk.stride(0):
        raise ValueError("dq and dk must share one row stride")
    dg = torch.empty((F, H), dtype=torch.float32, device=dev) if dg is None else dg
    dbeta = torch.empty((F, H), dtype=torch.float32, device=dev) if dbeta is None else dbeta
    for t, n in ((dg, "dg"), (dbeta, "dbeta")):
        _need(t, torch.float32, n, 2, cuda=False)
        _shape(t, (F, H), n)
    if not isinstance(state, torch.Tensor):
        raise TypeError("state must be the forward's workspace tensor")
    st_bytes = state.numel() * state.element_size()
    need_st = int(lib.tpk_gdn_workspace_bytes(dplan.plan.handle, H, dkk, dvv))
    if st_bytes < need_st:
        raise ValueError("state has %d bytes, the forward's workspace has %d" % (st_bytes, need_st))
    need = int(lib.tpk_gdn_bwd_workspace_bytes(dplan.plan.handle, H, dkk, dvv))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    if ws_bytes < need:
        raise ValueError("workspace has %d bytes, the delta rule's backward needs %d" % (ws_bytes, need))
    scale = 1.0 / math.sqrt(dkk) if scale is None else float(scale)
    _on_device(q, (k, "k"), (v, "v"), (g, "g"), (beta, "beta"), (dout, "dout"), (dq, "dq"), (dk, "dk"), (dv, "dv"),
               (dg, "dg"), (dbeta, "dbeta"), (state, "state"), (workspace, "workspace"),
               (dplan.image, "the plan image"))
    B.check(lib.tpk_gdn_delta_rule_bwd(dplan.plan.handle, _ptr(dplan.image), _ptr(q), _ptr(k), _ptr(v), q.stride(0),
                                       v.stride(0), _ptr(g), _ptr(beta), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                       dq.stride(0), dv.stride(0), _ptr(dg), _ptr(dbeta), H, dkk, dvv, scale,
                                       _ptr(state), st_bytes, _ptr(workspace), ws_bytes, _stream()),
            "tpk_gdn_delta_rule_bwd")
    return dq, dk, dv, dg, dbeta
