"""ctypes binding of libgva.so (include/gva.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module checks
shapes and dtypes, hands over device pointers and the current torch stream, and turns
status codes into exceptions. There is no fallback: if the library is missing or the
device is unsupported, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libgva.so")

GVA_OK, GVA_ERR_INVALID_ARG, GVA_ERR_UNSUPPORTED, GVA_ERR_CUDA, GVA_ERR_DEVICE_CHECK = range(5)
GVA_BF16, GVA_FP32 = 0, 1

# Every symbol include/gva.h declares.
EXPORTS = ("gva_plan", "gva_forward", "gva_lse_merge", "gva_plan_destroy", "gva_plan_get_info",
           "gva_device_status", "gva_status_string", "gva_last_error", "gva_forward_noalloc", "gva_plan_ranges",
           "gva_plan_causal", "gva_backward_workspace_size", "gva_backward", "gva_plan_inspect")
NOALLOC_MAX_WORK_ITEMS = 32768  # GVA_NOALLOC_MAX_WORK_ITEMS in include/gva.h


class GvaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_segments", ctypes.c_int32), ("num_heads_q", ctypes.c_int32),
                ("num_heads_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("total_q", ctypes.c_int64), ("total_k", ctypes.c_int64),
                ("num_work_items", ctypes.c_int32), ("num_merge_units", ctypes.c_int32),
                ("grid_ctas", ctypes.c_int32), ("sm_count", ctypes.c_int32),
                ("used_flops", ctypes.c_double)]


class WorkSummary(ctypes.Structure):
    _fields_ = [("num_work_items", ctypes.c_int32), ("num_key_blocks", ctypes.c_int32),
                ("num_merge_units", ctypes.c_int32), ("num_bwd_items", ctypes.c_int32),
                ("num_kv_units", ctypes.c_int32), ("backward_ok", ctypes.c_int32), ("used_flops", ctypes.c_double),
                ("num_walk_entries", ctypes.c_int32), ("num_kv_segs", ctypes.c_int32)]


_lib = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libgva.so (built by ``__graft_entry__.build()``); raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    i32, vp, f32 = ctypes.c_int32, ctypes.c_void_p, ctypes.c_float
    pi32 = ctypes.POINTER(ctypes.c_int32)
    lib.gva_plan.argtypes = [pi32, pi32, pi32, pi32, i32, i32, i32, i32, ctypes.POINTER(vp)]
    lib.gva_forward.argtypes = [vp, vp, vp, vp, vp, i32, vp, f32, vp]
    lib.gva_lse_merge.argtypes = [vp, i32, ctypes.POINTER(vp), i32, ctypes.POINTER(vp), vp, i32, vp, vp]
    lib.gva_plan_destroy.argtypes = [vp]
    lib.gva_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
    lib.gva_device_status.argtypes = [vp]
    lib.gva_status_string.argtypes = [i32]
    lib.gva_status_string.restype = ctypes.c_char_p
    lib.gva_last_error.argtypes = []
    lib.gva_last_error.restype = ctypes.c_char_p
    lib.gva_forward_noalloc.argtypes = [pi32, pi32, pi32, pi32, i32, i32, i32, i32, vp, vp, vp, vp, i32, vp, f32,
                                        vp]
    lib.gva_plan_causal.argtypes = [pi32, pi32, pi32, pi32, i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
    lib.gva_plan_ranges.argtypes = [pi32, pi32, i32, pi32, pi32, pi32, ctypes.c_int64, i32, i32, i32,
                                    ctypes.POINTER(vp)]
    lib.gva_backward_workspace_size.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
    lib.gva_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, vp, ctypes.c_size_t, f32, vp]
    lib.gva_plan_inspect.argtypes = [pi32, pi32, pi32, pi32, i32, pi32, pi32, pi32, ctypes.c_int64, i32, i32, i32,
                                     i32, i32, i32, ctypes.POINTER(WorkSummary), pi32, i32, pi32, i32, pi32, i32,
                                     pi32, i32, pi32, i32]
    for name in ("gva_plan", "gva_forward", "gva_lse_merge", "gva_plan_destroy", "gva_plan_get_info",
                 "gva_device_status", "gva_forward_noalloc", "gva_plan_ranges", "gva_plan_causal",
                 "gva_backward_workspace_size", "gva_backward", "gva_plan_inspect"):
        getattr(lib, name).restype = i32
    if path is None:
        _lib = lib
    return lib


def _check(lib, status: int, what: str):
    if status != GVA_OK:
        name = lib.gva_status_string(status).decode()
        detail = lib.gva_last_error().decode()
        raise GvaError(status, f"{what}: {name}: {detail}")


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


WORK_ITEM_FIELDS = ("q_row0", "q_rows", "blk0", "nblk", "head_kv", "n_tiles", "k_len", "q_pos0")
KV_UNIT_FIELDS = ("key_row0", "keys", "seg0", "n_tiles", "head_kv", "tile0", "key_pos0", "pos_shift")
KV_SEG_FIELDS = ("q_row0", "q_used")


def inspect_plan(cu_seqlens_q, seqused_q, cu_seqlens_k, seqused_k, num_heads_q: int, num_heads_kv: int,
                 head_dim: int, causal_block: int = 0, key_ranges=None, total_k: int = 0, grid: int = 152) -> dict:
    """``gva_plan_inspect``: the work lists a plan of this geometry holds, built on the
    host (no CUDA call). With ``key_ranges`` (per segment a list of ``(start, length)``
    K/V row ranges, as ``Plan.from_ranges``) the keys are those ranges and
    ``cu_seqlens_k`` / ``seqused_k`` are not used. Returns the counts, ``backward_ok``,
    ``used_flops`` and three int32 arrays of 8 columns in the kernels' order: ``items``
    (forward, fields ``WORK_ITEM_FIELDS``), ``bwd_items`` (dQ, same fields) and
    ``kv_units`` (dK / dV, ``KV_UNIT_FIELDS``), ``kv_segs`` (the segments the dK / dV
    units list, 2 columns ``KV_SEG_FIELDS``), plus ``walk``, ``bwd_walk`` and
    ``kv_walk``: each list as a grid of min(``grid``, its length) CTAs walks it (per
    entry the index into the list, -1 for padding)."""
    lib = load_library()
    q = [_i32(x) for x in (cu_seqlens_q, seqused_q)]
    n = int(q[1].shape[0])
    p = lambda x: x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    if key_ranges is not None:
        off = _i32(np.concatenate([[0], np.cumsum([len(r) for r in key_ranges])]))
        flat = [x for r in key_ranges for x in r]
        st = _i32([a for a, _ in flat]) if flat else _i32(np.zeros(1))
        ln = _i32([b for _, b in flat]) if flat else _i32(np.zeros(1))
        keys = [None, None, p(off), p(st), p(ln), int(total_k)]
    else:
        k = [_i32(x) for x in (cu_seqlens_k, seqused_k)]
        keys = [p(k[0]), p(k[1]), None, None, None, 0]
    summ = WorkSummary()
    args = [p(q[0]), p(q[1]), keys[0], keys[1], n, keys[2], keys[3], keys[4], keys[5], int(causal_block),
            int(num_heads_q), int(num_heads_kv), int(head_dim), int(grid)]
    _check(lib, lib.gva_plan_inspect(*args, 0, ctypes.byref(summ), None, 0, None, 0, None, 0, None, 0, None, 0),
           "gva_plan_inspect")
    items = np.zeros((max(summ.num_work_items, 1), 8), np.int32)
    segs = np.zeros((max(summ.num_kv_segs, 1), 2), np.int32)
    bwd = np.zeros((max(summ.num_bwd_items, 1), 8), np.int32)
    kvu = np.zeros((max(summ.num_kv_units, 1), 8), np.int32)
    walks = []
    for kind in range(3):  # forward items, dQ items, dK / dV units
        s2 = WorkSummary()
        _check(lib, lib.gva_plan_inspect(*args, kind, ctypes.byref(s2), None, 0, None, 0, None, 0, None, 0, None, 0),
               "gva_plan_inspect")
        walk = np.zeros(max(s2.num_walk_entries, 1), np.int32)
        _check(lib, lib.gva_plan_inspect(*args, kind, ctypes.byref(s2), p(items), summ.num_work_items, p(walk),
                                         s2.num_walk_entries, p(bwd), summ.num_bwd_items, p(kvu),
                                         summ.num_kv_units, p(segs), summ.num_kv_segs), "gva_plan_inspect")
        walks.append(walk[:s2.num_walk_entries])
    return {"num_work_items": summ.num_work_items, "num_key_blocks": summ.num_key_blocks,
            "num_merge_units": summ.num_merge_units, "num_bwd_items": summ.num_bwd_items,
            "num_kv_units": summ.num_kv_units, "backward_ok": bool(summ.backward_ok), "used_flops": summ.used_flops,
            "items": items[:summ.num_work_items], "walk": walks[0], "bwd_walk": walks[1], "kv_walk": walks[2],
            "bwd_items": bwd[:summ.num_bwd_items],
            "kv_units": kvu[:summ.num_kv_units], "kv_segs": segs[:summ.num_kv_segs]}


class Plan:
    """A validated segment geometry with its device work list (``gva_plan``)."""

    def __init__(self, cu_seqlens_q, seqused_q, cu_seqlens_k, seqused_k, num_heads_q: int, num_heads_kv: int,
                 head_dim: int, causal_block: int = 0):
        """``causal_block`` > 0 builds a block-causal plan (``gva_plan_causal``)."""
        self._lib = load_library()
        self.cu_q, self.used_q = _i32(cu_seqlens_q), _i32(seqused_q)
        self.cu_k, self.used_k = _i32(cu_seqlens_k), _i32(seqused_k)
        n = int(self.used_q.shape[0])
        if self.cu_q.shape[0] != n + 1 or self.cu_k.shape[0] != n + 1 or self.used_k.shape[0] != n:
            raise ValueError("cu_seqlens must have num_segments + 1 entries and seqused num_segments")
        ptr = ctypes.c_void_p()
        as_p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
        if causal_block:
            st = self._lib.gva_plan_causal(as_p(self.cu_q), as_p(self.used_q), as_p(self.cu_k), as_p(self.used_k),
                                           n, int(causal_block), int(num_heads_q), int(num_heads_kv), int(head_dim),
                                           ctypes.byref(ptr))
            _check(self._lib, st, "gva_plan_causal")
        else:
            st = self._lib.gva_plan(as_p(self.cu_q), as_p(self.used_q), as_p(self.cu_k), as_p(self.used_k), n,
                                    int(num_heads_q), int(num_heads_kv), int(head_dim), ctypes.byref(ptr))
            _check(self._lib, st, "gva_plan")
        self.causal_block = int(causal_block)
        self._handle = ptr
        self.num_heads_q, self.num_heads_kv, self.head_dim = int(num_heads_q), int(num_heads_kv), int(head_dim)
        self.total_q, self.total_k = int(self.cu_q[-1]), int(self.cu_k[-1])

    @classmethod
    def from_geometry(cls, g, causal_block: int = 0) -> "Plan":
        return cls(g.cu_q, g.used_q, g.cu_k, g.used_k, g.num_heads_q, g.num_heads_kv, g.head_dim, causal_block)

    @classmethod
    def from_ranges(cls, cu_seqlens_q, seqused_q, key_ranges, total_k: int, num_heads_q: int, num_heads_kv: int,
                    head_dim: int) -> "Plan":
        """``gva_plan_ranges``: segment b attends the concatenation of the K/V row ranges
        ``key_ranges[b]`` (a list of ``(start, length)`` pairs)."""
        self = cls.__new__(cls)
        self._lib = load_library()
        self.cu_q, self.used_q = _i32(cu_seqlens_q), _i32(seqused_q)
        n = int(self.used_q.shape[0])
        if self.cu_q.shape[0] != n + 1 or len(key_ranges) != n:
            raise ValueError("cu_seqlens_q must have num_segments + 1 entries, seqused_q and key_ranges num_segments")
        off = _i32(np.concatenate([[0], np.cumsum([len(r) for r in key_ranges])]))
        flat = [x for r in key_ranges for x in r]
        starts = _i32([st for st, _ in flat]) if flat else _i32(np.zeros(1))
        lens = _i32([ln for _, ln in flat]) if flat else _i32(np.zeros(1))
        ptr = ctypes.c_void_p()
        as_p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
        st = self._lib.gva_plan_ranges(as_p(self.cu_q), as_p(self.used_q), n, as_p(off), as_p(starts), as_p(lens),
                                       int(total_k), int(num_heads_q), int(num_heads_kv), int(head_dim),
                                       ctypes.byref(ptr))
        _check(self._lib, st, "gva_plan_ranges")
        self._handle = ptr
        self.num_heads_q, self.num_heads_kv, self.head_dim = int(num_heads_q), int(num_heads_kv), int(head_dim)
        self.total_q, self.total_k = int(self.cu_q[-1]), int(total_k)
        self.cu_k = self.used_k = None
        self.causal_block = 0
        return self

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._handle is None:
            raise RuntimeError("plan was destroyed")
        return self._handle

    def info(self) -> dict:
        inf = PlanInfo()
        _check(self._lib, self._lib.gva_plan_get_info(self.handle, ctypes.byref(inf)), "gva_plan_get_info")
        return {name: getattr(inf, name) for name, _ in PlanInfo._fields_}

    def close(self):
        if getattr(self, "_handle", None) is not None:
            self._lib.gva_plan_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _stream_ptr(stream) -> ctypes.c_void_p:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev_ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def forward(plan: Plan, q, k, v, out, lse, softmax_scale: float = 0.0, stream=None):
    """``gva_forward``: write O and LSE of the used rows into ``out`` / ``lse``.

    q [total_q, Hq, d] bf16, k / v [total_k, Hkv, d] bf16, out [total_q, Hq, d] bf16
    or fp32, lse [Hq, total_q] fp32, all contiguous CUDA tensors."""
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k and v must be bfloat16")
    if out.dtype not in (torch.bfloat16, torch.float32) or lse.dtype != torch.float32:
        raise TypeError("out must be bfloat16 or float32 and lse float32")
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    hq, hkv, d = plan.num_heads_q, plan.num_heads_kv, plan.head_dim
    if tuple(q.shape) != (plan.total_q, hq, d) or tuple(out.shape) != (plan.total_q, hq, d):
        raise ValueError(f"q / out must be [{plan.total_q}, {hq}, {d}]")
    if tuple(k.shape) != (plan.total_k, hkv, d) or tuple(v.shape) != (plan.total_k, hkv, d):
        raise ValueError(f"k / v must be [{plan.total_k}, {hkv}, {d}]")
    if tuple(lse.shape) != (hq, plan.total_q):
        raise ValueError(f"lse must be [{hq}, {plan.total_q}]")
    lib = plan._lib
    st = lib.gva_forward(plan.handle, _dev_ptr(q), _dev_ptr(k), _dev_ptr(v), _dev_ptr(out),
                         GVA_FP32 if out.dtype == torch.float32 else GVA_BF16, _dev_ptr(lse),
                         float(softmax_scale), _stream_ptr(stream))
    _check(lib, st, "gva_forward")
    return out, lse


def lse_merge(plan: Plan, outs: Sequence, lses: Sequence, out, lse, stream=None):
    """``gva_lse_merge``: combine partial results of disjoint key sets of plan's rows."""
    import torch
    if len(outs) != len(lses) or not outs:
        raise ValueError("need one LSE per partial output and at least one partition")
    in_dtype = outs[0].dtype
    for o, l in zip(outs, lses):
        if o.dtype != in_dtype or o.dtype not in (torch.bfloat16, torch.float32) or l.dtype != torch.float32:
            raise TypeError("partials must share one dtype (bf16 or fp32) with fp32 LSEs")
        if tuple(o.shape) != (plan.total_q, plan.num_heads_q, plan.head_dim) or tuple(l.shape) != (
                plan.num_heads_q, plan.total_q):
            raise ValueError("partial shapes do not match the plan")
        if not (o.is_cuda and l.is_cuda and o.is_contiguous() and l.is_contiguous()):
            raise ValueError("partials must be contiguous CUDA tensors")
    if tuple(out.shape) != tuple(outs[0].shape) or tuple(lse.shape) != tuple(lses[0].shape):
        raise ValueError("out / lse shapes do not match the plan")
    if not (out.is_cuda and lse.is_cuda and out.is_contiguous() and lse.is_contiguous()):
        raise ValueError("out / lse must be contiguous CUDA tensors")
    n = len(outs)
    po = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    pl = (ctypes.c_void_p * n)(*[l.data_ptr() for l in lses])
    lib = plan._lib
    st = lib.gva_lse_merge(plan.handle, n, po, GVA_FP32 if in_dtype == torch.float32 else GVA_BF16, pl,
                           _dev_ptr(out), GVA_FP32 if out.dtype == torch.float32 else GVA_BF16, _dev_ptr(lse),
                           _stream_ptr(stream))
    _check(lib, st, "gva_lse_merge")
    return out, lse


def backward_workspace_bytes(plan: Plan) -> int:
    """``gva_backward_workspace_size``: device scratch bytes ``backward`` needs."""
    n = ctypes.c_size_t()
    _check(plan._lib, plan._lib.gva_backward_workspace_size(plan.handle, ctypes.byref(n)),
           "gva_backward_workspace_size")
    return int(n.value)


def backward(plan: Plan, q, k, v, out, lse, d_out, dq, dk, dv, softmax_scale: float = 0.0, workspace=None,
             stream=None):
    """``gva_backward``: dQ, dK, dV of the forward (``out`` / ``lse`` from ``forward`` on
    the same inputs) for the output gradient ``d_out``.

    q, out, d_out [total_q, Hq, d] bf16; k, v [total_k, Hkv, d] bf16; lse [Hq, total_q]
    fp32; dq [total_q, Hq, d] and dk / dv [total_k, Hkv, d] bf16 or fp32 (dk and dv the
    same dtype). ``workspace``: a CUDA uint8 tensor of at least
    ``backward_workspace_bytes(plan)`` bytes, allocated here if None."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("d_out", d_out)):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
    if lse.dtype != torch.float32:
        raise TypeError("lse must be float32")
    if dq.dtype not in (torch.bfloat16, torch.float32) or dk.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("dq / dk / dv must be bfloat16 or float32")
    if dv.dtype != dk.dtype:
        raise TypeError("dk and dv must share one dtype")
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse), ("d_out", d_out), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    hq, hkv, d = plan.num_heads_q, plan.num_heads_kv, plan.head_dim
    for name, t in (("q", q), ("out", out), ("d_out", d_out), ("dq", dq)):
        if tuple(t.shape) != (plan.total_q, hq, d):
            raise ValueError(f"{name} must be [{plan.total_q}, {hq}, {d}]")
    for name, t in (("k", k), ("v", v), ("dk", dk), ("dv", dv)):
        if tuple(t.shape) != (plan.total_k, hkv, d):
            raise ValueError(f"{name} must be [{plan.total_k}, {hkv}, {d}]")
    if tuple(lse.shape) != (hq, plan.total_q):
        raise ValueError(f"lse must be [{hq}, {plan.total_q}]")
    need = backward_workspace_bytes(plan)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    lib = plan._lib
    st = lib.gva_backward(plan.handle, _dev_ptr(q), _dev_ptr(k), _dev_ptr(v), _dev_ptr(out), _dev_ptr(d_out),
                          _dev_ptr(lse), _dev_ptr(dq), GVA_FP32 if dq.dtype == torch.float32 else GVA_BF16,
                          _dev_ptr(dk), _dev_ptr(dv), GVA_FP32 if dk.dtype == torch.float32 else GVA_BF16,
                          _dev_ptr(workspace), workspace.numel() * workspace.element_size(), float(softmax_scale),
                          _stream_ptr(stream))
    _check(lib, st, "gva_backward")
    return dq, dk, dv


def device_status(plan: Plan = None):
    """Synchronise and raise if a kernel of this plan recorded a device-side failure;
    without a plan, the same for the last ``forward_noalloc`` launch on the current
    device (whose error word lives in the library's fixed scratch)."""
    lib = plan._lib if plan is not None else load_library()
    _check(lib, lib.gva_device_status(plan.handle if plan is not None else None), "gva_device_status")


def forward_noalloc(cu_seqlens_q, seqused_q, cu_seqlens_k, seqused_k, num_heads_q: int, num_heads_kv: int,
                    q, k, v, out, lse, softmax_scale: float = 0.0, stream=None):
    """``gva_forward_noalloc``: the forward without a plan, for callers that may not
    allocate device memory (the work list goes to a fixed scratch array inside the
    library). Same tensors as ``forward``; the geometry is given as host arrays."""
    import torch
    lib = load_library()
    a = [_i32(x) for x in (cu_seqlens_q, seqused_q, cu_seqlens_k, seqused_k)]
    n = int(a[1].shape[0])
    if a[0].shape[0] != n + 1 or a[2].shape[0] != n + 1 or a[3].shape[0] != n:
        raise ValueError("cu_seqlens must have num_segments + 1 entries and seqused num_segments")
    d = int(q.shape[-1])
    total_q, total_k = int(a[0][-1]), int(a[2][-1])
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k and v must be bfloat16")
    if out.dtype not in (torch.bfloat16, torch.float32) or lse.dtype != torch.float32:
        raise TypeError("out must be bfloat16 or float32 and lse float32")
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if tuple(q.shape) != (total_q, num_heads_q, d) or tuple(out.shape) != (total_q, num_heads_q, d):
        raise ValueError(f"q / out must be [{total_q}, {num_heads_q}, {d}]")
    if tuple(k.shape) != (total_k, num_heads_kv, d) or tuple(v.shape) != (total_k, num_heads_kv, d):
        raise ValueError(f"k / v must be [{total_k}, {num_heads_kv}, {d}]")
    if tuple(lse.shape) != (num_heads_q, total_q):
        raise ValueError(f"lse must be [{num_heads_q}, {total_q}]")
    as_p = lambda x: x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    st = lib.gva_forward_noalloc(as_p(a[0]), as_p(a[1]), as_p(a[2]), as_p(a[3]), n, int(num_heads_q),
                                 int(num_heads_kv), d, _dev_ptr(q), _dev_ptr(k), _dev_ptr(v), _dev_ptr(out),
                                 GVA_FP32 if out.dtype == torch.float32 else GVA_BF16, _dev_ptr(lse),
                                 float(softmax_scale), _stream_ptr(stream))
    _check(lib, st, "gva_forward_noalloc")
    return out, lse
