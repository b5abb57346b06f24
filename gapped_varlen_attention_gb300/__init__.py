"""Gapped variable-length attention forward (and backward) for GB300 (sm_103a).

Public API (a thin binding of the C ABI in include/gva.h):

    plan = Plan(cu_seqlens_q, seqused_q, cu_seqlens_k, seqused_k, Hq, Hkv, d)
    forward(plan, q, k, v, out, lse, softmax_scale=0.0)   # one sm_103a kernel
    lse_merge(plan, [o0, o1], [lse0, lse1], out, lse)      # FP32 LSE merge kernel
    backward(plan, q, k, v, out, lse, d_out, dq, dk, dv)   # dQ, dK, dV kernels

The library (libgva.so) is built in-tree by ``build()``; nothing here computes on the
CPU, and calls raise if the library or a supported GPU is missing.
"""
from ._lib import (GVA_BF16, GVA_FP32, EXPORTS, GvaError, Plan, backward, backward_workspace_bytes, device_status,
                   forward, forward_noalloc, inspect_plan, load_library, lse_merge)


def build(force: bool = False, verbose: bool = False) -> str:
    from ._build import build as _build
    return _build(force=force, verbose=verbose)


__all__ = ["Plan", "forward", "forward_noalloc", "lse_merge", "backward", "backward_workspace_bytes", "device_status",
           "inspect_plan", "load_library", "build", "GvaError", "EXPORTS",
           "GVA_BF16", "GVA_FP32"]
