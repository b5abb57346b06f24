"""FP64 CPU oracle for the gapped variable-length attention forward, its LSE merge and
its backward.

TEST INFRASTRUCTURE ONLY. This module is the correctness reference that the CUDA
path is checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import it; the library itself
never does, and it shares no code with the library.

What it computes (plain definition, FP64 throughout, bf16 inputs widened exactly):

cosmos-framework PR #302 ("fix(mot): gapped replay on GPUs FlashAttention-4 has no
kernels for (sm120)"), section "What": every segment ``b`` has query rows
``cu_q[b] .. cu_q[b+1]`` and key rows ``cu_k[b] .. cu_k[b+1]``; only the first
``used_q[b]`` query rows attend, and only to the first ``used_k[b]`` keys. Rows past
a segment's used length are left as they are; a segment with no keys gets a zero
output and a log-sum-exp of -inf. Its "Tests" section names the check used here:
a per-segment FP64 reference.

For query head ``h`` of a row ``r < cu_q[b] + used_q[b]`` (KV head ``h // (Hq/Hkv)``,
the contiguous GQA grouping):

    x_j   = s * <Q[r, h], K[cu_k[b] + j, h_kv]>      for j < used_k[b]
    M     = max_j x_j,   l = sum_j exp(x_j - M)
    O[r,h]= sum_j exp(x_j - M) V[cu_k[b] + j, h_kv] / l
    LSE[h, r] = M + ln l                             (natural log of scaled logits)

with ``s = 1/sqrt(d)`` unless given. Zero-padded keys are never part of the sum:
each one would add exp(0) = 1 to ``l`` (TensorRT-LLM issue #18687, "actual
behavior").

The LSE merge (cosmos-framework PR #312, "Problem and behavior": visibility
partitions combined by an FP32 LSE merge) combines partial results of disjoint key
sets of the same query rows:

    L = max_p lse_p;   if L = -inf:  O = 0, lse = -inf
    else  w_p = exp(lse_p - L),  lse = L + ln sum_p w_p,  O = sum_p w_p O_p / sum_p w_p

Block-causal masking within a segment (``causal_block``) restricts row i to keys
j < (floor(pos / B) + 1) * B with pos = i + used_k - used_q: a single launch covers the
causal replay that the visibility partitions of PR #312 split into maskless launches.

The backward (``attention_backward``) is the gradient of that definition: with P the
softmax and dO the output gradient, dP_ij = <dO_i, V_j>, D_i = <dO_i, O_i>,
dS_ij = P_ij (dP_ij - D_i), dQ_i = s sum_j dS_ij K_j, dK_j = s sum_i dS_ij Q_i and
dV_j = sum_i P_ij dO_i, the sums over i running over the query heads of the KV head.

Score blocks are sized from a byte budget rather than a fixed row count (the
review of PR #302 on the FP32 fallback's score block), so long segments do not
materialise a huge score matrix.

Every function here is pinned by ``tests/test_oracle.py`` against brute force,
closed forms, library routines and invariants.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

__all__ = ["attention_backward", "attention_backward_ranges", "attention_forward", "attention_forward_ranges",
           "attention_rows", "causal_limits", "lse_merge", "used_flops"]

DEFAULT_BUDGET_BYTES = 1 << 30


def _as_f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: widen through float32 (exact for bf16)
        x = x.detach().cpu().float().numpy()
    return np.asarray(x)


def used_flops(used_q, used_k, num_heads_q: int, head_dim: int) -> float:
    """Useful FLOPs: 2*d per score for QK^T and 2*d per score for PV."""
    uq = np.asarray(used_q, np.float64)
    uk = np.asarray(used_k, np.float64)
    return 4.0 * head_dim * num_heads_q * float(np.sum(uq * uk))


def _segment_attention(qs: np.ndarray, ks: np.ndarray, vs: np.ndarray, scale: float,
                       budget_bytes: int):
    """Softmax attention of ``qs`` [n, d] over ``ks``/``vs`` [m, d], FP64, m >= 1.

    Returns (O [n, d], LSE [n]). The score block holds at most ``budget_bytes``."""
    n, m = qs.shape[0], ks.shape[0]
    rows = max(1, int(budget_bytes) // (8 * max(m, 1)))
    o = np.empty((n, vs.shape[1]), np.float64)
    lse = np.empty(n, np.float64)
    kt = ks.T
    for r0 in range(0, n, rows):
        r1 = min(n, r0 + rows)
        x = (qs[r0:r1] @ kt) * scale  # [rows, m]
        mx = x.max(axis=1)
        e = np.exp(x - mx[:, None])
        l = e.sum(axis=1)
        o[r0:r1] = (e @ vs) / l[:, None]
        lse[r0:r1] = mx + np.log(l)
    return o, lse


def causal_limits(used_q: int, used_k: int, causal_block: int) -> np.ndarray:
    """Keys visible to each used query row of a segment under block-causal masking.

    Query row i sits at key position i + (used_k - used_q) (the queries are the last
    used_q positions of the key sequence); it sees keys j < (floor(pos / B) + 1) * B,
    capped at used_k, with B = ``causal_block`` (1: token-causal)."""
    pos = np.arange(used_q, dtype=np.int64) + (int(used_k) - int(used_q))
    lim = (np.floor_divide(pos, int(causal_block)) + 1) * int(causal_block)
    return np.clip(lim, 0, int(used_k))


def _masked_attention(qs: np.ndarray, ks: np.ndarray, vs: np.ndarray, scale: float, limits: np.ndarray):
    """Softmax attention where row r sees keys ``j < limits[r]``; rows with no key get
    O = 0 and LSE = -inf. FP64, one row block (causal workloads are small enough)."""
    x = (qs @ ks.T) * scale
    mask = np.arange(ks.shape[0])[None, :] < limits[:, None]
    x = np.where(mask, x, -np.inf)
    mx = x.max(axis=1)
    live = np.isfinite(mx)
    e = np.where(mask, np.exp(x - np.where(live, mx, 0.0)[:, None]), 0.0)
    l = e.sum(axis=1)
    o = np.where(live[:, None], (e @ vs) / np.where(live, l, 1.0)[:, None], 0.0)
    lse = np.where(live, np.where(live, mx, 0.0) + np.log(np.where(live, l, 1.0)), -np.inf)
    return o, lse


def attention_forward(q, k, v, cu_q, used_q, cu_k, used_k, *, scale: Optional[float] = None,
                      out=None, lse=None, num_heads_kv: Optional[int] = None,
                      budget_bytes: int = DEFAULT_BUDGET_BYTES, segments: Optional[Sequence[int]] = None,
                      causal_block: int = 0):
    """Gapped varlen attention forward over packed Q [total_q, Hq, d], K/V [total_k, Hkv, d].

    ``out`` ([total_q, Hq, d]) and ``lse`` ([Hq, total_q]) give the buffers' prior
    contents; rows past a segment's used length keep them (default: zeros). Returns
    FP64 (out, lse). ``segments`` restricts the work to a subset of segments.
    ``causal_block`` > 0 applies block-causal masking within each segment (see
    ``causal_limits``); 0 is the maskless forward."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    total_q, hq, d = q.shape
    hkv = k.shape[1] if num_heads_kv is None else num_heads_kv
    if hq % hkv:
        raise ValueError(f"Hq={hq} is not a multiple of Hkv={hkv}")
    g = hq // hkv
    s = 1.0 / math.sqrt(d) if scale is None else float(scale)
    cu_q = np.asarray(cu_q, np.int64)
    cu_k = np.asarray(cu_k, np.int64)
    used_q = np.asarray(used_q, np.int64)
    used_k = np.asarray(used_k, np.int64)
    o_out = np.zeros((total_q, hq, v.shape[2]), np.float64) if out is None else _as_f64(out).astype(np.float64, copy=True)
    l_out = np.zeros((hq, total_q), np.float64) if lse is None else _as_f64(lse).astype(np.float64, copy=True)
    segs = range(len(used_q)) if segments is None else segments
    for b in segs:
        r0, nq = int(cu_q[b]), int(used_q[b])
        k0, nk = int(cu_k[b]), int(used_k[b])
        if nq == 0:
            continue
        if nk == 0:  # keyless segment: zero output, -inf LSE on used rows only
            o_out[r0:r0 + nq] = 0.0
            l_out[:, r0:r0 + nq] = -np.inf
            continue
        lim = np.repeat(causal_limits(nq, nk, causal_block), g) if causal_block > 0 else None
        for hk in range(hkv):
            # the g query heads sharing KV head hk, folded into one row block
            qs = q[r0:r0 + nq, hk * g:(hk + 1) * g, :].astype(np.float64).reshape(nq * g, d)
            ks = k[k0:k0 + nk, hk, :].astype(np.float64)
            vs = v[k0:k0 + nk, hk, :].astype(np.float64)
            if lim is None:
                ob, lb = _segment_attention(qs, ks, vs, s, budget_bytes)
            else:
                ob, lb = _masked_attention(qs, ks, vs, s, lim)
            o_out[r0:r0 + nq, hk * g:(hk + 1) * g, :] = ob.reshape(nq, g, -1)
            l_out[hk * g:(hk + 1) * g, r0:r0 + nq] = lb.reshape(nq, g).T
    return o_out, l_out


def attention_forward_ranges(q, k, v, cu_q, used_q, key_ranges, *, scale: Optional[float] = None, out=None,
                             lse=None, num_heads_kv: Optional[int] = None,
                             budget_bytes: int = DEFAULT_BUDGET_BYTES):
    """The forward when a segment's keys are several row ranges of K/V.

    ``key_ranges[b]`` lists ``(start, length)`` pairs; segment b's keys are the
    concatenation of K/V rows ``start .. start + length`` over its pairs, in order.
    This is the single-launch form of the visibility partitions of cosmos-framework
    PR #312 ("Problem and behavior"), and covers valid keys that are not a prefix
    (TensorRT-LLM issue #18687, "additional notes": rank-major key order). With one
    ``(cu_k[b], used_k[b])`` pair per segment it is ``attention_forward``.
    Rows past a segment's used length keep ``out`` / ``lse``; no keys at all gives
    0 / -inf. FP64."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    total_q, hq, d = q.shape
    hkv = k.shape[1] if num_heads_kv is None else num_heads_kv
    if hq % hkv:
        raise ValueError(f"Hq={hq} is not a multiple of Hkv={hkv}")
    g = hq // hkv
    s = 1.0 / math.sqrt(d) if scale is None else float(scale)
    cu_q = np.asarray(cu_q, np.int64)
    used_q = np.asarray(used_q, np.int64)
    o_out = np.zeros((total_q, hq, v.shape[2]), np.float64) if out is None else _as_f64(out).astype(np.float64, copy=True)
    l_out = np.zeros((hq, total_q), np.float64) if lse is None else _as_f64(lse).astype(np.float64, copy=True)
    for b in range(len(used_q)):
        r0, nq = int(cu_q[b]), int(used_q[b])
        if nq == 0:
            continue
        rows = [np.arange(int(st), int(st) + int(n)) for st, n in key_ranges[b] if int(n) > 0]
        idx = np.concatenate(rows) if rows else np.zeros(0, np.int64)
        if idx.size == 0:
            o_out[r0:r0 + nq] = 0.0
            l_out[:, r0:r0 + nq] = -np.inf
            continue
        for hk in range(hkv):
            qs = q[r0:r0 + nq, hk * g:(hk + 1) * g, :].astype(np.float64).reshape(nq * g, d)
            ks = k[idx, hk, :].astype(np.float64)
            vs = v[idx, hk, :].astype(np.float64)
            ob, lb = _segment_attention(qs, ks, vs, s, budget_bytes)
            o_out[r0:r0 + nq, hk * g:(hk + 1) * g, :] = ob.reshape(nq, g, -1)
            l_out[hk * g:(hk + 1) * g, r0:r0 + nq] = lb.reshape(nq, g).T
    return o_out, l_out


def attention_rows(q, k, v, cu_q, used_q, cu_k, used_k, rows: Sequence[int], *,
                   scale: Optional[float] = None, num_heads_kv: Optional[int] = None,
                   budget_bytes: int = DEFAULT_BUDGET_BYTES, causal_block: int = 0):
    """The same definition evaluated for a list of global query rows (all heads).

    For spot checks of launches too large to evaluate in full. Every row must be a
    used row. Rows of one segment are evaluated together, with the segment's keys
    widened once per KV head. Returns (O [n, Hq, d], LSE [Hq, n]) in FP64."""
    hq, d = q.shape[1], q.shape[2]
    hkv = k.shape[1] if num_heads_kv is None else num_heads_kv
    g = hq // hkv
    s = 1.0 / math.sqrt(d) if scale is None else float(scale)
    cu_q = np.asarray(cu_q, np.int64)
    cu_k = np.asarray(cu_k, np.int64)
    used_q = np.asarray(used_q, np.int64)
    used_k = np.asarray(used_k, np.int64)
    rows = [int(r) for r in rows]
    o = np.zeros((len(rows), hq, v.shape[2]), np.float64)
    l = np.zeros((hq, len(rows)), np.float64)
    by_segment = {}
    for i, r in enumerate(rows):
        b = int(np.searchsorted(cu_q, r, side="right")) - 1  # last segment starting at or before r
        if not (0 <= b < len(used_q) and cu_q[b] <= r < cu_q[b] + used_q[b]):
            raise ValueError(f"row {r} is not a used row")
        by_segment.setdefault(b, []).append(i)
    for b, idx in by_segment.items():
        k0, nk = int(cu_k[b]), int(used_k[b])
        if nk == 0:
            l[:, idx] = -np.inf
            continue
        sel = [rows[i] for i in idx]
        lim = None
        if causal_block > 0:
            seg_lim = causal_limits(int(used_q[b]), nk, causal_block)
            lim = np.repeat(seg_lim[[r - int(cu_q[b]) for r in sel]], g)
        for hk in range(hkv):
            qs = np.concatenate([_as_f64(q[r, hk * g:(hk + 1) * g, :]) for r in sel]).astype(np.float64)
            ks = _as_f64(k[k0:k0 + nk, hk, :]).astype(np.float64)
            vs = _as_f64(v[k0:k0 + nk, hk, :]).astype(np.float64)
            if lim is None:
                ob, lb = _segment_attention(qs, ks, vs, s, budget_bytes)
            else:
                ob, lb = _masked_attention(qs, ks, vs, s, lim)
            o[idx, hk * g:(hk + 1) * g] = ob.reshape(len(sel), g, -1)
            l[hk * g:(hk + 1) * g, idx] = lb.reshape(len(sel), g).T
    return o, l


def lse_merge(outs: Sequence, lses: Sequence, cu_q, used_q, *, out=None, lse=None):
    """Combine partial results of disjoint key partitions of the same query rows.

    ``outs[p]`` is [total_q, Hq, d] and ``lses[p]`` is [Hq, total_q]. Only used rows
    are merged; the others keep ``out`` / ``lse`` (default zeros). FP64."""
    outs = [_as_f64(o).astype(np.float64) for o in outs]
    lses = [_as_f64(x).astype(np.float64) for x in lses]
    if len(outs) < 1 or len(outs) != len(lses):
        raise ValueError("need at least one partition, with one LSE per output")
    total_q, hq, d = outs[0].shape
    o_out = np.zeros((total_q, hq, d), np.float64) if out is None else _as_f64(out).astype(np.float64, copy=True)
    l_out = np.zeros((hq, total_q), np.float64) if lse is None else _as_f64(lse).astype(np.float64, copy=True)
    cu_q = np.asarray(cu_q, np.int64)
    used_q = np.asarray(used_q, np.int64)
    for b in range(len(used_q)):
        r0, r1 = int(cu_q[b]), int(cu_q[b]) + int(used_q[b])
        if r1 == r0:
            continue
        ls = np.stack([x[:, r0:r1] for x in lses])  # [P, Hq, n]
        big = ls.max(axis=0)  # [Hq, n]
        dead = np.isneginf(big)
        safe = np.where(dead, 0.0, big)
        w = np.where(np.isneginf(ls), 0.0, np.exp(ls - safe[None]))  # [P, Hq, n]
        tot = w.sum(axis=0)
        merged_lse = np.where(dead, -np.inf, safe + np.log(np.where(dead, 1.0, tot)))
        acc = np.zeros((r1 - r0, hq, d), np.float64)
        for p, o in enumerate(outs):
            wp = np.where(dead, 0.0, w[p] / np.where(dead, 1.0, tot)).T[:, :, None]  # [n, Hq, 1]
            # a partition with zero weight (no keys for the row) contributes nothing
            acc += np.where(wp > 0.0, wp * np.where(wp > 0.0, o[r0:r1], 0.0), 0.0)
        o_out[r0:r1] = acc
        l_out[:, r0:r1] = merged_lse
    return o_out, l_out


def attention_backward(q, k, v, d_out, cu_q, used_q, cu_k, used_k, *, scale: Optional[float] = None,
                       dq=None, dk=None, dv=None, num_heads_kv: Optional[int] = None, causal_block: int = 0):
    """Gradients of the gapped varlen forward with respect to Q, K and V. FP64.

    The backward the pages mark as missing on the non-FA4 paths (cosmos-framework
    PR #302 review, PR #312 "Problem and behavior": forward only), written from the
    forward's definition. For each segment, query head h and used row i, with P the
    softmax over the used keys and dO the output gradient:

        dP_ij = <dO_i, V_j>,   D_i = sum_j P_ij dP_ij,   dS_ij = P_ij (dP_ij - D_i)
        dQ_i  = s sum_j dS_ij K_j
        dK_j  = s sum_{i, h in the KV group} dS_ij Q_i
        dV_j  = sum_{i, h in the KV group} P_ij dO_i

    Only used rows of dQ and used keys of dK / dV are written (others keep ``dq`` /
    ``dk`` / ``dv``, default zeros); a keyless segment's used rows get dQ = 0 and the
    used keys of a segment without used rows get dK = dV = 0. Each
    segment's used keys must not overlap another segment's. ``causal_block`` > 0 takes
    the gradients of the block-causal forward (``causal_limits``): a row's P is zero
    past its limit, and a row that sees no key has P = 0 and so dQ = 0. Returns
    (dq, dk, dv)."""
    q, k, v, d_out = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(d_out)
    total_q, hq, d = q.shape
    hkv = k.shape[1] if num_heads_kv is None else num_heads_kv
    g = hq // hkv
    s = 1.0 / math.sqrt(d) if scale is None else float(scale)
    cu_q = np.asarray(cu_q, np.int64)
    cu_k = np.asarray(cu_k, np.int64)
    used_q = np.asarray(used_q, np.int64)
    used_k = np.asarray(used_k, np.int64)
    dq_out = np.zeros(q.shape, np.float64) if dq is None else _as_f64(dq).astype(np.float64, copy=True)
    dk_out = np.zeros(k.shape, np.float64) if dk is None else _as_f64(dk).astype(np.float64, copy=True)
    dv_out = np.zeros(v.shape, np.float64) if dv is None else _as_f64(dv).astype(np.float64, copy=True)
    for b in range(len(used_q)):
        r0, nq = int(cu_q[b]), int(used_q[b])
        k0, nk = int(cu_k[b]), int(used_k[b])
        if nk > 0:  # a used key no used row reads still has a (zero) gradient
            dk_out[k0:k0 + nk] = 0.0
            dv_out[k0:k0 + nk] = 0.0
        if nq == 0:
            continue
        if nk == 0:
            dq_out[r0:r0 + nq] = 0.0
            continue
        lim = np.repeat(causal_limits(nq, nk, causal_block), g) if causal_block > 0 else None
        for hk in range(hkv):
            qs = q[r0:r0 + nq, hk * g:(hk + 1) * g, :].astype(np.float64).reshape(nq * g, d)
            dos = d_out[r0:r0 + nq, hk * g:(hk + 1) * g, :].astype(np.float64).reshape(nq * g, d)
            ks = k[k0:k0 + nk, hk, :].astype(np.float64)
            vs = v[k0:k0 + nk, hk, :].astype(np.float64)
            x = (qs @ ks.T) * s
            if lim is None:
                x -= x.max(axis=1, keepdims=True)
                p = np.exp(x)
                p /= p.sum(axis=1, keepdims=True)
            else:  # keys past a row's limit leave its softmax; a row with none has P = 0
                vis = np.arange(nk)[None, :] < lim[:, None]
                live = vis.any(axis=1)
                x = np.where(vis, x, -np.inf)
                mx = np.where(live, x.max(axis=1), 0.0)
                p = np.exp(x - mx[:, None])
                p /= np.where(live, p.sum(axis=1), 1.0)[:, None]
            dp = dos @ vs.T
            dd = (p * dp).sum(axis=1, keepdims=True)
            ds = p * (dp - dd)
            dq_out[r0:r0 + nq, hk * g:(hk + 1) * g, :] = (s * (ds @ ks)).reshape(nq, g, d)
            dk_out[k0:k0 + nk, hk, :] = s * (ds.T @ qs)
            dv_out[k0:k0 + nk, hk, :] = p.T @ dos
    return dq_out, dk_out, dv_out


def attention_backward_ranges(q, k, v, d_out, cu_q, used_q, key_ranges, *, scale: Optional[float] = None,
                              dq=None, dk=None, dv=None, num_heads_kv: Optional[int] = None):
    """Gradients of ``attention_forward_ranges``: segment b's keys are the concatenation
    of the K/V row ranges ``key_ranges[b]``. The same formulas as ``attention_backward``
    per (segment, KV head); a K/V row that several ranges cover (of one segment or of
    several) receives the sum of its contributions. Rows no range covers keep ``dk`` /
    ``dv`` (default zeros); covered rows of a segment without used rows get 0; the used
    rows of a segment without keys get dQ = 0. FP64. Returns (dq, dk, dv)."""
    q, k, v, d_out = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(d_out)
    total_q, hq, d = q.shape
    hkv = k.shape[1] if num_heads_kv is None else num_heads_kv
    g = hq // hkv
    s = 1.0 / math.sqrt(d) if scale is None else float(scale)
    cu_q = np.asarray(cu_q, np.int64)
    used_q = np.asarray(used_q, np.int64)
    dq_out = np.zeros(q.shape, np.float64) if dq is None else _as_f64(dq).astype(np.float64, copy=True)
    dk_out = np.zeros(k.shape, np.float64) if dk is None else _as_f64(dk).astype(np.float64, copy=True)
    dv_out = np.zeros(v.shape, np.float64) if dv is None else _as_f64(dv).astype(np.float64, copy=True)
    seg_rows = []
    for b in range(len(used_q)):
        rows = [np.arange(int(st), int(st) + int(n)) for st, n in key_ranges[b] if int(n) > 0]
        seg_rows.append(np.concatenate(rows) if rows else np.zeros(0, np.int64))
    for idx in seg_rows:  # every covered row starts from zero, then sums its contributions
        dk_out[idx] = 0.0
        dv_out[idx] = 0.0
    for b in range(len(used_q)):
        r0, nq = int(cu_q[b]), int(used_q[b])
        idx = seg_rows[b]
        if nq == 0:
            continue
        if idx.size == 0:
            dq_out[r0:r0 + nq] = 0.0
            continue
        for hk in range(hkv):
            qs = q[r0:r0 + nq, hk * g:(hk + 1) * g, :].astype(np.float64).reshape(nq * g, d)
            dos = d_out[r0:r0 + nq, hk * g:(hk + 1) * g, :].astype(np.float64).reshape(nq * g, d)
            ks = k[idx, hk, :].astype(np.float64)
            vs = v[idx, hk, :].astype(np.float64)
            x = (qs @ ks.T) * s
            x -= x.max(axis=1, keepdims=True)
            p = np.exp(x)
            p /= p.sum(axis=1, keepdims=True)
            dp = dos @ vs.T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq_out[r0:r0 + nq, hk * g:(hk + 1) * g, :] = (s * (ds @ ks)).reshape(nq, g, d)
            np.add.at(dk_out, (idx, hk), s * (ds.T @ qs))
            np.add.at(dv_out, (idx, hk), p.T @ dos)
    return dq_out, dk_out, dv_out
