"""Seeded synthetic workloads for the gapped variable-length attention forward.

This module only draws segment geometries and random tensors. It holds none of
the attention arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing any of the method's code.

Geometry conventions (cosmos-framework PR #302, "What"; the FA4 varlen
forward's ``cu_seqlens`` / ``seqused`` arguments):

* segment ``b`` owns query rows ``cu_q[b] .. cu_q[b+1]`` (its capacity) and key
  rows ``cu_k[b] .. cu_k[b+1]``;
* only the first ``used_q[b]`` query rows attend, and only to the first
  ``used_k[b]`` keys of the segment; the rest of each range is a gap;
* Q / O are packed token-major ``[total_q, Hq, d]``, K / V ``[total_k, Hkv, d]``,
  the log-sum-exp is ``[Hq, total_q]`` (the PyTorch unpadded varlen layout
  named in the review of PR #302).

Every workload below is a synthetic stand-in for the pages' workloads (Cosmos3
CFG text cross-attention, multiview camera + LiDAR replay); those need model
weights and data that are not available.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np

try:  # torch is only needed to draw tensors, not to describe geometries
    import torch
except ImportError:  # pragma: no cover
    torch = None


@dataclasses.dataclass
class Geometry:
    """One launch's segment geometry (host ints) plus head layout."""

    cu_q: np.ndarray  # int32 [B+1]
    used_q: np.ndarray  # int32 [B]
    cu_k: np.ndarray  # int32 [B+1]
    used_k: np.ndarray  # int32 [B]
    num_heads_q: int
    num_heads_kv: int
    head_dim: int

    @property
    def num_segments(self) -> int:
        return int(self.used_q.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def total_k(self) -> int:
        return int(self.cu_k[-1])

    def used_flops(self) -> float:
        """Useful FLOPs of one forward: QK^T and PV over used rows and keys."""
        pairs = float(np.sum(self.used_q.astype(np.float64) * self.used_k.astype(np.float64)))
        return 4.0 * self.head_dim * self.num_heads_q * pairs

    def with_keys(self, cu_k: np.ndarray, used_k: np.ndarray) -> "Geometry":
        return dataclasses.replace(self, cu_k=np.asarray(cu_k, np.int32),
                                   used_k=np.asarray(used_k, np.int32))


def _geom(cq, uq, ck, uk, hq, hkv, d) -> Geometry:
    return Geometry(np.asarray(cq, np.int32), np.asarray(uq, np.int32),
                    np.asarray(ck, np.int32), np.asarray(uk, np.int32), hq, hkv, d)


def _cum(caps) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(caps, np.int64))]).astype(np.int32)


# --------------------------------------------------------------------------------------
# The five workloads.
# --------------------------------------------------------------------------------------

TINY_SENTINEL = 7.0


def tiny() -> Geometry:
    """Three segments with capacity 48 q / 48 k each and used (q, k) of (40, 48),
    (17, 33) and (12, 0): a partial tile, a ragged key tail and a keyless segment
    (PR #302, "What": rows past the used length, a segment with no keys).
    Hq=4, Hkv=2 (GQA), d=64."""
    cu = _cum([48, 48, 48])
    return _geom(cu, [40, 17, 12], cu, [48, 33, 0], 4, 2, 64)


def cfg_text_cross(pad_to: int = 1024) -> Geometry:
    """CFG B=2 text cross-attention (TensorRT-LLM issue #18687, "Code walk-through"):
    4096 video query rows per sample; text keys right-padded to ``pad_to`` with real
    lengths 700 (negative prompt) and 20 (positive prompt). Hq=16, Hkv=8, d=128."""
    return _geom(_cum([4096, 4096]), [4096, 4096], _cum([pad_to, pad_to]), [700, 20], 16, 8, 128)


def multiview_causal(seed: int = 1003) -> Tuple[Geometry, List[Geometry]]:
    """Multiview causal gapped replay: 7 camera segments, query capacity 2048 with
    used lengths uniform in [1024, 2048]; key capacity 8192 with a seeded 50-100 %
    used. Hq=32, Hkv=8, d=128.

    Returns the full geometry and its split into two visibility partitions over
    the same K/V buffers: partition 0 sees the first ``floor(used_k/2)`` keys of
    each segment, partition 1 the rest (cosmos-framework PR #312, "Problem and
    behavior": visibility partitions combined by an FP32 LSE merge)."""
    rng = np.random.default_rng(seed)
    B, cq, ck = 7, 2048, 8192
    uq = rng.integers(1024, 2048, size=B, endpoint=True)
    uk = np.floor(rng.uniform(0.5, 1.0, size=B) * ck).astype(np.int64)
    full = _geom(_cum([cq] * B), uq, _cum([ck] * B), uk, 32, 8, 128)
    return full, split_keys(full, uk // 2)


def split_keys(g: Geometry, sigma: np.ndarray) -> List[Geometry]:
    """Two zero-copy key partitions of ``g``: keys ``[0, sigma_b)`` and
    ``[sigma_b, used_k_b)`` of each segment, expressed by shifting ``cu_k``."""
    sigma = np.asarray(sigma, np.int64)
    uk = g.used_k.astype(np.int64)
    cu = g.cu_k.astype(np.int64)
    p0 = g.with_keys(cu, sigma)
    cu1 = cu.copy()
    cu1[:-1] = cu[:-1] + sigma
    p1 = g.with_keys(cu1, uk - sigma)
    return [p0, p1]


def lse_merge_union(seed: int = 1004, empty: str = "text") -> Tuple[Geometry, Geometry, Geometry, int]:
    """8192 query rows in 10 segments (9 x 820 + 1 x 812), each with its own text
    (1024 keys) and video (16384 keys) key set; Hq = Hkv = 24, d = 128.

    Returns (text partition, video partition, union, index of the keyless segment).
    The union geometry refers to a K/V buffer laid out per segment as
    [text keys | video keys]; a seeded 10 % of the rows (one segment) has an empty
    partition, chosen by ``empty`` ("text" or "video")."""
    rng = np.random.default_rng(seed)
    B = 10
    q_caps = [820] * 9 + [812]
    kt, kv = 1024, 16384
    dead = int(rng.integers(0, B))
    ut = np.full(B, kt)
    uv = np.full(B, kv)
    if empty == "text":
        ut[dead] = 0
    else:
        uv[dead] = 0
    cq = _cum(q_caps)
    text = _geom(cq, q_caps, _cum([kt] * B), ut, 24, 24, 128)
    video = _geom(cq, q_caps, _cum([kv] * B), uv, 24, 24, 128)
    union = _geom(cq, q_caps, _cum([kt + kv] * B), ut + uv, 24, 24, 128)
    return text, video, union, dead


def long_replay(seed: int = 1005) -> Geometry:
    """Long joint video + LiDAR replay: 4 segments of 32768 query rows with seeded
    used fractions in [0.6, 1.0]; 65536 keys per segment with used fractions in
    [0.5, 1.0]. Hq=32, Hkv=8, d=128, non-causal within a segment."""
    rng = np.random.default_rng(seed)
    B, cq, ck = 4, 32768, 65536
    uq = np.floor(rng.uniform(0.6, 1.0, size=B) * cq).astype(np.int64)
    uk = np.floor(rng.uniform(0.5, 1.0, size=B) * ck).astype(np.int64)
    return _geom(_cum([cq] * B), uq, _cum([ck] * B), uk, 32, 8, 128)


def long_replay_small(seed: int = 1006) -> Geometry:
    """A reduced long replay for profiling captures: 2 segments of 8192 query rows and
    32768 keys, used fractions drawn from the same ranges; Hq=32, Hkv=8, d=128 (Q + K + V about
    0.4 GB, above the 129 MB L2)."""
    rng = np.random.default_rng(seed)
    B, cq, ck = 2, 8192, 32768
    uq = np.floor(rng.uniform(0.6, 1.0, size=B) * cq).astype(np.int64)
    uk = np.floor(rng.uniform(0.5, 1.0, size=B) * ck).astype(np.int64)
    return _geom(_cum([cq] * B), uq, _cum([ck] * B), uk, 32, 8, 128)


def random_geometry(rng: np.random.Generator, num_segments: int, max_q: int, max_k: int,
                    num_heads_q: int, num_heads_kv: int, head_dim: int,
                    allow_empty: bool = True) -> Geometry:
    """A random gapped geometry for property tests: capacities and used lengths
    drawn independently, zero-length segments allowed."""
    lo = 0 if allow_empty else 1
    cq = rng.integers(lo, max_q, size=num_segments, endpoint=True)
    ck = rng.integers(lo, max_k, size=num_segments, endpoint=True)
    uq = np.array([rng.integers(lo if c > 0 else 0, c, endpoint=True) for c in cq])
    uk = np.array([rng.integers(lo if c > 0 else 0, c, endpoint=True) for c in ck])
    return _geom(_cum(cq), uq, _cum(ck), uk, num_heads_q, num_heads_kv, head_dim)


# --------------------------------------------------------------------------------------
# Tensors.
# --------------------------------------------------------------------------------------

def gap_rows(cu: np.ndarray, used: np.ndarray) -> np.ndarray:
    """Boolean mask over packed rows: True on rows past a segment's used length."""
    total = int(cu[-1])
    mask = np.zeros(total, dtype=bool)
    for b in range(len(used)):
        mask[int(cu[b]) + int(used[b]):int(cu[b + 1])] = True
    return mask


def make_qkv(g: Geometry, seed: int, device: str = "cpu", dtype=None,
             gap_fill: Optional[float] = None, k_pad_fill: Optional[float] = None):
    """Q, K, V ~ N(0, 1) in bf16 drawn from ``torch.Generator(device).manual_seed(seed)``.

    ``gap_fill`` overwrites Q / K / V rows past the used lengths (e.g. NaN to prove
    they never leak); ``k_pad_fill`` overwrites only the K / V gap rows (0.0 gives
    the exactly-zero text pads of TensorRT-LLM issue #18687, "Code walk-through"
    step 3)."""
    assert torch is not None
    dtype = dtype or torch.bfloat16
    gen = torch.Generator(device=device).manual_seed(seed)
    q = torch.randn((g.total_q, g.num_heads_q, g.head_dim), generator=gen, device=device,
                    dtype=torch.float32).to(dtype)
    k = torch.randn((g.total_k, g.num_heads_kv, g.head_dim), generator=gen, device=device,
                    dtype=torch.float32).to(dtype)
    v = torch.randn((g.total_k, g.num_heads_kv, g.head_dim), generator=gen, device=device,
                    dtype=torch.float32).to(dtype)
    if gap_fill is not None:
        qm = torch.from_numpy(gap_rows(g.cu_q, g.used_q)).to(device)
        q[qm] = gap_fill
    kfill = gap_fill if k_pad_fill is None else k_pad_fill
    if kfill is not None:
        km = torch.from_numpy(gap_rows(g.cu_k, g.used_k)).to(device)
        k[km] = kfill
        v[km] = kfill
    return q, k, v


def make_partials(g: Geometry, used_k_parts, seed: int, device: str = "cpu", dtype=None):
    """Partial results of ``len(used_k_parts)`` key partitions of ``g``'s rows, as the
    forward leaves them: O ~ N(0, 1) ``[total_q, Hq, d]`` (fp32 by default) and LSE ~
    N(0, 3^2) ``[Hq, total_q]``, except that the used rows of a segment whose partition
    has no keys (``used_k_parts[p][b] == 0``) hold O = 0 and LSE = -inf."""
    assert torch is not None
    dtype = dtype or torch.float32
    gen = torch.Generator(device=device).manual_seed(seed)
    outs, lses = [], []
    for uk in used_k_parts:
        o = torch.randn((g.total_q, g.num_heads_q, g.head_dim), generator=gen, device=device,
                        dtype=torch.float32).to(dtype)
        lse = 3.0 * torch.randn((g.num_heads_q, g.total_q), generator=gen, device=device, dtype=torch.float32)
        for b in range(g.num_segments):
            if int(uk[b]) == 0:
                r0, r1 = int(g.cu_q[b]), int(g.cu_q[b]) + int(g.used_q[b])
                o[r0:r1] = 0.0
                lse[:, r0:r1] = -float("inf")
        outs.append(o)
        lses.append(lse)
    return outs, lses


def make_outputs(g: Geometry, fill: float, device: str = "cpu", out_dtype=None):
    """O ``[total_q, Hq, d]`` and LSE ``[Hq, total_q]`` prefilled with a sentinel."""
    assert torch is not None
    out_dtype = out_dtype or torch.bfloat16
    o = torch.full((g.total_q, g.num_heads_q, g.head_dim), fill, dtype=out_dtype, device=device)
    lse = torch.full((g.num_heads_q, g.total_q), fill, dtype=torch.float32, device=device)
    return o, lse
