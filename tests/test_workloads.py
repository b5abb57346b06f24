"""The seeded input generators, on CPU: every workload has the shapes, lengths and head
layout its recipe states, is reproducible from its seed, and its partitions address the
same K/V buffers without copies."""
import numpy as np
import torch

from gapped_varlen_attention_gb300 import workloads as W


def _valid(g):
    assert g.cu_q[0] == 0 and g.cu_k[0] >= 0
    assert np.all(np.diff(g.cu_q) >= 0) and np.all(np.diff(g.cu_k) >= 0)
    assert np.all((g.used_q >= 0) & (g.used_q <= np.diff(g.cu_q)))
    assert np.all((g.used_k >= 0) & (g.used_k <= np.diff(g.cu_k)))
    assert g.num_heads_q % g.num_heads_kv == 0


def test_tiny():
    g = W.tiny()
    _valid(g)
    assert list(g.cu_q) == [0, 48, 96, 144] and list(g.cu_k) == [0, 48, 96, 144]
    assert list(g.used_q) == [40, 17, 12] and list(g.used_k) == [48, 33, 0]
    assert (g.num_heads_q, g.num_heads_kv, g.head_dim) == (4, 2, 64)


def test_cfg_text_cross():
    g = W.cfg_text_cross()
    _valid(g)
    assert list(np.diff(g.cu_q)) == [4096, 4096] and list(g.used_q) == [4096, 4096]
    assert list(np.diff(g.cu_k)) == [1024, 1024] and list(g.used_k) == [700, 20]
    assert (g.num_heads_q, g.num_heads_kv, g.head_dim) == (16, 8, 128)
    assert list(np.diff(W.cfg_text_cross(4096).cu_k)) == [4096, 4096]


def test_multiview_causal_and_its_partitions():
    full, parts = W.multiview_causal()
    _valid(full)
    assert full.num_segments == 7 and np.all(np.diff(full.cu_q) == 2048) and np.all(np.diff(full.cu_k) == 8192)
    assert np.all((full.used_q >= 1024) & (full.used_q <= 2048))
    assert np.all((full.used_k >= 4096) & (full.used_k <= 8192))
    assert (full.num_heads_q, full.num_heads_kv, full.head_dim) == (32, 8, 128)
    p0, p1 = parts
    for p in parts:
        _valid(p)
        assert np.array_equal(p.cu_q, full.cu_q) and np.array_equal(p.used_q, full.used_q)
    # partition 0 is the first half of each segment's used keys, partition 1 the rest,
    # both inside the full geometry's K/V rows
    assert np.array_equal(p0.cu_k, full.cu_k) and np.array_equal(p0.used_k, full.used_k // 2)
    assert np.array_equal(p1.cu_k[:-1], full.cu_k[:-1] + full.used_k // 2)
    assert np.array_equal(p0.used_k + p1.used_k, full.used_k)


def test_lse_merge_union():
    for empty in ("text", "video"):
        text, video, union, dead = W.lse_merge_union(empty=empty)
        for g in (text, video, union):
            _valid(g)
            assert g.total_q == 8192 and g.num_segments == 10
            assert (g.num_heads_q, g.num_heads_kv, g.head_dim) == (24, 24, 128)
        assert list(np.diff(text.cu_q)) == [820] * 9 + [812]
        assert np.all(np.diff(text.cu_k) == 1024) and np.all(np.diff(video.cu_k) == 16384)
        emptied = text if empty == "text" else video
        other = video if empty == "text" else text
        assert emptied.used_k[dead] == 0 and np.all(np.delete(emptied.used_k, dead) > 0)
        assert np.all(other.used_k > 0)
        assert np.array_equal(union.used_k, text.used_k + video.used_k)


def test_long_replay():
    g = W.long_replay()
    _valid(g)
    assert g.num_segments == 4 and np.all(np.diff(g.cu_q) == 32768) and np.all(np.diff(g.cu_k) == 65536)
    assert np.all((g.used_q >= 0.6 * 32768) & (g.used_q <= 32768))
    assert np.all((g.used_k >= 0.5 * 65536) & (g.used_k <= 65536))
    assert (g.num_heads_q, g.num_heads_kv, g.head_dim) == (32, 8, 128)
    # the benchmark's FLOP count for seed 1005
    assert g.used_flops() == 4.0 * 128 * 32 * float(np.sum(g.used_q.astype(np.float64) * g.used_k))
    assert abs(g.used_flops() - 91.377e12) < 0.01e12


def test_tensors_are_seeded_and_gap_filled():
    g = W.tiny()
    a = W.make_qkv(g, 1001)
    b = W.make_qkv(g, 1001)
    c = W.make_qkv(g, 1002)
    assert all(torch.equal(x, y) for x, y in zip(a, b)) and not torch.equal(a[0], c[0])
    q, k, v = W.make_qkv(g, 1001, gap_fill=float("nan"))
    gq, gk = torch.from_numpy(W.gap_rows(g.cu_q, g.used_q)), torch.from_numpy(W.gap_rows(g.cu_k, g.used_k))
    assert torch.isnan(q[gq].float()).all() and not torch.isnan(q[~gq].float()).any()
    assert torch.isnan(k[gk].float()).all() and torch.isnan(v[gk].float()).all()
    _, k0, v0 = W.make_qkv(W.cfg_text_cross(), 1002, k_pad_fill=0.0)
    gk0 = torch.from_numpy(W.gap_rows(W.cfg_text_cross().cu_k, W.cfg_text_cross().used_k))
    assert torch.all(k0[gk0] == 0) and torch.all(v0[gk0] == 0)


def test_partials_mark_keyless_partitions():
    text, video, union, dead = W.lse_merge_union()
    outs, lses = W.make_partials(union, [text.used_k, video.used_k], 3004)
    r0, r1 = int(union.cu_q[dead]), int(union.cu_q[dead]) + int(union.used_q[dead])
    assert torch.all(outs[0][r0:r1] == 0) and torch.all(torch.isneginf(lses[0][:, r0:r1]))
    assert torch.all(torch.isfinite(lses[1])) and torch.isfinite(lses[0][:, :r0]).all()
