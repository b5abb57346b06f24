"""Host-side pieces of the benchmark, on CPU: the merge's algorithmic bytes, the used-row
ranges the end-to-end steps copy, and the row-range copy itself."""
import types

import numpy as np
import pytest
import torch

import bench
from gapped_varlen_attention_gb300 import workloads as W


def test_merge_bytes_text_video():
    """8192 rows x 24 heads: two LSEs read and one written (12 bytes per row and head),
    each live FP32 partial read (512 bytes per row and head) and a bf16 output written
    (256); the segment whose text partition is keyless reads one partial only."""
    text, video, union, dead = W.lse_merge_union()
    got = bench.merge_bytes(union, [text.used_k, video.used_k], 2)
    rows = int(union.used_q.sum())
    dead_rows = int(union.used_q[dead])
    want = rows * 24 * (12 + 128 * (8 + 2)) - dead_rows * 24 * 128 * 4
    assert got == want
    # a sample of rows counts the same bytes per row
    some = np.arange(int(union.cu_q[dead]), int(union.cu_q[dead]) + 5)
    assert bench.merge_bytes(union, [text.used_k, video.used_k], 2, rows=some) == 5 * 24 * (12 + 128 * 6)


def test_job_rate():
    assert bench.job_rate(1, 2e12, 1000.0) == pytest.approx(2.0)
    assert bench.job_rate(4, 2e12, 1000.0) == pytest.approx(8.0)
    assert bench.job_rate(1, 5e9, 1.0, 1e9) == pytest.approx(5000.0)


def _stub(g, backward=False):
    s = types.SimpleNamespace(geoms=[g], parts=None, merge_only=False, backward=backward)
    t = lambda rows, heads: torch.empty((rows, heads, g.head_dim), dtype=torch.bfloat16, device="meta")  # noqa
    s.inputs = [t(g.total_q, g.num_heads_q), t(g.total_k, g.num_heads_kv), t(g.total_k, g.num_heads_kv)]
    s.outputs = [t(g.total_q, g.num_heads_q), torch.empty((g.num_heads_q, g.total_q), device="meta")]
    s.row_ranges = types.MethodType(bench.Workload.row_ranges, s)
    return s


def test_row_ranges_cover_used_rows_only():
    g = W.random_geometry(np.random.default_rng(3), 6, 50, 70, 8, 2, 64)
    s = _stub(g)
    (rq, rk, rv), (ro, rl) = s.row_ranges()
    assert rk == rv and ro == rq and rl is None

    def mask(ranges, total):
        m = np.zeros(total, bool)
        for r0, n in ranges:
            assert n > 0 and not m[r0:r0 + n].any()
            m[r0:r0 + n] = True
        return m
    assert np.array_equal(mask(rq, g.total_q), ~W.gap_rows(g.cu_q, g.used_q))
    assert np.array_equal(mask(rk, g.total_k), ~W.gap_rows(g.cu_k, g.used_k))
    h2d, d2h = bench.Workload.copy_bytes(s)
    row_q, row_k = g.num_heads_q * g.head_dim * 2, g.num_heads_kv * g.head_dim * 2
    assert h2d == int(g.used_q.sum()) * row_q + 2 * int(g.used_k.sum()) * row_k
    assert d2h == int(g.used_q.sum()) * row_q + g.num_heads_q * g.total_q * 4


def test_copy_rows_leaves_gaps():
    src = torch.arange(40.0).reshape(10, 4)
    dst = torch.full((10, 4), -1.0)
    bench.copy_rows(dst, src, [(1, 2), (6, 3)])
    assert torch.equal(dst[[1, 2, 6, 7, 8]], src[[1, 2, 6, 7, 8]])
    assert torch.all(dst[[0, 3, 4, 5, 9]] == -1.0)
    bench.copy_rows(dst, src, None)
    assert torch.equal(dst, src)
