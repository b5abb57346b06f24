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


def _roof_stub(work, dom_flops):
    s = types.SimpleNamespace(bound="tensor", unit="TFLOP/s", scale=1e12, merge_only=False, work=work,
                              kernel="gva_fwd_kernel", dominant=0)
    s.plans = [types.SimpleNamespace(info=lambda: {"used_flops": dom_flops})]
    s.dominant_bytes = lambda: 1.0e9
    return s


def test_roofline_peak_follows_the_kernels_own_timed_region():
    """Burst peak when the dominant kernel's timed launches last under a second,
    sustained above; both fractions are always given."""
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "hbm_gbs": 7000.0}
    wl = _roof_stub(1e14, 1e14)
    short = {"dom_ms": 60.0, "dom_launches": 10, "same_size_copy_gbs": None}  # 0.6 s
    r = bench.roofline_of(wl, short, peaks, "measured", None)
    assert r["peak"] == 2000.0 and "burst" in r["peak_source"]
    assert r["achieved"] == pytest.approx(1e14 / 0.06 / 1e12, abs=0.01)  # rounded to 0.01
    assert r["frac"] == r["frac_burst"] and r["frac_sustained"] == pytest.approx(r["achieved"] / 1600.0, abs=1e-4)
    long = {"dom_ms": 60.0, "dom_launches": 20, "same_size_copy_gbs": None}  # 1.2 s
    r = bench.roofline_of(wl, long, peaks, "measured", 2.0e9)
    assert r["peak"] == 1600.0 and "sustained" in r["peak_source"]
    assert r["traffic"] == 2.0e9 and r["traffic_over_algorithmic"] == 2.0


def test_dominant_bytes_of_the_long_replay():
    """Q, O (bf16) and LSE of the used rows plus K and V of the used keys: about 2.587 GB
    for the long replay's used lengths."""
    g = W.long_replay()
    s = types.SimpleNamespace(merge_only=False, geoms=[g], dominant=0, partials=None,
                              out=torch.empty(0, dtype=torch.bfloat16, device="meta"))
    got = bench.Workload.dominant_bytes(s)
    rows, keys = int(g.used_q.sum()), int(g.used_k.sum())
    assert got == rows * 32 * (128 * 2 + 128 * 2 + 4) + keys * 8 * 2 * 128 * 2
    assert got == pytest.approx(2.587e9, rel=1e-3)


def test_recorded_traffic_needs_the_current_kernel_sources(tmp_path, monkeypatch):
    import json
    rec = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(rec))
    assert bench.recorded_traffic("long_replay", "gva_fwd_kernel") is None  # no record
    h = bench.kernel_source_hash("gva_fwd_kernel")
    rec.write_text(json.dumps({"records": {"long_replay": {"kernel": "gva_fwd_kernel", "source_sha16": h,
                                                           "dram_bytes_per_launch": 3.1e9}}}))
    assert bench.recorded_traffic("long_replay", "gva_fwd_kernel") == 3.1e9
    assert bench.recorded_traffic("long_replay", "gva_backward") is None  # another kernel
    rec.write_text(json.dumps({"records": {"long_replay": {"kernel": "gva_fwd_kernel", "source_sha16": "0" * 16,
                                                           "dram_bytes_per_launch": 3.1e9}}}))
    assert bench.recorded_traffic("long_replay", "gva_fwd_kernel") is None  # taken on other sources


def test_kernel_hash_covers_code_not_comments(tmp_path, monkeypatch):
    """A comment edit keeps the hash (and so a recorded capture) valid; a code edit does
    not. String literals that hold comment markers are code."""
    src = 'int f() { return 1; }  // one\n/* block\n comment */\nconst char* s = "//x/*y*/";\n'
    assert bench.code_only(src) == 'int f() { return 1; }\nconst char* s = "//x/*y*/";'
    csrc = tmp_path / "csrc"
    csrc.mkdir()
    names = bench.KERNEL_SOURCES["gva_fwd_kernel"]
    for n in names:
        (csrc / n).write_text(src)
    monkeypatch.setattr(bench, "CSRC", str(csrc))
    h0 = bench.kernel_source_hash("gva_fwd_kernel")
    (csrc / names[0]).write_text(src.replace("// one", "// one, reworded\n// and a second line"))
    assert bench.kernel_source_hash("gva_fwd_kernel") == h0
    (csrc / names[0]).write_text(src.replace("return 1", "return 2"))
    assert bench.kernel_source_hash("gva_fwd_kernel") != h0
