"""GPU parity of the key-range forward (gva_plan_ranges + gva_forward) against the FP64
oracle: several K/V row ranges per segment, attended as one softmax in one launch."""
import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import workloads as W
from helpers_gpu import check_full, check_rows, gap_untouched, gpu_forward, sample_rows
from oracle import gva_oracle

pytestmark = pytest.mark.gpu
FILL = W.TINY_SENTINEL


@pytest.fixture(scope="module", autouse=True)
def _built():
    gva.build()


def _ranges_forward(g, ranges, total_k, q, k, v, out_dtype=torch.bfloat16):
    plan = gva.Plan.from_ranges(g.cu_q, g.used_q, ranges, total_k, g.num_heads_q, g.num_heads_kv, g.head_dim)
    o, l = W.make_outputs(g, FILL, device="cuda", out_dtype=out_dtype)
    gva.forward(plan, q.cuda(), k.cuda(), v.cuda(), o, l)
    gva.device_status(plan)
    return o, l


def _oracle(g, ranges, q, k, v):
    qn, kn, vn = (t.detach().cpu().float().numpy() for t in (q, k, v))
    return gva_oracle.attention_forward_ranges(qn, kn, vn, g.cu_q, g.used_q, ranges,
                                               out=np.full(qn.shape, FILL),
                                               lse=np.full((g.num_heads_q, g.total_q), FILL))


def _keyless_segments_check(g, ranges):
    # check_full finds keyless rows from used_k; give it the range totals
    return g.with_keys(g.cu_q, np.array([sum(n for _, n in r) for r in ranges], np.int32))


def test_prefix_ranges_match_the_plain_plan_bit_for_bit():
    rng = np.random.default_rng(51)
    g = W.random_geometry(rng, 6, 600, 900, 16, 4, 128)
    q, k, v = W.make_qkv(g, 51, gap_fill=float("nan"))
    ranges = [[(int(g.cu_k[b]), int(g.used_k[b]))] for b in range(g.num_segments)]
    o1, l1 = gpu_forward(g, q, k, v)
    o2, l2 = _ranges_forward(g, ranges, g.total_k, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("hq,hkv,d,seed", [(8, 2, 128, 61), (16, 16, 128, 62), (32, 8, 64, 63), (4, 4, 64, 64)])
def test_random_ranges(hq, hkv, d, seed):
    """Up to four ranges per segment anywhere in K/V (ragged lengths, empty ranges,
    overlaps with other segments); rows no range covers are NaN."""
    rng = np.random.default_rng(seed)
    g = W.random_geometry(rng, 5, 500, 10, hq, hkv, d)
    total_k = 3000
    ranges = []
    for _ in range(g.num_segments):
        rr = []
        for _ in range(int(rng.integers(0, 5))):
            st = int(rng.integers(0, total_k))
            rr.append((st, int(rng.integers(0, min(700, total_k - st) + 1))))
        ranges.append(rr)
    ranges[0] = []  # one keyless segment
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(g.total_q, hq, d, generator=gen).bfloat16()
    k = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    v = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    covered = np.zeros(total_k, bool)
    for rr in ranges:
        for st, n in rr:
            covered[st:st + n] = True
    k[torch.from_numpy(~covered)] = float("nan")
    v[torch.from_numpy(~covered)] = float("nan")
    o, l = _ranges_forward(g, ranges, total_k, q, k, v)
    o_ref, l_ref = _oracle(g, ranges, q, k, v)
    check_full(_keyless_segments_check(g, ranges), o, l, o_ref, l_ref, FILL)


def test_rank_major_keys():
    """Keys in the rank-major order an all-to-all leaves behind (per rank: text chunk,
    then video chunk); each sample's valid keys are its own text length in every text
    chunk plus all video keys, so they are not a prefix."""
    ranks, text_cap, video = 4, 64, 384
    text_len = [[37, 64, 5, 0], [64, 64, 64, 12]]  # per sample, per rank
    hq, hkv, d = 16, 8, 128
    cu_q = np.array([0, 1000, 2000], np.int32)
    used_q = np.array([1000, 777], np.int32)
    g = W.Geometry(cu_q, used_q, np.array([0, 0, 0], np.int32), np.array([0, 0], np.int32), hq, hkv, d)
    chunk = text_cap + video
    total_k = 2 * ranks * chunk  # each sample has its own gathered K/V
    ranges = []
    for b in range(2):
        rr = []
        for r in range(ranks):
            base = (b * ranks + r) * chunk
            rr.append((base, text_len[b][r]))
            rr.append((base + text_cap, video))
        ranges.append(rr)
    gen = torch.Generator().manual_seed(71)
    q = torch.randn(g.total_q, hq, d, generator=gen).bfloat16()
    k = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    v = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    for b in range(2):  # zero pads of the text chunks, as the text encoder leaves them
        for r in range(ranks):
            base = (b * ranks + r) * chunk
            k[base + text_len[b][r]:base + text_cap] = 0.0
            v[base + text_len[b][r]:base + text_cap] = 0.0
    o, l = _ranges_forward(g, ranges, total_k, q, k, v)
    o_ref, l_ref = _oracle(g, ranges, q, k, v)
    check_full(_keyless_segments_check(g, ranges), o, l, o_ref, l_ref, FILL)


@pytest.mark.slow
def test_multiview_partitions_fused_in_one_launch():
    """The two visibility partitions of the multiview workload as two ranges per segment
    of one launch: no partial outputs, no merge."""
    full, parts = W.multiview_causal()
    q, k, v = W.make_qkv(full, 1003, device="cuda", gap_fill=float("nan"))
    ranges = [[(int(p.cu_k[b]), int(p.used_k[b])) for p in parts] for b in range(full.num_segments)]
    o, l = _ranges_forward(full, ranges, full.total_k, q, k, v)
    assert gap_untouched(full, o, l, FILL)
    rows = sample_rows(full, np.random.default_rng(8), per_segment=3)
    o_ref, l_ref = gva_oracle.attention_rows(q.cpu(), k.cpu(), v.cpu(), full.cu_q, full.used_q, full.cu_k,
                                             full.used_k, rows)
    check_rows(o, l, rows, o_ref, l_ref)


@pytest.mark.slow
def test_text_and_video_keys_fused_in_one_launch():
    """The merge workload's text and video key sets as two ranges of one K/V buffer."""
    text, video, union, dead = W.lse_merge_union(empty="text")
    gen = torch.Generator(device="cuda").manual_seed(1004)
    q = torch.randn((text.total_q, 24, 128), generator=gen, device="cuda").bfloat16()
    k = torch.randn((text.total_k + video.total_k, 24, 128), generator=gen, device="cuda").bfloat16()
    v = torch.randn_like(k, dtype=torch.float32).bfloat16()
    ranges = [[(int(text.cu_k[b]), int(text.used_k[b])), (text.total_k + int(video.cu_k[b]), int(video.used_k[b]))]
              for b in range(text.num_segments)]
    o, l = _ranges_forward(text, ranges, k.shape[0], q, k, v)
    rows = sample_rows(union, np.random.default_rng(9), per_segment=3)
    qc, kc, vc = (t.cpu().float().numpy() for t in (q, k, v))  # widened once
    o_ref = np.zeros((len(rows), 24, 128))
    l_ref = np.zeros((24, len(rows)))
    for b in range(union.num_segments):
        idx = [i for i, r in enumerate(rows) if union.cu_q[b] <= r < union.cu_q[b + 1]]
        if not idx:
            continue
        oo, ll = gva_oracle.attention_forward_ranges(qc[union.cu_q[b]:union.cu_q[b + 1]], kc, vc,
                                                     [0, int(union.used_q[b])], [int(union.used_q[b])],
                                                     [ranges[b]])
        sel = [rows[i] - int(union.cu_q[b]) for i in idx]
        o_ref[idx], l_ref[:, idx] = oo[sel], ll[:, sel]
    check_rows(o, l, rows, o_ref, l_ref)
