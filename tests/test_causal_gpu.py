"""GPU parity of the block-causal forward (gva_plan_causal + gva_forward) against the
FP64 oracle: row i of a segment sits at key position i + used_k - used_q and sees keys
j < (floor(pos / B) + 1) * B."""
import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import workloads as W
from helpers_gpu import LSE_TOL, O_TOL, check_rows, gap_untouched, sample_rows
from oracle import gva_oracle

pytestmark = pytest.mark.gpu
FILL = W.TINY_SENTINEL


@pytest.fixture(scope="module", autouse=True)
def _built():
    gva.build()


def _causal_forward(g, q, k, v, block, out_dtype=torch.bfloat16):
    plan = gva.Plan.from_geometry(g, causal_block=block)
    o, l = W.make_outputs(g, FILL, device="cuda", out_dtype=out_dtype)
    gva.forward(plan, q.cuda(), k.cuda(), v.cuda(), o, l)
    gva.device_status(plan)
    return o, l, plan


def _check(g, o, l, o_ref, l_ref):
    o = o.float().cpu().numpy().astype(np.float64)
    l = l.cpu().numpy().astype(np.float64)
    gap = W.gap_rows(g.cu_q, g.used_q)
    assert np.all(o[gap] == FILL) and np.all(l[:, gap] == FILL), "a gap row was written"
    used = ~gap
    dead = np.isneginf(l_ref) & used[None, :]
    assert np.array_equal(np.isneginf(l) & used[None, :], dead), "rows without keys differ"
    assert np.all(o.transpose(1, 0, 2)[dead] == 0.0)
    live = np.isfinite(l_ref) & used[None, :]
    assert np.abs(l[live] - l_ref[live]).max() <= LSE_TOL
    rows_live = live.any(axis=0)
    assert np.abs(o[rows_live] - o_ref[rows_live]).max() <= O_TOL


CASES = [  # (Hq, Hkv, d, causal block, seed)
    (8, 2, 128, 1, 81),
    (16, 4, 128, 3, 82),
    (32, 8, 128, 64, 83),
    (8, 8, 64, 200, 84),
    (16, 8, 64, 1, 85),
    (4, 1, 128, 129, 86),
]


@pytest.mark.parametrize("hq,hkv,d,block,seed", CASES)
def test_random_block_causal(hq, hkv, d, block, seed):
    """Random gapped geometries; used_q may exceed used_k (early rows then see no key)."""
    rng = np.random.default_rng(seed)
    g = W.random_geometry(rng, 6, 600, 700, hq, hkv, d)
    q, k, v = W.make_qkv(g, seed, gap_fill=float("nan"))
    o, l, _ = _causal_forward(g, q, k, v, block)
    qn, kn, vn = (t.float().numpy() for t in (q, k, v))
    o_ref, l_ref = gva_oracle.attention_forward(qn, kn, vn, g.cu_q, g.used_q, g.cu_k, g.used_k,
                                                out=np.full(qn.shape, FILL),
                                                lse=np.full((g.num_heads_q, g.total_q), FILL), causal_block=block)
    _check(g, o, l, o_ref, l_ref)


def test_block_larger_than_segments_is_the_maskless_forward():
    """With used_q <= used_k every row sits at a non-negative key position, so a block
    longer than any segment masks nothing."""
    rng = np.random.default_rng(87)
    g = W.random_geometry(rng, 5, 500, 800, 16, 4, 128)
    g.used_q = np.minimum(g.used_q, g.used_k).astype(np.int32)
    q, k, v = W.make_qkv(g, 87)
    o1, l1, _ = _causal_forward(g, q, k, v, 1 << 20)
    plan = gva.Plan.from_geometry(g)
    o2, l2 = W.make_outputs(g, FILL, device="cuda")
    gva.forward(plan, q.cuda(), k.cuda(), v.cuda(), o2, l2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_causal_plan_counts_visible_keys_only():
    g = W.Geometry(np.array([0, 10], np.int32), np.array([10], np.int32), np.array([0, 10], np.int32),
                   np.array([10], np.int32), 4, 2, 64)
    plan = gva.Plan.from_geometry(g, causal_block=1)
    # token-causal, equal lengths: sum_i (i + 1) = 55 pairs
    assert plan.info()["used_flops"] == pytest.approx(4 * 64 * 4 * 55)


@pytest.mark.slow
def test_multiview_block_causal_full_size():
    """The multiview workload (7 segments with gaps) as one block-causal launch with
    512-token frames instead of partitions plus a merge."""
    full, _ = W.multiview_causal()
    q, k, v = W.make_qkv(full, 1003, device="cuda", gap_fill=float("nan"))
    o, l, _ = _causal_forward(full, q, k, v, 512)
    assert gap_untouched(full, o, l, FILL)
    rows = sample_rows(full, np.random.default_rng(10), per_segment=3)
    o_ref, l_ref = gva_oracle.attention_rows(q.cpu(), k.cpu(), v.cpu(), full.cu_q, full.used_q, full.cu_k,
                                             full.used_k, rows, causal_block=512)
    check_rows(o, l, rows, o_ref, l_ref)
