"""GPU parity of gva_lse_merge against the FP64 oracle merge, through the C ABI."""
import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import workloads as W
from oracle import gva_oracle

pytestmark = pytest.mark.gpu

FILL = 7.0


@pytest.fixture(scope="module", autouse=True)
def _built():
    gva.build()


def _partials(g, parts, rng, in_dtype, dead_frac=0.15):
    outs, lses = [], []
    for p in range(parts):
        o = torch.randn(g.total_q, g.num_heads_q, g.head_dim, generator=rng).to(in_dtype)
        l = torch.randn(g.num_heads_q, g.total_q, generator=rng) * 3.0
        dead = torch.rand(g.num_heads_q, g.total_q, generator=rng) < dead_frac
        l[dead] = -float("inf")
        o.permute(1, 0, 2)[dead] = 0.0  # a keyless partial has a zero output
        outs.append(o)
        lses.append(l)
    return outs, lses


@pytest.mark.parametrize("parts,in_dtype,out_dtype,hq,d", [
    (2, torch.float32, torch.bfloat16, 24, 128),
    (2, torch.bfloat16, torch.bfloat16, 8, 64),
    (3, torch.float32, torch.float32, 16, 128),
    (8, torch.bfloat16, torch.float32, 4, 64),
    (1, torch.float32, torch.float32, 32, 128),
    (8, torch.float32, torch.bfloat16, 256, 64),   # most weights: 8 x 256 heads, one chunk group
    (7, torch.float32, torch.float32, 48, 128),
])
def test_merge_matches_oracle(parts, in_dtype, out_dtype, hq, d):
    rng_np = np.random.default_rng(parts * 100 + hq)
    g = W.random_geometry(rng_np, 7 if hq <= 64 else 3, 90 if hq <= 64 else 40, 10, hq, hq, d)
    gen = torch.Generator().manual_seed(5)
    outs, lses = _partials(g, parts, gen, in_dtype)
    plan = gva.Plan.from_geometry(g)
    o, l = W.make_outputs(g, FILL, device="cuda", out_dtype=out_dtype)
    gva.lse_merge(plan, [x.cuda() for x in outs], [x.cuda() for x in lses], o, l)
    gva.device_status(plan)
    o_ref, l_ref = gva_oracle.lse_merge([x.float().numpy() for x in outs], [x.numpy() for x in lses], g.cu_q,
                                        g.used_q, out=np.full(o.shape, FILL), lse=np.full(l.shape, FILL))
    og = o.float().cpu().numpy().astype(np.float64)
    lg = l.cpu().numpy().astype(np.float64)
    gap = W.gap_rows(g.cu_q, g.used_q)
    assert np.all(og[gap] == FILL) and np.all(lg[:, gap] == FILL)
    used = ~gap
    assert np.array_equal(np.isneginf(lg[:, used]), np.isneginf(l_ref[:, used]))
    fin = np.isfinite(l_ref) & used[None, :]
    assert np.abs(lg[fin] - l_ref[fin]).max() <= 1e-5
    # fp32 output: FP32 arithmetic only; bf16 output: plus its own rounding (<= 2^-9 relative)
    rel = 2.0 ** -8 if out_dtype == torch.bfloat16 else 0.0
    assert np.all(np.abs(og[used] - o_ref[used]) <= rel * np.abs(o_ref[used]) + 1e-5)
    dead = np.isneginf(l_ref) & used[None, :]
    assert np.all(og.transpose(1, 0, 2)[dead] == 0.0)


def test_merge_in_place():
    """out may alias the first partition and lse the first LSE."""
    g = W.random_geometry(np.random.default_rng(3), 5, 64, 10, 8, 8, 128)
    gen = torch.Generator().manual_seed(6)
    outs, lses = _partials(g, 2, gen, torch.float32)
    o_ref, l_ref = gva_oracle.lse_merge([x.numpy() for x in outs], [x.numpy() for x in lses], g.cu_q, g.used_q,
                                        out=outs[0].numpy(), lse=lses[0].numpy())
    plan = gva.Plan.from_geometry(g)
    o0, l0 = outs[0].cuda(), lses[0].cuda()
    gva.lse_merge(plan, [o0, outs[1].cuda()], [l0, lses[1].cuda()], o0, l0)
    gva.device_status(plan)
    assert np.abs(o0.cpu().numpy() - o_ref).max() <= 1e-5
    lg = l0.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.abs(lg[fin] - l_ref[fin]).max() <= 1e-5


def test_merge_rejects_bad_counts():
    g = W.tiny()
    plan = gva.Plan.from_geometry(g)
    o, l = W.make_outputs(g, 0.0, device="cuda", out_dtype=torch.float32)
    with pytest.raises(ValueError):
        gva.lse_merge(plan, [], [], o, l)
    with pytest.raises(gva.GvaError, match="num_parts"):
        gva.lse_merge(plan, [o] * 9, [l] * 9, o, l)


@pytest.mark.parametrize("parts,in_dtype", [(2, torch.float32), (3, torch.bfloat16), (5, torch.float32)])
def test_merge_skips_keyless_partitions(parts, in_dtype):
    """A partition whose LSE is -inf for a row has no keys there: its output is never
    read (NaN there must not leak), and the merge is the other partitions' result."""
    g = W.random_geometry(np.random.default_rng(11 + parts), 6, 120, 10, 8, 8, 128, allow_empty=False)
    gen = torch.Generator().manual_seed(12)
    outs, lses = _partials(g, parts, gen, in_dtype, dead_frac=0.3)
    for o, l in zip(outs, lses):
        o.permute(1, 0, 2)[torch.isneginf(l)] = float("nan")
    o_ref, l_ref = gva_oracle.lse_merge([x.float().numpy() for x in outs], [x.numpy() for x in lses], g.cu_q,
                                        g.used_q, out=np.zeros((g.total_q, 8, 128)), lse=np.zeros((8, g.total_q)))
    plan = gva.Plan.from_geometry(g)
    o, l = W.make_outputs(g, 0.0, device="cuda", out_dtype=torch.float32)
    gva.lse_merge(plan, [x.cuda() for x in outs], [x.cuda() for x in lses], o, l)
    gva.device_status(plan)
    og = o.cpu().numpy()
    used = ~W.gap_rows(g.cu_q, g.used_q)
    assert not np.isnan(og[used]).any()
    assert np.all(np.abs(og[used] - o_ref[used]) <= 1e-5 * np.abs(o_ref[used]) + 1e-5)
    dead = np.isneginf(l_ref) & used[None, :]
    assert np.all(og.transpose(1, 0, 2)[dead] == 0.0)


def test_merge_in_place_output_only():
    """out aliases the first partition while the merged LSE goes to its own buffer (the
    merge may then share a unit among several CTAs)."""
    g = W.random_geometry(np.random.default_rng(8), 6, 100, 10, 16, 16, 64, allow_empty=False)
    gen = torch.Generator().manual_seed(9)
    outs, lses = _partials(g, 3, gen, torch.float32)
    o_ref, l_ref = gva_oracle.lse_merge([x.numpy() for x in outs], [x.numpy() for x in lses], g.cu_q, g.used_q,
                                        out=outs[0].numpy(), lse=np.zeros((16, g.total_q)))
    plan = gva.Plan.from_geometry(g)
    o0 = outs[0].cuda()
    lse = torch.zeros(16, g.total_q, device="cuda")
    gva.lse_merge(plan, [o0] + [x.cuda() for x in outs[1:]], [x.cuda() for x in lses], o0, lse)
    gva.device_status(plan)
    assert np.abs(o0.cpu().numpy() - o_ref).max() <= 1e-5
    lg = lse.cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.abs(lg[fin] - l_ref[fin]).max() <= 1e-5
