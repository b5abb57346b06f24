"""GPU parity of gva_forward against the FP64 oracle, through the C ABI.

Small workloads are compared element by element in full; the full-size workloads run in
the launch configuration the benchmark times and are spot-checked on sampled rows, plus
exact checks of every gap row."""
import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import workloads as W
from helpers_gpu import (LSE_TOL, O_TOL, check_full, check_rows, gap_untouched, gpu_forward, oracle_forward,
                         sample_rows)
from oracle import gva_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    gva.build()


def test_tiny_workload():
    """3 segments, ragged q / k tails, a keyless segment, 7.0 sentinels on gap rows."""
    g = W.tiny()
    q, k, v = W.make_qkv(g, 1001)
    o, l = gpu_forward(g, q, k, v)
    o_ref, l_ref = oracle_forward(g, q, k, v)
    check_full(g, o, l, o_ref, l_ref, W.TINY_SENTINEL)


def test_tiny_workload_fp32_output():
    g = W.tiny()
    q, k, v = W.make_qkv(g, 1001)
    o, l = gpu_forward(g, q, k, v, out_dtype=torch.float32)
    o_ref, l_ref = oracle_forward(g, q, k, v)
    check_full(g, o, l, o_ref, l_ref, W.TINY_SENTINEL)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 128), (12, 4, 128), (24, 1, 128), (5, 1, 64)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_output_only_16_byte_aligned(out_dtype, hq, hkv, d):
    """An output that is 16- but not 32-byte aligned: full tiles leave through TMA stores
    (which need 16 bytes), partial tiles through 16-byte row stores. The result is the
    same as through an aligned buffer, and the elements just before and after the output
    stay untouched. With groups that do not divide 128 (3, 24, 5) a TMA box covers only
    the T * G rows of a tile that hold data."""
    g = W.random_geometry(np.random.default_rng(77), 4, 300, 500, hq, hkv, d)
    q, k, v = W.make_qkv(g, 77)
    o_ref, l_ref = gpu_forward(g, q, k, v, out_dtype=out_dtype)
    pad = 16 // torch.tensor([], dtype=out_dtype).element_size()
    n = g.total_q * g.num_heads_q * g.head_dim
    buf = torch.full((n + 2 * pad,), W.TINY_SENTINEL, dtype=out_dtype, device="cuda")
    o = buf[pad:pad + n].view(g.total_q, g.num_heads_q, g.head_dim)
    assert o.data_ptr() % 32 == 16
    l = torch.full((g.num_heads_q, g.total_q), W.TINY_SENTINEL, device="cuda")
    plan = gva.Plan.from_geometry(g)
    gva.forward(plan, q.cuda(), k.cuda(), v.cuda(), o, l)
    gva.device_status(plan)
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
    assert torch.all(buf[:pad] == W.TINY_SENTINEL) and torch.all(buf[pad + n:] == W.TINY_SENTINEL)


def test_cfg_text_cross_attention():
    """CFG B=2: 4096 query rows per sample, text keys padded to 1024 with exact-zero pads,
    real lengths 700 and 20. Full comparison."""
    g = W.cfg_text_cross()
    q, k, v = W.make_qkv(g, 1002, k_pad_fill=0.0)
    o, l = gpu_forward(g, q, k, v)
    o_ref, l_ref = oracle_forward(g, q, k, v)
    check_full(g, o, l, o_ref, l_ref, W.TINY_SENTINEL)


def test_cfg_output_is_invariant_to_pad_length():
    """Growing the zero padding from 1024 to 4096 keys leaves O and LSE bit-identical."""
    g1 = W.cfg_text_cross(1024)
    g4 = W.cfg_text_cross(4096)
    q, k1, v1 = W.make_qkv(g1, 1002, k_pad_fill=0.0)
    k4 = torch.zeros((g4.total_k,) + tuple(k1.shape[1:]), dtype=k1.dtype)
    v4 = torch.zeros_like(k4)
    for b in range(2):
        n = int(g1.used_k[b])
        k4[g4.cu_k[b]:g4.cu_k[b] + n] = k1[g1.cu_k[b]:g1.cu_k[b] + n]
        v4[g4.cu_k[b]:g4.cu_k[b] + n] = v1[g1.cu_k[b]:g1.cu_k[b] + n]
    o1, l1 = gpu_forward(g1, q, k1, v1)
    o4, l4 = gpu_forward(g4, q, k4, v4)
    assert torch.equal(o1, o4) and torch.equal(l1, l4)


def test_attending_the_pads_would_dilute():
    """Including the 1004 zero pads of the short prompt (the issue's bug) changes its LSE
    by ln((e^lse + 1004) / e^lse): the kernel must not do that."""
    g = W.cfg_text_cross()
    q, k, v = W.make_qkv(g, 1002, k_pad_fill=0.0)
    _, l = gpu_forward(g, q, k, v)
    wrong = g.with_keys(g.cu_k, np.array([1024, 1024]))
    _, lw = gpu_forward(wrong, q, k, v)
    r = slice(int(g.cu_q[1]), int(g.cu_q[2]))
    expect = torch.log(torch.exp(l[:, r].double()) + (1024 - 20))
    assert torch.allclose(lw[:, r].double(), expect, atol=2e-3)
    assert float((lw[:, r] - l[:, r]).min()) > 1.0


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_nan_gaps_do_not_leak(seed):
    """Q / K / V gap rows filled with NaN give results bit-identical to zero-filled gaps."""
    rng = np.random.default_rng(seed)
    g = W.random_geometry(rng, 5, 300, 400, 8, 2, 128)
    qa, ka, va = W.make_qkv(g, seed, gap_fill=float("nan"))
    qb, kb, vb = W.make_qkv(g, seed, gap_fill=0.0)
    oa, la = gpu_forward(g, qa, ka, va)
    ob, lb = gpu_forward(g, qb, kb, vb)
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    o_ref, l_ref = oracle_forward(g, qb, kb, vb)
    check_full(g, oa, la, o_ref, l_ref, W.TINY_SENTINEL)


CASES = [  # (Hq, Hkv, d, out dtype, seed)
    (4, 4, 128, torch.bfloat16, 21),
    (8, 4, 128, torch.bfloat16, 22),
    (16, 4, 128, torch.float32, 23),
    (32, 4, 128, torch.bfloat16, 24),
    (8, 8, 64, torch.bfloat16, 25),
    (16, 8, 64, torch.float32, 26),
    (32, 8, 64, torch.bfloat16, 27),
    (128, 1, 128, torch.bfloat16, 28),
    # groups that do not divide the 128-row tile: floor(128 / g) tokens per tile
    (12, 4, 128, torch.bfloat16, 29),   # g = 3: 12 cross-attention heads split over 4 KV heads
    (24, 4, 128, torch.float32, 30),    # g = 6
    (12, 1, 64, torch.bfloat16, 31),    # g = 12
    (40, 8, 128, torch.bfloat16, 32),   # g = 5
    (100, 1, 128, torch.bfloat16, 33),  # g = 100: one token of 100 heads per tile
]


@pytest.mark.parametrize("hq,hkv,d,dtype,seed", CASES)
def test_random_gapped_geometries(hq, hkv, d, dtype, seed):
    """Random capacities and used lengths (zero-length segments included), spanning
    several tiles and key blocks with ragged tails."""
    rng = np.random.default_rng(seed)
    g = W.random_geometry(rng, 6, 700, 900, hq, hkv, d)
    q, k, v = W.make_qkv(g, seed, gap_fill=float("nan"))
    o, l = gpu_forward(g, q, k, v, out_dtype=dtype)
    o_ref, l_ref = oracle_forward(g, q, k, v)
    check_full(g, o, l, o_ref, l_ref, W.TINY_SENTINEL)


@pytest.mark.parametrize("scale", [0.02, 0.25])
def test_explicit_softmax_scale(scale):
    """A sharper softmax concentrates O on few values of |v| up to ~4, where rounding O
    itself to bf16 costs up to 1.6e-2; fp32 output measures the kernel's arithmetic."""
    rng = np.random.default_rng(31)
    g = W.random_geometry(rng, 3, 300, 500, 8, 2, 128, allow_empty=False)
    q, k, v = W.make_qkv(g, 31)
    o, l = gpu_forward(g, q, k, v, scale=scale, out_dtype=torch.float32)
    o_ref, l_ref = oracle_forward(g, q, k, v, scale=scale)
    check_full(g, o, l, o_ref, l_ref, W.TINY_SENTINEL)


def test_large_logits_rescale_path():
    """Scaled-up queries give logit ranges far beyond the rescale threshold, with the max
    growing along the keys (keys sorted by their logit), so O is rescaled many times."""
    rng = np.random.default_rng(32)
    g = W.random_geometry(rng, 2, 256, 1500, 8, 8, 128, allow_empty=False)
    q, k, v = W.make_qkv(g, 32)
    q = (q.float() * 4.0).bfloat16()
    k = k.clone()
    for b in range(g.num_segments):  # ascending norms along the keys of each segment
        k0, n = int(g.cu_k[b]), int(g.used_k[b])
        k[k0:k0 + n] = (k[k0:k0 + n].float() * torch.linspace(0.2, 3.0, n)[:, None, None]).bfloat16()
    o, l = gpu_forward(g, q, k, v)
    o_ref, l_ref = oracle_forward(g, q, k, v)
    check_full(g, o, l, o_ref, l_ref, W.TINY_SENTINEL)


def test_all_keyless_and_empty_segments():
    g = W.Geometry(np.array([0, 5, 5, 300], np.int32), np.array([5, 0, 200], np.int32),
                   np.array([0, 0, 0, 0], np.int32), np.array([0, 0, 0], np.int32), 8, 2, 128)
    q = torch.randn(g.total_q, 8, 128).bfloat16()
    k = torch.zeros(0, 2, 128, dtype=torch.bfloat16)
    o, l = gpu_forward(g, q, k, k)
    o_ref, l_ref = oracle_forward(g, q, k, k)
    check_full(g, o, l, o_ref, l_ref, W.TINY_SENTINEL)


def test_deterministic():
    rng = np.random.default_rng(41)
    g = W.random_geometry(rng, 4, 600, 900, 16, 4, 128)
    q, k, v = W.make_qkv(g, 41)
    o1, l1 = gpu_forward(g, q, k, v)
    o2, l2 = gpu_forward(g, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_plan_info():
    g = W.cfg_text_cross()
    plan = gva.Plan.from_geometry(g)
    info = plan.info()
    assert info["total_q"] == g.total_q and info["total_k"] == g.total_k
    # 2 segments x 8 KV heads x ceil(4096 / 128) items of 2 x 64 tokens
    assert info["num_work_items"] == 2 * 8 * 32
    assert info["used_flops"] == pytest.approx(g.used_flops())
    assert 0 < info["grid_ctas"] <= info["sm_count"]


# ------------------------------------------------------------------------------------
# Full-size workloads, sampled.
# ------------------------------------------------------------------------------------

def _device_inputs(g, seed, **kw):
    return W.make_qkv(g, seed, device="cuda", **kw)


@pytest.mark.slow
def test_long_replay_full_size_sampled():
    """4 segments of up to 32768 rows and 65536 keys, Hq=32, Hkv=8, d=128."""
    g = W.long_replay()
    q, k, v = _device_inputs(g, 1005, gap_fill=float("nan"))
    o, l = gpu_forward(g, q, k, v)
    assert gap_untouched(g, o, l, W.TINY_SENTINEL)
    rows = sample_rows(g, np.random.default_rng(5), per_segment=4)
    o_ref, l_ref = gva_oracle.attention_rows(q.cpu(), k.cpu(), v.cpu(), g.cu_q, g.used_q, g.cu_k, g.used_k, rows)
    check_rows(o, l, rows, o_ref, l_ref)
    assert not bool(torch.isnan(o.float()).any())


@pytest.mark.slow
def test_multiview_partitions_and_merge_full_size():
    """7 camera segments with gaps; two visibility partitions (fp32 partials) merged by
    gva_lse_merge equal attention over the union (oracle on sampled rows)."""
    full, parts = W.multiview_causal()
    q, k, v = _device_inputs(full, 1003, gap_fill=float("nan"))
    partials = [gpu_forward(p, q, k, v, out_dtype=torch.float32) for p in parts]
    plan = gva.Plan.from_geometry(full)
    o, l = W.make_outputs(full, W.TINY_SENTINEL, device="cuda")
    gva.lse_merge(plan, [p[0] for p in partials], [p[1] for p in partials], o, l)
    gva.device_status(plan)
    assert gap_untouched(full, o, l, W.TINY_SENTINEL)
    rows = sample_rows(full, np.random.default_rng(3), per_segment=3)
    o_ref, l_ref = gva_oracle.attention_rows(q.cpu(), k.cpu(), v.cpu(), full.cu_q, full.used_q, full.cu_k,
                                             full.used_k, rows)
    check_rows(o, l, rows, o_ref, l_ref)
    # the single-launch forward over the union agrees with the merged result
    o1, l1 = gpu_forward(full, q, k, v)
    check_rows(o1, l1, rows, o_ref, l_ref)


@pytest.mark.slow
@pytest.mark.parametrize("empty", ["text", "video"])
def test_lse_merge_union_full_size(empty):
    """8192 rows attending 1024 text + 16384 video keys (Hq = Hkv = 24) as two
    launches merged, against the oracle over the union; one segment has an empty
    partition (identity merge)."""
    text, video, union, dead = W.lse_merge_union(empty=empty)
    gen = torch.Generator(device="cuda").manual_seed(1004)
    q = torch.randn((text.total_q, 24, 128), generator=gen, device="cuda").bfloat16()
    kt = torch.randn((text.total_k, 24, 128), generator=gen, device="cuda").bfloat16()
    vt = torch.randn_like(kt, dtype=torch.float32).bfloat16()
    kv_ = torch.randn((video.total_k, 24, 128), generator=gen, device="cuda").bfloat16()
    vv = torch.randn_like(kv_, dtype=torch.float32).bfloat16()
    pt = gpu_forward(text, q, kt, vt, out_dtype=torch.float32)
    pv = gpu_forward(video, q, kv_, vv, out_dtype=torch.float32)
    plan = gva.Plan.from_geometry(union)
    o, l = W.make_outputs(union, 0.0, device="cuda")
    gva.lse_merge(plan, [pt[0], pv[0]], [pt[1], pv[1]], o, l)
    gva.device_status(plan)
    # oracle over the union: for each sampled row, the used text keys then the used
    # video keys of its segment
    rows = sample_rows(union, np.random.default_rng(4), per_segment=3)
    qc = q.cpu()
    o_ref = np.zeros((len(rows), 24, 128))
    l_ref = np.zeros((24, len(rows)))
    for b in range(union.num_segments):
        idx = [i for i, r in enumerate(rows) if union.cu_q[b] <= r < union.cu_q[b + 1]]
        if not idx:
            continue
        t0, nt = int(text.cu_k[b]), int(text.used_k[b])
        v0, nv = int(video.cu_k[b]), int(video.used_k[b])
        ks = torch.cat([kt[t0:t0 + nt], kv_[v0:v0 + nv]]).cpu()
        vs = torch.cat([vt[t0:t0 + nt], vv[v0:v0 + nv]]).cpu()
        q0, nq = int(union.cu_q[b]), int(union.used_q[b])
        oo, ll = gva_oracle.attention_rows(qc, ks, vs, np.array([q0, q0 + nq]), [nq], np.array([0, nt + nv]),
                                           [nt + nv], [rows[i] for i in idx])
        o_ref[idx], l_ref[:, idx] = oo, ll
    check_rows(o, l, rows, o_ref, l_ref)
    # the empty partition's segment: merged result equals the other partition's
    r0, r1 = int(union.cu_q[dead]), int(union.cu_q[dead]) + int(union.used_q[dead])
    other = pv if empty == "text" else pt
    assert torch.equal(l[:, r0:r1], other[1][:, r0:r1])
    assert torch.equal(o[r0:r1], other[0][r0:r1].bfloat16())
