"""GPU parity of the backward (gva_backward) against the FP64 oracle.

Tolerance, from the arithmetic: the kernels round P and dS to bf16 before the two
tensor-core products that use them (relative error 2^-9 per term, unbiased), read O
in bf16 for D = <dO, O>, and accumulate in FP32. For sums of many such terms the error
stays a small multiple of 2^-9 of the result's scale, so each gradient tensor must
satisfy max |g - g_ref| <= 2^-6 max |g_ref| (4 x the single rounding of a bf16 store
of the largest element) and rms(g - g_ref) <= 2^-8 rms(g_ref). Rows the backward must
not write keep their sentinel bit for bit; keyless rows get dQ = 0 exactly and the
keys of a segment without rows get dK = dV = 0 exactly."""
import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import workloads as W
from oracle import gva_oracle

pytestmark = pytest.mark.gpu
FILL = W.TINY_SENTINEL
MAX_REL = 2.0 ** -6
RMS_REL = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _built():
    gva.build()


def _make_dout(g, seed, gap_fill=float("nan"), device="cpu"):
    gen = torch.Generator(device=device).manual_seed(seed + 7)
    do = torch.randn((g.total_q, g.num_heads_q, g.head_dim), generator=gen, device=device).bfloat16()
    if gap_fill is not None:
        do[torch.from_numpy(W.gap_rows(g.cu_q, g.used_q)).to(device)] = gap_fill
    return do


def _masks(g):
    """Rows of dq and keys of dk / dv the backward writes."""
    dq_rows = ~W.gap_rows(g.cu_q, g.used_q)
    dk_rows = np.zeros(g.total_k, bool)
    for b in range(g.num_segments):
        dk_rows[g.cu_k[b]:g.cu_k[b] + g.used_k[b]] = True
    return dq_rows, dk_rows


def gpu_backward(g, q, k, v, do, scale=0.0, grad_dtype=torch.bfloat16, plan=None, causal_block=0):
    plan = plan or gva.Plan.from_geometry(g, causal_block=causal_block)
    qc, kc, vc, doc = (t.cuda() for t in (q, k, v, do))
    o, l = W.make_outputs(g, FILL, device="cuda")
    gva.forward(plan, qc, kc, vc, o, l, scale)
    dq = torch.full(qc.shape, FILL, dtype=grad_dtype, device="cuda")
    dk = torch.full(kc.shape, FILL, dtype=grad_dtype, device="cuda")
    dv = torch.full(vc.shape, FILL, dtype=grad_dtype, device="cuda")
    gva.backward(plan, qc, kc, vc, o, l, doc, dq, dk, dv, scale)
    gva.device_status(plan)
    return dq, dk, dv


def oracle_backward(g, q, k, v, do, scale=None, causal_block=0):
    qn, kn, vn, don = (t.detach().cpu().float().numpy() for t in (q, k, v, do))
    return gva_oracle.attention_backward(qn, kn, vn, don, g.cu_q, g.used_q, g.cu_k, g.used_k, scale=scale,
                                         dq=np.full(qn.shape, FILL), dk=np.full(kn.shape, FILL),
                                         dv=np.full(vn.shape, FILL), causal_block=causal_block)


def _close(name, got, ref, max_rel=MAX_REL, rms_rel=RMS_REL, atol=0.0):
    if ref.size == 0:
        return 0.0
    err = np.abs(got - ref)
    scale = max(np.abs(ref).max(), 1e-30)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    assert err.max() <= max_rel * scale + atol, f"{name}: max err {err.max():.3e} > {max_rel:.1e} x {scale:.3e}"
    rms_ref = max(np.sqrt(np.mean(ref ** 2)), 1e-30)
    rms_err = np.sqrt(np.mean(err ** 2))
    assert rms_err <= rms_rel * rms_ref + atol, f"{name}: rms err {rms_err:.3e} > {rms_rel:.1e} x {rms_ref:.3e}"
    return float(err.max() / scale)


def check_backward(g, got, ref, max_rel=MAX_REL, rms_rel=RMS_REL, atol=0.0):
    dq, dk, dv = (t.float().cpu().numpy().astype(np.float64) for t in got)
    dq_ref, dk_ref, dv_ref = ref
    dq_rows, dk_rows = _masks(g)
    fill32 = np.float64(np.float32(FILL))
    assert np.all(dq[~dq_rows] == fill32), "a gap row of dQ was written"
    assert np.all(dk[~dk_rows] == fill32) and np.all(dv[~dk_rows] == fill32), "a key past seqused_k was written"
    exact = []  # rows whose exact answer is 0: keyless segments' rows, row-less segments' keys
    for b in range(g.num_segments):
        r0, nq, k0, nk = int(g.cu_q[b]), int(g.used_q[b]), int(g.cu_k[b]), int(g.used_k[b])
        if nq and not nk:
            assert np.all(dq[r0:r0 + nq] == 0.0), "keyless segment: dQ must be 0"
        if nk and not nq:
            assert np.all(dk[k0:k0 + nk] == 0.0) and np.all(dv[k0:k0 + nk] == 0.0), "row-less segment: dK/dV must be 0"
            exact.append(b)
    errs = (_close("dQ", dq[dq_rows], dq_ref[dq_rows], max_rel, rms_rel, atol),
            _close("dK", dk[dk_rows], dk_ref[dk_rows], max_rel, rms_rel, atol),
            _close("dV", dv[dk_rows], dv_ref[dk_rows], max_rel, rms_rel, atol))
    print(f"max err / max |ref|: dQ {errs[0]:.2e}  dK {errs[1]:.2e}  dV {errs[2]:.2e}")
    return errs


def test_tiny():
    g = W.tiny()
    q, k, v = W.make_qkv(g, 1001, gap_fill=float("nan"))
    do = _make_dout(g, 1001)
    check_backward(g, gpu_backward(g, q, k, v, do), oracle_backward(g, q, k, v, do))


CASES = [  # (Hq, Hkv, d, seed)
    (8, 2, 128, 201),
    (16, 16, 128, 202),
    (32, 8, 64, 203),
    (4, 4, 64, 204),
    (16, 1, 128, 205),
    (128, 1, 64, 206),
    # groups that do not divide the 128-row tile: floor(128 / g) tokens per tile
    (12, 4, 128, 207),  # g = 3
    (24, 4, 64, 208),   # g = 6
    (12, 1, 128, 209),  # g = 12
    (96, 1, 64, 210),   # g = 96: one token of 96 heads per tile
]


@pytest.mark.parametrize("hq,hkv,d,seed", CASES)
def test_random_geometries(hq, hkv, d, seed):
    """Ragged segments spanning several Q tiles and key blocks, empty segments, NaN in
    every gap row of Q, K, V and dO."""
    rng = np.random.default_rng(seed)
    g = W.random_geometry(rng, 6, 600, 700, hq, hkv, d)
    q, k, v = W.make_qkv(g, seed, gap_fill=float("nan"))
    do = _make_dout(g, seed)
    check_backward(g, gpu_backward(g, q, k, v, do), oracle_backward(g, q, k, v, do))


def test_keyless_and_rowless_segments():
    """A segment with rows but no keys (dQ = 0) and one with keys but no rows (dK = dV = 0)."""
    cu_q = np.array([0, 100, 230, 230, 300], np.int32)
    used_q = np.array([90, 130, 0, 61], np.int32)
    cu_k = np.array([0, 150, 150, 400, 700], np.int32)
    used_k = np.array([150, 0, 250, 129], np.int32)
    g = W.Geometry(cu_q, used_q, cu_k, used_k, 8, 4, 128)
    q, k, v = W.make_qkv(g, 301, gap_fill=float("nan"))
    do = _make_dout(g, 301)
    check_backward(g, gpu_backward(g, q, k, v, do), oracle_backward(g, q, k, v, do))


def test_no_keys_at_all():
    """Every segment keyless: K / V are empty, dQ is zero on used rows only."""
    cu_q = np.array([0, 50, 50, 170], np.int32)
    g = W.Geometry(cu_q, np.array([31, 0, 100], np.int32), np.zeros(4, np.int32), np.zeros(3, np.int32), 16, 4, 128)
    q, k, v = W.make_qkv(g, 311, gap_fill=float("nan"))
    assert k.shape[0] == 0
    do = _make_dout(g, 311)
    check_backward(g, gpu_backward(g, q, k, v, do), oracle_backward(g, q, k, v, do))


def test_no_rows_at_all():
    """No used query row anywhere: the used keys get dK = dV = 0, nothing else is written."""
    g = W.Geometry(np.zeros(3, np.int32), np.zeros(2, np.int32), np.array([0, 130, 300], np.int32),
                   np.array([129, 77], np.int32), 8, 8, 64)
    q, k, v = W.make_qkv(g, 312, gap_fill=float("nan"))
    assert q.shape[0] == 0
    do = _make_dout(g, 312)
    check_backward(g, gpu_backward(g, q, k, v, do), oracle_backward(g, q, k, v, do))


def test_fp32_gradients_and_explicit_scale():
    rng = np.random.default_rng(401)
    g = W.random_geometry(rng, 4, 500, 500, 16, 4, 128, allow_empty=False)
    q, k, v = W.make_qkv(g, 401)
    do = _make_dout(g, 401)
    got = gpu_backward(g, q, k, v, do, scale=0.05, grad_dtype=torch.float32)
    # no bf16 store of the result: half the bound
    check_backward(g, got, oracle_backward(g, q, k, v, do, scale=0.05), max_rel=MAX_REL / 2, rms_rel=RMS_REL / 2)


def test_deterministic():
    rng = np.random.default_rng(501)
    g = W.random_geometry(rng, 5, 700, 900, 32, 8, 128, allow_empty=False)
    q, k, v = W.make_qkv(g, 501)
    do = _make_dout(g, 501)
    plan = gva.Plan.from_geometry(g)
    a = gpu_backward(g, q, k, v, do, plan=plan)
    b = gpu_backward(g, q, k, v, do, plan=plan)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_overlapping_ranges_tiny():
    """Two segments whose key ranges share rows 40 .. 47: those rows' dK / dV sum both
    segments' contributions (the oracle's summed gradient)."""
    g = W.tiny()
    ranges = [[(0, 48)], [(40, 33)], []]
    q, k, v = W.make_qkv(g, 1001)
    do = _make_dout(g, 1001)
    _check_ranges(g, ranges, _ranges_backward(g, ranges, g.total_k, q, k, v, do), q, k, v, do)


def _ranges_backward(g, ranges, total_k, q, k, v, do):
    plan = gva.Plan.from_ranges(g.cu_q, g.used_q, ranges, total_k, g.num_heads_q, g.num_heads_kv, g.head_dim)
    return gpu_backward(g, q, k, v, do, plan=plan)


def _check_ranges(g, ranges, got, q, k, v, do):
    qn, kn, vn, don = (t.detach().cpu().float().numpy() for t in (q, k, v, do))
    ref = gva_oracle.attention_backward_ranges(qn, kn, vn, don, g.cu_q, g.used_q, ranges,
                                               dq=np.full(qn.shape, FILL), dk=np.full(kn.shape, FILL),
                                               dv=np.full(vn.shape, FILL))
    dq, dk, dv = (t.float().cpu().numpy().astype(np.float64) for t in got)
    dq_rows = ~W.gap_rows(g.cu_q, g.used_q)
    covered = np.zeros(kn.shape[0], bool)
    for rr in ranges:
        for st, n in rr:
            covered[st:st + n] = True
    fill32 = np.float64(np.float32(FILL))
    assert np.all(dq[~dq_rows] == fill32) and np.all(dk[~covered] == fill32) and np.all(dv[~covered] == fill32)
    attended = np.zeros(kn.shape[0], bool)  # K/V rows some segment with used rows attends
    for b, rr in enumerate(ranges):
        if g.used_q[b]:
            for st, n in rr:
                attended[st:st + n] = True
    for b, rr in enumerate(ranges):  # exact zeros: keyless segments' rows, keys no used row attends
        if g.used_q[b] and not sum(n for _, n in rr):
            assert np.all(dq[g.cu_q[b]:g.cu_q[b] + g.used_q[b]] == 0.0)
    idle = covered & ~attended
    assert np.all(dk[idle] == 0.0) and np.all(dv[idle] == 0.0)
    _close("dQ", dq[dq_rows], ref[0][dq_rows])
    _close("dK", dk[covered], ref[1][covered])
    _close("dV", dv[covered], ref[2][covered])


@pytest.mark.parametrize("hq,hkv,d,seed", [(8, 2, 128, 801), (16, 16, 64, 802), (32, 8, 128, 803)])
def test_disjoint_key_ranges(hq, hkv, d, seed):
    """Up to four disjoint ranges per segment anywhere in K/V (ragged lengths, empty
    ranges, partial blocks in the middle of a segment's keys); rows no range covers are
    NaN and must stay untouched."""
    rng = np.random.default_rng(seed)
    g = W.random_geometry(rng, 5, 500, 10, hq, hkv, d)
    total_k = 3000
    cuts = np.sort(rng.choice(np.arange(1, total_k), size=2 * 4 * g.num_segments, replace=False))
    pieces = [(int(cuts[2 * i]), int(cuts[2 * i + 1] - cuts[2 * i])) for i in range(len(cuts) // 2)]
    rng.shuffle(pieces)
    ranges = []
    for b in range(g.num_segments):
        take = int(rng.integers(0, 5))
        ranges.append([(st, min(n, 400)) for st, n in pieces[:take]])
        pieces = pieces[take:]
    ranges[0] = []  # one keyless segment
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(g.total_q, hq, d, generator=gen).bfloat16()
    k = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    v = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    do = _make_dout(g, seed)
    covered = np.zeros(total_k, bool)
    for rr in ranges:
        for st, n in rr:
            covered[st:st + n] = True
    k[torch.from_numpy(~covered)] = float("nan")
    v[torch.from_numpy(~covered)] = float("nan")
    _check_ranges(g, ranges, _ranges_backward(g, ranges, total_k, q, k, v, do), q, k, v, do)


@pytest.mark.parametrize("hq,hkv,d,seed", [(8, 2, 128, 821), (16, 16, 64, 822), (12, 4, 128, 823)])
def test_overlapping_key_ranges(hq, hkv, d, seed):
    """Key ranges that overlap freely: every segment attends one shared range (a common
    prompt), plus up to three ranges of its own that may overlap other segments' ranges
    or its own (one range listed twice). A K/V row's dK / dV is the sum over every
    attending segment, counted once per covering range; rows no range covers stay
    untouched (NaN inputs there)."""
    rng = np.random.default_rng(seed)
    g = W.random_geometry(rng, 5, 500, 10, hq, hkv, d)
    total_k = 2000
    shared = (int(rng.integers(0, 400)), int(rng.integers(1, 300)))
    ranges = []
    for b in range(g.num_segments):
        rr = [shared]
        for _ in range(int(rng.integers(0, 4))):
            st = int(rng.integers(0, total_k - 1))
            rr.append((st, int(rng.integers(0, min(400, total_k - st) + 1))))
        ranges.append(rr)
    ranges[-1].append(ranges[-1][-1])  # a range listed twice: its keys enter the softmax twice
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(g.total_q, hq, d, generator=gen).bfloat16()
    k = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    v = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    do = _make_dout(g, seed)
    covered = np.zeros(total_k, bool)
    for rr in ranges:
        for st, n in rr:
            covered[st:st + n] = True
    k[torch.from_numpy(~covered)] = float("nan")
    v[torch.from_numpy(~covered)] = float("nan")
    _check_ranges(g, ranges, _ranges_backward(g, ranges, total_k, q, k, v, do), q, k, v, do)


def test_rank_major_keys_backward():
    """Keys in the rank-major order an all-to-all leaves (per rank: a text chunk, then a
    video chunk): each sample attends its text length of every text chunk plus all video
    keys; the zero pads of the text chunks are in no range and stay untouched."""
    ranks, text_cap, video = 4, 64, 384
    text_len = [[37, 64, 5, 0], [64, 64, 64, 12]]
    hq, hkv, d = 16, 8, 128
    cu_q = np.array([0, 1000, 2000], np.int32)
    g = W.Geometry(cu_q, np.array([1000, 777], np.int32), np.array([0, 0, 0], np.int32), np.array([0, 0], np.int32),
                   hq, hkv, d)
    chunk = text_cap + video
    total_k = 2 * ranks * chunk
    ranges = [[x for r in range(ranks) for x in (((b * ranks + r) * chunk, text_len[b][r]),
                                                 ((b * ranks + r) * chunk + text_cap, video))] for b in range(2)]
    gen = torch.Generator().manual_seed(811)
    q = torch.randn(g.total_q, hq, d, generator=gen).bfloat16()
    k = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    v = torch.randn(total_k, hkv, d, generator=gen).bfloat16()
    do = _make_dout(g, 811)
    _check_ranges(g, ranges, _ranges_backward(g, ranges, total_k, q, k, v, do), q, k, v, do)


CAUSAL_CASES = [  # (Hq, Hkv, d, causal block, seed)
    (8, 2, 128, 1, 601),
    (16, 4, 128, 3, 602),
    (32, 8, 128, 64, 603),
    (8, 8, 64, 200, 604),
    (16, 1, 64, 128, 605),
    (4, 1, 128, 129, 606),
    (12, 4, 128, 7, 607),  # g = 3
    (24, 2, 64, 50, 608),  # g = 12
]


@pytest.mark.parametrize("hq,hkv,d,block,seed", CAUSAL_CASES)
def test_block_causal_random_geometries(hq, hkv, d, block, seed):
    """Gradients of the block-causal forward: random gapped geometries where used_q may
    exceed used_k (early rows see no key: dQ = 0 there), NaN in every gap row."""
    rng = np.random.default_rng(seed)
    g = W.random_geometry(rng, 6, 600, 700, hq, hkv, d)
    q, k, v = W.make_qkv(g, seed, gap_fill=float("nan"))
    do = _make_dout(g, seed)
    check_backward(g, gpu_backward(g, q, k, v, do, causal_block=block),
                   oracle_backward(g, q, k, v, do, causal_block=block))


def test_block_causal_huge_block_is_the_maskless_backward():
    """With used_q <= used_k every row sits at a non-negative key position, so a block
    longer than any segment masks nothing: bit-identical to the maskless backward."""
    rng = np.random.default_rng(607)
    g = W.random_geometry(rng, 5, 500, 800, 16, 4, 128)
    g.used_q = np.minimum(g.used_q, g.used_k).astype(np.int32)
    q, k, v = W.make_qkv(g, 607)
    do = _make_dout(g, 607)
    a = gpu_backward(g, q, k, v, do, causal_block=1 << 20)
    b = gpu_backward(g, q, k, v, do)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_cfg_text_cross_full():
    """The CFG text cross-attention workload at full size (8192 rows, 700 / 20 used of
    1024 padded keys), every gradient element against the oracle."""
    g = W.cfg_text_cross()
    q, k, v = W.make_qkv(g, 1002, k_pad_fill=0.0)
    do = _make_dout(g, 1002)
    check_backward(g, gpu_backward(g, q, k, v, do), oracle_backward(g, q, k, v, do))


def _segment_properties(g, q, k, do, dq, dk, dv, b, s):
    """Identities of the exact gradients of one segment, per KV head:
    sum_j dV_j = sum_{i, h in group} dO_i (softmax rows sum to 1), sum_j dK_j = 0 (the
    rows of dS sum to 0), and sum_i <Q_i, dQ_i> = sum_j <K_j, dK_j> (both equal
    sum_ij dS_ij x_ij)."""
    r0, nq, k0, nk = int(g.cu_q[b]), int(g.used_q[b]), int(g.cu_k[b]), int(g.used_k[b])
    grp = g.num_heads_q // g.num_heads_kv
    f = lambda t: t.double()  # noqa: E731
    for hk in range(g.num_heads_kv):
        heads = slice(hk * grp, (hk + 1) * grp)
        sdo = f(do[r0:r0 + nq, heads]).sum(dim=(0, 1))
        sdv = f(dv[k0:k0 + nk, hk]).sum(dim=0)
        scale_dv = f(dv[k0:k0 + nk, hk]).abs().sum(dim=0).max().item()
        assert (sdv - sdo).abs().max().item() <= 1e-2 * scale_dv + 1e-3, "sum dV != sum dO"
        sdk = f(dk[k0:k0 + nk, hk]).sum(dim=0)
        scale_dk = f(dk[k0:k0 + nk, hk]).abs().sum(dim=0).max().item()
        assert sdk.abs().max().item() <= 1e-2 * scale_dk, "sum dK != 0"
        qdq = (f(q[r0:r0 + nq, heads]) * f(dq[r0:r0 + nq, heads])).sum().item()
        kdk = (f(k[k0:k0 + nk, hk]) * f(dk[k0:k0 + nk, hk])).sum().item()
        mag = (f(q[r0:r0 + nq, heads]) * f(dq[r0:r0 + nq, heads])).abs().sum().item()
        assert abs(qdq - kdk) <= 1e-2 * mag, f"<Q,dQ> {qdq:.4e} != <K,dK> {kdk:.4e}"


@pytest.mark.slow
def test_long_replay_full_size_sampled():
    """The long replay workload at full size (4 segments, up to 32768 rows and 65536
    keys each): dQ on sampled rows against the oracle (a row's dQ depends on that row
    only), dK / dV through identities that hold at any size."""
    g = W.long_replay()
    q, k, v = W.make_qkv(g, 1005, device="cuda", gap_fill=float("nan"))
    do = _make_dout(g, 1005, device="cuda")
    dq, dk, dv = gpu_backward(g, q, k, v, do)
    dq_rows, dk_rows = _masks(g)
    assert bool((dq[torch.from_numpy(~dq_rows).cuda()].float() == FILL).all())
    assert bool((dk[torch.from_numpy(~dk_rows).cuda()].float() == FILL).all())
    rng = np.random.default_rng(12)
    s = 1.0 / np.sqrt(g.head_dim)
    for b in range(g.num_segments):
        _segment_properties(g, q, k, do, dq, dk, dv, b, s)
        # sampled rows, each a one-row segment over the segment's keys
        rows = sorted(set(int(x) for x in rng.integers(0, g.used_q[b], size=3)) | {0, int(g.used_q[b]) - 1})
        k0, nk = int(g.cu_k[b]), int(g.used_k[b])
        sel = [int(g.cu_q[b]) + r for r in rows]
        qs, dos = q[sel].cpu(), do[sel].cpu()
        n = len(sel)
        ks, vs = k[k0:k0 + nk].cpu(), v[k0:k0 + nk].cpu()
        dq_ref, _, _ = gva_oracle.attention_backward(qs, ks, vs, dos, np.arange(n + 1), np.ones(n, np.int64),
                                                     np.zeros(n + 1, np.int64), np.full(n, nk))
        got = dq[sel].float().cpu().numpy().astype(np.float64)
        scale = np.abs(dq_ref).max()
        assert np.abs(got - dq_ref).max() <= MAX_REL * scale


@pytest.mark.slow
def test_multiview_block_causal_full_size_sampled():
    """The multiview workload (7 segments, 512-token frames) at full size: dQ on sampled
    rows against the oracle (each sampled row attends exactly its visible keys), dK / dV
    through the identities (every row sees at least its own frame here: used_q < used_k)."""
    full, _ = W.multiview_causal()
    blk = 512
    q, k, v = W.make_qkv(full, 1003, device="cuda", gap_fill=float("nan"))
    do = _make_dout(full, 1003, device="cuda")
    dq, dk, dv = gpu_backward(full, q, k, v, do, causal_block=blk)
    dq_rows, dk_rows = _masks(full)
    assert bool((dq[torch.from_numpy(~dq_rows).cuda()].float() == FILL).all())
    assert bool((dk[torch.from_numpy(~dk_rows).cuda()].float() == FILL).all())
    rng = np.random.default_rng(14)
    for b in range(full.num_segments):
        nq, nk = int(full.used_q[b]), int(full.used_k[b])
        lim = gva_oracle.causal_limits(nq, nk, blk)
        _segment_properties(full, q, k, do, dq, dk, dv, b, 1.0 / np.sqrt(full.head_dim))
        rows = sorted(set(int(x) for x in rng.integers(0, nq, size=3)) | {0, nq - 1})
        k0 = int(full.cu_k[b])
        for r in rows:
            sel = [int(full.cu_q[b]) + r]
            n = int(lim[r])
            dq_ref, _, _ = gva_oracle.attention_backward(q[sel].cpu(), k[k0:k0 + n].cpu(), v[k0:k0 + n].cpu(),
                                                         do[sel].cpu(), [0, 1], [1], [0, n], [n])
            got = dq[sel].float().cpu().numpy().astype(np.float64)
            assert np.abs(got - dq_ref).max() <= MAX_REL * max(np.abs(dq_ref).max(), 1e-30)


@pytest.mark.slow
def test_long_replay_small_one_segment_and_kv_head_elementwise():
    """dQ, dK and dV element by element at full size: the whole reduced long replay (2
    segments of up to 8192 rows and 32768 keys, Hq = 32, Hkv = 8) runs through the
    backward, and one whole segment of one KV head is checked against the oracle. Each
    dK / dV unit there sums over the segment's ~190 Q tiles (32 tokens x 4 heads each),
    so an error in one unit's accumulation or in any tile it streams shows up here,
    which the sum identities at the larger size cannot localise."""
    g = W.long_replay_small()
    q, k, v = W.make_qkv(g, 1006, device="cuda", gap_fill=float("nan"))
    do = _make_dout(g, 1006, device="cuda")
    dq, dk, dv = gpu_backward(g, q, k, v, do)
    b, hk = 0, int(np.random.default_rng(31).integers(0, g.num_heads_kv))
    grp = g.num_heads_q // g.num_heads_kv
    heads = slice(hk * grp, (hk + 1) * grp)
    r0, nq, k0, nk = int(g.cu_q[b]), int(g.used_q[b]), int(g.cu_k[b]), int(g.used_k[b])
    qs, dos = q[r0:r0 + nq, heads].cpu(), do[r0:r0 + nq, heads].cpu()
    ks, vs = k[k0:k0 + nk, hk:hk + 1].cpu(), v[k0:k0 + nk, hk:hk + 1].cpu()
    # the same problem with this KV head's group alone: Hq = grp, Hkv = 1
    dq_ref, dk_ref, dv_ref = gva_oracle.attention_backward(qs, ks, vs, dos, [0, nq], [nq], [0, nk], [nk])
    got = [t.float().cpu().numpy().astype(np.float64) for t in
           (dq[r0:r0 + nq, heads], dk[k0:k0 + nk, hk:hk + 1], dv[k0:k0 + nk, hk:hk + 1])]
    errs = (_close("dQ", got[0], dq_ref), _close("dK", got[1], dk_ref), _close("dV", got[2], dv_ref))
    print(f"segment {b}, KV head {hk}: max err / max |ref|: dQ {errs[0]:.2e}  dK {errs[1]:.2e}  dV {errs[2]:.2e}")
