"""Pins for the FP64 oracle: each check ties it to something other than itself.

* brute force on tiny inputs (pure-Python scalar loops with ``math.fsum``);
* closed forms: all-zero keys, a single key, the dilution worked example;
* exact special cases: keyless segments, untouched gap rows, pad invariance;
* a library routine: equal-length gap-free segments against
  ``torch.nn.functional.scaled_dot_product_attention`` in float64;
* invariants: GQA = repeated K/V, key permutation, merge of disjoint key
  partitions = attention over their union.

``test_pins_catch_planted_mistakes`` plants plausible mistakes in a copy of the
oracle's source and checks that at least one pin fails for each.
"""
import inspect
import json
import math
import os
import types

import numpy as np
import pytest
import torch

from gapped_varlen_attention_gb300 import workloads as W
from oracle import gva_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------------
# Independent brute force: scalar Python, no numpy arithmetic.
# ------------------------------------------------------------------------------------

def brute_force(q, k, v, cu_q, used_q, cu_k, used_k, scale, fill_o, fill_l):
    total_q, hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    o = [[[fill_o for _ in range(d)] for _ in range(hq)] for _ in range(total_q)]
    l = [[fill_l for _ in range(total_q)] for _ in range(hq)]
    for b in range(len(used_q)):
        for i in range(int(used_q[b])):
            r = int(cu_q[b]) + i
            for h in range(hq):
                hk = h // g
                keys = range(int(cu_k[b]), int(cu_k[b]) + int(used_k[b]))
                if len(keys) == 0:
                    o[r][h] = [0.0] * d
                    l[h][r] = -math.inf
                    continue
                x = [scale * math.fsum(float(q[r, h, t]) * float(k[j, hk, t]) for t in range(d)) for j in keys]
                m = max(x)
                e = [math.exp(xi - m) for xi in x]
                den = math.fsum(e)
                o[r][h] = [math.fsum(e[n] * float(v[j, hk, t]) for n, j in enumerate(keys)) / den for t in range(d)]
                l[h][r] = m + math.log(den)
    return np.array(o), np.array(l)


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ------------------------------------------------------------------------------------
# Pins, parameterised on the oracle module so planted mistakes can be checked.
# ------------------------------------------------------------------------------------

def pin_bruteforce(orc):
    rng = np.random.default_rng(7)
    for trial in range(4):
        hq, hkv = [(2, 1), (4, 2), (3, 3), (6, 2)][trial]
        d = [4, 8, 5, 6][trial]
        g = W.random_geometry(rng, 4, 5, 6, hq, hkv, d)
        q = _rand(rng, g.total_q, hq, d)
        k = _rand(rng, g.total_k, hkv, d)
        v = _rand(rng, g.total_k, hkv, d)
        scale = 0.3 + trial * 0.2
        o_ref, l_ref = brute_force(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k, scale, 0.5, 0.25)
        o, l = orc.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k, scale=scale,
                                     out=np.full(q.shape, 0.5), lse=np.full((hq, g.total_q), 0.25))
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, l_ref, rtol=0, atol=1e-12)


def pin_default_scale(orc):
    rng = np.random.default_rng(8)
    g = W.random_geometry(rng, 2, 4, 5, 2, 1, 9, allow_empty=False)
    q, k, v = _rand(rng, g.total_q, 2, 9), _rand(rng, g.total_k, 1, 9), _rand(rng, g.total_k, 1, 9)
    o_ref, l_ref = brute_force(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k, 1.0 / 3.0, 0.0, 0.0)
    o, l = orc.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k)
    np.testing.assert_allclose(o, o_ref, atol=1e-12)
    np.testing.assert_allclose(l, l_ref, atol=1e-12)


def pin_dilution_golden(orc):
    with open(os.path.join(GOLDEN, "dilution_worked_example.json")) as f:
        ex = json.load(f)
    q = np.array(ex["q"])[:, None, :]
    k = np.array(ex["k"])[:, None, :]
    v = np.array(ex["v"])[:, None, :]
    cap = k.shape[0]
    for used, eo, el in [(ex["used_k"], ex["expected_o"], ex["expected_lse_exp"]),
                         (ex["diluted_used_k"], ex["diluted_o"], ex["diluted_lse_exp"])]:
        o, l = orc.attention_forward(q, k, v, [0, 1], [1], [0, cap], [used], scale=ex["scale"])
        np.testing.assert_allclose(o[0, 0], eo, rtol=0, atol=1e-14)
        assert abs(l[0, 0] - math.log(el)) < 1e-14


def pin_zero_keys_closed_form(orc):
    """All used keys zero: every logit is 0, so O = mean of the used values and
    LSE = ln(used_k), whatever the query."""
    rng = np.random.default_rng(9)
    for uk in [1, 3, 17]:
        q = _rand(rng, 5, 4, 8)
        k = np.zeros((uk + 4, 2, 8))
        v = _rand(rng, uk + 4, 2, 8)
        o, l = orc.attention_forward(q, k, v, [0, 5], [5], [0, uk + 4], [uk])
        mean = v[:uk].mean(axis=0)  # [2, 8]
        for h in range(4):
            np.testing.assert_allclose(o[:, h, :], np.broadcast_to(mean[h // 2], (5, 8)), atol=1e-13)
        np.testing.assert_allclose(l, math.log(uk), atol=1e-13)


def pin_single_key(orc):
    rng = np.random.default_rng(10)
    q = _rand(rng, 3, 2, 6)
    k = _rand(rng, 2, 1, 6)
    v = _rand(rng, 2, 1, 6)
    o, l = orc.attention_forward(q, k, v, [0, 3], [3], [0, 2], [1], scale=0.7)
    for r in range(3):
        for h in range(2):
            np.testing.assert_allclose(o[r, h], v[0, 0], atol=1e-14)
            x0 = 0.7 * math.fsum(q[r, h, t] * k[0, 0, t] for t in range(6))
            assert abs(l[h, r] - x0) < 1e-13


def pin_keyless_and_gap_rows(orc):
    """The tiny workload: 7.0 sentinels survive on gap rows bit for bit; the keyless
    segment's used rows get +0.0 and -inf."""
    g = W.tiny()
    q, k, v = (t.float().numpy() for t in W.make_qkv(g, 1001))
    o0 = np.full(q.shape, W.TINY_SENTINEL)
    l0 = np.full((g.num_heads_q, g.total_q), W.TINY_SENTINEL)
    o, l = orc.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k, out=o0, lse=l0)
    gap = W.gap_rows(g.cu_q, g.used_q)
    assert np.array_equal(o[gap], o0[gap]) and np.array_equal(l[:, gap], l0[:, gap])
    r0 = int(g.cu_q[2])
    keyless = slice(r0, r0 + int(g.used_q[2]))
    assert np.all(o[keyless] == 0.0) and not np.any(np.signbit(o[keyless]))
    assert np.all(np.isneginf(l[:, keyless]))
    keyed = ~gap
    keyed[keyless] = False
    assert np.all(np.isfinite(o[~gap])) and np.all(np.isfinite(l[:, keyed]))


def pin_pad_invariance(orc):
    """Appending zero or NaN K/V rows past the used keys (growing the capacity)
    leaves O and LSE bit-identical."""
    rng = np.random.default_rng(11)
    q = _rand(rng, 6, 2, 8)
    k = _rand(rng, 5, 2, 8)
    v = _rand(rng, 5, 2, 8)
    base = orc.attention_forward(q, k, v, [0, 6], [6], [0, 5], [5])
    for pad, fill in [(3, 0.0), (40, 0.0), (7, np.nan), (2, np.inf)]:
        kp = np.concatenate([k, np.full((pad, 2, 8), fill)])
        vp = np.concatenate([v, np.full((pad, 2, 8), fill)])
        got = orc.attention_forward(q, kp, vp, [0, 6], [6], [0, 5 + pad], [5])
        assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1])


def pin_sdpa_equal_lengths(orc):
    """Equal-length, gap-free segments are a dense batch: compare with PyTorch's
    float64 scaled_dot_product_attention (GQA via enable_gqa)."""
    rng = np.random.default_rng(12)
    B, L, S, hq, hkv, d = 3, 7, 9, 6, 2, 16
    q = _rand(rng, B * L, hq, d)
    k = _rand(rng, B * S, hkv, d)
    v = _rand(rng, B * S, hkv, d)
    cu_q = np.arange(B + 1) * L
    cu_k = np.arange(B + 1) * S
    o, _ = orc.attention_forward(q, k, v, cu_q, [L] * B, cu_k, [S] * B, scale=0.2)
    tq = torch.from_numpy(q).view(B, L, hq, d).transpose(1, 2)
    tk = torch.from_numpy(k).view(B, S, hkv, d).transpose(1, 2)
    tv = torch.from_numpy(v).view(B, S, hkv, d).transpose(1, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.2, enable_gqa=True)
    np.testing.assert_allclose(o, ref.transpose(1, 2).reshape(B * L, hq, d).numpy(), atol=1e-12)


def pin_gqa_repeat(orc):
    rng = np.random.default_rng(13)
    g = W.random_geometry(rng, 3, 6, 7, 6, 3, 5, allow_empty=False)
    q = _rand(rng, g.total_q, 6, 5)
    k = _rand(rng, g.total_k, 3, 5)
    v = _rand(rng, g.total_k, 3, 5)
    a = orc.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k)
    b = orc.attention_forward(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1),
                              g.cu_q, g.used_q, g.cu_k, g.used_k)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def pin_key_permutation(orc):
    rng = np.random.default_rng(14)
    q = _rand(rng, 4, 2, 8)
    k = _rand(rng, 9, 1, 8)
    v = _rand(rng, 9, 1, 8)
    a = orc.attention_forward(q, k, v, [0, 4], [4], [0, 9], [7])
    perm = np.concatenate([rng.permutation(7), np.arange(7, 9)])
    b = orc.attention_forward(q, k[perm], v[perm], [0, 4], [4], [0, 9], [7])
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def pin_merge_union(orc):
    """Attention over disjoint key partitions, merged, equals attention over the union;
    a keyless partition makes the merge the identity; all-keyless gives 0 / -inf."""
    rng = np.random.default_rng(15)
    g = W.random_geometry(rng, 5, 8, 12, 4, 2, 8, allow_empty=False)
    q = _rand(rng, g.total_q, 4, 8)
    k = _rand(rng, g.total_k, 2, 8)
    v = _rand(rng, g.total_k, 2, 8)
    # split strictly inside where possible, and one segment entirely on each side
    sigma = np.array([rng.integers(1, u) if u >= 2 else u for u in g.used_k])
    sigma[0], sigma[1] = 0, g.used_k[1]
    assert np.any((sigma > 0) & (sigma < g.used_k))
    parts = W.split_keys(g, sigma)
    res = [orc.attention_forward(q, k, v, p.cu_q, p.used_q, p.cu_k, p.used_k) for p in parts]
    union = orc.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k)
    o, l = orc.lse_merge([r[0] for r in res], [r[1] for r in res], g.cu_q, g.used_q)
    np.testing.assert_allclose(o, union[0], atol=1e-12)
    assert np.array_equal(np.isneginf(l), np.isneginf(union[1]))
    fin = np.isfinite(union[1])
    np.testing.assert_allclose(l[fin], union[1][fin], atol=1e-12)
    # a keyless partition: identity, bit for bit
    empty = g.with_keys(g.cu_k, np.zeros_like(g.used_k))
    e = orc.attention_forward(q, k, v, empty.cu_q, empty.used_q, empty.cu_k, empty.used_k)
    o2, l2 = orc.lse_merge([union[0], e[0]], [union[1], e[1]], g.cu_q, g.used_q)
    used = ~W.gap_rows(g.cu_q, g.used_q)
    assert np.array_equal(o2[used], union[0][used]) and np.array_equal(l2[:, used], union[1][:, used])
    o3, l3 = orc.lse_merge([e[0], e[0]], [e[1], e[1]], g.cu_q, g.used_q)
    assert np.all(o3[used] == 0.0) and np.all(np.isneginf(l3[:, used]))


def pin_rows_match(orc):
    g = W.tiny()
    q, k, v = (t.float().numpy() for t in W.make_qkv(g, 1001))
    o, l = orc.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k)
    rows = [0, 39, 48, 64, 96, 107]
    o2, l2 = orc.attention_rows(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k, rows)
    assert np.array_equal(o2, o[rows]) and np.array_equal(l2, l[:, rows])


def pin_ranges(orc):
    """Key ranges: one prefix range per segment is the plain forward (bit for bit);
    several ranges equal the LSE merge of their separate forwards; an empty range list
    gives 0 / -inf."""
    rng = np.random.default_rng(16)
    g = W.random_geometry(rng, 4, 7, 30, 4, 2, 8, allow_empty=False)
    q = _rand(rng, g.total_q, 4, 8)
    k = _rand(rng, g.total_k, 2, 8)
    v = _rand(rng, g.total_k, 2, 8)
    prefix = [[(int(g.cu_k[b]), int(g.used_k[b]))] for b in range(g.num_segments)]
    a = orc.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k)
    b = orc.attention_forward_ranges(q, k, v, g.cu_q, g.used_q, prefix)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # arbitrary ranges anywhere in K/V (including overlaps across segments and gaps)
    ranges = []
    for b_ in range(g.num_segments):
        rr = []
        for _ in range(int(rng.integers(1, 4))):
            st = int(rng.integers(0, g.total_k))
            rr.append((st, int(rng.integers(0, g.total_k - st + 1))))
        if sum(n for _, n in rr) == 0:
            rr.append((0, 1))
        ranges.append(rr)
    full = orc.attention_forward_ranges(q, k, v, g.cu_q, g.used_q, ranges)
    parts = []
    for i in range(3):
        sub = [[rr[i]] if i < len(rr) else [] for rr in ranges]
        parts.append(orc.attention_forward_ranges(q, k, v, g.cu_q, g.used_q, sub))
    o, l = orc.lse_merge([x[0] for x in parts], [x[1] for x in parts], g.cu_q, g.used_q)
    used = ~W.gap_rows(g.cu_q, g.used_q)
    np.testing.assert_allclose(o[used], full[0][used], atol=1e-12)
    np.testing.assert_allclose(l[:, used], full[1][:, used], atol=1e-12)
    none = orc.attention_forward_ranges(q, k, v, g.cu_q, g.used_q, [[] for _ in range(g.num_segments)])
    assert np.all(none[0][used] == 0.0) and np.all(np.isneginf(none[1][:, used]))
    # the concatenation order of the ranges does not matter
    rev = orc.attention_forward_ranges(q, k, v, g.cu_q, g.used_q, [list(reversed(rr)) for rr in ranges])
    np.testing.assert_allclose(rev[0], full[0], atol=1e-12)


def pin_causal(orc):
    """Block-causal masking within a segment.

    * hand-written limits from the definition (queries are the last positions);
    * token-causal with equal lengths is float64 SDPA with is_causal;
    * every row equals the maskless forward over its own visible key prefix;
    * a block larger than any segment is the maskless forward;
    * a row that sees no key gets 0 / -inf."""
    assert list(orc.causal_limits(5, 8, 1)) == [4, 5, 6, 7, 8]
    assert list(orc.causal_limits(5, 8, 4)) == [4, 8, 8, 8, 8]
    assert list(orc.causal_limits(6, 4, 2)) == [0, 0, 2, 2, 4, 4]
    rng = np.random.default_rng(17)
    # equal lengths, token-causal: SDPA is_causal (row i sees keys 0..i)
    B, L, hq, hkv, d = 2, 9, 4, 2, 8
    q = _rand(rng, B * L, hq, d)
    k = _rand(rng, B * L, hkv, d)
    v = _rand(rng, B * L, hkv, d)
    cu = np.arange(B + 1) * L
    o, _ = orc.attention_forward(q, k, v, cu, [L] * B, cu, [L] * B, scale=0.3, causal_block=1)
    tq = torch.from_numpy(q).view(B, L, hq, d).transpose(1, 2)
    tk = torch.from_numpy(k).view(B, L, hkv, d).transpose(1, 2)
    tv = torch.from_numpy(v).view(B, L, hkv, d).transpose(1, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.3, is_causal=True, enable_gqa=True)
    np.testing.assert_allclose(o, ref.transpose(1, 2).reshape(B * L, hq, d).numpy(), atol=1e-12)
    # unequal lengths and blocks: each row equals the maskless forward over its prefix
    for (uq, uk, blk) in [(7, 10, 3), (6, 4, 2), (5, 5, 1), (4, 9, 100)]:
        q = _rand(rng, uq, hq, d)
        k = _rand(rng, uk + 2, hkv, d)
        v = _rand(rng, uk + 2, hkv, d)
        o, l = orc.attention_forward(q, k, v, [0, uq], [uq], [0, uk + 2], [uk], causal_block=blk)
        lim = orc.causal_limits(uq, uk, blk)
        for i in range(uq):
            oi, li = orc.attention_forward(q[i:i + 1], k, v, [0, 1], [1], [0, uk + 2], [int(lim[i])])
            np.testing.assert_allclose(o[i], oi[0], atol=1e-12)
            assert (np.isneginf(l[:, i]) == np.isneginf(li[:, 0])).all()
            fin = np.isfinite(li[:, 0])
            np.testing.assert_allclose(l[fin, i], li[fin, 0], atol=1e-12)
        if blk >= uq + uk:
            o2, l2 = orc.attention_forward(q, k, v, [0, uq], [uq], [0, uk + 2], [uk])
            np.testing.assert_allclose(o, o2, atol=1e-12)
            np.testing.assert_allclose(l, l2, atol=1e-12)
    # a row with no visible key
    q = _rand(rng, 6, 2, 4)
    k = _rand(rng, 4, 1, 4)
    o, l = orc.attention_forward(q, k, k, [0, 6], [6], [0, 4], [4], causal_block=2)
    assert np.all(o[:2] == 0.0) and np.all(np.isneginf(l[:, :2])) and np.all(np.isfinite(l[:, 2:]))
    # spot rows agree with the full evaluation
    rows = [0, 3, 5]
    o3, l3 = orc.attention_rows(q, k, k, [0, 6], [6], [0, 4], [4], rows, causal_block=2)
    np.testing.assert_array_equal(o3, o[rows])


def pin_backward(orc):
    """Gradients: central finite differences of sum(dO * O) on a tiny gapped geometry
    (GQA, a keyless segment, a segment with keys but no rows, gap rows), float64
    autograd of SDPA on equal lengths, and untouched gap rows."""
    rng = np.random.default_rng(18)
    cu_q, used_q = np.array([0, 4, 7, 9, 9]), np.array([3, 3, 2, 0])
    cu_k, used_k = np.array([0, 5, 9, 12, 14]), np.array([4, 3, 0, 2])
    hq, hkv, d, sc = 4, 2, 3, 0.7
    q = _rand(rng, 9, hq, d)
    k = _rand(rng, 14, hkv, d)
    v = _rand(rng, 14, hkv, d)
    do = _rand(rng, 9, hq, d)
    dq, dk, dv = orc.attention_backward(q, k, v, do, cu_q, used_q, cu_k, used_k, scale=sc,
                                        dq=np.full(q.shape, 3.0), dk=np.full(k.shape, 4.0), dv=np.full(v.shape, 5.0))

    def loss(qq, kk, vv):
        o, _ = orc.attention_forward(qq, kk, vv, cu_q, used_q, cu_k, used_k, scale=sc)
        return float(np.sum(o * do))
    eps = 1e-6
    for name, arr, grad, rows in [("q", q, dq, [0, 2, 4, 7, 8]), ("k", k, dk, [0, 3, 5, 7, 12]),
                                  ("v", v, dv, [1, 3, 6, 13])]:
        for r in rows:
            for h in range(arr.shape[1]):
                for t in range(d):
                    a, b_ = arr.copy(), arr.copy()
                    a[r, h, t] += eps
                    b_[r, h, t] -= eps
                    args_a = {"q": (a, k, v), "k": (q, a, v), "v": (q, k, a)}[name]
                    args_b = {"q": (b_, k, v), "k": (q, b_, v), "v": (q, k, b_)}[name]
                    fd = (loss(*args_a) - loss(*args_b)) / (2 * eps)
                    assert abs(fd - grad[r, h, t]) < 1e-6, (name, r, h, t, fd, grad[r, h, t])
    # untouched: gap q row 3; keys past used (4, 8) and the keyless segment's keys
    assert np.all(dq[3] == 3.0) and np.all(dk[[4, 8, 9, 10, 11]] == 4.0) and np.all(dv[[4, 8, 9, 10, 11]] == 5.0)
    assert np.all(dq[7:9] == 0.0)  # keyless segment: O = 0 does not depend on Q
    # equal lengths: float64 autograd of SDPA
    B, L, S = 2, 5, 6
    q = torch.randn(B, hq, L, d, dtype=torch.float64, requires_grad=True)
    kt = torch.randn(B, hkv, S, d, dtype=torch.float64, requires_grad=True)
    vt = torch.randn(B, hkv, S, d, dtype=torch.float64, requires_grad=True)
    gout = torch.randn(B, hq, L, d, dtype=torch.float64)
    torch.nn.functional.scaled_dot_product_attention(q, kt, vt, scale=sc, enable_gqa=True).backward(gout)
    pack = lambda t: t.detach().transpose(1, 2).reshape(-1, t.shape[1], d).numpy()  # noqa: E731
    dq2, dk2, dv2 = orc.attention_backward(pack(q), pack(kt), pack(vt), pack(gout), np.arange(B + 1) * L, [L] * B,
                                           np.arange(B + 1) * S, [S] * B, scale=sc)
    np.testing.assert_allclose(dq2, pack(q.grad), atol=1e-12)
    np.testing.assert_allclose(dk2, pack(kt.grad), atol=1e-12)
    np.testing.assert_allclose(dv2, pack(vt.grad), atol=1e-12)


def pin_backward_causal(orc):
    """Block-causal gradients: central finite differences of sum(dO * O) through the
    oracle's block-causal forward (rows with no visible key included), and float64
    autograd of SDPA with is_causal on equal lengths (token-causal)."""
    rng = np.random.default_rng(19)
    cu_q, used_q = np.array([0, 6, 9]), np.array([6, 3])
    cu_k, used_k = np.array([0, 4, 10]), np.array([4, 6])  # segment 0: two rows before the first key
    hq, hkv, d, sc = 4, 2, 3, 0.8
    q = _rand(rng, 9, hq, d)
    k = _rand(rng, 10, hkv, d)
    v = _rand(rng, 10, hkv, d)
    do = _rand(rng, 9, hq, d)
    for blk in (1, 2, 3):
        dq, dk, dv = orc.attention_backward(q, k, v, do, cu_q, used_q, cu_k, used_k, scale=sc, causal_block=blk)

        def loss(qq, kk, vv):
            o, _ = orc.attention_forward(qq, kk, vv, cu_q, used_q, cu_k, used_k, scale=sc, causal_block=blk)
            return float(np.sum(o * do))
        eps = 1e-6
        for name, arr, grad, rows in [("q", q, dq, [0, 2, 5, 6, 8]), ("k", k, dk, [0, 3, 4, 9]),
                                      ("v", v, dv, [1, 3, 5, 8])]:
            for r in rows:
                for h in range(arr.shape[1]):
                    for t in range(d):
                        a, b_ = arr.copy(), arr.copy()
                        a[r, h, t] += eps
                        b_[r, h, t] -= eps
                        args_a = {"q": (a, k, v), "k": (q, a, v), "v": (q, k, a)}[name]
                        args_b = {"q": (b_, k, v), "k": (q, b_, v), "v": (q, k, b_)}[name]
                        fd = (loss(*args_a) - loss(*args_b)) / (2 * eps)
                        assert abs(fd - grad[r, h, t]) < 1e-6, (blk, name, r, h, t, fd, grad[r, h, t])
        assert np.all(dq[0:2] == 0.0)  # rows 0, 1 sit before the segment's first key
    B, L = 2, 6
    qt = torch.randn(B, hq, L, d, dtype=torch.float64, requires_grad=True)
    kt = torch.randn(B, hkv, L, d, dtype=torch.float64, requires_grad=True)
    vt = torch.randn(B, hkv, L, d, dtype=torch.float64, requires_grad=True)
    gout = torch.randn(B, hq, L, d, dtype=torch.float64)
    torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=sc, is_causal=True,
                                                     enable_gqa=True).backward(gout)
    pack = lambda t: t.detach().transpose(1, 2).reshape(-1, t.shape[1], d).numpy()  # noqa: E731
    got = orc.attention_backward(pack(qt), pack(kt), pack(vt), pack(gout), np.arange(B + 1) * L, [L] * B,
                                 np.arange(B + 1) * L, [L] * B, scale=sc, causal_block=1)
    for g_, ref in zip(got, (qt.grad, kt.grad, vt.grad)):
        np.testing.assert_allclose(g_, pack(ref), atol=1e-12)


def pin_backward_ranges(orc):
    """Range gradients: one prefix range per segment is attention_backward bit for bit;
    overlapping ranges (shared by two segments and repeated inside one) match central
    finite differences through attention_forward_ranges, so a covered row sums its
    contributions."""
    rng = np.random.default_rng(20)
    g = W.random_geometry(rng, 3, 6, 9, 4, 2, 3, allow_empty=False)
    q = _rand(rng, g.total_q, 4, 3)
    k = _rand(rng, g.total_k, 2, 3)
    v = _rand(rng, g.total_k, 2, 3)
    do = _rand(rng, g.total_q, 4, 3)
    prefix = [[(int(g.cu_k[b]), int(g.used_k[b]))] for b in range(g.num_segments)]
    a = orc.attention_backward(q, k, v, do, g.cu_q, g.used_q, g.cu_k, g.used_k)
    b = orc.attention_backward_ranges(q, k, v, do, g.cu_q, g.used_q, prefix)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    total_k = 12
    k = _rand(rng, total_k, 2, 3)
    v = _rand(rng, total_k, 2, 3)
    ranges = [[(0, 4), (2, 3)], [(3, 5)], [(9, 2)]]  # rows 2, 3 twice in segment 0; 3..4 shared
    sc = 0.9
    dq, dk, dv = orc.attention_backward_ranges(q, k, v, do, g.cu_q, g.used_q, ranges, scale=sc,
                                               dk=np.full(k.shape, 4.0), dv=np.full(v.shape, 5.0))

    def loss(qq, kk, vv):
        o, _ = orc.attention_forward_ranges(qq, kk, vv, g.cu_q, g.used_q, ranges, scale=sc)
        return float(np.sum(o * do))
    eps = 1e-6
    for name, arr, grad, rows in [("q", q, dq, [0, int(g.cu_q[1]), int(g.cu_q[2])]), ("k", k, dk, [0, 2, 3, 4, 9]),
                                  ("v", v, dv, [2, 3, 7, 10])]:
        for r in rows:
            for h in range(arr.shape[1]):
                for t in range(3):
                    a_, b_ = arr.copy(), arr.copy()
                    a_[r, h, t] += eps
                    b_[r, h, t] -= eps
                    args_a = {"q": (a_, k, v), "k": (q, a_, v), "v": (q, k, a_)}[name]
                    args_b = {"q": (b_, k, v), "k": (q, b_, v), "v": (q, k, b_)}[name]
                    fd = (loss(*args_a) - loss(*args_b)) / (2 * eps)
                    assert abs(fd - grad[r, h, t]) < 1e-6, (name, r, h, t, fd, grad[r, h, t])
    assert np.all(dk[[8, 11]] == 4.0) and np.all(dv[[8, 11]] == 5.0)  # rows no range covers


def pin_used_flops(orc):
    """Useful FLOPs are 2·d per score for QK^T plus 2·d per score for PV, summed over
    every (used row, used key, query head): counted here one pair at a time, and checked
    against a closed form (the tiny workload: 40·48 + 17·33 + 12·0 pairs, 4 heads,
    d = 64)."""
    rng = np.random.default_rng(17)
    uq, uk = rng.integers(0, 9, size=5), rng.integers(0, 7, size=5)
    hq, d = 3, 8
    pairs = 0
    for b in range(5):
        for _ in range(int(uq[b])):
            for _ in range(int(uk[b])):
                pairs += 1
    assert orc.used_flops(uq, uk, hq, d) == 2 * d * 2 * hq * pairs
    g = W.tiny()
    assert orc.used_flops(g.used_q, g.used_k, g.num_heads_q, g.head_dim) == 4 * 64 * 4 * (40 * 48 + 17 * 33)


PINS = [pin_bruteforce, pin_default_scale, pin_dilution_golden, pin_zero_keys_closed_form,
        pin_single_key, pin_keyless_and_gap_rows, pin_pad_invariance, pin_sdpa_equal_lengths,
        pin_gqa_repeat, pin_key_permutation, pin_merge_union, pin_rows_match, pin_ranges, pin_causal,
        pin_backward, pin_backward_causal, pin_backward_ranges, pin_used_flops]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(gva_oracle)


def test_budgeted_blocks_agree():
    """A tiny score-block budget (one row per block) gives the same result."""
    g = W.tiny()
    q, k, v = (t.float().numpy() for t in W.make_qkv(g, 1001))
    a = gva_oracle.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k)
    b = gva_oracle.attention_forward(q, k, v, g.cu_q, g.used_q, g.cu_k, g.used_k, budget_bytes=8)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


# ------------------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin.
# ------------------------------------------------------------------------------------

MUTANTS = {
    "dropped_scale": ("x = (qs[r0:r1] @ kt) * scale", "x = (qs[r0:r1] @ kt)"),
    "log2_lse": ("lse[r0:r1] = mx + np.log(l)", "lse[r0:r1] = mx + np.log2(l)"),
    "no_normalisation": ("o[r0:r1] = (e @ vs) / l[:, None]", "o[r0:r1] = (e @ vs)"),
    "pad_key_attended": ("ks = k[k0:k0 + nk, hk, :].astype", "ks = k[k0:k0 + nk + 1, hk, :].astype"),
    "interleaved_gqa": ("qs = q[r0:r0 + nq, hk * g:(hk + 1) * g, :]", "qs = q[r0:r0 + nq, hk::hkv, :]"),
    "gap_row_written": ("o_out[r0:r0 + nq] = 0.0", "o_out[r0:r0 + nq + 1] = 0.0"),
    "keyless_lse_plus_inf": ("l_out[:, r0:r0 + nq] = -np.inf", "l_out[:, r0:r0 + nq] = np.inf"),
    "transposed_lse": ("lb.reshape(nq, g).T", "lb.reshape(g, nq)"),
    "merge_weight_sign": ("np.exp(ls - safe[None])", "np.exp(safe[None] - ls)"),
    "sqrt_d_scale": ("1.0 / math.sqrt(d) if scale is None", "1.0 / d if scale is None"),
    "causal_off_by_one": ("(np.floor_divide(pos, int(causal_block)) + 1)", "np.floor_divide(pos, int(causal_block))"),
    "causal_top_left": ("+ (int(used_k) - int(used_q))", "+ 0"),
    "backward_no_D": ("ds = p * (dp - dd)", "ds = p * dp"),
    "backward_dk_unscaled": ("dk_out[k0:k0 + nk, hk, :] = s * (ds.T @ qs)", "dk_out[k0:k0 + nk, hk, :] = ds.T @ qs"),
    "backward_dv_uses_ds": ("dv_out[k0:k0 + nk, hk, :] = p.T @ dos", "dv_out[k0:k0 + nk, hk, :] = ds.T @ dos"),
    "backward_rowless_keys_untouched": ("        if nk > 0:  # a used key", "        if nk > 0 and nq > 0:  # a used key"),
    "backward_causal_mask_dropped": ("                x = np.where(vis, x, -np.inf)\n                mx = np.where(live",
                                     "                x = x\n                mx = np.where(live"),
    "backward_ranges_overwrite": ("np.add.at(dk_out, (idx, hk), s * (ds.T @ qs))",
                                  "dk_out[idx, hk] = s * (ds.T @ qs)"),
    "range_end_dropped": ("np.arange(int(st), int(st) + int(n))", "np.arange(int(st), int(st) + int(n) - 1)"),
    "flops_one_product": ("return 4.0 * head_dim * num_heads_q", "return 2.0 * head_dim * num_heads_q"),
}


def _mutant(name):
    src = inspect.getsource(gva_oracle)
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name):
    mod = _mutant(name)
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception:  # any assertion or shape error counts as caught
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
