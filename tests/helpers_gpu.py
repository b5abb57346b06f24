"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI, run the
oracle on the same seeded inputs, and compare with the stated tolerances."""
import numpy as np
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import workloads as W
from oracle import gva_oracle

# Acceptance: max |O - O_ref| <= 1e-2 and max |LSE - LSE_ref| <= 1e-3 for bf16 inputs;
# exact on untouched rows and on the keyless 0 / -inf cases.
O_TOL = 1e-2
LSE_TOL = 1e-3


def gpu_forward(geom, q, k, v, fill=W.TINY_SENTINEL, out_dtype=torch.bfloat16, scale=0.0, plan=None):
    """Run gva_forward on device copies of q / k / v; outputs prefilled with ``fill``."""
    plan = plan or gva.Plan.from_geometry(geom)
    o, l = W.make_outputs(geom, fill, device="cuda", out_dtype=out_dtype)
    gva.forward(plan, q.cuda(), k.cuda(), v.cuda(), o, l, scale)
    gva.device_status(plan)
    return o, l


def oracle_forward(geom, q, k, v, fill=W.TINY_SENTINEL, scale=None):
    qn, kn, vn = (t.detach().cpu().float().numpy() for t in (q, k, v))
    o0 = np.full(qn.shape, fill)
    l0 = np.full((geom.num_heads_q, geom.total_q), fill)
    return gva_oracle.attention_forward(qn, kn, vn, geom.cu_q, geom.used_q, geom.cu_k, geom.used_k,
                                        scale=scale, out=o0, lse=l0)


def check_full(geom, o, l, o_ref, l_ref, fill, o_tol=O_TOL, lse_tol=LSE_TOL):
    """Element-wise parity on used rows; bit-exact sentinels on gap rows; exact 0 / -inf
    on keyless rows."""
    o = o.float().cpu().numpy().astype(np.float64)
    l = l.cpu().numpy().astype(np.float64)
    gap = W.gap_rows(geom.cu_q, geom.used_q)
    fill32 = np.float64(np.float32(fill))
    assert np.all(o[gap] == fill32), "a gap row of O was written"
    assert np.all(l[:, gap] == fill32), "a gap row of LSE was written"
    used = ~gap
    keyless = np.zeros_like(gap)
    for b in range(geom.num_segments):
        if geom.used_k[b] == 0:
            keyless[geom.cu_q[b]:geom.cu_q[b] + geom.used_q[b]] = True
    if keyless.any():
        assert np.all(o[keyless] == 0.0) and not np.any(np.signbit(o[keyless]))
        assert np.all(np.isneginf(l[:, keyless]))
    keyed = used & ~keyless
    if keyed.any():
        assert np.all(np.isfinite(o[keyed])) and np.all(np.isfinite(l[:, keyed]))
        eo = np.abs(o[keyed] - o_ref[keyed]).max()
        el = np.abs(l[:, keyed] - l_ref[:, keyed]).max()
        assert eo <= o_tol, f"max |O err| = {eo:.3e}"
        assert el <= lse_tol, f"max |LSE err| = {el:.3e}"
        return float(eo), float(el)
    return 0.0, 0.0


def sample_rows(geom, rng, per_segment=6, tokens_per_tile=None):
    """Used rows to spot-check: first, last, tile edges and random rows of each segment."""
    rows = []
    T = tokens_per_tile or 128 // (geom.num_heads_q // geom.num_heads_kv)
    for b in range(geom.num_segments):
        uq = int(geom.used_q[b])
        if uq == 0:
            continue
        cand = {0, uq - 1, min(T, uq - 1), min(2 * T - 1, uq - 1), min(2 * T, uq - 1), uq // 2}
        cand |= set(int(x) for x in rng.integers(0, uq, size=per_segment))
        rows += [int(geom.cu_q[b]) + c for c in sorted(cand)]
    return rows


def check_rows(o, l, rows, o_ref, l_ref, o_tol=O_TOL, lse_tol=LSE_TOL):
    idx = torch.as_tensor(rows, device=o.device)
    og = o.index_select(0, idx).float().cpu().numpy().astype(np.float64)
    lg = l.index_select(1, idx).cpu().numpy().astype(np.float64)
    dead = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(lg), dead), "-inf LSE pattern differs"
    if dead.any():
        assert np.all(og[dead.T] == 0.0)
    live = ~dead
    eo = np.abs(og[live.T] - o_ref[live.T]).max() if live.any() else 0.0
    el = np.abs(lg[live] - l_ref[live]).max() if live.any() else 0.0
    assert eo <= o_tol, f"max |O err| = {eo:.3e}"
    assert el <= lse_tol, f"max |LSE err| = {el:.3e}"
    return float(eo), float(el)


def gap_untouched(geom, o, l, fill):
    gap = torch.from_numpy(W.gap_rows(geom.cu_q, geom.used_q)).to(o.device)
    if not bool(gap.any()):
        return True
    f = torch.tensor(fill, dtype=torch.float32)
    return bool((o[gap].float() == f.to(o.device)).all()) and bool((l[:, gap] == f.to(l.device)).all())
