"""gva_forward_noalloc, the entry point for callers that cannot allocate device memory
(a runtime that owns every device byte through its own pool, code under a fixed memory
budget, a loop that must not take cudaMalloc's implicit synchronisation). Its work list
lives in a fixed scratch array inside the library instead of a plan's cudaMalloc'd
buffer. It runs the same kernel over the same rows as gva_forward, so its output must
be bit-identical to gva_forward's, and within the brief's bounds of the FP64 oracle, on
two calls in a row (the second overwriting the first call's scratch contents). This
file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import _lib
from gapped_varlen_attention_gb300 import workloads as W
from oracle import gva_oracle

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL = 1e-2, 1e-3
FILL = 7.0


@pytest.fixture(scope="module")
def lib():
    gva.build()
    return _lib.load_library()


def _via_plan(g, q, k, v):
    plan = gva.Plan.from_geometry(g)
    o, l = W.make_outputs(g, FILL, device="cuda")
    gva.forward(plan, q, k, v, o, l)
    gva.device_status(plan)
    return o, l


def _via_noalloc(g, q, k, v):
    o, l = W.make_outputs(g, FILL, device="cuda")
    gva.forward_noalloc(g.cu_q, g.used_q, g.cu_k, g.used_k, g.num_heads_q, g.num_heads_kv, q, k, v, o, l)
    gva.device_status()  # the no-alloc launch's own error word: synchronises, raises if set
    return o, l


def _oracle(g, q, k, v):
    qn, kn, vn = (t.float().cpu().numpy() for t in (q, k, v))
    return gva_oracle.attention_forward(qn, kn, vn, g.cu_q, g.used_q, g.cu_k, g.used_k,
                                        out=np.full(qn.shape, FILL), lse=np.full((g.num_heads_q, g.total_q), FILL))


def test_noalloc_matches_forward_on_two_calls_in_a_row(lib):
    rng = np.random.default_rng(77)
    geoms = [W.cfg_text_cross(), W.random_geometry(rng, 6, 700, 900, 32, 8, 128)]
    inputs = [W.make_qkv(geoms[0], 1002, device="cuda", k_pad_fill=0.0),
              W.make_qkv(geoms[1], 77, device="cuda", gap_fill=float("nan"))]
    for g, (q, k, v) in zip(geoms, inputs):
        o_ref, l_ref = _via_plan(g, q, k, v)
        o, l = _via_noalloc(g, q, k, v)
        used = torch.from_numpy(~W.gap_rows(g.cu_q, g.used_q)).cuda()
        assert bool((o[~used].float() == FILL).all()) and bool((l[:, ~used] == FILL).all())
        # same kernel, same arithmetic per row: bit-identical to gva_forward
        assert torch.equal(o, o_ref) and torch.equal(l, l_ref)
        # and within the brief's bounds of the FP64 oracle
        oo, lo = _oracle(g, q, k, v)
        un = used.cpu().numpy()
        og, lg = o.float().cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64)
        live = np.isfinite(lo[:, un])
        assert np.array_equal(np.isneginf(lg[:, un]), np.isneginf(lo[:, un]))
        assert np.abs(og[un] - oo[un]).max() <= O_TOL
        assert np.abs(lg[:, un][live] - lo[:, un][live]).max() <= LSE_TOL


def test_noalloc_refuses_launches_beyond_its_scratch(lib):
    # Hq = Hkv = 128: 256 tokens per item, 257 items per head -> 32896 > 32768 items
    cu = np.array([0, 256 * 257], np.int32)
    used = np.array([256 * 257], np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    st = lib.gva_forward_noalloc(p(cu), p(used), p(cu), p(used), 1, 128, 128, 128, None, None, None, None, 0,
                                 None, 0.0, None)
    assert st == _lib.GVA_ERR_INVALID_ARG
    assert "at most 32768" in lib.gva_last_error().decode()
    # a refused call launches nothing: the error word of the last launch stays clear
    assert lib.gva_device_status(None) == _lib.GVA_OK
