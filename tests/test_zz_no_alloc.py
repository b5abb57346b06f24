"""gva_forward_noalloc, the entry point for callers that cannot allocate device memory
(its work list lives in a fixed scratch array inside the library instead of a plan's
cudaMalloc'd buffer). Its output must match gva_forward's on two calls in a row, the
second overwriting the first call's scratch contents. This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import _lib
from gapped_varlen_attention_gb300 import workloads as W

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
    torch.cuda.synchronize()
    return o, l


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
        assert float((o[used].float() - o_ref[used].float()).abs().max()) <= O_TOL
        both = torch.isfinite(l_ref[:, used])
        assert torch.equal(torch.isneginf(l[:, used]), torch.isneginf(l_ref[:, used]))
        assert float((l[:, used][both] - l_ref[:, used][both]).abs().max()) <= LSE_TOL


def test_noalloc_refuses_launches_beyond_its_scratch(lib):
    # Hq = Hkv = 128: 256 tokens per item, 257 items per head -> 32896 > 32768 items
    cu = np.array([0, 256 * 257], np.int32)
    used = np.array([256 * 257], np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    st = lib.gva_forward_noalloc(p(cu), p(used), p(cu), p(used), 1, 128, 128, 128, None, None, None, None, 0,
                                 None, 0.0, None)
    assert st == _lib.GVA_ERR_INVALID_ARG
    assert "at most 32768" in lib.gva_last_error().decode()
