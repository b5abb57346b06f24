"""The C ABI without a GPU: the library builds, loads, exports every declared symbol,
and rejects bad geometry on the host before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import gapped_varlen_attention_gb300 as gva
from gapped_varlen_attention_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gva.build()
    return _lib.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gva.h")).read()
    return sorted(set(re.findall(r"^\s*(?:GVA_API\s+)?(?:gva_status|const char\s*\*)\s*(gva_\w+)\s*\(", src, re.M)))


def test_header_declares_the_api():
    names = declared_functions()
    assert {"gva_plan", "gva_forward", "gva_lse_merge", "gva_plan_destroy"} <= set(names)
    assert set(names) == set(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_only_the_api_is_exported(lib):
    out = os.popen(f"nm -D --defined-only {_lib.LIB_PATH}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    gva_syms = {s for s in exported if s.startswith("gva_")}
    assert gva_syms == set(declared_functions())


def test_status_strings(lib):
    for code, name in enumerate(["GVA_OK", "GVA_ERR_INVALID_ARG", "GVA_ERR_UNSUPPORTED", "GVA_ERR_CUDA",
                                 "GVA_ERR_DEVICE_CHECK"]):
        assert lib.gva_status_string(code).decode() == name
    assert lib.gva_status_string(99).decode() == "GVA_UNKNOWN_STATUS"


def _plan_status(lib, cu_q, uq, cu_k, uk, hq=4, hkv=2, d=64):
    a = [np.ascontiguousarray(np.asarray(x, np.int32)) for x in (cu_q, uq, cu_k, uk)]
    p = lambda x: x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    h = ctypes.c_void_p()
    st = lib.gva_plan(p(a[0]), p(a[1]), p(a[2]), p(a[3]), len(a[1]), hq, hkv, d, ctypes.byref(h))
    if st == 0:
        lib.gva_plan_destroy(h)
    else:
        assert not h.value
    return st, lib.gva_last_error().decode()


BAD = [
    ("negative cu_q start", ([-1, 48], [10], [0, 48], [10], 4, 2, 64), 1, "cu_seqlens_q[0]"),
    ("decreasing cu_k", ([0, 48, 96], [1, 1], [0, 48, 40], [1, 1], 4, 2, 64), 1, "decreases"),
    ("used_q > capacity", ([0, 48], [49], [0, 48], [1], 4, 2, 64), 1, "seqused_q"),
    ("negative used_k", ([0, 48], [4], [0, 48], [-1], 4, 2, 64), 1, "seqused_k"),
    ("Hq not a multiple of Hkv", ([0, 8], [8], [0, 8], [8], 6, 4, 64), 1, "divisible"),
    ("zero heads", ([0, 8], [8], [0, 8], [8], 0, 1, 64), 1, "positive"),
    ("head_dim 96", ([0, 8], [8], [0, 8], [8], 4, 2, 96), 2, "head_dim"),
    ("group 256 exceeds a tile", ([0, 8], [8], [0, 8], [8], 256, 1, 64), 2, "at most 128"),
    ("more than 256 query heads", ([0, 8], [8], [0, 8], [8], 512, 256, 64), 2, "too large"),
]


@pytest.mark.parametrize("name,args,status,msg", BAD, ids=[b[0] for b in BAD])
def test_plan_rejects_bad_geometry_on_the_host(lib, name, args, status, msg):
    st, err = _plan_status(lib, *args)
    assert st == status, (st, err)
    assert msg in err


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.gva_plan(None, None, None, None, 1, 4, 2, 64, ctypes.byref(h)) == 1
    assert lib.gva_plan(None, None, None, None, 1, 4, 2, 64, None) == 1
    assert lib.gva_forward(None, None, None, None, None, 0, None, 0.0, None) == 1
    assert lib.gva_lse_merge(None, 1, None, 0, None, None, 0, None, None) == 1
    assert lib.gva_plan_destroy(None) == 0
    if not torch.cuda.is_available():
        # a NULL plan reads gva_forward_noalloc's error word on the current device
        assert lib.gva_device_status(None) == 2 and "CUDA device" in lib.gva_last_error().decode()
    n = ctypes.c_size_t(7)
    assert lib.gva_backward_workspace_size(None, ctypes.byref(n)) == 1 and n.value == 7
    assert lib.gva_backward(None, None, None, None, None, None, None, None, 0, None, None, 0, None, 0, 0.0,
                            None) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_plan_without_a_gpu_is_refused_cleanly(lib):
    st, err = _plan_status(lib, [0, 48], [40], [0, 48], [48])
    assert st == 2 and "CUDA device" in err


def test_python_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load_library(str(tmp_path / "libgva.so"))


def _ranges_status(lib, cu_q, uq, off, starts, lens, total_k, hq=4, hkv=2, d=64):
    a = [np.ascontiguousarray(np.asarray(x, np.int32)) for x in (cu_q, uq, off, starts, lens)]
    p = lambda x: x.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))  # noqa: E731
    h = ctypes.c_void_p()
    st = lib.gva_plan_ranges(p(a[0]), p(a[1]), len(a[1]), p(a[2]), p(a[3]), p(a[4]), total_k, hq, hkv, d,
                             ctypes.byref(h))
    if st == 0:
        lib.gva_plan_destroy(h)
    return st, lib.gva_last_error().decode()


BAD_RANGES = [
    ("range past total_k", ([0, 8], [8], [0, 1], [90], [20], 100), "outside"),
    ("negative start", ([0, 8], [8], [0, 1], [-1], [2], 100), "outside"),
    ("negative length", ([0, 8], [8], [0, 1], [3], [-2], 100), "outside"),
    ("offsets not from 0", ([0, 8], [8], [1, 1], [3], [2], 100), "key_range_offsets[0]"),
    ("decreasing offsets", ([0, 4, 8], [4, 4], [0, 2, 1], [3, 5], [2, 2], 100), "decreases"),
    ("negative total_k", ([0, 8], [8], [0, 0], [0], [0], -1), "total_k"),
]


@pytest.mark.parametrize("name,args,msg", BAD_RANGES, ids=[b[0] for b in BAD_RANGES])
def test_plan_ranges_rejects_bad_ranges_on_the_host(lib, name, args, msg):
    st, err = _ranges_status(lib, *args)
    assert st == 1, (st, err)
    assert msg in err
