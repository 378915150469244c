"""The C ABI without a GPU: the library builds, loads and exports every symbol
that include/trellis.h declares, and argument errors return their status
codes before any CUDA call (nothing is launched)."""
import ctypes
import os
import re

import pytest

from trellis_coded_weight_gb300 import binding
from trellis_coded_weight_gb300 import build as tbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "include", "trellis.h")


@pytest.fixture(scope="module")
def lib():
    tbuild.build()
    return binding.load()


def declared_functions():
    txt = open(HDR).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(trellis_[a-z0-9_]+)\s*\(", txt)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("trellis_matvec_axis1", "trellis_matvec_axis0", "trellis_gateup_swiglu",
                     "trellis_expand_bf16", "trellis_gemm_prefill"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(binding.EXPORTS) <= set(declared_functions())


def test_version_and_status_strings(lib):
    assert lib.trellis_abi_version() >= 100
    for s in range(-8, 1):
        assert lib.trellis_status_string(s)
    assert lib.trellis_status_string(-99) == b"unknown status"


def G(**kw):
    base = dict(k=2, L=16, T=256, axis=1, rows=64, cols=512)
    base.update(kw)
    return binding.TrellisGeom(**base)


@pytest.mark.parametrize("kw,ok", [({}, True), ({"k": 3}, True), ({"k": 4, "L": 12}, True), ({"k": 1}, False),
                                   ({"k": 5}, False), ({"L": 20}, False), ({"T": 128}, False),
                                   ({"cols": 500}, False), ({"rows": 0}, False), ({"axis": 2}, False),
                                   ({"rows": 1 << 32}, False)])
def test_check_geom(lib, kw, ok):
    assert (lib.trellis_check_geom(ctypes.byref(G(**kw))) == 0) == ok


A = 1 << 20  # a 16-byte aligned fake address: never dereferenced, calls fail before any launch


def test_errors_before_launch(lib):
    g = G()
    assert lib.trellis_matvec_axis1(A, A, A, A, 1, None, None) == -7
    assert lib.trellis_matvec_axis1(A, A, A, A, 1, ctypes.byref(G(cols=300)), None) == -1
    assert lib.trellis_matvec_axis1(A, A, A, A, 1, ctypes.byref(G(axis=0)), None) == -4
    assert lib.trellis_matvec_axis1(A, A, A, A, 0, ctypes.byref(g), None) == -2
    assert lib.trellis_matvec_axis1(A, A, A, A, 5, ctypes.byref(g), None) == -2
    assert lib.trellis_matvec_axis1(None, A, A, A, 1, ctypes.byref(g), None) == -7
    assert lib.trellis_matvec_axis1(A + 4, A, A, A, 1, ctypes.byref(g), None) == -3
    assert lib.trellis_gateup_swiglu(A, A, A, A, A, A, 5, ctypes.byref(g), None) == -2
    assert lib.trellis_gateup_swiglu(A, A, A, A + 2, A, A, 1, ctypes.byref(g), None) == -3
    assert lib.trellis_gateup_swiglu(A, A, A, A, A, A, 1, ctypes.byref(G(axis=0)), None) == -4
    assert lib.trellis_expand_bf16(A, A, A + 8, ctypes.byref(g), None) == -3
    assert lib.trellis_expand_bf16(A, A, A, ctypes.byref(G(k=7)), None) == -1
    assert lib.trellis_gemm_prefill(A, A, A, A, 0, ctypes.byref(g), None) == -2
    assert lib.trellis_gemm_prefill(A, A, A, A, 64, ctypes.byref(G(axis=0, rows=60)), None) == -1  # rows % 8
    assert lib.trellis_gemm_prefill(A, A, A, A, 64, ctypes.byref(G(k=3, axis=0, cols=1024, interleave=2)), None) == -1
    g0 = G(axis=0)
    need = lib.trellis_workspace_bytes(4, ctypes.byref(g0))
    assert need > 0 and lib.trellis_workspace_bytes(5, ctypes.byref(g0)) == 0
    assert lib.trellis_matvec_axis0(A, A, A, A, 4, ctypes.byref(g0), None, need, None) == -5
    assert lib.trellis_matvec_axis0(A, A, A, A, 4, ctypes.byref(g0), A, need - 1, None) == -5
    assert lib.trellis_matvec_axis0(A, A, A, A, 4, ctypes.byref(g0), A + 4, need, None) == -5
    assert lib.trellis_matvec_axis0(A, A, A, A, 4, ctypes.byref(g), A, need, None) == -4


def test_host_buffer_matvec_errors_before_any_copy(lib):
    g = G()
    H = 12345  # host pointers carry no alignment rule
    f = lib.trellis_matvec_axis1_host
    assert f(A, A, H, H, 1, None, A, A, None) == -7
    assert f(A, A, H, H, 1, ctypes.byref(G(axis=0)), A, A, None) == -4
    assert f(A, A, H, H, 5, ctypes.byref(g), A, A, None) == -2
    assert f(A, A, None, H, 1, ctypes.byref(g), A, A, None) == -7
    assert f(A, A, H, None, 1, ctypes.byref(g), A, A, None) == -7
    assert f(A, A, H, H, 1, ctypes.byref(g), None, A, None) == -7
    assert f(A, A, H, H, 1, ctypes.byref(g), A + 2, A, None) == -3
    assert f(A, A, H, H, 1, ctypes.byref(g), A, A + 8, None) == -3


def test_no_usable_device_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.trellis_matvec_axis1(A, A, A, A, 1, ctypes.byref(G()), None) == -8
    assert lib.trellis_matvec_axis1_host(A, A, 7, 7, 1, ctypes.byref(G()), A, A, None) == -8


def test_workspace_grows_with_M(lib):
    g0 = G(axis=0, rows=17408, cols=5120)
    sizes = [lib.trellis_workspace_bytes(m, ctypes.byref(g0)) for m in (1, 2, 3, 4)]
    assert sizes == sorted(sizes) and sizes[0] > 0


def test_mlp_decode_errors_before_launch(lib):
    gu, gd = G(axis=1), G(axis=0)
    need = lib.trellis_workspace_bytes(2, ctypes.byref(gd))
    args = [A] * 9
    assert lib.trellis_mlp_decode(*args, 2, ctypes.byref(gu), ctypes.byref(G(axis=0, rows=32)), A, need, None) == -1
    assert lib.trellis_mlp_decode(*args, 2, ctypes.byref(gd), ctypes.byref(gd), A, need, None) == -4
    assert lib.trellis_mlp_decode(*args, 5, ctypes.byref(gu), ctypes.byref(gd), A, need, None) == -2
    assert lib.trellis_mlp_decode(*args, 2, ctypes.byref(gu), ctypes.byref(gd), A, need - 16, None) == -5


@pytest.mark.parametrize("kw,ok", [({"k": 3, "axis": 0, "cols": 1024, "interleave": 2}, True),
                                   ({"k": 3, "axis": 0, "cols": 1024, "interleave": 2, "L": 12}, True),
                                   ({"k": 2, "axis": 0, "cols": 1024, "interleave": 2}, False),
                                   ({"k": 3, "axis": 1, "cols": 1024, "interleave": 2}, False),
                                   ({"k": 3, "axis": 0, "cols": 768, "interleave": 2}, False),
                                   ({"k": 3, "axis": 0, "cols": 1024, "interleave": 1}, False),
                                   ({"reserved": 1}, False)])
def test_interleaved_geometry_rules(lib, kw, ok):
    assert (lib.trellis_check_geom(ctypes.byref(G(**kw))) == 0) == ok


@pytest.mark.parametrize("fn", ["trellis_load_floor", "trellis_load_floor_rows"])
def test_load_floor_errors_before_launch(lib, fn):
    gu = G(axis=1)
    f = getattr(lib, fn)
    assert f(A, A, ctypes.byref(G(axis=0)), None) == -4  # EAXIS
    assert f(None, A, ctypes.byref(gu), None) == -7      # ENULL
    assert f(A + 4, A, ctypes.byref(gu), None) == -3     # EALIGN
    assert f(A, A, ctypes.byref(G(axis=1, cols=100)), None) == -1  # EGEOM


def test_wait_limit_setter_needs_no_device(lib):
    # a host-side setting read by later prefill launches; 0 restores the default
    lib.trellis_set_wait_limit.argtypes = [ctypes.c_uint64]
    assert lib.trellis_set_wait_limit(1000) == 0
    assert lib.trellis_set_wait_limit(0) == 0
