"""trellis_matvec_axis0_noalloc: the axis-0 matvec for callers that cannot
allocate device memory (an engine's custom-operator slot that only passes
input and output tensors, or a runtime that forbids cudaMalloc after start-up).

The call keeps its split-row partial sums in a fixed device array inside the
library instead of a caller workspace.  This file is collected last so that a
run stopping at the first failure has run every other test; it also passes
alone in a fresh process.  It calls the entry point through the C ABI and
checks it against trellis_matvec_axis0 and the oracle on two calls in a row,
the second with a different geometry so that the shared array's counters must
have been cleared between them.
"""
import ctypes

import numpy as np
import pytest
import torch

from trellis_coded_weight_gb300 import binding as tb
from trellis_coded_weight_gb300 import inputs
from util import bf16_bits, check_band, to_dev_bf16, to_dev_f16, to_dev_u32

pytestmark = pytest.mark.gpu
L, T = 16, 256
SCRATCH_MAX = 4 << 20  # TRELLIS_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def lib():
    from trellis_coded_weight_gb300 import build
    build.build()
    lib = tb.load()
    fn = lib.trellis_matvec_axis0_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.POINTER(tb.TrellisGeom), ctypes.c_void_p]
    return lib


def _noalloc(lib, dc, ds, dx, g, M):
    out = torch.full((M, g.cols), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = lib.trellis_matvec_axis0_noalloc(dc.data_ptr(), ds.data_ptr(), dx.data_ptr(), out.data_ptr(), M,
                                          ctypes.byref(g.c()), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.trellis_status_string(st)
    return out


@pytest.mark.parametrize("first,second", [((17408, 5120, 2, 4), (300, 768, 3, 2)),
                                          ((77, 512, 4, 3), (17408, 5120, 3, 1))])
def test_noalloc_matches_workspace_call_twice(oracle_mod, lib, first, second):
    for rows, cols, k, M in (first, second):
        codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=70 + k, seed_x=71 + M, sigma=0.5,
                                              x_len=rows)
        g = tb.Geometry(k, L, T, 0, rows, cols)
        assert tb.workspace_bytes(M, g) <= SCRATCH_MAX
        dc, ds, dx = to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x)
        got = bf16_bits(_noalloc(lib, dc, ds, dx, g, M))
        want = bf16_bits(tb.matvec_axis0(dc, ds, dx, g, tb.new_workspace(M, g, "cuda")))
        assert np.array_equal(got, want)
        idx = np.unique(np.concatenate([np.arange(0, cols, max(1, cols // 40)), [cols - 1]])).astype(np.int64)
        ref, ab = oracle_mod.matvec_axis0(codes, scales, x, k, L, T, cols=idx)
        check_band(oracle_mod, got[:, idx], ref, ab, f"noalloc {rows}x{cols} k={k} M={M}")


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    g = tb.Geometry(2, L, T, 0, 131072, 262144)
    assert tb.workspace_bytes(4, g) > SCRATCH_MAX
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    st = lib.trellis_matvec_axis0_noalloc(p, p, p, p, 4, ctypes.byref(g.c()), None)
    assert st == -5  # TRELLIS_EWORKSPACE, returned before any launch
