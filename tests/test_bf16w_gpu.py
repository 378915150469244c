"""The bf16-rounded weight numerics (the pages' decoder variants 0-3): weights
are the bf16 expand weights; sums in fp32.  Against the oracle's sums over
the same bf16 weights in double."""
import numpy as np
import pytest

from trellis_coded_weight_gb300 import binding as tb
from trellis_coded_weight_gb300 import inputs
from util import bf16_bits, check_band, to_dev_bf16, to_dev_f16, to_dev_u32

pytestmark = pytest.mark.gpu
T = 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_coded_weight_gb300 import build
    build.build()
    tb.load()


@pytest.mark.parametrize("k,L", [(2, 16), (3, 16), (4, 12)])
@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("rows,cols", [(45, 768), (130, 1280)])
def test_axis1_bf16w(oracle_mod, k, L, M, rows, cols):
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=101 + k, seed_x=102)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = tb.matvec_axis1(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g, bf16_weights=True)
    ref, ab = oracle_mod.matvec_axis1_bf16w(codes, scales, x, k, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"axis1 bf16w k={k} M={M}")


@pytest.mark.parametrize("k,L", [(2, 16), (3, 16), (4, 12)])
@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("rows,cols", [(77, 512), (1000, 768)])
def test_axis0_bf16w(oracle_mod, k, L, M, rows, cols):
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=111 + k, seed_x=112, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    out = tb.matvec_axis0(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g, tb.new_workspace(M, g, "cuda"),
                          bf16_weights=True)
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"axis0 bf16w k={k} M={M}")


def test_bf16w_full_size_sampled(oracle_mod):
    rows, cols, M, k = 17408, 5120, 2, 2
    codes, scales, x = inputs.make_linear(rows, cols, k, M)
    g = tb.Geometry(k, 16, T, 1, rows, cols)
    out = bf16_bits(tb.matvec_axis1(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g, bf16_weights=True))
    idx = np.unique(np.r_[np.arange(0, rows, 613), rows - 1]).astype(np.int64)
    ref, ab = oracle_mod.matvec_axis1_bf16w(codes, scales, x, k, 16, T, rows=idx)
    check_band(oracle_mod, out[:, idx], ref, ab, "axis1 bf16w full")
    x0 = inputs.normal_bf16(5, (M, rows), 0.5)
    g0 = tb.Geometry(k, 16, T, 0, rows, cols)
    out0 = bf16_bits(tb.matvec_axis0(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x0), g0,
                                     tb.new_workspace(M, g0, "cuda"), bf16_weights=True))
    cidx = np.unique(np.r_[np.arange(0, cols, 307), cols - 1]).astype(np.int64)
    ref0, ab0 = oracle_mod.matvec_axis0_bf16w(codes, scales, x0, k, 16, T, cols=cidx)
    check_band(oracle_mod, out0[:, cidx], ref0, ab0, "axis0 bf16w full")
