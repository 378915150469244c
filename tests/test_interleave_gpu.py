"""The interleaved k=3 axis-0 layout [cols/512][rows][48] ("trellis-linear.ts"
format comment: two coded blocks of a row side by side, the rows of each
512-column group contiguous).  The GPU reads the interleaved array; the oracle
reads the same codes in row-major order."""
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


def interleave(rowmajor: np.ndarray) -> np.ndarray:
    """[rows][cols*3/32] -> [cols/512][rows][48]: group g holds blocks 2g, 2g+1 of every row."""
    rows, words = rowmajor.shape
    return np.ascontiguousarray(rowmajor.reshape(rows, words // 48, 48).transpose(1, 0, 2))


def test_interleave_permutation_by_hand():
    rm = np.arange(3 * 96, dtype=np.uint32).reshape(3, 96)  # 3 rows x 4 blocks of 24 words
    il = interleave(rm)
    assert il.shape == (2, 3, 48)
    assert il[1, 2, 0] == rm[2, 48] and il[1, 2, 24] == rm[2, 72] and il[0, 1, 47] == rm[1, 47]


@pytest.mark.parametrize("L", [16, 12])
@pytest.mark.parametrize("rows,cols", [(37, 512), (300, 1536)])
def test_expand_interleaved_bit_exact(oracle_mod, L, rows, cols):
    codes, scales, _ = inputs.make_linear(rows, cols, 3, 1, seed_codes=91)
    g = tb.Geometry(3, L, T, 0, rows, cols, interleave=2)
    out = tb.expand_bf16(to_dev_u32(interleave(codes)), to_dev_f16(scales), g)
    assert np.array_equal(bf16_bits(out), oracle_mod.expand_bf16(codes, scales, 3, L, T))


@pytest.mark.parametrize("L", [16, 12])
@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("rows,cols", [(45, 512), (777, 1024)])
def test_axis0_interleaved(oracle_mod, L, M, rows, cols):
    codes, scales, x = inputs.make_linear(rows, cols, 3, M, seed_codes=92, seed_x=93, sigma=0.5, x_len=rows)
    g = tb.Geometry(3, L, T, 0, rows, cols, interleave=2)
    dc, ds, dx = to_dev_u32(interleave(codes)), to_dev_f16(scales), to_dev_bf16(x)
    out = tb.matvec_axis0(dc, ds, dx, g, tb.new_workspace(M, g, "cuda"))
    ref, ab = oracle_mod.matvec_axis0(codes, scales, x, 3, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"axis0 interleaved L={L} M={M}")


def test_axis0_interleaved_full_size_sampled(oracle_mod):
    rows, cols, M = 17408, 5120, 4
    codes, scales, x = inputs.make_linear(rows, cols, 3, M, sigma=0.5, x_len=rows)
    g = tb.Geometry(3, 16, T, 0, rows, cols, interleave=2)
    out = bf16_bits(tb.matvec_axis0(to_dev_u32(interleave(codes)), to_dev_f16(scales), to_dev_bf16(x), g,
                                    tb.new_workspace(M, g, "cuda")))
    idx = np.unique(np.r_[np.arange(0, cols, 157), cols - 1]).astype(np.int64)
    ref, ab = oracle_mod.matvec_axis0(codes, scales, x, 3, 16, T, cols=idx)
    check_band(oracle_mod, out[:, idx], ref, ab, "axis0 interleaved full")
