"""Parity past 32-bit offsets: a code stream of more than 2^31 words (8.6 GB) through the matvecs, the fused
gate/up layer and the prefill on both axes, and an expand whose output has more than 2^32 elements (8.6 GB).

The matrices are periodic in the stored row: row r holds the code words of row r mod 4099 of a seeded base
matrix (4099 is prime, so no power-of-two distance maps a row onto a row with the same words), and every row
has its own seeded scale.  Results are checked on sampled rows or columns, including those whose offsets cross
2^31 and 2^32 words or bytes; the oracle gets exactly the words of the sampled rows (axis 1) or the sampled
columns' blocks of every row (axis 0), taken from the base matrix on the host.
"""
import numpy as np
import pytest
import torch

from test_parity_gpu import check_gateup
from trellis_coded_weight_gb300 import binding as tb
from trellis_coded_weight_gb300 import inputs
from util import bf16_bits, check_band, to_dev_bf16, to_dev_f16

pytestmark = pytest.mark.gpu
L, T = 16, 256
B = 4099  # rows of the base matrix


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_coded_weight_gb300 import build
    build.build()
    tb.load()
    tb.device_error(reset=True)
    yield
    assert tb.device_error() == 0, "a bounded wait in a tensor-core kernel gave up"


def _periodic(rows, cols, k, seed):
    """(base words [B, cols*k/32] on the host, the periodic [rows, cols*k/32] int32 matrix on the device)."""
    base = inputs.random_words(seed, (B, cols * k // 32))
    dev = torch.from_numpy(base.view(np.int32)).cuda()
    big = dev.repeat((rows + B - 1) // B, 1)[:rows]
    assert big.is_contiguous()
    return base, big


class Big:
    """k = 4, 8192 coded columns (1024 words a row), 2^21 + 40 stored rows: 2^31 + 40960 words."""
    k, cols = 4, 8192
    rows = (1 << 21) + 40


@pytest.fixture(scope="module")
def big():
    base, codes = _periodic(Big.rows, Big.cols, Big.k, 7001)
    scales = inputs.uniform_f16(7002, (Big.rows,))
    up_scales = inputs.uniform_f16(7003, (Big.rows,))
    yield base, codes, scales, to_dev_f16(scales), up_scales, to_dev_f16(up_scales)
    del codes
    torch.cuda.empty_cache()


def _rows_to_check(rows, wpr, seed):
    """Random rows plus those around word offsets 2^31 and byte offsets 2^32, and the last rows."""
    rng = np.random.default_rng(seed)
    w31, b32 = (1 << 31) // wpr, (1 << 32) // (4 * wpr)
    edges = [0, 1, B - 1, B, b32 - 1, b32, b32 + 1, w31 - 1, w31, w31 + 1, rows - 65, rows - 2, rows - 1]
    idx = np.concatenate([rng.choice(rows, 20, replace=False), [r for r in edges if 0 <= r < rows]])
    return np.unique(idx).astype(np.int64)


@pytest.mark.parametrize("M", [1, 4])
def test_axis1_matvec_past_2e31_words(oracle_mod, big, M):
    base, codes, scales, d_scales, _, _ = big
    g = tb.Geometry(Big.k, L, T, 1, Big.rows, Big.cols)
    x = inputs.normal_bf16(7100 + M, (M, Big.cols))
    out = bf16_bits(tb.matvec_axis1(codes, d_scales, to_dev_bf16(x), g))
    idx = _rows_to_check(Big.rows, g.words_per_row, M)
    ref, ab = oracle_mod.matvec_axis1(base[idx % B], scales[idx], x, Big.k, L, T)
    check_band(oracle_mod, out[:, idx], ref, ab, f"axis1 past 2^31 words M={M}")


@pytest.mark.parametrize("M", [1, 3])
def test_gateup_past_2e31_words(oracle_mod, big, M):
    """The same words as gate and up matrices, with different scales."""
    base, codes, scales, d_scales, up_scales, d_up = big
    g = tb.Geometry(Big.k, L, T, 1, Big.rows, Big.cols)
    x = inputs.normal_bf16(7200 + M, (M, Big.cols))
    out = bf16_bits(tb.gateup_swiglu(codes, d_scales, codes, d_up, to_dev_bf16(x), g))
    idx = _rows_to_check(Big.rows, g.words_per_row, 10 + M)
    sub = base[idx % B]
    sums = oracle_mod.gateup_sums(sub, scales[idx], sub, up_scales[idx], x, Big.k, L, T)
    check_gateup(oracle_mod, out[:, idx], *sums, f"gateup past 2^31 words M={M}")


@pytest.mark.parametrize("M", [8, 40])
def test_axis1_prefill_past_2e31_words(oracle_mod, big, M):
    """M = 8 on the register-decode kernel, M = 40 on the tcgen05 kernel."""
    base, codes, scales, d_scales, _, _ = big
    g = tb.Geometry(Big.k, L, T, 1, Big.rows, Big.cols)
    x = inputs.normal_bf16(7300 + M, (M, Big.cols), 0.5)
    out = bf16_bits(tb.gemm_prefill(codes, d_scales, to_dev_bf16(x), g))
    idx = _rows_to_check(Big.rows, g.words_per_row, 20 + M)
    ref, ab = oracle_mod.prefill(base[idx % B], scales[idx], x, Big.k, L, T)
    check_band(oracle_mod, out[:, idx], ref, ab, f"prefill axis1 past 2^31 words M={M}")


def _axis0_columns(cols, seed):
    """Sampled output columns in the first and the last column block, as (global, block-local in the
    two-block host matrix) indices."""
    rng = np.random.default_rng(seed)
    last = cols // T - 1
    loc = np.unique(np.concatenate([[0, T - 1, T, 2 * T - 1], rng.choice(2 * T, 12, replace=False)])).astype(np.int64)
    glob = np.where(loc < T, loc, last * T + (loc - T))
    return glob, loc


def _axis0_host_blocks(base, rows, k):
    """Every stored row's words of the first and the last column block, [rows, 2 * T*k/32] on the host."""
    wpb = T * k // 32
    two = np.concatenate([base[:, :wpb], base[:, -wpb:]], axis=1)
    return np.ascontiguousarray(np.tile(two, ((rows + B - 1) // B, 1))[:rows])


@pytest.mark.parametrize("M", [1, 4])
def test_axis0_matvec_past_2e31_words(oracle_mod, big, M):
    """The stored matrix read as W^T (2^21 + 40 inputs, 8192 outputs): every stored row enters each output."""
    base, codes, scales, d_scales, _, _ = big
    g = tb.Geometry(Big.k, L, T, 0, Big.rows, Big.cols)
    x = inputs.normal_bf16(7400 + M, (M, Big.rows), 0.5)
    ws = tb.new_workspace(M, g, codes.device)
    out = bf16_bits(tb.matvec_axis0(codes, d_scales, to_dev_bf16(x), g, ws))
    glob, loc = _axis0_columns(Big.cols, 30 + M)
    ref, ab = oracle_mod.matvec_axis0(_axis0_host_blocks(base, Big.rows, Big.k), scales, x, Big.k, L, T, cols=loc)
    check_band(oracle_mod, out[:, glob], ref, ab, f"axis0 past 2^31 words M={M}")


@pytest.mark.parametrize("M", [8, 32, 40])
def test_axis0_prefill_past_2e31_words(oracle_mod, big, M):
    """M = 8 and 32 on the register-decode kernel (cluster fold), M = 40 on the tcgen05 kernel."""
    base, codes, scales, d_scales, _, _ = big
    g = tb.Geometry(Big.k, L, T, 0, Big.rows, Big.cols)
    x = inputs.normal_bf16(7500 + M, (M, Big.rows), 0.5)
    out = bf16_bits(tb.gemm_prefill(codes, d_scales, to_dev_bf16(x), g))
    glob, loc = _axis0_columns(Big.cols, 40 + M)
    ref, ab = oracle_mod.matvec_axis0_bf16w(_axis0_host_blocks(base, Big.rows, Big.k), scales, x, Big.k, L, T,
                                            cols=loc)
    check_band(oracle_mod, out[:, glob], ref, ab, f"prefill axis0 past 2^31 words M={M}")


def test_expand_past_2e32_elements(oracle_mod):
    """k = 2, 4096 columns, 2^20 + 5 rows: 2^32 + 20480 decoded weights (8.6 GB of bf16), bit-exact."""
    rows, cols, k = (1 << 20) + 5, 4096, 2
    base, codes = _periodic(rows, cols, k, 7601)
    scales = inputs.uniform_f16(7602, (rows,))
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = tb.expand_bf16(codes, to_dev_f16(scales), g)
    rng = np.random.default_rng(5)
    e32 = (1 << 32) // cols  # the first row whose elements lie past 2^32
    idx = np.unique(np.concatenate([rng.choice(rows, 16, replace=False),
                                    [0, B, e32 // 2 - 1, e32 // 2, e32 - 1, e32, rows - 1]])).astype(np.int64)
    got = out[torch.from_numpy(idx).cuda()].cpu().view(torch.int16).numpy().view(np.uint16)
    want = oracle_mod.expand_bf16(base[idx % B], scales[idx], k, L, T)
    assert np.array_equal(got, want)
    del out, codes
    torch.cuda.empty_cache()
