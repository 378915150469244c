"""Parity of the tcgen05 prefill GEMM against the oracle (bf16 expand weights,
fp64 sums) and against the expand + torch.matmul comparator."""
import numpy as np
import pytest
import torch

from trellis_coded_weight_gb300 import binding as tb
from trellis_coded_weight_gb300 import inputs
from util import bf16_bits, check_band, to_dev_bf16, to_dev_f16, to_dev_u32

pytestmark = pytest.mark.gpu
L, T = 16, 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_coded_weight_gb300 import build
    build.build()
    tb.load()
    tb.device_error(reset=True)
    yield
    assert tb.device_error() == 0, "a bounded wait in the prefill kernel gave up"


@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("M,rows,cols", [(1, 64, 512), (5, 128, 256), (12, 77, 512), (16, 200, 5120), (17, 130, 768),
                                         (24, 77, 1024), (25, 130, 512),
                                         (32, 200, 768), (33, 128, 512), (100, 257, 1024),
                                         (300, 136, 512), (64, 64, 2048), (600, 130, 1024)])
def test_prefill_small(oracle_mod, k, M, rows, cols):
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=61 + k, seed_x=62 + M)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    ref, ab = oracle_mod.prefill(codes, scales, x, k, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"prefill k={k} M={M} {rows}x{cols}")


@pytest.mark.parametrize("M", [32, 512, 2048])
def test_prefill_full_size_sampled(oracle_mod, M):
    rows, cols, k = 17408, 5120, 2
    codes, scales, x = inputs.make_linear(rows, cols, k, M)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = bf16_bits(tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g))
    rng = np.random.default_rng(M)
    idx = np.unique(np.concatenate([rng.choice(rows, 24, replace=False), [0, 127, 128, 255, 256, 383, 384, rows - 1]])).astype(np.int64)
    ref, ab = oracle_mod.prefill(codes, scales, x, k, L, T, rows=idx)
    check_band(oracle_mod, out[:, idx], ref, ab, f"prefill full M={M}")


def test_prefill_matches_expand_then_matmul():
    rows, cols, M, k = 1024, 2048, 256, 3
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=9)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    dc, ds, dx = to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x)
    w = tb.expand_bf16(dc, ds, g)
    ref = dx.float() @ w.float().t()
    out = tb.gemm_prefill(dc, ds, dx, g).float()
    scale = dx.float().abs() @ w.float().abs().t()
    assert torch.all((out - ref).abs() <= 1e-5 * scale + 1e-6 + ref.abs() * 2 ** -8)


def test_prefill_L12(oracle_mod):
    codes, scales, x = inputs.make_linear(130, 512, 4, 40, seed_codes=3)
    g = tb.Geometry(4, 12, T, 1, 130, 512)
    out = tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    ref, ab = oracle_mod.prefill(codes, scales, x, 4, 12, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, "prefill L=12")


@pytest.mark.parametrize("k", [2, 3, 4])
def test_prefill_small_M_L12(oracle_mod, k):
    """The register-decode path (axis 1, M <= 24) with 12-bit windows: neighbouring positions pair up."""
    codes, scales, x = inputs.make_linear(70, 768, k, 9, seed_codes=5 + k)
    g = tb.Geometry(k, 12, T, 1, 70, 768)
    out = tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    ref, ab = oracle_mod.prefill(codes, scales, x, k, 12, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"prefill L=12 k={k} M=9")


@pytest.mark.parametrize("M", [8, 16, 24])
def test_prefill_small_M_full_size_sampled(oracle_mod, M):
    rows, cols = 17408, 5120
    codes, scales, x = inputs.make_linear(rows, cols, 2, M)
    g = tb.Geometry(2, L, T, 1, rows, cols)
    out = bf16_bits(tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g))
    idx = np.sort(np.random.default_rng(M).choice(rows, 40, replace=False))
    ref, ab = oracle_mod.prefill(codes, scales, x, 2, L, T, rows=idx)
    check_band(oracle_mod, out[:, idx], ref, ab, f"prefill full M={M}")


@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("M,rows,cols", [(1, 64, 256), (5, 256, 256), (8, 1000, 512), (12, 8, 256), (16, 520, 768),
                                         (17, 1000, 512), (24, 520, 768), (32, 8, 256), (32, 1000, 1024),
                                         (40, 1000, 512), (300, 520, 768), (33, 8, 256)])
def test_prefill_axis0_small(oracle_mod, k, M, rows, cols):
    """Axis 0 (stored W^T): out[m][c] = sum_r e(r,c) x[m][r] over bf16 expand weights."""
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=121 + k, seed_x=122, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    out = tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"prefill axis0 k={k} M={M} {rows}x{cols}")


@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("M", [11, 28])
def test_prefill_axis0_small_M_L12(oracle_mod, k, M):
    """The register-decode path of axis 0 (M <= 32) with 12-bit windows."""
    codes, scales, x = inputs.make_linear(296, 512, k, M, seed_codes=9 + k, seed_x=10, sigma=0.5, x_len=296)
    g = tb.Geometry(k, 12, T, 0, 296, 512)
    out = tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, 12, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"prefill axis0 L=12 k={k} M={M}")


@pytest.mark.parametrize("M", [8, 16, 24, 32])
def test_prefill_axis0_small_M_full_size_sampled(oracle_mod, M):
    """The down projection (17408 stored rows, 5120 outputs) at small M: 20 column blocks, each a cluster whose
    CTAs split the 17408 rows and fold their partials; sampled outputs against the oracle, repeated calls equal."""
    rows, cols, k = 17408, 5120, 3
    codes, scales, x = inputs.make_linear(rows, cols, k, M, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    dc, ds, dx = to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x)
    first = tb.gemm_prefill(dc, ds, dx, g)
    assert torch.equal(tb.gemm_prefill(dc, ds, dx, g).view(torch.int16), first.view(torch.int16))
    idx = np.sort(np.random.default_rng(M + 1).choice(cols, 40, replace=False))
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, L, T, cols=idx)
    check_band(oracle_mod, bf16_bits(first)[:, idx], ref, ab, f"prefill axis0 full M={M}")


def test_prefill_axis0_split_is_deterministic():
    # 4 output tiles leave SMs idle, so each tile's 1000-row reduction is split over a cluster of CTAs
    # whose partial accumulators are summed in a fixed CTA order: repeated calls give identical bits.
    codes, scales, x = inputs.make_linear(1000, 512, 3, 300, seed_codes=7, seed_x=8, sigma=0.5, x_len=1000)
    g = tb.Geometry(3, L, T, 0, 1000, 512)
    dc, ds, dx = to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x)
    first = tb.gemm_prefill(dc, ds, dx, g)
    for _ in range(3):
        assert torch.equal(tb.gemm_prefill(dc, ds, dx, g).view(torch.int16), first.view(torch.int16))


@pytest.mark.parametrize("M", [64, 512, 2048])
def test_prefill_axis0_full_size_sampled(oracle_mod, M):
    # M=2048: 160 tiles on the SMs run as a full unsplit wave plus the leftover tiles with split
    # reductions (features 4096.. of the last token tile); the sampled columns reach into both.
    rows, cols, k = 17408, 5120, 3
    codes, scales, x = inputs.make_linear(rows, cols, k, M, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    out = bf16_bits(tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g))
    idx = np.unique(np.r_[np.arange(0, cols, 331), 127, 128, 255, 256, cols - 1]).astype(np.int64)
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, L, T, cols=idx)
    check_band(oracle_mod, out[:, idx], ref, ab, f"prefill axis0 full M={M}")


def test_prefill_axis0_leftover_tiles_short_reduction(oracle_mod):
    # 42 feature tiles x 4 token tiles (the last one ragged: 1600 = 3*512 + 64) = 168 tiles: a full unsplit
    # wave, then the leftover tiles split over clusters whose size the 3-stage reduction caps.
    rows, cols, M, k = 96, 5376, 1600, 3
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=141, seed_x=142, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    dc, ds, dx = to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x)
    out = tb.gemm_prefill(dc, ds, dx, g)
    assert torch.equal(tb.gemm_prefill(dc, ds, dx, g).view(torch.int16), out.view(torch.int16))
    assert tb.device_error(reset=True) == 0
    idx = np.unique(np.r_[np.arange(0, cols, 97), 127, 128, 5247, 5248, cols - 1]).astype(np.int64)
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, L, T, cols=idx)
    check_band(oracle_mod, bf16_bits(out)[:, idx], ref, ab, f"prefill axis0 leftover M={M} {rows}x{cols}")


def test_prefill_axis0_L12_split(oracle_mod):
    # L = 12 through the axis-0 decoder (4 tiles, each reduction split over 4 CTAs)
    rows, cols, M, k = 256, 512, 40, 3
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=151, seed_x=152, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, 12, T, 0, rows, cols)
    out = tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    assert tb.device_error(reset=True) == 0
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, 12, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, "prefill axis0 L=12")


def test_prefill_axis0_leftover_tiles_one_stage(oracle_mod):
    # a 32-row reduction is a single stage: the leftover tiles run unsplit, as a second persistent launch
    # that starts at a tile offset
    rows, cols, M, k = 32, 5376, 1600, 2
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=161, seed_x=162, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    out = tb.gemm_prefill(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    assert tb.device_error(reset=True) == 0
    idx = np.unique(np.r_[np.arange(0, cols, 89), 127, 128, 5247, 5248, cols - 1]).astype(np.int64)
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, L, T, cols=idx)
    check_band(oracle_mod, bf16_bits(out)[:, idx], ref, ab, f"prefill axis0 one-stage leftover M={M}")


# ------------------------------------------------------------------ bounded waits (failure detection)

@pytest.mark.parametrize("axis,M", [(1, 40), (0, 40)])
def test_bounded_waits_run_out_and_the_next_call_is_correct(oracle_mod, axis, M):
    """Failure detection without a GPU fault: with every pipeline wait limited to 200 ns the waits of an
    ordinary problem run out; the kernel records a non-zero error word, lets its copies and MMAs finish and
    returns with the context intact.  The next call, at the default limit, is correct and clean.  Axis 0 at
    M = 40 runs the cluster-split reduction (8-CTA clusters), whose waits run out too."""
    rows, cols, k = 512, 2048, 2
    codes, scales, _ = inputs.make_linear(rows, cols, k, 1, seed_codes=880 + axis, seed_scales=881)
    n_in = cols if axis == 1 else rows
    x = inputs.normal_bf16(882 + axis, (M, n_in), 1.0 if axis == 1 else 0.5)
    g = tb.Geometry(k, L, T, axis, rows, cols)
    dc, ds, dx = to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x)
    tb.device_error(reset=True)
    try:
        tb.set_wait_limit(200)
        tb.gemm_prefill(dc, ds, dx, g)
        torch.cuda.synchronize()  # a clean return: no CUDA error
    finally:
        tb.set_wait_limit(0)
    assert tb.device_error(reset=True) != 0, "no bounded wait ran out at a 200 ns limit"
    out = tb.gemm_prefill(dc, ds, dx, g)
    torch.cuda.synchronize()
    assert tb.device_error() == 0
    if axis == 1:
        ref, ab = oracle_mod.prefill(codes, scales, x, k, L, T)
    else:
        ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"prefill axis{axis} after a run-out")
    bn, plan = tb.prefill_plan(M, g)
    if axis == 0:
        assert plan[0][2] > 1, "the axis-0 case is meant to run the cluster split"
