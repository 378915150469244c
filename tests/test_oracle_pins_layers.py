"""Pins of the oracle's number formats and layers (run without a GPU).

Library routines (numpy/torch dtype conversions and matmuls in float64) and
special cases (one-hot inputs, zero inputs, zero scales) pin the oracle's
expand, matvec, gate/up and prefill against the pages' definitions in the
"trellis-linear.ts" and "trellis-tiled-prefill.ts" diff pages.
"""
import numpy as np
import pytest
import torch

from trellis_coded_weight_gb300 import inputs

D32 = np.float32(147.800537109375)


def _bf16_torch(a_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------- number formats

def test_bf16_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(11)
    v = (rng.standard_normal(4000) * np.exp(rng.uniform(-20, 20, 4000))).astype(np.float32)
    # exact ties: low half exactly 0x8000 with odd and even kept halves
    ties = (np.arange(1000, dtype=np.uint32) * 0x00010000 + 0x3F808000).view(np.float32)
    v = np.concatenate([v, ties, np.float32([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40])])
    want = _bf16_torch(v)
    got = np.array([oracle_mod.bf16_rne(float(t)) for t in v], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_f16_widening_matches_numpy(oracle_mod):
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle_mod.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))


def test_bf16_rne_f64_single_rounding(oracle_mod):
    """double -> bf16 rounds once: compare with the exact nearest of the two
    bracketing bf16 values."""
    rng = np.random.default_rng(5)
    v = rng.standard_normal(3000) * 10.0 ** rng.uniform(-6, 6, 3000)
    for d in v:
        b = oracle_mod.bf16_rne_f64(float(d))
        val = float(inputs.bf16_bits_to_f32(np.uint16(b)))
        lo = np.float32(abs(d))
        if float(lo) > abs(d):
            lo = np.nextafter(lo, np.float32(0))
        lo_b = int(lo.view(np.uint32)) >> 16
        cands = [float(np.uint32(c << 16).view(np.float32)) for c in (lo_b, lo_b + 1)]
        best = min(abs(c - abs(d)) for c in cands)
        assert abs(abs(val) - abs(d)) == best
        assert (val < 0) == (d < 0) or val == 0


# ------------------------------------------------------------- decoded weights

def _small(k, rows=24, cols=512, M=3, seed=0):
    return inputs.make_linear(rows, cols, k, M, seed_codes=100 + seed, seed_scales=200 + seed,
                              seed_x=300 + seed)


@pytest.mark.parametrize("k", [2, 3, 4])
def test_weights_are_fp32_value_times_scale(oracle_mod, k):
    """Packed-matvec weight = fp32(y / d) * fp32(scale), not bf16-rounded (the
    default decoder of the HEADER source); numpy float32 division and
    multiplication are IEEE correctly rounded."""
    codes, scales, _ = _small(k)
    st, ys, ws = oracle_mod.decode_rows(codes, scales, k, 16, 256)
    ylut, _ = oracle_mod.lut(16)
    assert np.array_equal(ylut[st], ys)  # dense decode through the table = bit walk
    want = (ys.astype(np.float32) / D32) * inputs.f16_bits_to_f32(scales)[:, None]
    assert np.array_equal(ws, want.astype(np.float32))


@pytest.mark.parametrize("k", [2, 3, 4])
def test_expand_is_bf16_of_weight(oracle_mod, k):
    """EXPAND_SOURCE: out[r][c] = bf16(value * scale[r]); torch's fp32->bf16."""
    codes, scales, _ = _small(k)
    _, ys, _ = oracle_mod.decode_rows(codes, scales, k, 16, 256)
    w = (ys.astype(np.float32) / D32) * inputs.f16_bits_to_f32(scales)[:, None]
    assert np.array_equal(oracle_mod.expand_bf16(codes, scales, k, 16, 256), _bf16_torch(w))
    sub = oracle_mod.expand_bf16(codes, scales, k, 16, 256, rows=[5, 0, 23])
    assert np.array_equal(sub, oracle_mod.expand_bf16(codes, scales, k, 16, 256)[[5, 0, 23]])


# ------------------------------------------------------------- matvecs

@pytest.mark.parametrize("k", [2, 3, 4])
def test_matvec_axis1_equals_dense_gemv(oracle_mod, k):
    """REDUCE_SOURCE: out[m][r] = sum_c w(r,c) x[m][c] -- against numpy's float64
    matmul of the dense decoded matrix (the expand-then-matmul path)."""
    codes, scales, x = _small(k)
    _, _, ws = oracle_mod.decode_rows(codes, scales, k, 16, 256)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    ref, ab = oracle_mod.matvec_axis1(codes, scales, x, k, 16, 256)
    want = xf @ ws.astype(np.float64).T
    assert np.allclose(ref, want, rtol=0, atol=1e-12 * ab.max())
    assert np.allclose(ab, np.abs(xf) @ np.abs(ws.astype(np.float64)).T, rtol=1e-12)
    assert np.all(ab >= np.abs(ref))


def test_matvec_axis1_special_cases(oracle_mod):
    k = 2
    codes, scales, x = _small(k, M=1)
    _, _, ws = oracle_mod.decode_rows(codes, scales, k, 16, 256)
    cols = ws.shape[1]
    for j in (0, 1, 255, 256, cols - 1):  # one-hot x picks one stored column
        e = np.zeros((1, cols), dtype=np.uint16)
        e[0, j] = 0x3F80  # bf16 1.0
        ref, _ = oracle_mod.matvec_axis1(codes, scales, e, k, 16, 256)
        assert np.array_equal(ref[0], ws[:, j].astype(np.float64))
    zero = np.zeros((2, cols), dtype=np.uint16)
    assert np.all(oracle_mod.matvec_axis1(codes, scales, zero, k, 16, 256)[0] == 0)
    zs = np.zeros_like(scales)
    assert np.all(oracle_mod.matvec_axis1(codes, zs, x, k, 16, 256)[0] == 0)
    # rows subset = the same rows of the full result
    full, _ = oracle_mod.matvec_axis1(codes, scales, x, k, 16, 256)
    part, _ = oracle_mod.matvec_axis1(codes, scales, x, k, 16, 256, rows=[7, 3])
    assert np.array_equal(part, full[:, [7, 3]])


@pytest.mark.parametrize("k", [2, 3])
def test_matvec_axis0_equals_transposed_gemv(oracle_mod, k):
    """SCATTER_SOURCE: the stored matrix is W^T [in, out]; out[m][c] =
    sum_r w(r,c) x[m][r] -- against numpy's float64 x @ W^T."""
    rows, cols = 40, 512
    codes, scales, x = inputs.make_linear(rows, cols, k, 4, seed_codes=9, seed_scales=8, seed_x=7,
                                          sigma=0.5, x_len=rows)
    _, _, ws = oracle_mod.decode_rows(codes, scales, k, 16, 256)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    ref, ab = oracle_mod.matvec_axis0(codes, scales, x, k, 16, 256)
    assert ref.shape == (4, cols)
    want = xf @ ws.astype(np.float64)
    assert np.allclose(ref, want, rtol=0, atol=1e-12 * ab.max())
    e = np.zeros((1, rows), dtype=np.uint16)
    e[0, 13] = 0x3F80
    one, _ = oracle_mod.matvec_axis0(codes, scales, e, k, 16, 256)
    assert np.array_equal(one[0], ws[13].astype(np.float64))
    part, _ = oracle_mod.matvec_axis0(codes, scales, x, k, 16, 256, cols=[511, 0, 300])
    assert np.array_equal(part, ref[:, [511, 0, 300]])


def test_shared_m_equals_independent_runs(oracle_mod):
    """Shared-M kernels must equal M separate M=1 runs (trellis-shared-m.ts)."""
    codes, scales, x = _small(3, M=4)
    ref, _ = oracle_mod.matvec_axis1(codes, scales, x, 3, 16, 256)
    for m in range(4):
        one, _ = oracle_mod.matvec_axis1(codes, scales, x[m:m + 1], 3, 16, 256)
        assert np.array_equal(one[0], ref[m])


# ------------------------------------------------------------- gate/up chain

def test_swiglu_chain_matches_torch(oracle_mod):
    """GATEUP_SOURCE cast chain: bf16 after sigmoid, silu and product.  Torch's
    fp32 sigmoid may differ from 1/(1+expf(-g)) by an fp32 ulp, so compare
    within one bf16 ulp and require near-total exact agreement."""
    rng = np.random.default_rng(3)
    g = inputs._f32_to_bf16_bits((rng.standard_normal(5000) * 4).astype(np.float32))
    u = inputs._f32_to_bf16_bits((rng.standard_normal(5000) * 4).astype(np.float32))
    got = oracle_mod.swiglu_bf16(g, u)
    gt = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).float()
    ut = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).float()
    sig = torch.sigmoid(gt).to(torch.bfloat16).float()
    silu = (gt * sig).to(torch.bfloat16).float()
    want = (silu * ut).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    diff = np.abs(got.view(np.int16).astype(np.int32) - want.view(np.int16).astype(np.int32))
    assert diff.max() <= 1
    assert (diff == 0).mean() > 0.99


def test_swiglu_special_values(oracle_mod):
    one, ten, zero = 0x3F80, 0x4120, 0x0000
    assert oracle_mod.swiglu_bf16(np.uint16([zero]), np.uint16([ten]))[0] == 0  # silu(0) = 0
    # sigmoid(10) rounds to bf16 1.0, so the output is bf16(10 * u)
    assert oracle_mod.swiglu_bf16(np.uint16([ten]), np.uint16([one]))[0] == ten
    # sigmoid(1) = 0.7311 -> bf16 0.73046875; silu = bf16(0.73046875) ; * 1
    assert inputs.bf16_bits_to_f32(oracle_mod.swiglu_bf16(np.uint16([one]), np.uint16([one])))[0] == np.float32(0.73046875)


def test_gateup_sums_are_two_axis1_matvecs(oracle_mod):
    g_codes, g_scales, x = _small(2, M=2, seed=1)
    u_codes, u_scales, _ = _small(2, M=2, seed=2)
    gr, ga, ur, ua = oracle_mod.gateup_sums(g_codes, g_scales, u_codes, u_scales, x, 2, 16, 256)
    assert np.array_equal(gr, oracle_mod.matvec_axis1(g_codes, g_scales, x, 2, 16, 256)[0])
    assert np.array_equal(ur, oracle_mod.matvec_axis1(u_codes, u_scales, x, 2, 16, 256)[0])


# ------------------------------------------------------------- prefill

def test_prefill_equals_expand_then_matmul(oracle_mod):
    """trellis-tiled-prefill.ts: out[m][r] = sum_c bf16 weight(r,c) x[m][c];
    against numpy float64 matmul of the bf16 expand (the pages' expand + matmul
    path)."""
    codes, scales, x = _small(2, rows=20, cols=768, M=9)
    e = inputs.bf16_bits_to_f32(oracle_mod.expand_bf16(codes, scales, 2, 16, 256)).astype(np.float64)
    ref, ab = oracle_mod.prefill(codes, scales, x, 2, 16, 256)
    want = inputs.bf16_bits_to_f32(x).astype(np.float64) @ e.T
    assert np.allclose(ref, want, rtol=0, atol=1e-12 * ab.max())
    part, _ = oracle_mod.prefill(codes, scales, x, 2, 16, 256, rows=[19, 4])
    assert np.array_equal(part, ref[:, [19, 4]])


@pytest.mark.parametrize("k", [2, 3])
def test_matvec_axis0_bf16w_equals_expand_then_gemv(oracle_mod, k):
    """Variants 0-3 (TRELLIS_ROUND): weights are the bf16 expand weights;
    against numpy's float64 x @ E for the stored W^T."""
    rows, cols = 33, 512
    codes, scales, x = inputs.make_linear(rows, cols, k, 3, seed_codes=12, sigma=0.5, x_len=rows)
    e = inputs.bf16_bits_to_f32(oracle_mod.expand_bf16(codes, scales, k, 16, 256)).astype(np.float64)
    ref, ab = oracle_mod.matvec_axis0_bf16w(codes, scales, x, k, 16, 256)
    want = inputs.bf16_bits_to_f32(x).astype(np.float64) @ e
    assert np.allclose(ref, want, rtol=0, atol=1e-12 * ab.max())
