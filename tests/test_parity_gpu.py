"""Parity of the CUDA path (through the C ABI) against the oracle.

Small cases are compared element by element in full: they span several
blocks, ragged row counts (not a multiple of 32), one-block rows, and M = 1..4.
Full-size cases (the 27B-class MLP shapes, in the launch configuration the
bench times) are compared on sampled rows or columns that the oracle computes
one by one.
"""
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


def _sample(n, count, seed):
    rng = np.random.default_rng(seed)
    idx = set(rng.choice(n, size=min(count, n), replace=False).tolist()) | {0, n - 1}
    return np.array(sorted(idx), dtype=np.int64)


# ------------------------------------------------------------------ expand

@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("rows,cols", [(1, 256), (333, 256), (37, 768), (64, 2048)])
def test_expand_bit_exact_small(oracle_mod, k, rows, cols):
    codes, scales, _ = inputs.make_linear(rows, cols, k, 1, seed_codes=11 + k, seed_scales=12)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = tb.expand_bf16(to_dev_u32(codes), to_dev_f16(scales), g)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(out), oracle_mod.expand_bf16(codes, scales, k, L, T))


@pytest.mark.parametrize("k", [2, 3, 4])
def test_expand_bit_exact_full_size_sampled(oracle_mod, k):
    rows, cols = 17408, 5120
    codes, scales, _ = inputs.make_linear(rows, cols, k, 1)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = bf16_bits(tb.expand_bf16(to_dev_u32(codes), to_dev_f16(scales), g))
    idx = _sample(rows, 48, k)
    assert np.array_equal(out[idx], oracle_mod.expand_bf16(codes, scales, k, L, T, rows=idx))


def test_expand_L12(oracle_mod):
    codes, scales, _ = inputs.make_linear(40, 512, 3, 1, seed_codes=77)
    out = tb.expand_bf16(to_dev_u32(codes), to_dev_f16(scales), tb.Geometry(3, 12, T, 1, 40, 512))
    assert np.array_equal(bf16_bits(out), oracle_mod.expand_bf16(codes, scales, 3, 12, T))


# ------------------------------------------------------------------ axis 1

@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("rows,cols", [(1, 256), (45, 768), (100, 1280)])
def test_matvec_axis1_small(oracle_mod, k, M, rows, cols):
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=21 + k, seed_x=22 + M)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = tb.matvec_axis1(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    ref, ab = oracle_mod.matvec_axis1(codes, scales, x, k, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"axis1 k={k} M={M} {rows}x{cols}")


def test_matvec_axis1_config_smoke_shape(oracle_mod):
    """R=512, C=2048, k=2, M=1: the small full-check configuration."""
    codes, scales, x = inputs.make_linear(512, 2048, 2, 1)
    g = tb.Geometry(2, L, T, 1, 512, 2048)
    out = tb.matvec_axis1(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g)
    ref, ab = oracle_mod.matvec_axis1(codes, scales, x, 2, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, "axis1 512x2048")


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("pinned", [True, False])
def test_matvec_axis1_host_buffers(oracle_mod, M, pinned):
    """The host-buffer call: x from host memory, out back to host memory, in one call; the same bits as the
    device call and within the oracle's band."""
    rows, cols, k = 300, 1280, 3
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=91, seed_x=92 + M)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    dc, ds = to_dev_u32(codes), to_dev_f16(scales)
    x_host = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    out_host = torch.full((M, rows), -1.0, dtype=torch.bfloat16)
    if pinned:
        x_host, out_host = x_host.pin_memory(), out_host.pin_memory()
    x_dev = torch.empty((M, cols), dtype=torch.bfloat16, device="cuda")
    out_dev = torch.empty((M, rows), dtype=torch.bfloat16, device="cuda")
    tb.matvec_axis1_host(dc, ds, x_host, g, out_host, x_dev, out_dev)
    torch.cuda.current_stream().synchronize()
    dev = tb.matvec_axis1(dc, ds, to_dev_bf16(x), g)
    assert torch.equal(out_host.view(torch.int16), dev.cpu().view(torch.int16))
    ref, ab = oracle_mod.matvec_axis1(codes, scales, x, k, L, T)
    check_band(oracle_mod, bf16_bits(out_host), ref, ab, f"axis1 host buffers M={M}")


def _host_view(a: np.ndarray, pinned: bool, shift: int) -> torch.Tensor:
    """A bf16 host tensor holding `a`'s bits, `shift` elements into its (pinned or pageable) allocation."""
    flat = torch.empty(a.size + shift, dtype=torch.int16)
    if pinned:
        flat = flat.pin_memory()
    v = flat[shift:].view(a.shape)
    v.copy_(torch.from_numpy(a.view(np.int16)))
    return v.view(torch.bfloat16)


@pytest.mark.parametrize("x_pinned,out_pinned,shift", [
    (True, False, 0), (False, True, 0),  # one side through its mapping, the other through the copy engines
    (True, True, 8),                     # 16 bytes into a pinned allocation: the mapping's offset
    (True, True, 1),                     # 2 bytes in: not 16-byte aligned, the copy engines
])
def test_matvec_axis1_host_buffer_forms(oracle_mod, x_pinned, out_pinned, shift):
    """Every combination of how the host call reaches x_host and out_host gives the device call's bits."""
    rows, cols, k, M = 272, 1536, 2, 3
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=93, seed_x=94)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    dc, ds = to_dev_u32(codes), to_dev_f16(scales)
    x_host = _host_view(x, x_pinned, shift)
    out_host = _host_view(np.full((M, rows), 0xBF80, dtype=np.uint16), out_pinned, shift)
    x_dev = torch.empty((M, cols), dtype=torch.bfloat16, device="cuda")
    out_dev = torch.empty((M, rows), dtype=torch.bfloat16, device="cuda")
    tb.matvec_axis1_host(dc, ds, x_host, g, out_host, x_dev, out_dev)
    torch.cuda.current_stream().synchronize()
    dev = tb.matvec_axis1(dc, ds, to_dev_bf16(x), g)
    assert torch.equal(out_host.view(torch.int16), dev.cpu().view(torch.int16))


@pytest.mark.parametrize("pinned", [True, False])
def test_matvec_axis1_host_chain_reuses_buffers(pinned):
    """Calls queued back to back without a synchronisation, each taking the previous call's host output as its
    input and sharing one pair of device buffers: stream order holds (each call reads what the previous call
    wrote), as in a chain of device calls."""
    n, k, M, calls = 512, 3, 2, 4
    codes, scales, x = inputs.make_linear(n, n, k, M, seed_codes=95, seed_x=96)
    g = tb.Geometry(k, L, T, 1, n, n)
    dc, ds = to_dev_u32(codes), to_dev_f16(scales)
    bufs = [_host_view(x if i == 0 else np.zeros((M, n), dtype=np.uint16), pinned, 0) for i in range(calls + 1)]
    x_dev = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    out_dev = torch.empty((M, n), dtype=torch.bfloat16, device="cuda")
    for i in range(calls):
        tb.matvec_axis1_host(dc, ds, bufs[i], g, bufs[i + 1], x_dev, out_dev)
    torch.cuda.current_stream().synchronize()
    want = to_dev_bf16(x)
    for i in range(calls):
        want = tb.matvec_axis1(dc, ds, want, g)
        assert torch.equal(bufs[i + 1].view(torch.int16), want.cpu().view(torch.int16)), f"call {i}"


@pytest.mark.parametrize("k", [2, 3, 4])
def test_matvec_axis1_full_size_sampled(oracle_mod, k):
    rows, cols, M = 17408, 5120, 4
    codes, scales, x = inputs.make_linear(rows, cols, k, M)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    dc, ds = to_dev_u32(codes), to_dev_f16(scales)
    idx = _sample(rows, 40, 100 + k)
    for m in (1, 4):
        out = bf16_bits(tb.matvec_axis1(dc, ds, to_dev_bf16(x[:m]), g))
        ref, ab = oracle_mod.matvec_axis1(codes, scales, x[:m], k, L, T, rows=idx)
        check_band(oracle_mod, out[:, idx], ref, ab, f"axis1 full k={k} M={m}")


def test_matvec_axis1_special_inputs(oracle_mod):
    rows, cols = 64, 512
    codes, scales, _ = inputs.make_linear(rows, cols, 2, 1)
    g = tb.Geometry(2, L, T, 1, rows, cols)
    dc, ds = to_dev_u32(codes), to_dev_f16(scales)
    zero = torch.zeros((2, cols), dtype=torch.bfloat16, device="cuda")
    assert torch.all(tb.matvec_axis1(dc, ds, zero, g) == 0)
    e = np.zeros((1, cols), dtype=np.uint16)
    e[0, 300] = 0x3F80
    out = tb.matvec_axis1(dc, ds, to_dev_bf16(e), g)
    ref, ab = oracle_mod.matvec_axis1(codes, scales, e, 2, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, "one-hot")


def test_matvec_axis1_L12(oracle_mod):
    codes, scales, x = inputs.make_linear(50, 1024, 4, 3, seed_codes=5)
    out = tb.matvec_axis1(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), tb.Geometry(4, 12, T, 1, 50, 1024))
    ref, ab = oracle_mod.matvec_axis1(codes, scales, x, 4, 12, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, "axis1 L=12")


# ------------------------------------------------------------------ load floor

@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("rows,cols", [(45, 768), (17408, 5120)])
def test_load_floor_reads_every_word(k, rows, cols):
    """The load-only floor folds by XOR every word it loads: all of the row's words, plus each block's
    two spill reads (word 4K with the first half block, word 0 with the second), which cancel those
    two words -- so the fold is the XOR of each block's words other than 0 and 4K."""
    codes, _, _ = inputs.make_linear(rows, cols, k, 1, seed_codes=61 + k)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    got = tb.load_floor(to_dev_u32(codes), g).cpu().numpy().view(np.uint32)
    blocks = np.ascontiguousarray(codes).view(np.uint32).reshape(rows, cols // T, T * k // 32).copy()
    blocks[:, :, 0] = 0
    blocks[:, :, 4 * k] = 0
    want = np.bitwise_xor.reduce(blocks.reshape(rows, -1), axis=1)
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ gate/up

def check_gateup(oracle, gpu_bits, gref, gab, uref, uab, what):
    """Accept an output if it is within one bf16 ulp of the activation chain
    evaluated at some pair of bf16 gate/up values that a correctly rounded
    cast of sums inside the tolerance band can give.  Returns the fraction of
    outputs whose gate or up band held more than one bf16 value.

    The band ends and the reference itself are tried first.  An output they
    do not explain is checked against every bf16 gate value of its band: for
    a fixed gate the chain bf16(silu(g) * u) is monotone in u and moves by at
    most two ulps per bf16 step of u, so the outputs reachable over the up
    band are those between the chain at its two ends, give or take one ulp."""
    from util import ABS_TOL, REL_TOL, _bits_of_ordered, _ordered, bf16_of_f64
    tg, tu = REL_TOL * gab + ABS_TOL, REL_TOL * uab + ABS_TOL
    cands_g = [bf16_of_f64(oracle, gref - tg), bf16_of_f64(oracle, gref), bf16_of_f64(oracle, gref + tg)]
    cands_u = [bf16_of_f64(oracle, uref - tu), bf16_of_f64(oracle, uref), bf16_of_f64(oracle, uref + tu)]
    gpu = _ordered(np.asarray(gpu_bits, dtype=np.uint16))
    ok = np.zeros(gpu.shape, dtype=bool)
    for cg in cands_g:
        for cu in cands_u:
            want = _ordered(oracle.swiglu_bf16(cg, cu))
            ok |= np.abs(gpu - want) <= 1
    glo, ghi = _ordered(cands_g[0]), _ordered(cands_g[2])
    for idx in zip(*np.nonzero(~ok)):
        gvals = np.arange(glo[idx], ghi[idx] + 1)
        gbits = _bits_of_ordered(gvals)
        a = _ordered(oracle.swiglu_bf16(gbits, np.full(gbits.shape, cands_u[0][idx], dtype=np.uint16)))
        b = _ordered(oracle.swiglu_bf16(gbits, np.full(gbits.shape, cands_u[2][idx], dtype=np.uint16)))
        ok[idx] = bool(((gpu[idx] >= np.minimum(a, b) - 1) & (gpu[idx] <= np.maximum(a, b) + 1)).any())
    assert ok.all(), f"{what}: {int((~ok).sum())} of {ok.size} outputs off the chain"
    multi = (cands_g[0] != cands_g[2]) | (cands_u[0] != cands_u[2])
    return float(multi.mean())


@pytest.mark.parametrize("k", [2, 3])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("rows,cols", [(33, 512), (96, 1536)])
def test_gateup_small(oracle_mod, k, M, rows, cols):
    gc, gs, x = inputs.make_linear(rows, cols, k, M, seed_codes=31, seed_scales=32, seed_x=33 + M)
    uc, us, _ = inputs.make_linear(rows, cols, k, M, seed_codes=41, seed_scales=42, seed_x=43)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = tb.gateup_swiglu(to_dev_u32(gc), to_dev_f16(gs), to_dev_u32(uc), to_dev_f16(us), to_dev_bf16(x), g)
    sums = oracle_mod.gateup_sums(gc, gs, uc, us, x, k, L, T)
    check_gateup(oracle_mod, bf16_bits(out), *sums, f"gateup k={k} M={M}")


@pytest.mark.parametrize("k", [2, 3])
def test_gateup_full_size_sampled(oracle_mod, k):
    rows, cols, M = 17408, 5120, 4
    gc, gs, x = inputs.make_linear(rows, cols, k, M, seed_codes=inputs.SEED_GATE)
    uc, us, _ = inputs.make_linear(rows, cols, k, M, seed_codes=inputs.SEED_UP, seed_scales=inputs.SEED_SCALES + 1)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    out = bf16_bits(tb.gateup_swiglu(to_dev_u32(gc), to_dev_f16(gs), to_dev_u32(uc), to_dev_f16(us),
                                     to_dev_bf16(x), g))
    idx = _sample(rows, 40, 200 + k)
    sums = oracle_mod.gateup_sums(gc, gs, uc, us, x, k, L, T, rows=idx)
    check_gateup(oracle_mod, out[:, idx], *sums, f"gateup full k={k}")


# ------------------------------------------------------------------ axis 0

@pytest.mark.parametrize("k", [2, 3, 4])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("rows,cols", [(1, 256), (77, 512), (300, 768)])
def test_matvec_axis0_small(oracle_mod, k, M, rows, cols):
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=51 + k, seed_x=52 + M, sigma=0.5,
                                          x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    ws = tb.new_workspace(M, g, "cuda")
    dc, ds, dx = to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x)
    ref, ab = oracle_mod.matvec_axis0(codes, scales, x, k, L, T)
    for _ in range(2):  # the workspace is reused: the second call must match too
        out = tb.matvec_axis0(dc, ds, dx, g, ws)
        check_band(oracle_mod, bf16_bits(out), ref, ab, f"axis0 k={k} M={M} {rows}x{cols}")


@pytest.mark.parametrize("k", [2, 3])
def test_matvec_axis0_full_size_sampled(oracle_mod, k):
    rows, cols, M = 17408, 5120, 4
    codes, scales, x = inputs.make_linear(rows, cols, k, M, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    ws = tb.new_workspace(M, g, "cuda")
    dc, ds = to_dev_u32(codes), to_dev_f16(scales)
    idx = _sample(cols, 40, 300 + k)
    for m in (1, 4):
        out = bf16_bits(tb.matvec_axis0(dc, ds, to_dev_bf16(x[:m]), g, ws))
        ref, ab = oracle_mod.matvec_axis0(codes, scales, x[:m], k, L, T, cols=idx)
        check_band(oracle_mod, out[:, idx], ref, ab, f"axis0 full k={k} M={m}")


@pytest.mark.parametrize("k", [2, 3, 4])
def test_matvec_axis0_L12(oracle_mod, k):
    rows, cols, M = 333, 768, 3
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=61 + k, seed_x=62, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, 12, T, 0, rows, cols)
    out = tb.matvec_axis0(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g, tb.new_workspace(M, g, "cuda"))
    ref, ab = oracle_mod.matvec_axis0(codes, scales, x, k, 12, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"axis0 L=12 k={k}")


# Work ranges that cross column blocks (several segments per CTA), a single column block shared by many CTAs,
# and staged pieces with a ragged last 8-row step.
@pytest.mark.parametrize("k", [2, 3])
@pytest.mark.parametrize("rows,cols,M", [(77, 256 * 40, 2), (5000, 256, 4), (1001, 1280, 1), (259, 512, 3)])
def test_matvec_axis0_segments_and_pieces(oracle_mod, k, rows, cols, M):
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=71 + k, seed_x=72 + M, sigma=0.5,
                                          x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    out = tb.matvec_axis0(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g, tb.new_workspace(M, g, "cuda"))
    ref, ab = oracle_mod.matvec_axis0(codes, scales, x, k, L, T)
    check_band(oracle_mod, bf16_bits(out), ref, ab, f"axis0 segments k={k} M={M} {rows}x{cols}")


def test_matvec_axis0_long_ranges(oracle_mod):
    """Each CTA's range is longer than one tensor-core accumulation chain (100000 rows over at most 256 CTAs)."""
    rows, cols, M, k = 100000, 1024, 2, 2
    codes, scales, x = inputs.make_linear(rows, cols, k, M, seed_codes=81, seed_x=82, sigma=0.5, x_len=rows)
    g = tb.Geometry(k, L, T, 0, rows, cols)
    out = bf16_bits(tb.matvec_axis0(to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g,
                                    tb.new_workspace(M, g, "cuda")))
    idx = _sample(cols, 24, 83)
    ref, ab = oracle_mod.matvec_axis0(codes, scales, x, k, L, T, cols=idx)
    check_band(oracle_mod, out[:, idx], ref, ab, "axis0 long ranges")


def test_matvec_axis0_is_deterministic():
    rows, cols = 2000, 1024
    codes, scales, x = inputs.make_linear(rows, cols, 3, 2, sigma=0.5, x_len=rows)
    g = tb.Geometry(3, L, T, 0, rows, cols)
    ws = tb.new_workspace(2, g, "cuda")
    args = (to_dev_u32(codes), to_dev_f16(scales), to_dev_bf16(x), g, ws)
    a = tb.matvec_axis0(*args).clone()
    b = tb.matvec_axis0(*args)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------ load-only floors (measurement aids)

@pytest.mark.parametrize("k", [2, 3, 4])
def test_load_floors_fold_the_words_they_read(k):
    """Both floors read the stream and fold every loaded word by XOR: the coalesced floor all words of the
    row; the M = 1 pattern each block's words plus the spill reads of words 4k and 0, which cancel those two."""
    rows, cols = 300, 1280
    codes, _, _ = inputs.make_linear(rows, cols, k, 1, seed_codes=600 + k)
    g = tb.Geometry(k, L, T, 1, rows, cols)
    dc = to_dev_u32(codes)
    got = tb.load_floor(dc, g, coalesced=True).cpu().numpy().view(np.uint32)
    assert np.array_equal(got, np.bitwise_xor.reduce(codes, axis=1))
    wpb = 8 * k
    keep = np.ones(wpb, dtype=bool)
    keep[0] = keep[4 * k] = False
    want = np.bitwise_xor.reduce(codes.reshape(rows, -1, wpb)[:, :, keep].reshape(rows, -1), axis=1)
    assert np.array_equal(tb.load_floor(dc, g).cpu().numpy().view(np.uint32), want)


# ------------------------------------------------------------------ back-to-back launches

@pytest.mark.parametrize("consumer_axis", [1, 0])
def test_chained_matvecs_read_the_previous_output(oracle_mod, consumer_axis):
    """A matvec whose x is the output of the matvec just ahead of it on the stream (both launched with
    programmatic dependent launch): the consumer must see the producer's finished output.  Repeated with
    fresh inputs so that a consumer reading early would see stale values."""
    M, k = 4, 2
    r1, c1 = 1024, 768  # producer: out1 [M, 1024]
    codes1, scales1, _ = inputs.make_linear(r1, c1, k, M, seed_codes=101, seed_x=102)
    if consumer_axis == 1:
        r2, c2 = 512, r1  # consumer reads out1 as x [M, 1024]
        codes2, scales2, _ = inputs.make_linear(r2, c2, k, M, seed_codes=103, seed_x=104)
        g2 = tb.Geometry(k, L, T, 1, r2, c2)
    else:
        r2, c2 = r1, 512  # axis-0 consumer: stored rows = 1024 = len(x)
        codes2, scales2, _ = inputs.make_linear(r2, c2, k, M, seed_codes=105, seed_x=106, x_len=r2)
        g2 = tb.Geometry(k, L, T, 0, r2, c2)
    g1 = tb.Geometry(k, L, T, 1, r1, c1)
    d1c, d1s, d2c, d2s = to_dev_u32(codes1), to_dev_f16(scales1), to_dev_u32(codes2), to_dev_f16(scales2)
    ws = tb.new_workspace(M, g2, "cuda") if consumer_axis == 0 else None
    for rep in range(3):
        x = inputs.normal_bf16(110 + rep, (M, c1))
        out1 = tb.matvec_axis1(d1c, d1s, to_dev_bf16(x), g1)
        out2 = tb.matvec_axis1(d2c, d2s, out1, g2) if consumer_axis == 1 else tb.matvec_axis0(d2c, d2s, out1, g2, ws)
        mid = bf16_bits(out1)
        if consumer_axis == 1:
            ref, ab = oracle_mod.matvec_axis1(codes2, scales2, mid, k, L, T)
        else:
            ref, ab = oracle_mod.matvec_axis0(codes2, scales2, mid, k, L, T)
        check_band(oracle_mod, bf16_bits(out2), ref, ab, f"chained axis1 -> axis{consumer_axis} rep {rep}")
