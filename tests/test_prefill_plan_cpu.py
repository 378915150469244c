"""The prefill GEMM's tile plan (trellis_prefill_plan), checked on the CPU.

The plan is the host arithmetic trellis_gemm_prefill launches by:
- tokens per tile from M;
- one persistent launch on axis 1;
- on axis 0, thread-block clusters that split each tile's reduction when
  the tiles leave SMs idle, and a second, split launch for the tiles left
  over after whole waves.

These tests pin the policy and the invariants every plan must keep: each
tile in exactly one launch, clusters that fit the SMs, and cluster sizes
within the portable limit (8, whose reduction slots fit in the stage ring) and
the reduction's stage count.
"""
import ctypes

import pytest

from trellis_coded_weight_gb300 import binding as tb


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_coded_weight_gb300 import build
    build.build()
    tb.load()


def _tiles(M, g):
    # the smallest of 32..512 tokens covering M, but 128 rather than 64 on axis 1
    bn = 32 if M <= 32 else (128 if g.axis == 1 else 64) if M <= 64 else 128 if M <= 128 else 256 if M <= 256 else 512
    feats = g.rows if g.axis == 1 else g.cols
    return bn, -(-feats // 128) * -(-M // bn)


def _stages(M, g):
    bn, _ = _tiles(M, g)
    bk = 32 if bn == 512 else 64
    kd = g.cols if g.axis == 1 else g.rows
    return -(-kd // bk)


@pytest.mark.parametrize("M,tokens", [(25, 32), (32, 32), (33, 64), (64, 64), (65, 128), (128, 128),
                                      (129, 256), (256, 256), (257, 512), (2048, 512), (100000, 512)])
def test_tokens_per_tile(M, tokens):
    """The smallest of 32..512 tokens covering M, except that axis 1 takes 128 where that is 64."""
    bn, _ = tb.prefill_plan(M, tb.Geometry(2, 16, 256, 1, 17408, 5120), 152)
    assert bn == (128 if tokens == 64 else tokens)
    if M > 32:  # axis 0 keeps the register-decode kernel up to 32 tokens
        assert tb.prefill_plan(M, tb.Geometry(2, 16, 256, 0, 17408, 5120), 152)[0] == tokens


SMALL_M_MAX = {1: 24, 0: 32}  # the register-decode kernels' range per axis


@pytest.mark.parametrize("M", [1, 5, 16, 17, 24, 25, 32, 33])
@pytest.mark.parametrize("axis", [0, 1])
def test_small_M_has_no_tiles(M, axis):
    # up to 24 tokens on axis 1 and 32 on axis 0 the register-decode kernels run: no tile plan
    bn, plan = tb.prefill_plan(M, tb.Geometry(2, 16, 256, axis, 17408, 5120), 152)
    if M <= SMALL_M_MAX[axis]:
        assert (bn, plan) == (0, [])
    else:
        assert bn == (32 if M <= 32 else 128 if axis == 1 else 64) and len(plan) >= 1


@pytest.mark.parametrize("M", [25, 32, 512, 2048, 5000])
def test_axis1_is_one_persistent_launch(M):
    g = tb.Geometry(2, 16, 256, 1, 17408, 5120)
    _, plan = tb.prefill_plan(M, g, 152)
    assert plan == [(0, _tiles(M, g)[1], 1)]


def test_axis0_pages_shapes():
    # the down projection, stored W^T [17408 in][5120 out]: 40 feature tiles
    g = tb.Geometry(3, 16, 256, 0, 17408, 5120)
    assert tb.prefill_plan(24, g, 152) == (0, [])                 # the register-decode kernel up to 32 tokens
    assert tb.prefill_plan(40, g, 152) == (64, [(0, 40, 3)])      # 3 CTAs per tile fill 120 of 152 SMs
    assert tb.prefill_plan(64, g, 152) == (64, [(0, 40, 3)])
    assert tb.prefill_plan(512, g, 152) == (512, [(0, 40, 3)])
    assert tb.prefill_plan(1024, g, 152) == (512, [(0, 80, 1)])   # 80 tiles: no room for 2 CTAs each
    # 160 tiles: the full wave unsplit, then the 8 leftover tiles split over 8-CTA clusters
    assert tb.prefill_plan(2048, g, 152) == (512, [(0, 152, 1), (152, 8, 8)])
    assert tb.prefill_plan(2048, g, 148) == (512, [(0, 148, 1), (148, 12, 8)])
    assert tb.prefill_plan(2048, g, 160) == (512, [(0, 160, 1)])  # whole waves: nothing left over


def test_split_caps():
    # every BN: at most the portable cluster size 8; short reductions: at most nk
    g = tb.Geometry(3, 16, 256, 0, 17408, 1024)                   # 8 feature tiles
    assert tb.prefill_plan(200, g, 152)[1] == [(0, 8, 8)]
    assert tb.prefill_plan(100, g, 152)[1] == [(0, 8, 8)]
    assert tb.prefill_plan(600, g, 152)[1] == [(0, 16, 8)]
    assert tb.prefill_plan(600, g, 100)[1] == [(0, 16, 6)]        # 16 tiles x 6 CTAs fill 96 of 100 SMs
    short = tb.Geometry(3, 16, 256, 0, 96, 5376)                  # 96 rows: 3 stages of 32 at BN = 512
    assert tb.prefill_plan(1600, short, 152) == (512, [(0, 152, 1), (152, 16, 3)])
    assert tb.prefill_plan(40, tb.Geometry(2, 16, 256, 0, 64, 5120), 152)[1] == [(0, 40, 1)]  # 1 stage of 64


@pytest.mark.parametrize("sms", [1, 7, 132, 148, 152, 160])
@pytest.mark.parametrize("axis", [0, 1])
def test_plan_invariants(sms, axis):
    for rows, cols in ((17408, 5120), (96, 5376), (1000, 768), (8, 256), (5120, 17408)):
        if axis == 0 and rows % 8:
            continue
        g = tb.Geometry(3, 16, 256, axis, rows, cols)
        for M in (1, 31, 64, 200, 300, 512, 777, 1024, 2048, 4096):
            bn, plan = tb.prefill_plan(M, g, sms)
            if M <= SMALL_M_MAX[axis]:  # the register-decode kernels: no tiles
                assert (bn, plan) == (0, [])
                continue
            _, ntiles = _tiles(M, g)
            nk = _stages(M, g)
            assert bn == _tiles(M, g)[0]
            assert 1 <= len(plan) <= 2
            covered = [t for t0, n, _ in plan for t in range(t0, t0 + n)]
            assert covered == list(range(ntiles)), "every tile exactly once, in order"
            for t0, n, S in plan:
                assert n >= 1 and 1 <= S <= 8 and S <= max(nk, 1)
                if axis == 1:
                    assert S == 1
                if S > 1:
                    assert n * S <= sms, "the clusters of a split launch run at once"


def test_plan_argument_errors():
    g = tb.Geometry(3, 16, 256, 0, 17408, 5120)
    lib = tb.load()
    bn, buf = ctypes.c_int32(0), (ctypes.c_int32 * 6)()
    assert lib.trellis_prefill_plan(0, ctypes.byref(g.c()), 152, ctypes.byref(bn), buf) == -2       # EM
    assert lib.trellis_prefill_plan(8, ctypes.byref(g.c()), 152, None, buf) == -7                   # ENULL
    assert lib.trellis_prefill_plan(8, ctypes.byref(g.c()), 152, ctypes.byref(bn), None) == -7      # ENULL
    assert lib.trellis_prefill_plan(8, None, 152, ctypes.byref(bn), buf) == -7                      # ENULL
    odd = tb.Geometry(3, 16, 256, 0, 17407, 5120)  # axis-0 rows must keep x rows 16-byte multiples
    assert lib.trellis_prefill_plan(8, ctypes.byref(odd.c()), 152, ctypes.byref(bn), buf) == -1     # EGEOM
    bad = tb.Geometry(5, 16, 256, 1, 17408, 5120)
    assert lib.trellis_prefill_plan(8, ctypes.byref(bad.c()), 152, ctypes.byref(bn), buf) == -1     # EGEOM
