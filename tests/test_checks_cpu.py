"""The parity checkers themselves, on the CPU: they must accept every output
the tolerance reading allows and reject what it does not."""
import numpy as np
import pytest

from test_parity_gpu import check_gateup
import util
from util import ABS_TOL, REL_TOL, _bits_of_ordered, _ordered, check_band


@pytest.fixture(autouse=True)
def _keep_band_stats_for_parity_checks():
    """The planted cases here are not parity results: keep them out of the
    session's bf16-distance summary."""
    n = len(util.BAND_STATS)
    yield
    del util.BAND_STATS[n:]


def _bf16_bits(v):
    a = np.asarray(v, dtype=np.float32).view(np.uint32)
    return ((a + 0x7FFF + ((a >> 16) & 1)) >> 16).astype(np.uint16)  # RNE, finite inputs


def test_ordered_round_trip():
    b = np.array([0x0000, 0x0001, 0x3F80, 0x7F7F, 0x8001, 0xBF80, 0xFF7F], dtype=np.uint16)
    assert np.array_equal(_bits_of_ordered(_ordered(b)), b)
    assert np.all(np.diff(_ordered(_bf16_bits([-3.0, -1.0, -1e-30, 0.0, 1e-30, 1.0, 3.0]))) > 0)


def test_gateup_check_takes_the_whole_band(oracle_mod):
    # An up sum of 1e-5 whose band (absolute sum 4) crosses zero holds thousands
    # of bf16 values; a result computed at one inside it -- not a band end, not
    # the reference -- is legitimate and must pass; an output two values off
    # every reachable one must not.
    gref = np.array([[-0.144722]])
    gab = np.array([[8.0]])
    uref = np.array([[1.0e-5]])
    uab = np.array([[4.0]])
    tu = REL_TOL * uab + ABS_TOL
    inner_u = _bf16_bits(uref - 0.5 * tu)
    g_bits = _bf16_bits(gref)
    legit = oracle_mod.swiglu_bf16(g_bits.ravel(), inner_u.ravel()).reshape(1, 1)
    check_gateup(oracle_mod, legit, gref, gab, uref, uab, "interior up value")
    # the largest output the band can reach, moved three values further out
    g_lo = _ordered(_bf16_bits(gref - (REL_TOL * gab + ABS_TOL)))
    g_hi = _ordered(_bf16_bits(gref + (REL_TOL * gab + ABS_TOL)))
    u_ends = [_bf16_bits(uref - tu), _bf16_bits(uref + tu)]
    reach = [_ordered(oracle_mod.swiglu_bf16(_bits_of_ordered(np.array([gv])), ue.ravel()))[0]
             for gv in range(int(g_lo[0, 0]), int(g_hi[0, 0]) + 1) for ue in u_ends]
    off = _bits_of_ordered(np.array([[max(reach) + 3]]))
    with pytest.raises(AssertionError):
        check_gateup(oracle_mod, off, gref, gab, uref, uab, "planted")


# ------------------------------------------------------------- check_band

def _ref_bf16_values(v):
    """Exact fp64 value of bf16 bit patterns."""
    return (np.asarray(v, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_band_narrow_accepts_the_rounding_and_rejects_neighbours(oracle_mod):
    # |ref| ~ 1 with sum|w*x| = 1: the band (1.1e-5) is far inside one bf16
    # ulp (2^-7), so only bf16(ref) itself passes; one or two ulps off fail.
    ref = np.array([[1.0 + 3.0e-4, -2.5 + 1.0e-3]])
    ab = np.ones_like(ref)
    mid = _bf16_bits(ref)
    check_band(oracle_mod, mid, ref, ab, "exact rounding")
    for d in (1, 2):
        planted = _bits_of_ordered(_ordered(mid) + d)
        with pytest.raises(AssertionError):
            check_band(oracle_mod, planted, ref, ab, f"{d} ulp off, narrow band")


def test_band_on_a_rounding_tie_accepts_both_neighbours(oracle_mod):
    # ref exactly halfway between two bf16 values: a value inside the fp32 band
    # on either side rounds to either neighbour, so both are legitimate.
    lo_b, hi_b = np.uint16(0x3F80), np.uint16(0x3F81)
    ref = np.array([[0.5 * (_ref_bf16_values(lo_b) + _ref_bf16_values(hi_b))]])
    ab = np.ones_like(ref)
    check_band(oracle_mod, np.array([[lo_b]]), ref, ab, "tie, low side")
    check_band(oracle_mod, np.array([[hi_b]]), ref, ab, "tie, high side")
    with pytest.raises(AssertionError):
        check_band(oracle_mod, np.array([[np.uint16(0x3F82)]]), ref, ab, "tie, two off")


def test_band_wide_accepts_the_interior_and_rejects_outside(oracle_mod):
    # Cancellation: ref = 0.01 from terms whose absolute sum is 1e4, so the
    # band is +-0.1 (hundreds of bf16 ulps at 0.01).  Any output inside it is
    # legitimate; one just past its end is not.
    ref = np.array([[0.01]])
    ab = np.array([[1.0e4]])
    tol = REL_TOL * ab + ABS_TOL
    inner = _bf16_bits(ref + 0.6 * tol)
    assert abs(int(_ordered(inner)[0, 0]) - int(_ordered(_bf16_bits(ref))[0, 0])) > 100
    assert check_band(oracle_mod, inner, ref, ab, "interior of a wide band") > 100
    outside = _bits_of_ordered(_ordered(_bf16_bits(ref + tol)) + 2)
    with pytest.raises(AssertionError):
        check_band(oracle_mod, outside, ref, ab, "past the band's end")
    with pytest.raises(AssertionError):
        check_band(oracle_mod, _bf16_bits(-ref - 1.5 * tol), ref, ab, "wrong sign, outside")
