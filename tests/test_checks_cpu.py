"""The parity checkers themselves, on the CPU: they must accept every output
the tolerance reading allows and reject what it does not."""
import numpy as np
import pytest

from test_parity_gpu import check_gateup
from util import ABS_TOL, REL_TOL, _bits_of_ordered, _ordered


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
