"""Pins of the oracle to facts other than itself (run without a GPU).

Each test names the passage of the reference pages it follows ("trellis-linear.ts"
and the other diff pages of mlx-bun 0.2.0 -> 0.4.0) and pins the oracle with a
worked example, a closed form, an invariant, a library routine or brute force.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from trellis_coded_weight_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
A, B = 34038481, 76625530
D = 147.800537109375
A_INV = pow(A, -1, 1 << 32)  # a is odd, so s -> s*a+b is a bijection mod 2^32


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _round_f32(q: Fraction) -> np.float32:
    """Exact round-to-nearest-even of a rational to fp32."""
    f = np.float32(float(q))
    best = None
    for cand in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        err = abs(Fraction(float(cand)) - q)
        key = (err, int(np.float32(cand).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


# ------------------------------------------------------------------ 1MAD code

def test_decode_worked_examples(oracle_mod):
    """Hand-derived examples of trellis_y (HEADER source, trellis-linear.ts)."""
    rows = _rows("decode_1mad.txt")
    assert len(rows) >= 7
    for s, xhex, b0, b1, b2, b3, y in rows:
        s, x, y = int(s), int(xhex, 16), int(y)
        assert [int(b0), int(b1), int(b2), int(b3)] == [(x >> (8 * i)) & 255 for i in range(4)]
        assert oracle_mod.code_y(s) == y, (s, y)


@pytest.mark.parametrize("x,y", [(0x00000000, -510), (0xFFFFFFFF, 510), (0x01000000, -509),
                                 (0x00000100, -509), (0x80808080, 2), (0x00FF00FF, 0),
                                 (0xFF000000, -255), (0x000000FF, -255), (0x12345678, -234)])
def test_decode_targets_each_byte(oracle_mod, x, y):
    """Closed form: choose x, solve s = (x - b) * a^-1 mod 2^32, so y is the
    byte sum of the chosen x minus 510 (trellis_y).  A dropped or doubled byte,
    a wrong offset or a wrong constant fails one of these."""
    s = ((x - B) * A_INV) % (1 << 32)
    assert (s * A + B) % (1 << 32) == x
    assert oracle_mod.code_y(s) == y


@pytest.mark.parametrize("L", [12, 16])
def test_decode_range_and_independent_table_all_states(oracle_mod, L):
    """Every state of a 2^L table: y stays in [-510, 510] (byte sums lie in
    [0, 1020]), and the table -- built by walking x = b + s*a incrementally and
    summing bytes with the two byte-pair adds of trellis_y (HEADER source) --
    equals the per-state decode (multiply, then bytes by division and
    remainder) at all 2^L states."""
    ys, vs = oracle_mod.lut(L)
    assert ys.size == 1 << L
    assert ys.min() >= -510 and ys.max() <= 510
    per_state = np.array([oracle_mod.code_y(s) for s in range(1 << L)], dtype=np.int32)
    assert np.array_equal(ys, per_state)
    # the table's values are the correctly rounded y/d of its own y
    vals = {y: oracle_mod.code_val(y) for y in np.unique(ys).tolist()}
    assert np.array_equal(vs, np.array([vals[int(y)] for y in ys], dtype=np.float32))


def _numpy_y(L):
    """A third formulation for the regression values: numpy uint64 products,
    bytes by shifts, vectorised over all 2^L states."""
    s = np.arange(1 << L, dtype=np.uint64)
    x = (s * np.uint64(A) + np.uint64(B)) % np.uint64(1 << 32)
    return sum(((x >> np.uint64(8 * i)) & np.uint64(255)).astype(np.int64) for i in range(4)) - 510


@pytest.mark.parametrize("L,lo,hi,distinct", [(16, -483, 469, 908), (12, -448, 454, 713)])
def test_decode_regression_values(oracle_mod, L, lo, hi, distinct):
    """Regression values of the code, fixed by enumerating all 2^L states
    outside this repository's code: the range of y,
    the number of distinct y, and at L = 16 mean(y) = -0.0582 and
    var(y/d) = 1.00018 (the code is built to have unit variance; d is the
    fp32 rounding of sqrt(21845), the standard deviation of a sum of four
    uniform bytes)."""
    ys, vs = oracle_mod.lut(L)
    assert (int(ys.min()), int(ys.max()), int(np.unique(ys).size)) == (lo, hi, distinct)
    assert np.array_equal(ys, _numpy_y(L))
    if L == 16:
        assert abs(float(ys.mean()) - (-0.0582275390625)) < 1e-12
        assert abs(float(np.var(vs.astype(np.float64))) - 1.00018) < 5e-6


def test_decode_statistics_over_the_full_state_space(oracle_mod):
    """Closed form: x runs over all of Z/2^32 as s does, so y has mean 0 and
    variance 4*(256^2-1)/12 = 21845; d is the fp32 rounding of sqrt(21845)."""
    assert np.float32(D) == np.float32(math.sqrt(21845.0))
    rng = np.random.default_rng(7)
    s = rng.integers(0, 1 << 32, size=200_000, dtype=np.uint64)
    y = np.array([oracle_mod.code_y(int(v)) for v in s], dtype=np.float64)
    assert abs(y.mean()) < 4 * math.sqrt(21845.0 / y.size)
    assert abs(y.var() - 21845.0) < 400.0


def test_code_val_is_correctly_rounded(oracle_mod):
    """value = y / d as one correctly rounded fp32 division (trellis_val), for
    all 1021 reachable y; checked against exact rational rounding."""
    dq = Fraction(D)
    for y in range(-510, 511):
        assert oracle_mod.code_val(y) == _round_f32(Fraction(y) / dq), y


def test_pages_claim_refined_reciprocal_is_correctly_rounded():
    """The pages state that y*(1/d) refined by one residual step (trellis_val_rcp)
    is correctly rounded for every y in [-510, 510], and that the unrefined
    product is within 1 ulp.  Checked exactly with rationals."""
    dq = Fraction(D)
    r = _round_f32(1 / dq)
    d32 = np.float32(D)

    def fma(a, b, c):
        return _round_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))

    miss_unrefined = 0
    for y in range(-510, 511):
        yf = np.float32(y)
        exact = _round_f32(Fraction(y) / dq)
        q = _round_f32(Fraction(y) * Fraction(float(r)))
        e = fma(-q, d32, yf)
        assert fma(e, r, q) == exact, y
        if q != exact:
            miss_unrefined += 1
            assert abs(int(q.view(np.int32)) - int(exact.view(np.int32))) == 1
    assert 0 < miss_unrefined < 1021


# ------------------------------------------------------------------ bitstream

def test_state_worked_examples(oracle_mod):
    """Hand-derived window states (header comment + trellis_state)."""
    rows = _rows("state_examples.txt")
    assert len(rows) >= 14
    for row in rows:
        T, k, L, t = map(int, row[:4])
        want = int(row[4], 16)
        words = np.array([int(w, 16) for w in row[5:]], dtype=np.uint32)
        assert oracle_mod.state(words, T, k, L, t) == want, row


def _rot_state(words, T, k, L, t):
    """Independent formulation: the block as one integer, rotated right."""
    n = T * k
    B_ = 0
    for i, w in enumerate(words):
        B_ |= int(w) << (32 * i)
    off = (T - 1 - t) * k
    rot = ((B_ >> off) | (B_ << (n - off))) & ((1 << n) - 1)
    return rot & ((1 << L) - 1)


@pytest.mark.parametrize("T,k", [(8, 4), (16, 2), (32, 1), (32, 3), (32, 4), (64, 2), (256, 2), (256, 3)])
def test_state_matches_block_rotation(oracle_mod, T, k):
    rng = np.random.default_rng(T * 10 + k)
    wpb = T * k // 32
    for L in sorted({k, min(8, T * k), min(12, T * k), min(16, T * k), min(24, T * k)}):
        for _ in range(6):
            words = rng.integers(0, 1 << 32, size=wpb, dtype=np.uint64).astype(np.uint32)
            for t in range(T):
                assert oracle_mod.state(words, T, k, L, t) == _rot_state(words, T, k, L, t)


@pytest.mark.parametrize("T,k,L", [(16, 2, 6), (256, 2, 16), (256, 3, 16), (256, 4, 16), (32, 4, 12)])
def test_state_one_hot_bits(oracle_mod, T, k, L):
    """Brute force: with only bit j set, state_t has bit i set exactly when
    (T-1-t)*k + i == j modulo T*k."""
    wpb = T * k // 32
    for j in range(0, T * k, max(1, T * k // 97)):
        words = np.zeros(wpb, dtype=np.uint32)
        words[j // 32] = np.uint32(1 << (j % 32))
        for t in range(T):
            s = oracle_mod.state(words, T, k, L, t)
            for i in range(L):
                want = ((T - 1 - t) * k + i) % (T * k) == j
                assert bool((s >> i) & 1) == want


@pytest.mark.parametrize("k", [2, 3, 4])
def test_shift_register_and_tail_biting(oracle_mod, k):
    """Trellis invariants: state_{t+1} >> k equals the low L-k bits of state_t,
    and the same holds from state_{T-1} to state_0 (the path is a closed cycle)."""
    T, L = 256, 16
    rng = np.random.default_rng(k)
    words = rng.integers(0, 1 << 32, size=T * k // 32, dtype=np.uint64).astype(np.uint32)
    st = [oracle_mod.state(words, T, k, L, t) for t in range(T)]
    mask = (1 << (L - k)) - 1
    for t in range(T - 1):
        assert st[t + 1] >> k == st[t] & mask
    assert st[0] >> k == st[T - 1] & mask


def test_geometry_rules(oracle_mod):
    assert oracle_mod.geom_check(2, 16, 256, 4, 512) == 0
    assert oracle_mod.geom_check(2, 16, 256, 4, 500) != 0   # cols not whole blocks
    assert oracle_mod.geom_check(3, 16, 16, 4, 512) != 0    # T*k not whole words
    assert oracle_mod.geom_check(2, 0, 256, 4, 512) != 0
    assert oracle_mod.geom_check(2, 16, 256, 0, 512) != 0


def test_split_reciprocal_is_correctly_rounded():
    """y/d as fma(y, r_hi, y * r_lo), with r_hi the fp32 nearest to 1/d and
    r_lo the fp32 nearest to (1/d in double) - r_hi, is the correctly rounded
    quotient for every reachable y (the value step of trellis_val).  Exact
    rational arithmetic; the constants are formed as a C++ compiler forms them."""
    dq = Fraction(D)
    r_hi = np.float32(1.0) / np.float32(D)
    r_lo = np.float32(1.0 / D - float(r_hi))
    assert r_hi == _round_f32(1 / dq)
    for y in range(-510, 511):
        t = _round_f32(Fraction(y) * Fraction(float(r_lo)))
        v = _round_f32(Fraction(y) * Fraction(float(r_hi)) + Fraction(float(t)))
        assert v == _round_f32(Fraction(y) / dq), y
