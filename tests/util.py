"""Shared helpers of the parity tests (no method arithmetic: conversions and
the tolerance rule).

Tolerance rule (matching rules of the measured path): a matvec or GEMM
output accumulated in fp32 must satisfy |gpu - ref| <= 1e-5 * sum|w*x| + 1e-6
before its final bf16 cast.  Only the bf16 result is observable, so the test
accepts exactly the bf16 values that a correctly rounded cast of some value in
[ref - tol, ref + tol] can give: every bf16 between bf16(ref - tol) and
bf16(ref + tol).  That is also the reading of "stored bf16 outputs within one
bf16 ulp": the output is the correct rounding of a value the fp32 rule allows.
Where the band is narrower than one ulp this is within one ulp of bf16(ref);
where cancellation makes the result small against sum|w*x| the band spans
several bf16 ulps and the check is the band itself.
"""
from __future__ import annotations

import numpy as np
import torch

from trellis_coded_weight_gb300 import inputs

REL_TOL = 1e-5
ABS_TOL = 1e-6

# One entry per check_band call: (what, outputs, outputs more than one bf16
# ulp from bf16(ref), largest distance in ulps).  The session's terminal
# summary prints them (tests/conftest.py).
BAND_STATS: list = []


def to_dev_u32(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)


def to_dev_bf16(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def to_dev_f16(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.float16).to(dev)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_of_f64(oracle, v: np.ndarray) -> np.ndarray:
    """Single-rounding double -> bf16 bits (the oracle's routine)."""
    return oracle.bf16_rne_f64_many(np.asarray(v, dtype=np.float64))


def _ordered(bits: np.ndarray) -> np.ndarray:
    """Map bf16 bit patterns to integers that order like their values."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def _bits_of_ordered(o: np.ndarray) -> np.ndarray:
    """Inverse of _ordered (zero maps to +0)."""
    o = np.asarray(o).astype(np.int32)
    return np.where(o < 0, (-o) | 0x8000, o).astype(np.uint16)


def check_band(oracle, gpu_bits: np.ndarray, ref: np.ndarray, absum: np.ndarray, what: str = ""):
    """Assert the tolerance rule for every element; return the max |ulp| distance."""
    gpu_bits = np.asarray(gpu_bits, dtype=np.uint16)
    tol = REL_TOL * absum + ABS_TOL
    lo = _ordered(bf16_of_f64(oracle, ref - tol))
    hi = _ordered(bf16_of_f64(oracle, ref + tol))
    mid = _ordered(bf16_of_f64(oracle, ref))
    g = _ordered(gpu_bits)
    bad = (g < lo) | (g > hi)
    if bad.any():
        i = np.flatnonzero(bad.reshape(-1))[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs outside the tolerance band; first at {i}: "
            f"gpu={inputs.bf16_bits_to_f32(gpu_bits.reshape(-1)[i])} ref={ref.reshape(-1)[i]} "
            f"tol={tol.reshape(-1)[i]}")
    ulps = np.abs(g - mid)
    allowed = np.maximum(1, np.maximum(hi - mid, mid - lo))
    assert np.all(ulps <= allowed), f"{what}: output farther from bf16(ref) than the band allows"
    BAND_STATS.append((what, int(ulps.size), int((ulps > 1).sum()), int(ulps.max()) if ulps.size else 0))
    return int(ulps.max()) if ulps.size else 0
