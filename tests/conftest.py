import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Per parity check: outputs compared, how many sit more than one bf16 ulp
    from bf16(ref) (allowed only where the fp32 band is wider than an ulp),
    and the largest distance."""
    try:
        from util import BAND_STATS
    except Exception:
        return
    if not BAND_STATS:
        return
    tr = terminalreporter
    tr.section("bf16 distance from bf16(ref) per parity check")
    total = sum(n for _, n, _, _ in BAND_STATS)
    over = sum(o for _, _, o, _ in BAND_STATS)
    worst = max(m for _, _, _, m in BAND_STATS)
    tr.write_line(f"{len(BAND_STATS)} checks, {total} outputs, {over} more than 1 ulp away, largest {worst} ulp")
    for what, n, o, m in BAND_STATS:
        if o or m > 1:
            tr.write_line(f"  {what}: {o} of {n} outputs more than 1 ulp away, largest {m} ulp")
