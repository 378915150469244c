"""The product path fails loudly and stands apart from the oracle (CPU).

- A missing library is an error, never a silent fallback.
- Every compute call refuses host tensors: there is no CPU path to fall
  back on.
- Nothing in the package imports or loads the oracle; only tests, the smoke
  check and the bench's CPU-baseline leg use it.
"""
import os
import re
import subprocess
import sys

import pytest
import torch

from trellis_coded_weight_gb300 import binding as tb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "trellis_coded_weight_gb300")


def _py(code):
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)


def test_missing_library_raises():
    r = _py("from trellis_coded_weight_gb300 import binding as tb\n"
            "try:\n"
            "    tb.load('/nonexistent/libtrellis.so')\n"
            "except RuntimeError as e:\n"
            "    print('raised', e)\n")
    assert r.returncode == 0 and r.stdout.startswith("raised"), r.stdout + r.stderr


def test_package_does_not_import_the_oracle():
    r = _py("import sys\n"
            "from trellis_coded_weight_gb300 import binding, build, inputs, shard\n"
            "print('oracle' in sys.modules)\n")
    assert r.returncode == 0 and r.stdout.strip() == "False", r.stdout + r.stderr
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "liboracle" not in text and "trellis_oracle" not in text, f


def _host(shape, dtype):
    return torch.zeros(shape, dtype=dtype)


def test_compute_calls_refuse_host_tensors():
    g1 = tb.Geometry(2, 16, 256, 1, 64, 512)
    g0 = tb.Geometry(2, 16, 256, 0, 64, 512)
    codes = _host((64, 512 * 2 // 32), torch.int32)
    scales = _host((64,), torch.float16)
    calls = [
        lambda: tb.expand_bf16(codes, scales, g1),
        lambda: tb.matvec_axis1(codes, scales, _host((2, 512), torch.bfloat16), g1),
        lambda: tb.matvec_axis1(codes, scales, _host((2, 512), torch.bfloat16), g1, bf16_weights=True),
        lambda: tb.gateup_swiglu(codes, scales, codes, scales, _host((1, 512), torch.bfloat16), g1),
        lambda: tb.gemm_prefill(codes, scales, _host((40, 512), torch.bfloat16), g1),
        lambda: tb.load_floor(codes, g1),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
    with pytest.raises(ValueError, match="CUDA tensor"):
        tb.matvec_axis0(codes, scales, _host((2, 64), torch.bfloat16), g0, _host((1 << 20,), torch.uint8))
