"""Every entry point on every visible GPU of one process.

Kernel attributes (the dynamic shared-memory limit of the axis-0 and prefill
kernels) and occupancy figures are per device, so the library sets them up
once per device.  This test switches the current device and runs each call
on a small problem there, checked against the oracle.  With one visible GPU
it is skipped."""
import numpy as np
import pytest
import torch

from trellis_coded_weight_gb300 import binding as tb
from trellis_coded_weight_gb300 import inputs
from util import bf16_bits, check_band, to_dev_bf16, to_dev_f16, to_dev_u32

pytestmark = pytest.mark.gpu
L, T = 16, 256


@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs two or more visible GPUs")
def test_every_entry_point_on_every_device(oracle_mod):
    from trellis_coded_weight_gb300 import build
    build.build()
    tb.load()
    rows, cols, k = 96, 768, 2
    codes, scales, x = inputs.make_linear(rows, cols, k, 2, seed_codes=901, seed_x=902)
    x0 = inputs.normal_bf16(903, (2, rows), 0.5)
    xp = inputs.normal_bf16(904, (40, cols))
    x0p = inputs.normal_bf16(905, (24, rows), 0.5)
    g1, g0 = tb.Geometry(k, L, T, 1, rows, cols), tb.Geometry(k, L, T, 0, rows, cols)
    want_e = oracle_mod.expand_bf16(codes, scales, k, L, T)
    r1, a1 = oracle_mod.matvec_axis1(codes, scales, x, k, L, T)
    r0, a0 = oracle_mod.matvec_axis0(codes, scales, x0, k, L, T)
    rp, ap = oracle_mod.prefill(codes, scales, xp, k, L, T)
    rp0, ap0 = oracle_mod.matvec_axis0_bf16w(codes, scales, x0p, k, L, T)
    sums = oracle_mod.gateup_sums(codes, scales, codes, scales, x, k, L, T)
    from test_parity_gpu import check_gateup
    for d in range(torch.cuda.device_count()):
        dev = torch.device("cuda", d)
        with torch.cuda.device(dev):
            dc, ds = to_dev_u32(codes, dev), to_dev_f16(scales, dev)
            assert np.array_equal(bf16_bits(tb.expand_bf16(dc, ds, g1)), want_e)
            check_band(oracle_mod, bf16_bits(tb.matvec_axis1(dc, ds, to_dev_bf16(x, dev), g1)), r1, a1, f"axis1 dev{d}")
            ws = tb.new_workspace(2, g0, dev)
            check_band(oracle_mod, bf16_bits(tb.matvec_axis0(dc, ds, to_dev_bf16(x0, dev), g0, ws)), r0, a0,
                       f"axis0 dev{d}")
            check_gateup(oracle_mod, bf16_bits(tb.gateup_swiglu(dc, ds, dc, ds, to_dev_bf16(x, dev), g1)), *sums,
                         f"gateup dev{d}")
            check_band(oracle_mod, bf16_bits(tb.gemm_prefill(dc, ds, to_dev_bf16(xp, dev), g1)), rp, ap,
                       f"prefill dev{d}")
            check_band(oracle_mod, bf16_bits(tb.gemm_prefill(dc, ds, to_dev_bf16(x0p, dev), g0)), rp0, ap0,
                       f"prefill axis0 dev{d}")
            torch.cuda.synchronize(dev)
            assert tb.device_error(reset=True) == 0
