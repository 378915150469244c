"""The decode MLP chain (gate/up SwiGLU then the axis-0 down projection) and
its CUDA-graph replay.  Each stage is checked against the oracle with the
stage's own input: hidden against the gate/up rule, out against the oracle's
axis-0 matvec of the GPU's hidden."""
import numpy as np
import pytest
import torch

from trellis_coded_weight_gb300 import binding as tb
from trellis_coded_weight_gb300 import inputs
from test_parity_gpu import check_gateup
from util import bf16_bits, check_band, to_dev_bf16, to_dev_f16, to_dev_u32

pytestmark = pytest.mark.gpu
L, T = 16, 256


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from trellis_coded_weight_gb300 import build
    build.build()
    tb.load()


def _mlp(I, H, ku, kd, M, seed=0):
    gc, gs, x = inputs.make_linear(I, H, ku, M, seed_codes=81 + seed, seed_scales=82 + seed, seed_x=83 + seed)
    uc, us, _ = inputs.make_linear(I, H, ku, M, seed_codes=84 + seed, seed_scales=85 + seed)
    dc, ds, _ = inputs.make_linear(I, H, kd, M, seed_codes=86 + seed, seed_scales=87 + seed)
    return gc, gs, uc, us, dc, ds, x


@pytest.mark.parametrize("I,H,ku,kd,M", [(96, 512, 2, 3, 1), (300, 768, 3, 2, 4), (17408, 5120, 2, 3, 2)])
def test_mlp_decode_stages(oracle_mod, I, H, ku, kd, M):
    gc, gs, uc, us, dc, ds, x = _mlp(I, H, ku, kd, M)
    g_up, g_dn = tb.Geometry(ku, L, T, 1, I, H), tb.Geometry(kd, L, T, 0, I, H)
    d = [to_dev_u32(gc), to_dev_f16(gs), to_dev_u32(uc), to_dev_f16(us), to_dev_u32(dc), to_dev_f16(ds)]
    ws = tb.new_workspace(M, g_dn, "cuda")
    hidden, out = tb.mlp_decode(*d, to_dev_bf16(x), g_up, g_dn, ws)
    hb, ob = bf16_bits(hidden), bf16_bits(out)
    rows = None if I <= 512 else np.unique(np.r_[np.arange(0, I, 997), I - 1]).astype(np.int64)
    sums = oracle_mod.gateup_sums(gc, gs, uc, us, x, ku, L, T, rows=rows)
    check_gateup(oracle_mod, hb if rows is None else hb[:, rows], *sums, "mlp hidden")
    cols = None if H <= 1024 else np.unique(np.r_[np.arange(0, H, 211), H - 1]).astype(np.int64)
    ref, ab = oracle_mod.matvec_axis0(dc, ds, hb, kd, L, T, cols=cols)
    check_band(oracle_mod, ob if cols is None else ob[:, cols], ref, ab, "mlp out")


def test_mlp_graph_replay_matches_direct_calls():
    I, H, M = 2048, 1024, 3
    gc, gs, uc, us, dc, ds, _ = _mlp(I, H, 2, 3, M, seed=5)
    g_up, g_dn = tb.Geometry(2, L, T, 1, I, H), tb.Geometry(3, L, T, 0, I, H)
    d = [to_dev_u32(gc), to_dev_f16(gs), to_dev_u32(uc), to_dev_f16(us), to_dev_u32(dc), to_dev_f16(ds)]
    graph = tb.MlpDecodeGraph(*d, g_up, g_dn, M)
    ws = tb.new_workspace(M, g_dn, "cuda")
    for step in range(3):
        xs = to_dev_bf16(inputs.normal_bf16(900 + step, (M, H)))
        graph.x.copy_(xs)
        got = graph.replay().clone()
        _, want = tb.mlp_decode(*d, xs, g_up, g_dn, ws)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
