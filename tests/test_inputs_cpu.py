"""The seeded input generators shared by the tests, the bench and the smoke
check (trellis_coded_weight_gb300/inputs.py), pinned on the CPU.

They hold no trellis arithmetic. What matters is that they are the published
generator, deterministic per seed, and produce the value distributions and
storage roundings that the input recipe states."""
import numpy as np
import torch

from trellis_coded_weight_gb300 import inputs


def test_splitmix64_reference_stream():
    # the first outputs of SplitMix64 from state 0 (Steele, Lea & Flood; the reference splitmix64.c)
    got = [int(v) for v in inputs.splitmix64(0, 4)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]


def test_streams_are_deterministic_and_keyed():
    a = inputs.random_words(1001, (64, 80))
    assert np.array_equal(a, inputs.random_words(1001, (64, 80)))
    assert not np.array_equal(a, inputs.random_words(1002, (64, 80)))
    assert a.dtype == np.uint32 and a.flags["C_CONTIGUOUS"]
    # a prefix of a stream does not depend on how much of it is drawn
    assert np.array_equal(inputs.splitmix64(7, 10), inputs.splitmix64(7, 1000)[:10])


def test_code_words_are_uniform_bits():
    w = inputs.random_words(1001, (1000, 1000))
    bits = np.unpackbits(w.view(np.uint8))
    assert abs(bits.mean() - 0.5) < 1e-3
    # every bit position of the words is balanced, not just the total
    per_bit = np.array([((w >> np.uint32(b)) & np.uint32(1)).mean() for b in range(32)])
    assert np.all(np.abs(per_bit - 0.5) < 3e-3)


def test_uniform01_range():
    u = inputs.uniform01(5, 200000)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 3e-3 and abs(u.var() - 1.0 / 12.0) < 2e-3


def test_scales_are_fp16_of_the_stated_range():
    s = inputs.uniform_f16(2001, (100000,))
    assert s.dtype == np.uint16
    f = s.view(np.float16).astype(np.float64)
    lo, hi = float(np.float16(0.005)), float(np.float16(0.02))
    assert f.min() >= lo and f.max() <= hi
    assert abs(f.mean() - 0.0125) < 1e-4
    # stored values are fp16 roundings of doubles in the range: re-rounding is the identity
    assert np.array_equal(f.astype(np.float16).view(np.uint16), s)


def test_x_is_rne_bf16_of_normal_draws():
    for sigma in (1.0, 0.5):
        x = inputs.normal_bf16(3001, (8, 50000), sigma)
        assert x.dtype == np.uint16
        f = inputs.bf16_bits_to_f32(x).astype(np.float64)
        assert np.all(np.isfinite(f))
        assert abs(f.mean()) < 0.01 * sigma and abs(f.std() / sigma - 1.0) < 0.01
        # the stored bits are the round-to-nearest-even bf16 of an fp32 value: torch's own conversion of
        # the decoded value gives the same bits back
        t = torch.from_numpy(f.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(t, x)


def test_make_linear_shapes():
    codes, scales, x = inputs.make_linear(33, 768, 3, 4)
    assert codes.shape == (33, 768 * 3 // 32) and codes.dtype == np.uint32
    assert scales.shape == (33,) and x.shape == (4, 768)
    _, _, x0 = inputs.make_linear(40, 512, 2, 2, sigma=0.5, x_len=40)
    assert x0.shape == (2, 40)
