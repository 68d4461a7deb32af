"""The seeded input generator: splitmix64 test vector, Box--Muller statistics, bf16
rounding, slicing, and (on a GPU) bit-identity of the device twin."""
import numpy as np
import pytest

import synth


def test_splitmix64_reference_output():
    # First output of splitmix64 from state 0 (Steele et al. 2014 reference generator).
    assert synth.mix64_int(0 + synth.GOLDEN) == 0xE220A8397B1DCDAF


def test_vector_mix_matches_scalar():
    z = np.arange(1, 50, dtype=np.uint64) * np.uint64(0x1234567)
    with np.errstate(over="ignore"):
        v = synth._mix64(z.copy())
    assert [int(a) for a in v] == [synth.mix64_int(int(a)) for a in z]


def test_bf16_round_to_nearest_even():
    v = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(v)
    # 1 + 2^-8 is half-way between 1 and 1 + 2^-7: ties to even -> 1.0
    assert bits[0] == 0x3F80 and bits[1] == 0x3F80
    # 1 + 3*2^-8 is half-way between 1 + 2^-7 and 1 + 2^-6: ties to even -> 1 + 2^-6
    assert bits[2] == 0x3F82
    assert synth.bf16_bits_to_f32(bits[3:4])[0] == -2.5


def test_normal_statistics_and_slicing():
    a = synth.normal_bf16(0, synth.TAG_X, 1 << 18, 1.0)
    f = synth.bf16_bits_to_f32(a).astype(np.float64)
    assert abs(f.mean()) < 0.01 and abs(f.std() - 1.0) < 0.01
    s = synth.normal_bf16(0, synth.TAG_X, 1000, 1.0, start=5000)
    assert np.array_equal(s, a[5000:6000])
    w = synth.bf16_bits_to_f32(synth.normal_bf16(3, synth.TAG_GATE, 1 << 16, 0.02)).astype(np.float64)
    assert abs(w.std() - 0.02) < 0.0005
    assert not np.array_equal(a[:100], synth.normal_bf16(1, synth.TAG_X, 100, 1.0))


def test_permutation_is_a_permutation():
    p = synth.permutation(5, 256)
    assert sorted(p.tolist()) == list(range(256))


@pytest.mark.gpu
def test_device_twin_bit_identical():
    import torch
    for seed, tag, sigma, n, start in [(0, synth.TAG_X, 1.0, 100_003, 0),
                                       (7, synth.TAG_GATE, 0.02, 65_536, 123_456_789),
                                       (101, synth.TAG_ROUTER, synth.SIGMA_ROUTER, 4096, 3)]:
        t = synth.torch_normal_bf16((n,), seed, tag, sigma, device="cuda", start=start)
        torch.cuda.synchronize()
        dev = t.cpu().view(torch.int16).numpy().view(np.uint16)
        host = synth.normal_bf16(seed, tag, n, sigma, start=start)
        assert np.array_equal(dev, host)
