"""Pins of the oracle's NVFP4 decoding (oracle_e2m1_to_f64, oracle_e4m3_to_f64,
oracle_nvfp4_dequant) to the format's definition: hand-computed values, every E4M3 byte against
torch's float8_e4m3fn (a library routine), a hand-built block, and a round trip through a numpy
quantiser written here from the definition (which must also agree bit for bit with the input
generator's quantiser).  A plausible slip -- the nibbles swapped, the scale applied per row
instead of per 16 rows, an exponent bias off by one -- fails one of them."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_codes_by_hand():
    for c in range(16):
        v = oracle.e2m1_to_f64(c)
        mag = E2M1[c & 7]
        assert v == (-mag if c & 8 else mag)
        assert math.copysign(1.0, v) == (-1.0 if c & 8 else 1.0)


def test_e4m3_by_hand_and_every_byte_against_torch():
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0,
            0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for b, v in hand.items():
        assert oracle.e4m3_to_f64(b) == v
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_f64(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])


def test_dequant_of_a_hand_built_block():
    # K = 32 (two scale groups), N = 4 columns; K-major: codes [N][K/2], scales [N][K/16]
    codes = np.zeros((4, 16), np.uint8)
    codes[0, 0] = 0x7 | (0xB << 4)   # column 0: k = 0 -> +6, k = 1 -> -1.5
    codes[2, 8] = 0x2 | (0x9 << 4)   # column 2: k = 16 -> +1, k = 17 -> -0.5
    codes[3, 0] = 0x5                # column 3: k = 0 -> +3
    scales = np.zeros((4, 2), np.uint8)
    scales[0] = [0x38, 0x40]   # column 0: group 0 -> 1, group 1 -> 2
    scales[2] = [0x38, 0x3C]   # column 2: 1, 1.5
    scales[3] = [0x01, 0x38]   # column 3: 2^-9, 1
    w = oracle.nvfp4_dequant(codes, scales, 0.25)
    want = np.zeros((32, 4))
    want[0, 0] = 6 * 1 * 0.25
    want[1, 0] = -1.5 * 1 * 0.25
    want[16, 2] = 1 * 1.5 * 0.25
    want[17, 2] = -0.5 * 1.5 * 0.25
    want[0, 3] = 3 * 2.0 ** -9 * 0.25
    assert np.array_equal(w, want)


def numpy_quantize(w):
    """NVFP4 quantiser from the definition, numpy float64, for one matrix [K, N]."""
    K, N = w.shape
    amax = np.abs(w).max()
    ts = 2.0 ** math.ceil(math.log2(amax / (6 * 448))) if amax > 0 else 1.0
    e4m3 = np.array([oracle.e4m3_to_f64(b) for b in range(0x7F)])  # positive values, ascending
    codes = np.zeros((K, N), np.uint8)
    scales = np.zeros((K // 16, N), np.uint8)
    for g in range(K // 16):
        blk = w[16 * g:16 * g + 16]
        need = np.abs(blk).max(axis=0) / 6 / ts
        for n in range(N):
            b = int(np.searchsorted(e4m3, np.float32(need[n]), side="left"))  # smallest >= need
            scales[g, n] = b
            s = e4m3[b] * ts
            for r in range(16):
                v = blk[r, n] / s if s > 0 else 0.0
                a = abs(v)
                dist = [abs(a - m) for m in E2M1]
                best = min(range(8), key=lambda i: (dist[i], i % 2))  # nearest, ties to the even code
                codes[16 * g + r, n] = (best | (8 if v < 0 and best else 0))
    # K-major encoding: codes [N][K/2] (the lower k in the low nibble), scales [N][K/16]
    ct = codes.T
    return (ct[:, 0::2] | (ct[:, 1::2] << 4)).astype(np.uint8), np.ascontiguousarray(scales.T), ts


def test_round_trip_through_a_numpy_quantiser_and_the_generator_agrees():
    K, N = 64, 24
    w = synth.normal_bf16(3, synth.TAG_GATE, K * N, 0.02).reshape(K, N)
    w64 = oracle.bf16_to_f64(w)
    codes, scales, ts = numpy_quantize(w64)
    dq = oracle.nvfp4_dequant(codes, scales, ts)
    # error bound: half the widest E2M1 step (4 -> 6) times the block's scale
    s = np.repeat(np.array([[oracle.e4m3_to_f64(b) for b in row] for row in scales.T]), 16, axis=0) * ts
    assert np.all(np.abs(dq - w64) <= 1.0 * s + 1e-30)
    assert np.max(np.abs(dq - w64)) > 0
    # the block scale is rounded up: no element needed clamping at 6
    assert np.all(np.abs(w64) <= 6.0 * s)
    # the input generator's torch quantiser gives the same bits
    c2, s2, t2 = synth.nvfp4_quantize(torch.from_numpy(w.view(np.int16)).view(torch.bfloat16))
    assert np.array_equal(c2.numpy(), codes) and np.array_equal(s2.numpy(), scales) and float(t2) == ts
    # power-of-two tensor scale: the dequantised values are bf16 values (exact in the bf16 oracle)
    oracle.f64_to_bf16_exact(dq)


def test_dequant_rejects_bad_shapes():
    with pytest.raises(RuntimeError):  # K = 4 is not a multiple of the 16-weight scale block
        oracle.nvfp4_dequant(np.zeros((8, 2), np.uint8), np.zeros((8, 1), np.uint8), 1.0)
