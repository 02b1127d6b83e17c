"""Pins for the oracle's fp8 e4m3 encode/decode and per-row quantisation.

The oracle's e4m3 arithmetic is written from the OCP 8-bit floating point
format definition.  It is pinned here against things that are not itself:
PyTorch's float8_e4m3fn conversion (an independent library implementation of
the same format, round-to-nearest-even), hand-checked code points, and
properties of the per-token quantisation that the 132-byte fp8 record of
"The Pivot: A Single Edit That Finally Fixed DeepSeek V4's Long-Context Recall
Failure" (section "Assumptions and Input Knowledge") implies: 128 one-byte
codes plus one fp32 scale, the largest element mapping to the format's largest
finite value.
"""
import numpy as np
import pytest
import torch

import oracle


def torch_encode(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_decode(c: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(c, np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float32).numpy()


def test_decode_all_codes_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_decode_code_points():
    # largest finite, one, smallest normal, smallest subnormal, signed zero
    pts = {0x7E: 448.0, 0x38: 1.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9,
           0x07: 7 * 2.0 ** -9, 0x77: 240.0, 0x00: 0.0}
    for c, v in pts.items():
        assert oracle.e4m3_decode(np.array([c], np.uint8))[0] == v
        assert oracle.e4m3_decode(np.array([c | 0x80], np.uint8))[0] == -v
    neg0 = oracle.e4m3_decode(np.array([0x80], np.uint8))[0]
    assert np.signbit(neg0)
    # monotone over the non-negative finite codes
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(vals) > 0)


def test_encode_code_points():
    cases = [(448.0, 0x7E), (240.0, 0x77), (2.0 ** -9, 0x01), (2.0 ** -10, 0x00),
             (3 * 2.0 ** -10, 0x02), (-0.0, 0x80), (0.0, 0x00), (1.0, 0x38),
             (1.0625, 0x38),     # halfway 1 and 1.125: ties to even mantissa 0
             (1.1875, 0x3A),     # halfway 1.125 and 1.25: ties to even mantissa 2
             (460.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE),  # saturation
             (float("inf"), 0x7E), (float("-inf"), 0xFE), (float("nan"), 0x7F),
             (-2.0 ** -11, 0x80)]  # negative value rounding to zero keeps the sign
    x = np.array([c[0] for c in cases], np.float32)
    got = oracle.e4m3_encode(x)
    for (v, want), g in zip(cases, got):
        assert g == want, (v, hex(g), hex(want))


@pytest.mark.slow
def test_encode_exhaustive_positive_against_torch():
    # Every non-negative fp32 bit pattern below the saturation threshold 464
    # (torch's conversion and the format agree there; above it the
    # saturating rule is pinned separately), in chunks.
    lim = int(np.array([464.0], np.float32).view(np.uint32)[0])
    step = 1 << 26
    for lo in range(0, lim, step):
        hi = min(lo + step, lim)
        bits = np.arange(lo, hi, dtype=np.uint32)
        x = bits.view(np.float32)
        a = oracle.e4m3_encode(x)
        b = torch_encode(x)
        bad = np.nonzero(a != b)[0]
        assert bad.size == 0, (hex(int(bits[bad[0]])), a[bad[0]], b[bad[0]])


def test_encode_sign_symmetry_and_saturation():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 31, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    a = oracle.e4m3_encode(x)
    b = oracle.e4m3_encode(-x)
    assert np.array_equal(a | 0x80, b)
    big = np.abs(x) >= 464.0
    assert np.all(a[big] == 0x7E)
    small = ~big
    assert np.array_equal(a[small], torch_encode(x[small]))


def test_encode_decode_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_quant_rows_properties():
    from sparse_attention_top_idx_gb300.workloads import f32_to_bf16_bits
    rng = np.random.default_rng(3)
    x32 = rng.standard_normal((500, 128)).astype(np.float32) * rng.uniform(
        0.01, 100, (500, 1)).astype(np.float32)
    xb = f32_to_bf16_bits(x32)
    codes, scales = oracle.quantize_rows(xb)
    xf = oracle.bf16_to_f32(xb)
    amax = np.abs(xf).max(axis=1)
    # the scale is the one IEEE fp32 division amax / 448
    assert np.array_equal(scales, (amax / np.float32(448.0)).astype(np.float32))
    # the largest-magnitude element maps to +-448
    j = np.abs(xf).argmax(axis=1)
    top = codes[np.arange(500), j]
    assert np.all((top & 0x7F) == 0x7E)
    assert np.array_equal(top >> 7, (xf[np.arange(500), j] < 0).astype(np.uint8))
    # each code is the RNE e4m3 of x / scale (torch as the independent encoder)
    y = (xf / scales[:, None]).astype(np.float32)
    assert np.array_equal(codes, torch_encode(y))
    # dequantised values are within half an e4m3 step of the input
    deq = torch_decode(codes) * scales[:, None]
    err = np.abs(deq - xf)
    assert np.all(err <= np.maximum(np.abs(xf) * 2.0 ** -4, scales[:, None] * 2.0 ** -10) * 1.0001)


def test_quant_zero_row():
    codes, scales = oracle.quantize_rows(np.zeros((2, 128), np.uint16))
    assert np.all(codes == 0) and np.all(scales == 0)
