"""Pins of the oracle's FP8 E4M3 weight codec (CPU only).

The library pin is PyTorch's own float32 -> float8_e4m3fn cast (round to
nearest even; it returns NaN instead of saturating above the largest finite
value, so saturation is pinned by hand)."""
import numpy as np
import pytest
import torch

import oracle as O


def torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_decode_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])
    assert O.e4m3_decode(np.uint8(0x7E)) == 448.0 and O.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9


def test_encode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = O.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(O.e4m3_encode(vals), codes)        # includes -0 -> 0x80


def test_encode_matches_torch_random_and_ties():
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.normal(size=20000).astype(np.float32) * np.float32(60.0),
        rng.uniform(-2.0 ** -5, 2.0 ** -5, size=5000).astype(np.float32),   # subnormal range
        rng.uniform(-463.0, 463.0, size=5000).astype(np.float32)])
    # exact midpoints between neighbouring codes (ties go to the even code)
    finite = O.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    assert np.array_equal(O.e4m3_encode(v), torch_e4m3(v))


def test_encode_saturates():
    v = np.array([448.0, 463.9, 464.0, 1e6, -500.0, np.float32(3.4e38)], dtype=np.float32)
    assert list(O.e4m3_encode(v)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E]


def test_quantize_scale_and_error_bound():
    rng = np.random.default_rng(12)
    w = (rng.normal(size=(64, 48)) * 0.02).astype(np.float32)
    q, s = O.quantize_fp8(w)
    assert s == np.float32(np.float32(np.abs(w).max()) / np.float32(448.0))
    # the largest element maps to 448 (code 0x7E or 0xFE)
    i = np.unravel_index(np.argmax(np.abs(w)), w.shape)
    assert q[i] & 0x7F == 0x7E
    # round to nearest: error at most half a step of the value's binade (relative
    # 2^-4 for normals; 2^-10 * scale absolute in the subnormal range)
    deq = O.dequantize_fp8(q, s)
    a = np.abs(w.astype(np.float64)) / float(s)
    step = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3))
    assert np.all(np.abs(deq - w) <= 0.5 * step * float(s) * (1 + 1e-6))


def test_quantize_zero_and_hand_case():
    q, s = O.quantize_fp8(np.zeros((3, 4), np.float32))
    assert s == 1.0 and not q.any()
    # amax 7 -> scale 7/448 = 1/64; 3.5 -> 224 = 1.75*2^7 (code 0x76), -0.0078125 -> -0.5 (0xB0)
    w = np.array([[7.0, 3.5, -0.0078125, 0.0]], np.float32)
    q, s = O.quantize_fp8(w)
    assert s == np.float32(1 / 64)
    assert list(q[0]) == [0x7E, 0x76, 0xB0, 0x00]
    assert np.array_equal(O.dequantize_fp8(q, s), w.astype(np.float64))
