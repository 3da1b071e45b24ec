"""Pins for the oracle's number formats (CPU only).

What pins what:
  * E2M1 decode: the 16 nibbles against the E2M1 grid {0, 0.5, 1, 1.5, 2, 3,
    4, 6} with a sign bit ("Quantising the KV cache", section "FP4 with a
    fine-grained scale": E2M1 elements).
  * E4M3 decode: all 256 bytes against torch.float8_e4m3fn (a library routine)
    plus the closed-form landmarks 448 = 0x7E and 2^-9 = 0x01 that the
    quantiser of section "Code" relies on (saturation, min_sub).
  * Encoders: the direct encoders against brute-force nearest search on every
    bf16 bit pattern; the E4M3 encoder against torch's fp32 -> float8_e4m3fn
    cast; the E2M1 encoder against an exact threshold formulation; the tie
    and saturation points by hand.
"""
import math
import warnings

import numpy as np
import pytest
import torch

import oracle

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


warnings.filterwarnings("ignore", message="overflow encountered", category=RuntimeWarning)


def all_bf16_as_f32() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32) << 16
    return bits.view(np.float32)


def e2m1_code_by_thresholds(absv: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Exact RNE onto the E2M1 grid (times s), saturating: count the rounding
    midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 that |v| passes; at a
    midpoint the even code wins (0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2,
    2.5->2, 3.5->4, 5->4).  Products tau*s are exact in float64."""
    absv = absv.astype(np.float64)
    s = np.asarray(s, dtype=np.float64)
    c = ((absv > 0.25 * s).astype(np.int32) + (absv >= 0.75 * s) + (absv > 1.25 * s)
         + (absv >= 1.75 * s) + (absv > 2.5 * s) + (absv >= 3.5 * s) + (absv > 5.0 * s))
    return c.astype(np.uint8)


def test_e2m1_grid():
    for nib in range(16):
        mag = E2M1_GRID[nib & 7]
        want = -mag if nib & 8 else mag
        got = oracle.e2m1_value(nib)
        assert got == want and math.copysign(1.0, got) == (-1.0 if nib & 8 else 1.0)


def test_e4m3_decode_all_bytes_vs_torch():
    lib_vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for b in range(256):
        got = oracle.e4m3_value(b)
        want = float(lib_vals[b])
        if math.isnan(want):
            assert math.isnan(got), b
        else:
            assert got == want, (b, got, want)
            assert math.copysign(1.0, got) == math.copysign(1.0, want)


def test_e4m3_landmarks():
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x38) == 1.0
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    finite_pos = [oracle.e4m3_value(b) for b in range(1, 0x7F)]
    assert len(finite_pos) == 126 and all(a < b for a, b in zip(finite_pos, finite_pos[1:]))


@pytest.mark.parametrize("enc", ["e2m1", "e4m3"])
def test_direct_encoder_equals_brute_force_on_all_bf16(enc):
    x = all_bf16_as_f32()
    f = oracle.e2m1_encode if enc == "e2m1" else oracle.e4m3_encode
    direct = f(x)
    brute = f(x, brute=True)
    finite = np.isfinite(x)
    assert np.array_equal(direct[finite], brute[finite])
    # scaled copies exercise other binades of the E2M1 grid
    if enc == "e2m1":
        for scale in (0.5, 0.75, 1.5, 3.0):
            y = (x[finite] * np.float32(scale)).astype(np.float32)
            y = y[np.isfinite(y)]
            assert np.array_equal(f(y), f(y, brute=True))


def test_direct_encoder_equals_brute_force_on_random_fp32():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    y = bits.view(np.float32)
    y = y[np.isfinite(y)]
    for scale in (1.0, 2.0 ** -120, 2.0 ** -100):  # pull values into both grids' range
        z = (y * np.float32(scale)).astype(np.float32)
        z = z[np.isfinite(z)]
        assert np.array_equal(oracle.e2m1_encode(z), oracle.e2m1_encode(z, brute=True))
        assert np.array_equal(oracle.e4m3_encode(z), oracle.e4m3_encode(z, brute=True))


def test_e4m3_encoder_vs_torch_cast():
    x = all_bf16_as_f32()
    x = x[np.isfinite(x) & (np.abs(x) <= 448.0)]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x)
    assert np.array_equal(got, want)
    # random fp32 inside the finite range, including the subnormal binade
    rng = np.random.default_rng(2)
    y = np.concatenate([rng.uniform(-448, 448, 100_000), rng.uniform(-2 ** -5, 2 ** -5, 100_000)])
    y = y.astype(np.float32)
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(y), want)


def test_e4m3_saturation_and_specials():
    enc = oracle.e4m3_encode
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, np.inf], np.float32)
    assert np.all(enc(big) == 0x7E)
    assert np.all(enc(-big) == 0xFE)
    assert enc(np.array([np.nan], np.float32))[0] == 0x7F
    assert enc(np.array([0.0], np.float32))[0] == 0x00
    assert enc(np.array([-0.0], np.float32))[0] == 0x80
    # half of the min subnormal is a tie between 0 (even) and 2^-9 (odd): -> 0
    assert enc(np.array([2.0 ** -10], np.float32))[0] == 0x00
    assert enc(np.array([3 * 2.0 ** -10], np.float32))[0] == 0x02  # tie 1 vs 2 -> 2


def test_e2m1_ties_saturation_sign():
    enc = oracle.e2m1_encode
    cases = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             0.2499: 0, 0.2501: 1, 5.0001: 7, 6.0: 7, 6.5: 7, 100.0: 7, np.inf: 7,
             0.0: 0, 1.0: 2, 3.0: 5}
    for y, code in cases.items():
        assert enc(np.array([y], np.float32))[0] == code, y
        assert enc(np.array([-y], np.float32))[0] == (code | 8), -y
    # sign kept when the magnitude rounds to zero
    assert enc(np.array([-0.0, -0.1, -0.25], np.float32)).tolist() == [8, 8, 8]


def test_e2m1_encoder_vs_exact_thresholds():
    x = all_bf16_as_f32()
    x = x[np.isfinite(x)]
    for s in (1.0, 0.5, 2.0 ** -9, 3 * 2.0 ** -9, 448.0, 1.125, 13.0):
        y = (x / np.float32(s)).astype(np.float32)  # fp32 IEEE division
        ok = np.isfinite(y)
        got = oracle.e2m1_encode(y[ok]) & 7
        want = e2m1_code_by_thresholds(np.abs(x[ok]), s)
        assert np.array_equal(got, want), s
