"""Pins of the oracle's bit-width-sweep quantisers ("Quantising the KV cache",
results table rows INT8 / INT4 / INT2 per token and "K per channel, V per
token", section "Per token or per channel?", section "Maths": b + s/g bits
with a 16-bit scale per group).

The pages print the storage cost of these formats but not their rounding.
The reading here is symmetric absmax quantisation: s = FP16_RNE(amax / qmax),
qmax = 2^(b-1) - 1, codes RNE(x / s) clamped to +-qmax, both divisions IEEE
fp32, a zero scale replaced by the smallest FP16 subnormal.  These tests pin
that reading against numpy's float16 conversion, brute-force nearest-level
search and an explicit index loop over the groups of both layouts.
"""
import numpy as np
import pytest

import oracle
from tests.test_oracle_formats import all_bf16_as_f32


def test_fp16_value_of_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_value(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_fp16_encode_every_bf16_value_against_numpy():
    x = all_bf16_as_f32()
    x = x[np.isfinite(x)]
    got = oracle.fp16_encode(x)
    inrange = np.abs(x) < 65520.0  # numpy rounds these to a finite value
    want = x[inrange].astype(np.float16).view(np.uint16)
    assert np.array_equal(got[inrange], want)
    # beyond: saturate to +-65504 (reading), keeping the sign
    sat = got[~inrange]
    assert np.all((sat & 0x7FFF) == 0x7BFF)
    assert np.array_equal(sat >> 15, (x[~inrange] < 0).astype(np.uint16))


def test_fp16_encode_random_fp32_against_numpy():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(400_000) * np.exp2(rng.integers(-30, 16, 400_000))).astype(np.float32)
    x = x[np.abs(x) < 65520.0]
    assert np.array_equal(oracle.fp16_encode(x), x.astype(np.float16).view(np.uint16))


def test_fp16_encode_ties_and_specials():
    # ties at the subnormal spacing 2^-24 and at 1 + 2^-11 go to the even pattern
    x = np.array([2.0 ** -25, 3 * 2.0 ** -25, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 65519.0, 65520.0, -0.0],
                 np.float32)
    assert [int(v) for v in oracle.fp16_encode(x)] == [0x0000, 0x0002, 0x3C00, 0x3C02, 0x7BFF, 0x7BFF, 0x8000]
    assert int(oracle.fp16_encode(np.array([np.nan], np.float32))[0]) == 0x7E00
    # infinities saturate like every other magnitude above 65504
    assert [int(v) for v in oracle.fp16_encode(np.array([np.inf, -np.inf, 3.0e38], np.float32))] == \
        [0x7BFF, 0xFBFF, 0x7BFF]
    codes, sb, bad = oracle.int_quantize_group(np.array([np.inf, 1.0, -2.0], np.float32), 4)
    assert sb == 0x7BFF and bad == 1 and codes.tolist() == [7, 0, 0]


def _brute_codes(x: np.ndarray, s: float, qmax: int) -> np.ndarray:
    """Nearest integer level of the fp32 quotient x / s among -qmax..qmax,
    ties to the even level (searched, not rounded)."""
    y = (x.astype(np.float32) / np.float32(s)).astype(np.float64)
    levels = np.arange(-qmax, qmax + 1, dtype=np.float64)
    dist = np.abs(y[:, None] - levels[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = np.where(dist == best, levels[None, :], np.nan)
    even = np.where(np.mod(cand, 2) == 0, cand, np.nan)
    with np.errstate(invalid="ignore"):
        lo = np.nanmin(cand, axis=1)  # the nearest level when it is unique
        pick = np.where(np.isnan(even).all(axis=1), lo, np.nanmax(np.where(np.isnan(even), -np.inf, even), axis=1))
    return pick.astype(np.int64)


@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_int_group_against_brute_force(bits):
    qmax = (1 << (bits - 1)) - 1
    rng = np.random.default_rng(bits)
    for trial in range(300):
        n = int(rng.integers(1, 40))
        x = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 12))).astype(np.float32)
        if trial % 7 == 0:  # put values exactly on rounding midpoints of the level grid
            codes, sb, _ = oracle.int_quantize_group(x, bits)
            s = oracle.fp16_value(sb)
            x[: n // 2] = (np.float32(s) * (rng.integers(-qmax, qmax, n // 2) + 0.5)).astype(np.float32)
        x = x.astype(np.float32)
        codes, sb, bad = oracle.int_quantize_group(x, bits)
        assert bad == 0
        amax = np.float32(np.abs(x).max())
        want_sb = int((amax / np.float32(qmax)).astype(np.float16).view(np.uint16)) if amax > 0 else 0
        if want_sb & 0x7FFF == 0:
            want_sb = 1
        assert sb == want_sb
        assert np.array_equal(codes.astype(np.int64), _brute_codes(x, oracle.fp16_value(sb), qmax))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_int_group_error_bound_and_extremes(bits):
    qmax = (1 << (bits - 1)) - 1
    x = np.random.default_rng(11).standard_normal((500, 16)).astype(np.float32)
    for row in x:
        codes, sb, _ = oracle.int_quantize_group(row, bits)
        s = oracle.fp16_value(sb)
        err = np.abs(codes * s - row.astype(np.float64))
        inside = np.abs(row) <= qmax * s
        assert np.all(err[inside] <= s / 2 + 1e-12)
        assert np.all(np.abs(codes) <= qmax)
        assert np.abs(codes).max() >= qmax - 1  # the amax lands on (or next to) the top level
    codes, sb, _ = oracle.int_quantize_group(np.zeros(8, np.float32), bits)
    assert sb == 1 and not codes.any()
    codes, sb, _ = oracle.int_quantize_group(np.array([0.0, -0.0, 1e-30], np.float32), bits)
    assert sb == 1 and not codes.any()


@pytest.mark.parametrize("per", ["token", "channel"])
def test_int_layouts_are_groups_of_the_right_axis(per):
    rng = np.random.default_rng(2)
    B, T, H, d = 2, 9, 3, 16
    x = rng.standard_normal((B, T, H, d)).astype(np.float32)
    x[:, :, :, 5] *= 40  # an outlier channel: visible in every per-token scale, only its own per-channel scale
    codes, scales, bad = oracle.int_quantize(x, 4, per)
    assert bad == 0
    for b in range(B):
        for h in range(H):
            if per == "token":
                for t in range(T):
                    c, sb, _ = oracle.int_quantize_group(x[b, t, h], 4)
                    assert sb == scales[b, t, h] and np.array_equal(c, codes[b, t, h])
            else:
                for ch in range(d):
                    c, sb, _ = oracle.int_quantize_group(x[b, :, h, ch], 4)
                    assert sb == scales[b, h, ch] and np.array_equal(c, codes[b, :, h, ch])
    xh = oracle.int_dequantize(codes, scales, per)
    assert xh.shape == x.shape
    if per == "token":
        assert np.allclose(xh[1, 4, 2], codes[1, 4, 2] * oracle.fp16_value(scales[1, 4, 2]))
    else:
        assert np.allclose(xh[1, :, 2, 7], codes[1, :, 2, 7] * oracle.fp16_value(scales[1, 2, 7]))


def test_outlier_channel_destroys_per_token_groups_not_per_channel():
    """The "DEBUG: an outlier channel destroying a group" case of the week's
    plan: one channel 100x larger sets the scale of every per-token group it
    joins, so at 4 bits the other channels mostly round to 0; per-channel
    scales leave them intact."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 64, 1, 32)).astype(np.float32)
    x[..., 3] *= 100
    others = np.delete(np.arange(32), 3)
    rel = {}
    for per in ("token", "channel"):
        codes, scales, _ = oracle.int_quantize(x, 4, per)
        xh = oracle.int_dequantize(codes, scales, per)
        rel[per] = np.abs(xh[..., others] - x[..., others]).mean() / np.abs(x[..., others]).mean()
    assert rel["token"] > 0.7
    assert rel["channel"] < 0.2


def test_bits_per_number_of_the_sweep_layouts():
    """b + s/g with a 16-bit scale: per token over a head of d channels, per
    channel over T tokens (the table's 10 / 6 / 4 at d = 8)."""
    def bits(b, g):
        return b + 16.0 / g
    assert [bits(8, 8), bits(4, 8), bits(2, 8)] == [10.0, 6.0, 4.0]
    assert bits(4, 128) == 4.125 and bits(2, 4096) == pytest.approx(2.00390625)
