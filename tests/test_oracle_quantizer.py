"""Pins for the oracle's block quantiser and the FP8 window quantiser (CPU only).

The quantiser follows "Quantising the KV cache", section "Code": per block of
16 channels, s = RNE_e4m3(amax/6) saturating, s == 0 replaced by the E4M3 min
subnormal, then each value RNE_e2m1(v/s) saturating; its storage cost is
4 + 8/16 = 4.5 bits per number (section "Maths").

Pins (each chosen so a dropped term, a wrong sign, a swapped nibble or a
wrong rounding direction fails one of them):
  * every bf16 amax: the scale byte against torch's float8_e4m3fn cast of the
    fp32 quotient amax/6 (library routine), 448 saturation, zero -> 0x01;
  * every reachable (bf16 value, scale) pair: the code against the exact
    threshold formulation of RNE onto the E2M1 grid;
  * packing order (even channel in the low nibble) and the sign bit;
  * invariants: |dequant| <= 6 s, error bound, round trip of grid blocks,
    idempotence except for the one exception class, 9 bytes per 16 values;
  * fp32 division agrees with exact rational division on the code decision;
  * the FP8 window: codes against torch's float8_e4m3fn cast of x/s_h.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle
from tests.test_oracle_formats import all_bf16_as_f32, e2m1_code_by_thresholds

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def unpack_nibbles(codes: np.ndarray) -> np.ndarray:
    lo = codes & 0x0F
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))


def e4m3_bytes_to_f64(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).double().numpy()


def test_scale_byte_for_every_bf16_amax():
    x = all_bf16_as_f32()
    x = x[np.isfinite(x)]
    blocks = np.zeros((x.size, 16), np.float32)
    blocks[:, 5] = x  # position inside the block must not matter
    _, scales, bad = oracle.quantize_rows(blocks)
    assert bad == 0
    t = (np.abs(x) / np.float32(6.0)).astype(np.float32)  # fp32 IEEE division
    want = torch.from_numpy(np.minimum(t, np.float32(448.0))).to(torch.float8_e4m3fn)
    want = want.view(torch.uint8).numpy().copy()
    want[want == 0] = 0x01
    assert np.array_equal(scales[:, 0], want)
    assert scales.max() == 0x7E and scales.min() == 0x01


def test_codes_for_every_reachable_value_scale_pair():
    allv = all_bf16_as_f32()
    allv = allv[np.isfinite(allv)]
    for sb in range(1, 0x7F):
        s = oracle.e4m3_value(sb)
        a = np.float32(6.0 * s)  # exact; a/6 == s exactly
        v = allv[np.abs(allv) <= a]
        pad = (-v.size) % 15
        v = np.concatenate([v, np.zeros(pad, np.float32)])
        blocks = np.empty((v.size // 15, 16), np.float32)
        blocks[:, 0] = -a if sb % 2 else a  # amax carrier, either sign
        blocks[:, 1:] = v.reshape(-1, 15)
        codes, scales, _ = oracle.quantize_rows(blocks)
        assert np.all(scales == sb), sb
        nib = unpack_nibbles(codes)
        want_mag = e2m1_code_by_thresholds(np.abs(blocks), s)
        want = want_mag | (np.signbit(blocks).astype(np.uint8) << 3)
        assert np.array_equal(nib, want), sb


def test_packing_order_and_sign():
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 6.0   # code 7 in the low nibble of byte 0
    x[0, 1] = -1.0  # code 0xA in the high nibble of byte 0
    x[0, 14] = 0.5  # code 1, low nibble of byte 7
    x[0, 15] = -0.0  # sign kept: 0x8, high nibble of byte 7
    codes, scales, _ = oracle.quantize_rows(x)
    assert scales[0, 0] == 0x38  # amax 6 -> s = 1.0
    assert codes[0, 0] == 0xA7
    assert codes[0, 7] == 0x81
    assert np.all(codes[0, 1:7] == 0)


def test_zero_blocks_use_min_subnormal_scale():
    codes, scales, _ = oracle.quantize_rows(np.zeros((2, 32), np.float32))
    assert np.all(scales == 0x01) and np.all(codes == 0)
    codes, scales, _ = oracle.quantize_rows(np.full((1, 16), -0.0, np.float32))
    assert scales[0, 0] == 0x01 and np.all(codes == 0x88)
    # a block whose amax/6 rounds to zero also gets 0x01
    codes, scales, _ = oracle.quantize_rows(np.full((1, 16), 2.0 ** -12, np.float32))
    assert scales[0, 0] == 0x01


def _random_blocks(n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, 16, generator=g)
    x[: n // 4] *= 20.0
    x[n // 4: n // 2] *= 1e-3
    x[n // 2: 3 * n // 4] *= 3000.0  # saturating scales
    return x.to(torch.bfloat16).float().numpy()


def test_block_invariants():
    x = _random_blocks(40_000, 3)
    codes, scales, _ = oracle.quantize_rows(x)
    xh = oracle.dequantize_rows(codes, scales)
    s = e4m3_bytes_to_f64(scales[:, 0])[:, None]
    assert np.all(np.abs(xh) <= 6.0 * s)
    # dequant equals grid[code] * s with the value's sign
    nib = unpack_nibbles(codes)
    recon = np.where(nib & 8, -1.0, 1.0) * E2M1_GRID[nib & 7] * s
    assert np.array_equal(xh, recon)
    # sign of every nonzero reconstruction matches the input
    nz = xh != 0
    assert np.all(np.sign(xh[nz]) == np.sign(x[nz]))
    # error bound: half a grid step below 4*s (1 step above), or saturation
    err = np.abs(xh - x)
    ax = np.abs(x) / s
    bound = np.where(ax <= 2.0, 0.25, np.where(ax <= 4.0, 0.5, 1.0)) * s
    bound = np.maximum(bound, (np.abs(x) - 6.0 * s))
    assert np.all(err <= bound)
    # scale is RNE(amax/6) unless it rounded to zero
    amax = np.abs(x).max(axis=1)
    t = (amax / np.float32(6.0)).astype(np.float32)
    want = torch.from_numpy(np.minimum(t, np.float32(448))).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    want[want == 0] = 1
    assert np.array_equal(scales[:, 0], want)


def test_round_trip_of_grid_blocks():
    rng = np.random.default_rng(4)
    for sb in range(1, 0x7F):
        s = oracle.e4m3_value(sb)
        nib = rng.integers(0, 16, size=(64, 16)).astype(np.uint8)
        nib[:, rng.integers(0, 16)] = 7 | (8 * (sb & 1))  # one element at +-6s fixes the scale
        vals = (np.where(nib & 8, -1.0, 1.0) * E2M1_GRID[nib & 7] * s).astype(np.float32)
        codes, scales, _ = oracle.quantize_rows(vals)
        assert np.all(scales == sb)
        got = unpack_nibbles(codes)
        # zero magnitudes keep their sign bit, everything else is identical
        assert np.array_equal(got, nib)


def test_idempotence_with_single_exception_class():
    """Q(D(Q(x))) == Q(x) for every block, except blocks whose scale is
    2^-8 (byte 0x02) with amax in [9, 10] * 2^-9: there the max code 4 gives
    D = 2^-6, whose requantisation picks s = 2^-9 and code 6."""
    x = _random_blocks(20_000, 5)
    singles = all_bf16_as_f32()
    singles = singles[np.isfinite(singles)]
    sblocks = np.zeros((singles.size, 16), np.float32)
    sblocks[:, 0] = singles
    for blocks in (x, sblocks):
        c1, s1, _ = oracle.quantize_rows(blocks)
        d1 = oracle.dequantize_rows(c1, s1).astype(np.float32)  # exact in fp32
        c2, s2, _ = oracle.quantize_rows(d1)
        same = np.all(c1 == c2, axis=1) & (s1[:, 0] == s2[:, 0])
        amax = np.abs(blocks).max(axis=1)
        exception = (s1[:, 0] == 0x02) & (amax >= 9 * 2.0 ** -9) & (amax <= 10 * 2.0 ** -9)
        assert np.all(same | exception)
        assert not np.any(same[exception])
    # the exception class among single-nonzero bf16 blocks: the 17 bf16
    # magnitudes in [9, 10] * 2^-9, each with both signs
    c1, s1, _ = oracle.quantize_rows(sblocks)
    d1 = oracle.dequantize_rows(c1, s1).astype(np.float32)
    c2, s2, _ = oracle.quantize_rows(d1)
    assert int(np.sum(~(np.all(c1 == c2, axis=1) & (s1[:, 0] == s2[:, 0])))) == 34


def test_storage_is_nine_bytes_per_sixteen_values():
    codes, scales, _ = oracle.quantize_rows(np.ones((3, 128), np.float32))
    assert codes.nbytes + scales.nbytes == 3 * 128 // 16 * 9
    bits_per_number = 8 * (codes.nbytes + scales.nbytes) / (3 * 128)
    assert bits_per_number == 4.5


def test_fp32_division_matches_exact_division_on_the_code():
    rng = np.random.default_rng(6)
    allv = all_bf16_as_f32()
    allv = allv[np.isfinite(allv)]
    for _ in range(3000):
        sb = int(rng.integers(1, 0x7F))
        s = oracle.e4m3_value(sb)
        v = float(allv[rng.integers(0, allv.size)])
        y32 = np.float32(np.float32(v) / np.float32(s))
        code32 = int(oracle.e2m1_encode(np.array([y32], np.float32))[0]) & 7
        q = abs(Fraction(v) / Fraction(s))
        dist = [abs(q - Fraction(g)) for g in E2M1_GRID]
        best = min(range(8), key=lambda c: (dist[c], c & 1))
        assert code32 == best, (v, s)


def test_nonfinite_blocks_are_counted():
    x = np.ones((3, 16), np.float32)
    x[1, 3] = np.inf
    x[2, 7] = np.nan
    _, _, bad = oracle.quantize_rows(x)
    assert bad == 2


def test_fp8_window_quantiser_vs_torch():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(4096, generator=g).to(torch.bfloat16).float().numpy()
    s = oracle.fp8_head_scale(x)
    assert s == np.float32(np.abs(x).max()) / np.float32(448.0)
    c, bad = oracle.fp8_quantize(x, s)
    assert bad == 0
    y = (x / np.float32(s)).astype(np.float32)
    want = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(c, want)
    # later values beyond the initial range saturate
    c2, _ = oracle.fp8_quantize(np.array([10 * np.abs(x).max(), -10 * np.abs(x).max()], np.float32), s)
    assert c2.tolist() == [0x7E, 0xFE]
    xh = oracle.fp8_dequantize(c, s)
    want_h = (e4m3_bytes_to_f64(c).astype(np.float32) * np.float32(s)).astype(np.float64)
    assert np.array_equal(xh, want_h)
    assert oracle.fp8_head_scale(np.zeros(8, np.float32)) == 1.0
