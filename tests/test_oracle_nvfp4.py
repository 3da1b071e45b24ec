"""Pins of the oracle's NVFP4 variant: the FP4 block quantiser ("Quantising
the KV cache", section "Code") applied to x / S with one fp32 second-level
scale S per tensor ("KV Cache Quantisation": the cache stored in FP8 or
NVFP4, scales handled at read time).  Reading: S = amax / (6 * 448), x / S
in fp32, values read back as fp32(fp32(e2m1 * e4m3) * S).

Pinned against the plain FP4 quantiser in the cases where the definitions
coincide (S = 1; S a power of two, where x / S is exact), the position of
the largest block scale, the rounding error bound, and the underflow that
the second level exists to avoid.
"""
import numpy as np

import oracle


def _x(seed, shape=(40, 128), mag=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * mag).astype(np.float32)


def test_unit_scale_is_plain_fp4():
    x = _x(0)
    c, s, _ = oracle.nvfp4_quantize_rows(x, 1.0)
    c1, s1, _ = oracle.quantize_rows(x)
    assert np.array_equal(c, c1) and np.array_equal(s, s1)
    assert np.array_equal(oracle.nvfp4_dequantize_rows(c, s, 1.0), oracle.dequantize_rows(c1, s1))


def test_power_of_two_scale_is_fp4_of_the_scaled_tensor():
    x = _x(1)
    for k in (-12, -3, 5, 20):
        S = float(2.0 ** k)
        c, s, _ = oracle.nvfp4_quantize_rows(x, S)
        c1, s1, _ = oracle.quantize_rows(x / np.float32(S))  # exact: a power of two
        assert np.array_equal(c, c1) and np.array_equal(s, s1)
        assert np.array_equal(oracle.nvfp4_dequantize_rows(c, s, S), oracle.dequantize_rows(c1, s1) * S)


def test_global_scale_puts_the_largest_block_on_the_top_e4m3_scale():
    for seed, mag in [(2, 1.0), (3, 1e-7), (4, 3e4)]:
        x = _x(seed, mag=mag)
        S = oracle.nvfp4_global_scale(x)
        assert S == np.float32(np.abs(x).max()) / np.float32(2688.0)
        _, s, _ = oracle.nvfp4_quantize_rows(x, S)
        assert s.max() == 0x7E  # 448
    assert oracle.nvfp4_global_scale(np.zeros(32, np.float32)) == 1.0


def test_rounding_error_bound():
    x = _x(5, mag=0.01)
    S = oracle.nvfp4_global_scale(x)
    c, s, _ = oracle.nvfp4_quantize_rows(x, S)
    xh = oracle.nvfp4_dequantize_rows(c, s, S)
    blk_scale = np.repeat(np.vectorize(oracle.e4m3_value)(s), 16, axis=1) * S
    # the widest E2M1 gap is 2 (between 4 and 6): half of it, times the
    # block's scale, plus the final fp32 rounding
    assert np.all(np.abs(xh - x) <= blk_scale * 1.0 * (1 + 1e-6) + 1e-30)


def test_second_level_avoids_scale_underflow():
    """Tiny values: the plain E4M3 block scale bottoms out at 2^-9 and every
    code rounds to zero; with S the blocks keep their resolution."""
    x = _x(6, mag=1e-6)
    c1, s1, _ = oracle.quantize_rows(x)
    assert np.all(s1 == 0x01) and not np.any(c1 & 0x77)
    S = oracle.nvfp4_global_scale(x)
    c, s, _ = oracle.nvfp4_quantize_rows(x, S)
    err = np.abs(oracle.nvfp4_dequantize_rows(c, s, S) - x)
    assert err.mean() < 0.12 * np.abs(x).mean()
