"""NVFP4 caches (the FP4 layout plus one fp32 second-level scale per kv head
for K and for V; "KV Cache Quantisation": FP8 or NVFP4 with the scales
handled at read time) through the C ABI against the oracle: second-level
scales and codes bit for bit, dequantised values exactly, decode attention
within 2e-3 * max|V^|.  Magnitudes far from 1 are where the second level
matters: plain FP4 scales underflow or saturate there."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import TOL, ensure_built, gather_unit_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


BASE = workloads.WORKLOADS["gqa_outliers"]


def _build(w, T, mag, seed, split=None):
    """All sequences T long; second-level scales from every token; appended
    in one call, or first `split` tokens then one token per call."""
    B = w.batch
    ks, vs = [], []
    for b in range(B):
        k, v = workloads.sequence_kv(w, b, T, seed=seed, device="cuda")
        ks.append((k.float() * mag).to(torch.bfloat16))
        vs.append((v.float() * mag).to(torch.bfloat16))
    K, V = torch.stack(ks).contiguous(), torch.stack(vs).contiguous()
    P = w.page_size
    max_pages = -(-T // P)
    cache = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, P, B * max_pages, max_pages, nvfp4=True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.fp8_set_scales(cache, K, V, err=err)
    if split is None:
        kvq.append(cache, torch.zeros(B, dtype=torch.int32, device="cuda"), K, V, err=err)
    else:
        kvq.append(cache, torch.zeros(B, dtype=torch.int32, device="cuda"), K[:, :split].contiguous(),
                   V[:, :split].contiguous(), err=err)
        for t in range(split, T):
            kvq.append(cache, torch.full((B,), t, dtype=torch.int32, device="cuda"), K[:, t:t + 1].contiguous(),
                       V[:, t:t + 1].contiguous(), err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return cache, K, V


@pytest.mark.parametrize("mag", [1.0, 1e-6, 3e3])
@pytest.mark.parametrize("d", [64, 128])
def test_scales_codes_dequant_and_decode(mag, d):
    w = workloads.scaled(BASE, batch=3, num_kv_heads=2, num_q_heads=8, head_dim=d,
                         k_outlier_channels=(3, 17, 40) if d == 64 else (3, 17, 64, 101))
    T = 300
    cache, K, V = _build(w, T, mag, seed=d)
    Kh, Vh = K.float().cpu().numpy(), V.float().cpu().numpy()
    Sk = cache.k_gscale.cpu().numpy()
    Sv = cache.v_gscale.cpu().numpy()
    for h in range(w.num_kv_heads):
        assert Sk[h] == np.float32(oracle.nvfp4_global_scale(Kh[:, :, h]))
        assert Sv[h] == np.float32(oracle.nvfp4_global_scale(Vh[:, :, h]))
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            kc, ks, vc, vs = gather_unit_bytes(cache, None, b, h, T)
            okc, oks, _ = oracle.nvfp4_quantize_rows(Kh[b, :, h], float(Sk[h]))
            ovc, ovs, _ = oracle.nvfp4_quantize_rows(Vh[b, :, h], float(Sv[h]))
            assert np.array_equal(ks, oks) and np.array_equal(kc, okc)
            assert np.array_equal(vs, ovs) and np.array_equal(vc, ovc)
    lens = torch.full((w.batch,), T, dtype=torch.int32, device="cuda")
    kd, vd = kvq.dequant(cache, lens, T)
    kd, vd = kd.cpu().numpy(), vd.cpu().numpy()
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            okc, oks, _ = oracle.nvfp4_quantize_rows(Kh[b, :, h], float(Sk[h]))
            assert np.array_equal(kd[b, :, h].astype(np.float64), oracle.nvfp4_dequantize_rows(okc, oks, float(Sk[h])))
    q = workloads.queries(w, seed=d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    out = kvq.decode_attn(cache, lens, q, scale).cpu().numpy()
    qh = q.float().cpu().numpy()
    G = w.group
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            ref, vmax = oracle.decode_unit(qh[b, h * G:(h + 1) * G], Kh[b, :, h], Vh[b, :, h], scale,
                                           nvfp4_scales=(float(Sk[h]), float(Sv[h])))
            assert np.abs(out[b, h * G:(h + 1) * G] - ref).max() <= TOL * vmax


def test_single_token_appends_at_odd_positions():
    """Token-pair V rows filled one token per call (the read-modify-write of
    the partner token's nibbles) give the same bytes as one bulk append."""
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8)
    T = 70
    cache, K, V = _build(w, T, 1.0, seed=3, split=33)
    Kh, Vh = K.float().cpu().numpy(), V.float().cpu().numpy()
    Sv = cache.v_gscale.cpu().numpy()
    for b in range(2):
        for h in range(2):
            _, _, vc, vs = gather_unit_bytes(cache, None, b, h, T)
            ovc, ovs, _ = oracle.nvfp4_quantize_rows(Vh[b, :, h], float(Sv[h]))
            assert np.array_equal(vs, ovs) and np.array_equal(vc, ovc)


def test_nvfp4_needs_its_scales():
    cache = kvq.Fp4Cache(2, 128, 64, 4, 2, nvfp4=True)
    s = cache.struct()
    s.k_scale = None
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.zeros((1, 1, 2, 128), dtype=torch.bfloat16, device="cuda")
    st = kvq.load().kvq_append(ctypes.byref(s), 1, 1, start.data_ptr(), k.data_ptr(), k.data_ptr(), None,
                               torch.cuda.current_stream().cuda_stream)
    assert st == 1  # KVQ_ERR_INVALID_ARGUMENT, nothing enqueued


# One second-level scale per kv head across the fp32 range, with the decimal
# span of x / S its blocks take: the division-free path's ends 2^-90 (tiny
# x included: x below 2^-102 gives |x / S| < 2^-12) and 2^126, just outside
# them 2^-91 and 1e38 (IEEE path), a subnormal S, S = 1e-37 with x / S
# overflowing for the larger blocks (flagged, saturated codes), and two
# ordinary scales.
RANGE_SCALES = [(2.0 ** -90, -14, 12), (2.0 ** -91, -14, 12), (1e-37, -10, 41), (1e-38, -10, 10),
                (3.7e-20, -12, 12), (0.3, -30, 30), (2.0 ** 126, -12, 1), (1e38, -12, 1)]


def _range_blocks(scales, n, d, g):
    """bf16-valued [n][Hkv][d]: per 16-value block, N(0,1) times 10^u with
    u uniform in log10(S_h) + [lo, hi] (kept inside the bf16 range)."""
    out = np.empty((n, len(scales), d), np.float32)
    for h, (S, lo, hi) in enumerate(scales):
        u = torch.empty(n, d // 16).uniform_(lo, hi, generator=g) + math.log10(S)
        u = u.clamp(-45.0, 37.5).repeat_interleave(16, dim=-1)
        x = torch.randn(n, d, generator=g, dtype=torch.float64) * 10.0 ** u.double()
        out[:, h] = x.float().to(torch.bfloat16).float().numpy()
    return out


def _append_with_scales(k: np.ndarray, v: np.ndarray, Sk, Sv):
    """Append bf16-valued arrays [n][Hkv][d] as one sequence under the given
    per-head second-level scales; return the cache and the error flag."""
    n, hkv, d = k.shape
    P = 64
    pages = -(-n // P)
    cache = kvq.Fp4Cache(hkv, d, P, pages, pages, nvfp4=True)
    cache.k_gscale.copy_(torch.tensor(Sk, dtype=torch.float32))
    cache.v_gscale.copy_(torch.tensor(Sv, dtype=torch.float32))
    kt = torch.from_numpy(k).to(torch.bfloat16)
    vt = torch.from_numpy(v).to(torch.bfloat16)
    assert torch.equal(kt.float(), torch.from_numpy(k)) and torch.equal(vt.float(), torch.from_numpy(v))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append(cache, torch.zeros(1, dtype=torch.int32, device="cuda"), kt[None].cuda(), vt[None].cuda(), err=err)
    torch.cuda.synchronize()
    return cache, int(err.item())


def _check_against_oracle(cache, k, v, Sk, Sv):
    n, hkv, _ = k.shape
    bad = 0
    for h in range(hkv):
        kc, ks, vc, vs = gather_unit_bytes(cache, None, 0, h, n)
        okc, oks, kbad = oracle.nvfp4_quantize_rows(k[:, h], float(np.float32(Sk[h])))
        ovc, ovs, vbad = oracle.nvfp4_quantize_rows(v[:, h], float(np.float32(Sv[h])))
        assert np.array_equal(ks, oks) and np.array_equal(kc, okc), ("K", h, Sk[h])
        assert np.array_equal(vs, ovs) and np.array_equal(vc, ovc), ("V", h, Sv[h])
        bad += kbad + vbad
    return bad


def test_second_level_scales_across_the_fp32_range():
    """Blocks around each scale of RANGE_SCALES (V takes them in reverse
    order): codes and scale bytes equal the oracle's IEEE divisions bit for
    bit, and the non-finite flag is raised exactly when some x / S
    overflows.  Every branch of the append's NVFP4 path runs here; the rare
    inputs where a one-ulp error in x / S would move a code across an E2M1
    midpoint are pinned by the host check in test_quotient_exhaustive.py."""
    hkv, d, n = len(RANGE_SCALES), 128, 96
    g = torch.Generator().manual_seed(21)
    k = _range_blocks(RANGE_SCALES, n, d, g)
    v = _range_blocks(RANGE_SCALES[::-1], n, d, g)
    Sk = [S for S, _, _ in RANGE_SCALES]
    Sv = Sk[::-1]
    cache, flag = _append_with_scales(k, v, Sk, Sv)
    bad = _check_against_oracle(cache, k, v, Sk, Sv)
    assert bad > 0  # the 1e-37 head overflows
    assert flag == kvq.FLAG_NONFINITE


def test_ties_and_special_blocks_under_a_second_level_scale():
    """Every E2M1 tie, saturation, signed zeros and tiny values, scaled by an
    exact power of two so that x / S lands on them exactly, through the
    division-free path."""
    rows = [np.zeros(16), np.full(16, -0.0), np.full(16, 2.0 ** -12),
            np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0]),
            np.array([3000.0] + [1.0] * 15), np.array([2688.0, -2688.0] + [0.0] * 14),
            np.array([9 * 2.0 ** -9] + [0.0] * 15), np.array([1e-30] * 8 + [-1e-30] * 8)]
    S = 0.25
    blk = np.array(rows, np.float64) * S
    blk = torch.tensor(blk, dtype=torch.float32).to(torch.bfloat16).float().numpy()
    n = blk.shape[0]
    k = np.zeros((n, 2, 128), np.float32)
    k[:, :, :16] = blk[:, None, :]
    k[:, :, 64:80] = -blk[:, None, :]
    v = k[::-1].copy()
    cache, flag = _append_with_scales(k, v, [S, 3.0 * S], [S, S])
    assert _check_against_oracle(cache, k, v, [S, 3.0 * S], [S, S]) == 0
    assert flag == 0


@pytest.mark.parametrize("d,mag,T", [(128, 1.0, 300), (64, 3e3, 300), (128, 3e3, 50)])
def test_decode_with_fp8_window(d, mag, T):
    """An NVFP4 global cache with the FP8 sliding window (W = 64): positions
    before the window from the NVFP4 cache with both second-level scales,
    the last min(W, T) from the FP8 ring, one softmax; T = 50 reads the
    window alone."""
    W = 64
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8, head_dim=d,
                         k_outlier_channels=(3, 17, 40) if d == 64 else (3, 17, 64, 101))
    cache, K, V = _build(w, T, mag, seed=7 + d)
    B, hkv, G = w.batch, w.num_kv_heads, w.group
    swa = kvq.Fp8WindowCache(B, hkv, d, W)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    w0 = min(W, T)
    kw, vw = K[:, T - w0:].contiguous(), V[:, T - w0:].contiguous()
    kvq.fp8_set_scales(swa, kw, vw, err=err)
    kvq.append(swa, torch.full((B,), T - w0, dtype=torch.int32, device="cuda"), kw, vw, err=err)
    lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
    q = workloads.queries(w, seed=d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    out = kvq.decode_attn(cache, lens, q, scale, swa=swa, err=err).cpu().numpy()
    torch.cuda.synchronize()
    assert err.item() == 0
    Kh, Vh = K.float().cpu().numpy(), V.float().cpu().numpy()
    kwh, vwh = kw.float().cpu().numpy(), vw.float().cpu().numpy()
    Sk, Sv = cache.k_gscale.cpu().numpy(), cache.v_gscale.cpu().numpy()
    qh = q.float().cpu().numpy()
    for h in range(hkv):
        sk = oracle.fp8_head_scale(kwh[:, :, h])
        sv = oracle.fp8_head_scale(vwh[:, :, h])
        assert swa.k_scales[h].item() == sk and swa.v_scales[h].item() == sv
        for b in range(B):
            ref, vmax = oracle.decode_unit(qh[b, h * G:(h + 1) * G], Kh[b, :, h], Vh[b, :, h], scale, window=W,
                                           swa_scales=(sk, sv), nvfp4_scales=(float(Sk[h]), float(Sv[h])))
            assert np.abs(out[b, h * G:(h + 1) * G] - ref).max() <= TOL * vmax
