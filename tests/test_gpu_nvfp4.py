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
