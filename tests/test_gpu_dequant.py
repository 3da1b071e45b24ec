"""kvq_dequant against the oracle's dequantiser: exact equality (the FP4
products are exact in fp32 and bf16), zeros past each sequence's length, and
the FP8 window's fp32 products."""
import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import build_fp4, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


@pytest.mark.parametrize("paged,page_size,d", [(True, 64, 128), (False, 32, 64), (True, 256, 128)])
def test_fp4_dequant_exact(paged, page_size, d):
    w = workloads.scaled(workloads.WORKLOADS["gqa_outliers"], batch=4, paged=paged, page_size=page_size,
                         head_dim=d, k_outlier_channels=(3, 17) if d == 64 else (3, 17, 64, 101))
    lens = [1, 130, 0, 517]
    built = build_fp4(w, lens, seed=2)
    max_len = max(lens) + 3
    for dtype in (torch.float32, torch.bfloat16):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kd, vd = kvq.dequant(built.cache, built.lens_dev, max_len, dtype=dtype, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        kd, vd = kd.float().cpu().numpy(), vd.float().cpu().numpy()
        for b, n in enumerate(lens):
            for h in range(w.num_kv_heads):
                kc, ks, _ = oracle.quantize_rows(built.seq_k[b][:, h].float().cpu().numpy())
                vc, vs, _ = oracle.quantize_rows(built.seq_v[b][:, h].float().cpu().numpy())
                assert np.array_equal(kd[b, :n, h], oracle.dequantize_rows(kc, ks).astype(np.float32))
                assert np.array_equal(vd[b, :n, h], oracle.dequantize_rows(vc, vs).astype(np.float32))
            assert not kd[b, n:].any() and not vd[b, n:].any()


def test_fp8_dequant_matches_fp32_products():
    g = torch.Generator().manual_seed(4)
    B, Hkv, D, W = 2, 3, 64, 32
    k = torch.randn(B, W, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, W, Hkv, D, generator=g).to(torch.bfloat16)
    cache = kvq.Fp8WindowCache(B, Hkv, D, W)
    kvq.fp8_set_scales(cache, k.cuda(), v.cuda())
    kvq.append(cache, torch.zeros(B, dtype=torch.int32, device="cuda"), k.cuda(), v.cuda())
    kd, vd = kvq.dequant(cache, None, W)
    torch.cuda.synchronize()
    for h in range(Hkv):
        sk = np.float32(cache.k_scales[h].item())
        sv = np.float32(cache.v_scales[h].item())
        for b in range(B):
            ck, _ = oracle.fp8_quantize(k[b, :, h].float().numpy(), sk)
            cv, _ = oracle.fp8_quantize(v[b, :, h].float().numpy(), sv)
            assert np.array_equal(kd[b, :, h].cpu().numpy(), oracle.fp8_dequantize(ck, sk).astype(np.float32))
            assert np.array_equal(vd[b, :, h].cpu().numpy(), oracle.fp8_dequantize(cv, sv).astype(np.float32))
