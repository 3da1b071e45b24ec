"""kvq_prefill_attn (chunked prefill over the FP4 cache, tensor cores) against
fp64 attention over the oracle's own dequantised cache: every query row
attends its causal prefix, max |err| <= 2e-3 * max|V^| over that prefix.

Covers head_dim 64 and 128, GQA groups 1/2/4/8, page sizes 16..256, paged
and contiguous layouts, chunks that are not a multiple of a CTA's query
tokens, a chunk with no earlier context, prefixes shorter and longer than one
128-position tile, several sequences of different lengths, NVFP4 caches, and
the bad-length flag."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import TOL, build_fp4, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


BASE = workloads.WORKLOADS["gqa_outliers"]


def _check(out, q, built_k, built_v, lens, chunk, G, scale, nvfp4_scales=None):
    """out [B][chunk][Hq][d] vs the oracle, unit by unit."""
    out = out.cpu().numpy()
    qh = q.float().cpu().numpy()
    B, _, Hq, d = q.shape
    Hkv = Hq // G
    worst = 0.0
    for b in range(B):
        T = lens[b]
        for h in range(Hkv):
            k = built_k[b][:, h].float().cpu().numpy()
            v = built_v[b][:, h].float().cpu().numpy()
            if nvfp4_scales is None:
                kc, ks, _ = oracle.quantize_rows(k)
                vc, vs, _ = oracle.quantize_rows(v)
                kh, vh = oracle.dequantize_rows(kc, ks), oracle.dequantize_rows(vc, vs)
            else:
                Sk, Sv = nvfp4_scales[0][h], nvfp4_scales[1][h]
                kc, ks, _ = oracle.nvfp4_quantize_rows(k, Sk)
                vc, vs, _ = oracle.nvfp4_quantize_rows(v, Sv)
                kh, vh = oracle.nvfp4_dequantize_rows(kc, ks, Sk), oracle.nvfp4_dequantize_rows(vc, vs, Sv)
            vabs = np.maximum.accumulate(np.abs(vh).max(axis=1))  # max |V^| over each prefix
            for i in range(chunk):
                n = T - chunk + i + 1
                ref, _, _ = oracle.attend(qh[b, i, h * G:(h + 1) * G], kh[:n], vh[:n], scale)
                err = np.abs(out[b, i, h * G:(h + 1) * G] - ref).max()
                ratio = err / vabs[n - 1] if vabs[n - 1] > 0 else err
                worst = max(worst, ratio)
                assert ratio <= TOL, (b, h, i, err, vabs[n - 1])
    return worst


def _run(w, lens, chunk, seed=0, paged=None, nvfp4=False):
    if paged is not None:
        w = workloads.scaled(w, paged=paged)
    if nvfp4:
        return _run_nvfp4(w, lens, chunk, seed)
    built = build_fp4(w, lens, seed=seed)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 77)
    q = torch.randn((w.batch, chunk, w.num_q_heads, w.head_dim), generator=g, device="cuda").to(torch.bfloat16)
    scale = 1.0 / math.sqrt(w.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # decode against the paged table the cache was built with
    if built.table is not None:
        built.cache.page_table = built.table
    out = kvq.prefill_attn(built.cache, built.lens_dev, q, scale, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return _check(out, q, built.seq_k, built.seq_v, lens, chunk, w.group, scale)


def _run_nvfp4(w, lens, chunk, seed):
    T = lens[0]
    assert all(n == T for n in lens)
    B = w.batch
    ks, vs = [], []
    for b in range(B):
        k, v = workloads.sequence_kv(w, b, T, seed=seed, device="cuda")
        ks.append(k)
        vs.append(v)
    K, V = torch.stack(ks).contiguous(), torch.stack(vs).contiguous()
    P = w.page_size
    max_pages = -(-T // P)
    cache = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, P, B * max_pages, max_pages, nvfp4=True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.fp8_set_scales(cache, K, V, err=err)
    kvq.append(cache, torch.zeros(B, dtype=torch.int32, device="cuda"), K, V, err=err)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 78)
    q = torch.randn((B, chunk, w.num_q_heads, w.head_dim), generator=g, device="cuda").to(torch.bfloat16)
    scale = 1.0 / math.sqrt(w.head_dim)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = kvq.prefill_attn(cache, lens_dev, q, scale, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    Sk = [float(x) for x in cache.k_gscale.cpu().numpy()]
    Sv = [float(x) for x in cache.v_gscale.cpu().numpy()]
    return _check(out, q, ks, vs, lens, chunk, w.group, scale, nvfp4_scales=(Sk, Sv))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_head_dims_and_groups(d, g):
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=2 * g, head_dim=d,
                         k_outlier_channels=(3, 17, 40) if d == 64 else (3, 17, 64, 101))
    _run(w, [300, 181], chunk=37, seed=g + d)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("paged", [False, True])
def test_page_sizes_and_layouts(page_size, paged):
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=16, page_size=page_size)
    _run(w, [520, 129], chunk=40, seed=page_size, paged=paged)


def test_chunk_without_earlier_context_and_long_chunks():
    w = workloads.scaled(BASE, batch=2, num_kv_heads=1, num_q_heads=8)
    _run(w, [45, 300], chunk=45, seed=3)          # first sequence: the whole cache is the chunk
    _run(w, [700, 700], chunk=300, seed=4)        # 19 query blocks of 16 tokens, 6 tiles


def test_single_query_token_matches_decode():
    """A chunk of 1 is a decode step: compare with kvq_decode_attn too."""
    w = workloads.scaled(BASE, batch=3, num_kv_heads=2, num_q_heads=8)
    lens = [1000, 77, 129]
    built = build_fp4(w, lens, seed=5)
    q = workloads.queries(w, seed=5, device="cuda")
    dec = kvq.decode_attn(built.cache, built.lens_dev, q)
    pre = kvq.prefill_attn(built.cache, built.lens_dev, q[:, None].contiguous())
    torch.cuda.synchronize()
    vmax = max(float(v.float().abs().max()) for v in built.seq_v) * 1.2
    assert (pre[:, 0] - dec).abs().max().item() <= 2 * TOL * vmax


def test_nvfp4_cache():
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=16)
    _run(w, [400, 400], chunk=33, seed=6, nvfp4=True)


def test_bad_length_flag():
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8)
    built = build_fp4(w, [64, 64], seed=7)
    lens = torch.tensor([64, 10], dtype=torch.int32, device="cuda")  # second: shorter than the chunk
    q = torch.ones((2, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvq.prefill_attn(built.cache, lens, q, err=err)
    torch.cuda.synchronize()
    assert err.item() & kvq.FLAG_BAD_LENGTH
    assert not out[1].any() and torch.isfinite(out[0]).all()


def test_full_size_sampled_rows():
    """The benchmark's configuration (B4, Hkv8, Hq64, d128, a 1024-token chunk
    over 16384 positions, page 64) in its launch configuration; sampled rows
    (first, middle and last chunk tokens, several heads) against the oracle."""
    w = workloads.WORKLOADS["prefill_attn"]
    B, T, C, d = w.batch, w.context, w.chunk, w.head_dim
    mp = -(-T // w.page_size)
    cache = kvq.Fp4Cache(w.num_kv_heads, d, w.page_size, B * mp, mp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.empty((B, T, w.num_kv_heads, d), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    for b in range(B):
        k[b], v[b] = workloads.sequence_kv(w, b, T, seed=0, device="cuda")
    kvq.append(cache, torch.zeros(B, dtype=torch.int32, device="cuda"), k, v, err=err)
    g = torch.Generator(device="cuda")
    g.manual_seed(4242)
    q = torch.randn((B, C, w.num_q_heads, d), generator=g, device="cuda").to(torch.bfloat16)
    lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
    out = kvq.prefill_attn(cache, lens, q, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out, qh = out.cpu().numpy(), q.float().cpu().numpy()
    G = w.group
    scale = 1.0 / math.sqrt(d)
    for b, h in ((0, 0), (3, 7)):
        kc, ks, _ = oracle.quantize_rows(k[b, :, h].float().cpu().numpy())
        vc, vs, _ = oracle.quantize_rows(v[b, :, h].float().cpu().numpy())
        kh, vh = oracle.dequantize_rows(kc, ks), oracle.dequantize_rows(vc, vs)
        vabs = np.maximum.accumulate(np.abs(vh).max(axis=1))
        for i in (0, 511, C - 1):
            n = T - C + i + 1
            hh = h * G + (i % G)
            ref, _, _ = oracle.attend(qh[b, i, hh:hh + 1], kh[:n], vh[:n], scale)
            assert np.abs(out[b, i, hh] - ref[0]).max() <= TOL * vabs[n - 1], (b, h, i)
