"""kvq_append and kvq_fp8_set_scales against the oracle, bit for bit.

Covers the exhaustive sets of the oracle's pins run through the GPU
quantiser: every finite bf16 amax (scale byte), every reachable (bf16 value,
E4M3 scale) pair (codes), special blocks (zeros, -0.0, saturation, ties),
paged layouts with random page tables and ragged start positions, the FP8
window codes over every finite bf16 value, the device error flags, and the
prefill appends at their full sizes in the benchmark's launch (sampled pages
bit for bit, every scale byte in range).
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import ensure_built, gather_unit_bytes, unpack_pool_rows
from tests.test_oracle_formats import all_bf16_as_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _rows_through_gpu(blocks: np.ndarray, head_dim: int = 64):
    """Append rows of `head_dim` values (as K, and -rows as V) to a contiguous
    one-head cache; return (k_codes, k_scales, v_codes, v_scales) per row."""
    x = torch.from_numpy(np.ascontiguousarray(blocks, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.from_numpy(blocks.astype(np.float32)))  # inputs are bf16 values
    n = x.shape[0]
    P = 64
    pages = (n + P - 1) // P
    cache = kvq.Fp4Cache(1, head_dim, P, pages, pages, device="cuda")
    k = x.reshape(1, n, 1, head_dim).cuda()
    v = (-x).reshape(1, n, 1, head_dim).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append(cache, torch.zeros(1, dtype=torch.int32, device="cuda"), k, v, err=err)
    torch.cuda.synchronize()
    out = gather_unit_bytes(cache, None, 0, 0, n)
    return out, int(err.item())


def _compare_rows(blocks):
    if blocks.shape[1] == 16:  # pack four 16-value blocks per 64-channel row
        pad = (-blocks.shape[0]) % 4
        blocks = np.concatenate([blocks, np.zeros((pad, 16), blocks.dtype)]).reshape(-1, 64)
    (kc, ks, vc, vs), flag = _rows_through_gpu(blocks, blocks.shape[1])
    okc, oks, _ = oracle.quantize_rows(blocks)
    ovc, ovs, _ = oracle.quantize_rows(-blocks)
    assert np.array_equal(ks, oks)
    assert np.array_equal(kc, okc)
    assert np.array_equal(vs, ovs)
    assert np.array_equal(vc, ovc)
    return flag


def test_every_bf16_amax_scale_byte():
    x = all_bf16_as_f32()
    x = x[np.isfinite(x)]
    blocks = np.zeros((x.size, 16), np.float32)
    blocks[:, 5] = x
    assert _compare_rows(blocks) == 0


def test_every_reachable_value_scale_pair():
    allv = all_bf16_as_f32()
    allv = allv[np.isfinite(allv)]
    chunks = []
    for sb in range(1, 0x7F):
        s = oracle.e4m3_value(sb)
        a = np.float32(6.0 * s)
        v = allv[np.abs(allv) <= a]
        pad = (-v.size) % 15
        v = np.concatenate([v, np.zeros(pad, np.float32)])
        blk = np.empty((v.size // 15, 16), np.float32)
        blk[:, 0] = -a if sb % 2 else a
        blk[:, 1:] = v.reshape(-1, 15)
        chunks.append(blk)
    blocks = np.concatenate(chunks)
    assert _compare_rows(blocks) == 0


def test_special_blocks_and_ties():
    rows = []
    rows.append(np.zeros(16))
    rows.append(np.full(16, -0.0))
    rows.append(np.full(16, 2.0 ** -12))                      # amax/6 rounds to zero -> 0x01
    rows.append(np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5,
                          -5.0, -6.0]))                        # s = 1: every E2M1 tie
    rows.append(np.array([3000.0] + [1.0] * 15))              # saturating scale (448)
    rows.append(np.array([2688.0, -2688.0] + [0.0] * 14))     # 6 * 448 exactly
    rows.append(np.array([9 * 2.0 ** -9] + [0.0] * 15))       # the requantisation exception class
    rows.append(np.array([1e-30] * 8 + [-1e-30] * 8))         # tiny values, sign kept
    blocks = torch.tensor(np.array(rows), dtype=torch.float32).to(torch.bfloat16).float().numpy()
    assert _compare_rows(blocks) == 0


def test_random_blocks_d128_with_outliers():
    g = torch.Generator().manual_seed(11)
    x = torch.randn(20000, 128, generator=g)
    x[:, [3, 17, 64, 101]] *= 20.0
    x[:5000] *= 1e-3
    x[5000:6000] *= 3000.0
    blocks = x.to(torch.bfloat16).float().numpy()
    assert _compare_rows(blocks) == 0


@pytest.mark.parametrize("page_size", [16, 64, 256])
def test_paged_append_ragged_starts(page_size):
    w = workloads.scaled(workloads.WORKLOADS["paged_ragged"], page_size=page_size, batch=5, ragged=None)
    lens = [0, 1, 63, 200, 517]
    n_new = 37
    table_cpu, num_pages, max_pages = workloads.page_layout(w, lens, reserve=n_new, seed=3)
    table = table_cpu.cuda()
    cache = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, page_size, num_pages, max_pages, page_table=table)
    g = torch.Generator().manual_seed(5)
    k = torch.randn(w.batch, n_new, w.num_kv_heads, w.head_dim, generator=g).to(torch.bfloat16)
    v = torch.randn(w.batch, n_new, w.num_kv_heads, w.head_dim, generator=g).to(torch.bfloat16) * 7
    start = torch.tensor(lens, dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.append(cache, start.cuda(), k.cuda(), v.cuda(), err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            kc, ks, vc, vs = gather_unit_bytes(cache, table_cpu[b].numpy(), b, h, lens[b] + n_new)
            sl = slice(lens[b], lens[b] + n_new)
            okc, oks, _ = oracle.quantize_rows(k[b, :, h].float().numpy())
            ovc, ovs, _ = oracle.quantize_rows(v[b, :, h].float().numpy())
            assert np.array_equal(kc[sl], okc) and np.array_equal(ks[sl], oks)
            assert np.array_equal(vc[sl], ovc) and np.array_equal(vs[sl], ovs)
            # positions before the start keep their (zero) bytes, including the
            # other nibble of a V byte shared with the first new token
            assert not kc[: lens[b]].any() and not ks[: lens[b]].any()
            assert not vc[: lens[b]].any() and not vs[: lens[b]].any()


def test_flags_page_oob_bad_start_nonfinite():
    cache = kvq.Fp4Cache(1, 64, 16, 2, 2, page_table=torch.tensor([[0, 5]], dtype=torch.int32, device="cuda"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.ones(1, 20, 1, 64, dtype=torch.bfloat16, device="cuda")
    kvq.append(cache, torch.zeros(1, dtype=torch.int32, device="cuda"), k, k, err=err)
    torch.cuda.synchronize()
    assert err.item() == kvq.FLAG_PAGE_OOB       # page id 5 >= num_pages: tokens 16.. skipped
    assert not cache.pool[1].any()               # nothing written to the other page
    err.zero_()
    kvq.append(cache, torch.full((1,), -4, dtype=torch.int32, device="cuda"), k, k, err=err)
    torch.cuda.synchronize()
    assert err.item() == kvq.FLAG_BAD_LENGTH
    err.zero_()
    k2 = k.clone()
    k2[0, 3, 0, 7] = float("nan")
    k2[0, 4, 0, 1] = float("inf")
    kvq.append(cache, torch.zeros(1, dtype=torch.int32, device="cuda"), k2[:, :16].contiguous(),
               k[:, :16].contiguous(), err=err)
    torch.cuda.synchronize()
    assert err.item() == kvq.FLAG_NONFINITE
    # a position past the table's last page
    err.zero_()
    kvq.append(cache, torch.full((1,), 31, dtype=torch.int32, device="cuda"), k[:, :2].contiguous(),
               k[:, :2].contiguous(), err=err)
    torch.cuda.synchronize()
    assert err.item() & kvq.FLAG_PAGE_OOB


def test_fp8_window_codes_every_bf16():
    x = all_bf16_as_f32()
    x = x[np.isfinite(x)]
    D, W = 32, 64
    n = x.size // D
    x = x[: n * D].reshape(n, D)
    for s in (1.0, 0.0078125, 3.7e-3, 1234.5):
        cache = kvq.Fp8WindowCache(1, 1, D, W)
        cache.k_scales.fill_(s)
        cache.v_scales.fill_(s * 2)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kx = torch.from_numpy(x).to(torch.bfloat16)
        for t0 in range(0, n, W):
            blk = kx[t0:t0 + W]
            m = blk.shape[0]
            kvq.append(cache, torch.tensor([t0], dtype=torch.int32, device="cuda"),
                       blk.reshape(1, m, 1, D).cuda(), (-blk).reshape(1, m, 1, D).cuda(), err=err)
            torch.cuda.synchronize()
            got_k = cache.k_codes[0, 0, :m].cpu().numpy()
            got_v = cache.v_codes[0, 0, :m].cpu().numpy()
            want_k, _ = oracle.fp8_quantize(blk.float().numpy(), np.float32(s))
            want_v, _ = oracle.fp8_quantize((-blk).float().numpy(), np.float32(s * 2))
            assert np.array_equal(got_k, want_k), (s, t0)
            assert np.array_equal(got_v, want_v), (s, t0)
        assert err.item() == 0


def test_fp8_set_scales_and_ring_slots():
    g = torch.Generator().manual_seed(9)
    B, Hkv, D, W, n = 3, 4, 128, 16, 40
    k = torch.randn(B, n, Hkv, D, generator=g).to(torch.bfloat16)
    v = (torch.randn(B, n, Hkv, D, generator=g) * 3).to(torch.bfloat16)
    v[:, :, 2] = 0  # an all-zero head -> scale 1
    cache = kvq.Fp8WindowCache(B, Hkv, D, W)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.fp8_set_scales(cache, k[:, n - W:].contiguous().cuda(), v[:, n - W:].contiguous().cuda(), err=err)
    start = torch.tensor([0, 5, 1000], dtype=torch.int32)
    kvq.append(cache, start.cuda(), k.cuda(), v.cuda(), err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    for h in range(Hkv):
        assert cache.k_scales[h].item() == oracle.fp8_head_scale(k[:, n - W:, h].float().numpy())
        assert cache.v_scales[h].item() == oracle.fp8_head_scale(v[:, n - W:, h].float().numpy())
    for b in range(B):
        for h in range(Hkv):
            sk = np.float32(cache.k_scales[h].item())
            for t in range(n - W, n):  # the last W positions occupy every slot once
                slot = (int(start[b]) + t) % W
                want, _ = oracle.fp8_quantize(k[b, t, h].float().numpy(), sk)
                assert np.array_equal(cache.k_codes[b, h, slot].cpu().numpy(), want)


@pytest.mark.parametrize("name,nv", [("prefill", False), ("prefill", True), ("prefill_b1", False)])
def test_prefill_append_full_size_sampled(name, nv):
    """The benchmark's prefill append (B16 or B1 x 16384 tokens, Hkv 8, d 128,
    the whole batch in one call) at full size: 26 sampled (sequence, kv head,
    page) blocks -- the first and last pages among them -- bit for bit
    against the oracle's quantiser (NVFP4: with the second-level scales,
    themselves checked against the oracle from each head's amax), and every
    scale byte of the pool a positive finite E4M3 value (0x01..0x7E)."""
    w = workloads.WORKLOADS[name]
    B, T, H, D, P = w.batch, w.context, w.num_kv_heads, w.head_dim, w.page_size
    max_pages = -(-T // P)
    cache = kvq.Fp4Cache(H, D, P, B * max_pages, max_pages, device="cuda", nvfp4=nv)
    k = torch.empty((B, T, H, D), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    for b in range(B):
        k[b], v[b] = workloads.sequence_kv(w, b, T, seed=0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if nv:
        kvq.fp8_set_scales(cache, k, v, err=err)
    kvq.append(cache, torch.zeros(B, dtype=torch.int32, device="cuda"), k, v, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    if nv:
        Sk, Sv = cache.k_gscale.cpu().numpy(), cache.v_gscale.cpu().numpy()
        for h in range(H):
            ak = k[:, :, h].float().abs().amax().item()
            av = v[:, :, h].float().abs().amax().item()
            assert Sk[h] == np.float32(oracle.nvfp4_global_scale(np.array([ak], np.float32)))
            assert Sv[h] == np.float32(oracle.nvfp4_global_scale(np.array([av], np.float32)))
    G, nb = cache.group, D // 16
    blocks = cache.pool.reshape(-1, cache.pool.shape[-1])
    for lo, hi in ((G * D // 2, G * (D // 2 + nb)), (G * (D + nb), blocks.shape[1])):
        sc = blocks[:, lo:hi]
        assert int(sc.min().item()) >= 0x01 and int(sc.max().item()) <= 0x7E
    rng = np.random.default_rng(23)
    picks = [(0, 0, 0), (B - 1, H - 1, max_pages - 1)]
    picks += [(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(max_pages))) for _ in range(24)]
    for b, h, pg in picks:
        kc, ks, vc, vs = unpack_pool_rows(cache, [b * max_pages + pg], h, P)
        xk = k[b, pg * P:(pg + 1) * P, h].float().cpu().numpy()
        xv = v[b, pg * P:(pg + 1) * P, h].float().cpu().numpy()
        if nv:
            okc, oks, _ = oracle.nvfp4_quantize_rows(xk, float(Sk[h]))
            ovc, ovs, _ = oracle.nvfp4_quantize_rows(xv, float(Sv[h]))
        else:
            okc, oks, _ = oracle.quantize_rows(xk)
            ovc, ovs, _ = oracle.quantize_rows(xv)
        assert np.array_equal(ks, oks) and np.array_equal(kc, okc), (b, h, pg)
        assert np.array_equal(vs, ovs) and np.array_equal(vc, ovc), (b, h, pg)
