"""The bounds-checked build of the library (-DKVQ_DEBUG_BOUNDS, built here as
libkvq_bounds.so) on the small cases of the other GPU tests.

In that build every checked index or address range -- the bulk copies'
sources and stage slots, the consumers' shared-memory reads of a stage, the
query rows, the split partials and unit records, the window rings, the
append's pool groups and input rows, the dequantiser's groups -- raises
KVQ_FLAG_BOUNDS and skips the access when it falls outside its buffer
(nothing traps).  On every case the flag must stay clear and the results must
equal the normal build's bit for bit (the checks only guard accesses).
"""
import math

import pytest
import torch

from fp4_kv_cache_kvq_gb300 import build, kvq, workloads
from tests.helpers import build_fp4, ensure_built

pytestmark = pytest.mark.gpu

BASE = workloads.WORKLOADS["gqa_outliers"]


@pytest.fixture(scope="module")
def libs():
    normal = ensure_built()
    path = build.build(bounds=True)
    saved, old = kvq._lib, kvq.LIB_PATH
    kvq._lib, kvq.LIB_PATH = None, path
    try:
        checked = kvq.load()
    finally:
        kvq._lib, kvq.LIB_PATH = saved, old
    return normal, checked


def _with(lib, fn):
    saved = kvq._lib
    kvq._lib = lib
    try:
        return fn()
    finally:
        kvq._lib = saved


def _twin(cache):
    c = kvq.Fp4Cache(cache.num_kv_heads, cache.head_dim, cache.page_size, cache.num_pages, cache.max_pages_per_seq,
                     page_table=cache.page_table, nvfp4=cache.nvfp4)
    c.pool.copy_(cache.pool)
    return c


@pytest.mark.parametrize("d,g,page_size,paged", [(64, 1, 16, True), (64, 8, 256, False), (128, 4, 64, True),
                                                 (128, 8, 128, False), (128, 2, 32, True)])
def test_decode_and_dequant(libs, d, g, page_size, paged):
    normal, checked = libs
    w = workloads.scaled(BASE, batch=6, num_kv_heads=2, num_q_heads=2 * g, head_dim=d, page_size=page_size,
                         paged=paged, k_outlier_channels=(3, 17, 40) if d == 64 else (3, 17, 64, 101))
    lens = [0, 1, 17, 300, 1000, 129]
    built = build_fp4(w, lens, seed=d + page_size, keep_kv=False)
    q = workloads.queries(w, seed=3, device="cuda")
    outs, flags, deq = [], [], []
    for lib in (normal, checked):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs.append(_with(lib, lambda: kvq.decode_attn(built.cache, built.lens_dev, q, err=err)))
        deq.append(_with(lib, lambda: kvq.dequant(built.cache, built.lens_dev, max(lens), err=err)))
        torch.cuda.synchronize()
        flags.append(err.item())
    assert flags == [0, 0]
    assert torch.equal(outs[0], outs[1])
    for a, b in zip(deq[0], deq[1]):
        assert torch.equal(a, b)


@pytest.mark.parametrize("reserve", [2, 100_000])
def test_append_and_fused_decode(libs, reserve):
    """kvq_append (several tokens, odd starts) and kvq_append_decode_attn by its
    separate-append path and by the fused kernel (large capacity)."""
    normal, checked = libs
    w = workloads.scaled(BASE, batch=5, num_kv_heads=2, num_q_heads=8, paged=True)
    lens0 = [63, 64, 1, 300, 127]
    pools, outs, flags = [], [], []
    for lib in (normal, checked):
        built = build_fp4(w, lens0, seed=5, reserve=reserve + 8, keep_kv=False)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kn, vn = workloads.step_tokens(w, 1, seed=5, device="cuda")
        k3 = torch.cat([kn] * 3, dim=1).contiguous()
        v3 = torch.cat([vn] * 3, dim=1).contiguous()
        start = torch.tensor(lens0, dtype=torch.int32, device="cuda")
        _with(lib, lambda: kvq.append(built.cache, start, k3, v3, err=err))
        lens = torch.tensor([n + 4 for n in lens0], dtype=torch.int32, device="cuda")
        q = workloads.queries(w, seed=5, device="cuda")
        outs.append(_with(lib, lambda: kvq.append_decode_attn(built.cache, lens, kn[:, 0].contiguous(),
                                                              vn[:, 0].contiguous(), q, err=err)))
        torch.cuda.synchronize()
        pools.append(built.cache.pool)
        flags.append(err.item())
    assert flags == [0, 0]
    assert torch.equal(pools[0], pools[1])
    assert torch.equal(outs[0], outs[1])


def test_window_merge(libs):
    normal, checked = libs
    w = workloads.scaled(workloads.WORKLOADS["swa_append"], batch=3, num_kv_heads=2, num_q_heads=16, context=300,
                         window=128)
    built = build_fp4(w, [300] * 3, seed=9, keep_kv=True)
    swa = kvq.Fp8WindowCache(3, 2, w.head_dim, 128)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = torch.stack([built.seq_k[b][300 - 128:] for b in range(3)]).contiguous()
    vw = torch.stack([built.seq_v[b][300 - 128:] for b in range(3)]).contiguous()
    kvq.fp8_set_scales(swa, kw, vw, err=err)
    kvq.append(swa, torch.full((3,), 300 - 128, dtype=torch.int32, device="cuda"), kw, vw, err=err)
    q = workloads.queries(w, seed=9, device="cuda")
    outs, flags = [], []
    for lib in (normal, checked):
        e = torch.zeros(1, dtype=torch.int32, device="cuda")
        outs.append(_with(lib, lambda: kvq.decode_attn(built.cache, built.lens_dev, q, 1.0 / math.sqrt(w.head_dim),
                                                       swa=swa, err=e)))
        torch.cuda.synchronize()
        flags.append(e.item())
    assert flags == [0, 0] and err.item() == 0
    assert torch.equal(outs[0], outs[1])
