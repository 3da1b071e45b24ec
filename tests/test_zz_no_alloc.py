"""The allocation-free decode entry point (kvq_decode_attn_noalloc), called
through the C ABI, against the regular entry point (kvq_decode_attn).

It serves callers that cannot allocate device memory when they call decode --
a plug-in whose host framework owns every device allocation, or code under a
fixed memory budget -- so it keeps its scratch in a fixed device array inside
the library.  It launches the same kernels with the same grid as
kvq_decode_attn, so the outputs must be identical bit for bit: on two calls in
a row on one stream (the second reusing the array the first left behind), with
and without the FP8 window.  After one warm-up call (which may load the
library's device module), further calls must not lower the device's free
memory.  This file runs last so a failure here comes after every other test.
"""
import ctypes
import math

import pytest
import torch

from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import build_fp4, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    L = ensure_built()
    fn = L.kvq_decode_attn_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(kvq.KvqCacheStruct), ctypes.POINTER(kvq.KvqCacheStruct), ctypes.c_int32,
                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                   ctypes.c_void_p, ctypes.c_void_p]
    return L


def _noalloc(lib, cache, lens, q, scale, out, err, swa=None):
    g = cache.struct()
    w = swa.struct() if swa is not None else None
    st = lib.kvq_decode_attn_noalloc(ctypes.byref(g), ctypes.byref(w) if w is not None else None, q.shape[0],
                                     q.shape[1], lens.data_ptr(), q.data_ptr(), scale, out.data_ptr(),
                                     err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.kvq_status_string(st)


def _case():
    w = workloads.scaled(workloads.WORKLOADS["gqa_outliers"], batch=5, num_kv_heads=4, num_q_heads=16,
                         paged=True)
    built = build_fp4(w, [300, 1, 77, 1000, 129], seed=21)
    return w, built, 1.0 / math.sqrt(w.head_dim)


def test_noalloc_matches_decode_attn_twice(lib):
    w, built, scale = _case()
    qs = [workloads.queries(w, seed=21, step=c, device="cuda") for c in range(2)]
    lens = [built.lens_dev, torch.tensor([17, 1, 64, 999, 128], dtype=torch.int32, device="cuda")]
    outs = [torch.full(qs[0].shape, float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
    errs = [torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(2)]
    for c in range(2):  # back to back on one stream, no synchronisation between
        _noalloc(lib, built.cache, lens[c], qs[c], scale, outs[c], errs[c])
    refs = [kvq.decode_attn(built.cache, lens[c], qs[c], scale) for c in range(2)]
    torch.cuda.synchronize()
    for c in range(2):
        assert errs[c].item() == 0
        assert torch.equal(outs[c], refs[c]), f"call {c}"


def test_noalloc_with_fp8_window_matches_decode_attn(lib):
    w = workloads.scaled(workloads.WORKLOADS["swa_append"], batch=3, num_kv_heads=2, num_q_heads=16, context=300,
                         window=128)
    built = build_fp4(w, [300] * 3, seed=22)
    swa = kvq.Fp8WindowCache(3, 2, w.head_dim, 128)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = torch.stack([built.seq_k[b][300 - 128:] for b in range(3)]).contiguous()
    vw = torch.stack([built.seq_v[b][300 - 128:] for b in range(3)]).contiguous()
    kvq.fp8_set_scales(swa, kw, vw, err=err)
    kvq.append(swa, torch.full((3,), 300 - 128, dtype=torch.int32, device="cuda"), kw, vw, err=err)
    scale = 1.0 / math.sqrt(w.head_dim)
    outs, refs = [], []
    for c in range(2):
        q = workloads.queries(w, seed=22, step=c, device="cuda")
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        _noalloc(lib, built.cache, built.lens_dev, q, scale, out, err, swa=swa)
        outs.append(out)
        refs.append(kvq.decode_attn(built.cache, built.lens_dev, q, scale, swa=swa))
    torch.cuda.synchronize()
    assert err.item() == 0
    for o, r in zip(outs, refs):
        assert torch.equal(o, r)


def test_noalloc_calls_allocate_nothing(lib):
    w, built, scale = _case()
    q = workloads.queries(w, seed=23, device="cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _noalloc(lib, built.cache, built.lens_dev, q, scale, out, err)  # warm-up: may load the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        _noalloc(lib, built.cache, built.lens_dev, q, scale, out, err)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert err.item() == 0
    assert free1 >= free0, f"device free memory fell by {free0 - free1} bytes across the calls"


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    cache = kvq.Fp4Cache(8, 128, 64, 4096, 1)  # 4096 sequences x 8 kv heads x 64 q heads: ~137 MB of scratch
    lens = torch.ones(4096, dtype=torch.int32, device="cuda")
    q = torch.zeros(4096, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(4096, 64, 128, dtype=torch.float32, device="cuda")
    g = cache.struct()
    st = lib.kvq_decode_attn_noalloc(ctypes.byref(g), None, 4096, 64, lens.data_ptr(), q.data_ptr(), 0.1,
                                     out.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert st == 3  # KVQ_ERR_WORKSPACE: beyond the built-in 8 MiB, nothing enqueued
