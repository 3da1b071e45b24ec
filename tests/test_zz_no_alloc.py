"""The allocation-free decode entry point (kvq_decode_attn_noalloc), called
through the C ABI, against the regular entry point (kvq_decode_attn).

It serves callers that cannot allocate device memory when they call decode, so
it keeps its scratch in a fixed device array inside the library.  Two calls in
a row with different inputs must both agree with kvq_decode_attn within the
tolerance the decode tests use (2e-3 of the largest dequantised |V| of the
unit).  This file runs last so a failure here comes after every other test.
"""
import ctypes
import math

import pytest
import torch

from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import TOL, build_fp4, ensure_built

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


def _noalloc(lib, cache, lens, q, scale, swa=None):
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=q.device)
    err = torch.zeros(1, dtype=torch.int32, device=q.device)
    g = cache.struct()
    w = swa.struct() if swa is not None else None
    st = lib.kvq_decode_attn_noalloc(ctypes.byref(g), ctypes.byref(w) if w is not None else None, q.shape[0],
                                     q.shape[1], lens.data_ptr(), q.data_ptr(), scale, out.data_ptr(),
                                     err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.kvq_status_string(st)
    return out, err


def _check(out, ref, cache, lens, w):
    kd, vd = kvq.dequant(cache, lens, int(lens.max().item()))
    G = w.group
    for b in range(out.shape[0]):
        for h in range(w.num_kv_heads):
            vmax = vd[b, :, h].abs().max().item()
            err = (out[b, h * G:(h + 1) * G] - ref[b, h * G:(h + 1) * G]).abs().max().item()
            assert err <= TOL * max(vmax, 1e-30), (b, h, err, vmax)


def test_noalloc_matches_decode_attn_twice(lib):
    w = workloads.scaled(workloads.WORKLOADS["gqa_outliers"], batch=5, num_kv_heads=4, num_q_heads=16,
                         paged=True)
    built = build_fp4(w, [300, 1, 77, 1000, 129], seed=21)
    scale = 1.0 / math.sqrt(w.head_dim)
    for call in range(2):
        q = workloads.queries(w, seed=21, step=call, device="cuda")
        lens = built.lens_dev if call == 0 else torch.tensor([17, 1, 64, 999, 128], dtype=torch.int32,
                                                              device="cuda")
        out, err = _noalloc(lib, built.cache, lens, q, scale)
        ref = kvq.decode_attn(built.cache, lens, q, scale)
        torch.cuda.synchronize()
        assert err.item() == 0 and torch.isfinite(out).all()
        _check(out, ref, built.cache, lens, w)


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    cache = kvq.Fp4Cache(8, 128, 64, 4096, 1)  # 4096 sequences x 8 kv heads x 64 q heads: ~137 MB of scratch
    lens = torch.ones(4096, dtype=torch.int32, device="cuda")
    q = torch.zeros(4096, 64, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(4096, 64, 128, dtype=torch.float32, device="cuda")
    g = cache.struct()
    st = lib.kvq_decode_attn_noalloc(ctypes.byref(g), None, 4096, 64, lens.data_ptr(), q.data_ptr(), 0.1,
                                     out.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert st == 3  # KVQ_ERR_WORKSPACE: beyond the built-in 8 MiB, nothing enqueued
