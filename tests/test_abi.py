"""The C ABI without a GPU: libkvq.so builds (nvcc cross-compiles for
sm_103a), loads, exports every function include/kvq.h declares, matches the
binding's struct layout, and rejects invalid arguments on the host before
touching the device."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from fp4_kv_cache_kvq_gb300 import build, kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kvq.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted([
        "kvq_append", "kvq_append_decode_attn", "kvq_attn_dense", "kvq_decode_attn", "kvq_decode_attn_noalloc", "kvq_decode_attn_tc",
        "kvq_decode_workspace_bytes",
        "kvq_dequant", "kvq_fake_quant", "kvq_fp4_pool_bytes", "kvq_fp8_set_scales", "kvq_prefill_attn",
        "kvq_status_string", "kvq_swa_replay", "kvq_swa_replay_workspace_bytes", "kvq_test_set_wait_limit_ns",
        "kvq_version"])


def test_library_exports_every_declared_function(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (kvq_[a-z0-9_]+)\b", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_struct_layout_matches_header():
    src = r'''
#include <stddef.h>
#include <stdio.h>
#include "kvq.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu\n", sizeof(kvq_cache), offsetof(kvq_cache, num_pages),
         offsetof(kvq_cache, max_pages_per_seq), offsetof(kvq_cache, page_table),
         offsetof(kvq_cache, data), offsetof(kvq_cache, k_scale), offsetof(kvq_cache, v_scale));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    S = kvq.KvqCacheStruct
    want = [ctypes.sizeof(S), S.num_pages.offset, S.max_pages_per_seq.offset, S.page_table.offset,
            S.data.offset, S.k_scale.offset, S.v_scale.offset]
    assert got == want


def test_sweep_entry_points_refuse_bad_arguments_on_the_host(lib):
    # layout / bits / head_dim are checked before anything is enqueued
    assert lib.kvq_fake_quant(9, 4, 1, 2, 1, 64, 16, 32, None, None, None, None) == 1
    assert lib.kvq_fake_quant(2, 1, 1, 2, 1, 64, 16, 32, None, None, None, None) == 1
    assert lib.kvq_fake_quant(2, 4, 1, 2, 1, 24, 16, 32, None, None, None, None) == 1
    assert lib.kvq_fake_quant(1, 8, 1, 2, 1, 64, 16, 32, None, None, None, None) == 1  # FP8 needs its scale pair
    assert lib.kvq_fake_quant(2, 4, 0, 2, 1, 64, None, None, None, None, None, None) == 0  # empty: no-op
    assert lib.kvq_attn_dense(1, 16385, 2, 1, 64, 16, 32, 64, 0.1, 128, None, None) == 2
    assert lib.kvq_attn_dense(1, 8, 3, 2, 64, 16, 32, 64, 0.1, 128, None, None) == 1
    assert lib.kvq_attn_dense(1, 8, 2, 1, 64, 16, 32, 64, -1.0, 128, None, None) == 1


def test_prefill_refuses_bad_arguments_on_the_host(lib):
    s = _fp4_struct()
    assert lib.kvq_prefill_attn(ctypes.byref(s), 2, 16, 0, 16, 32, 0.1, 64, None, None) == 1   # chunk 0
    assert lib.kvq_prefill_attn(ctypes.byref(s), 2, 3, 4, 16, 32, 0.1, 64, None, None) == 1    # Hq % Hkv
    assert lib.kvq_prefill_attn(ctypes.byref(s), 2, 32, 4, 16, 32, 0.1, 64, None, None) == 2   # G = 16
    assert lib.kvq_prefill_attn(ctypes.byref(s), 2, 16, 4, None, 32, 0.1, 64, None, None) == 1  # no lengths


def test_replay_refuses_bad_arguments_on_the_host(lib):
    # (pointers are fake: every one of these is refused before any launch)
    w, e, st, ws = 256, 512, 1024, 2048
    need = lib.kvq_swa_replay_workspace_bytes(2, 100, 128)
    assert need == (4 * 100 * 128 + 4 * 2 * 128 * 128) * 4
    assert lib.kvq_swa_replay_workspace_bytes(2, 100, 96) == 0
    assert lib.kvq_swa_replay(w, 2, 96, e, 100, 16, st, None, ws, need, None) == 1    # d
    assert lib.kvq_swa_replay(w, 0, 128, e, 100, 16, st, None, ws, need, None) == 1   # layers
    assert lib.kvq_swa_replay(w, 2, 128, e, 100, 101, st, None, ws, need, None) == 1  # n_win > n
    assert lib.kvq_swa_replay(w, 2, 128, e, 9000, 4097, st, None, ws, 1 << 30, None) == 1  # n_win > 4096
    assert lib.kvq_swa_replay(w, 2, 128, e, 100, 16, None, None, ws, need, None) == 1  # no states
    assert lib.kvq_swa_replay(w, 2, 128, e, 100, 16, st, None, ws + 4, need, None) == 1  # workspace alignment
    assert lib.kvq_swa_replay(w, 2, 128, e, 100, 16, st, None, ws, need - 4, None) == 3  # too small


def test_fp4_pool_bytes(lib):
    assert lib.kvq_fp4_pool_bytes(10, 8, 64, 128) == 10 * 8 * 64 * 144
    assert lib.kvq_fp4_pool_bytes(3, 2, 16, 64) == 3 * 2 * 16 * 72
    assert lib.kvq_fp4_pool_bytes(3, 2, 48, 64) == 0
    assert lib.kvq_fp4_pool_bytes(3, 2, 64, 80) == 0


def test_status_strings_and_version(lib):
    assert lib.kvq_version() == 1
    assert lib.kvq_status_string(0) == b"ok"
    assert lib.kvq_status_string(1) == b"invalid argument"
    assert lib.kvq_status_string(3) == b"workspace too small"


def _fp4_struct(**kw):
    fields = dict(format=kvq.FORMAT_FP4, num_kv_heads=2, head_dim=128, page_size=64, num_pages=4,
                  max_pages_per_seq=2, reserved=0, page_table=None, data=4096, v_data=None,
                  k_scale=None, v_scale=None)
    fields.update(kw)
    return kvq.KvqCacheStruct(**fields)


@pytest.mark.parametrize("bad", [
    dict(head_dim=24), dict(head_dim=0), dict(head_dim=96), dict(page_size=48), dict(num_kv_heads=0),
    dict(reserved=1), dict(data=None), dict(data=4097), dict(v_data=8192), dict(k_scale=64), dict(format=7),
    dict(num_pages=1)])
def test_invalid_cache_is_rejected_on_the_host(lib, bad):
    s = _fp4_struct(**bad)
    st = lib.kvq_append(ctypes.byref(s), 2, 1, 16, 32, 64, None, None)
    assert st == 1  # KVQ_ERR_INVALID_ARGUMENT, nothing enqueued


def test_invalid_sizes_are_rejected_on_the_host(lib):
    s = _fp4_struct()
    assert lib.kvq_append(ctypes.byref(s), -1, 1, 16, 32, 64, None, None) == 1
    assert lib.kvq_append(ctypes.byref(s), 2, -3, 16, 32, 64, None, None) == 1
    assert lib.kvq_append(ctypes.byref(s), 2, 1, None, 32, 64, None, None) == 1
    # one sequence's 16-value blocks must fit the kernel's 32-bit item index
    assert lib.kvq_append(ctypes.byref(s), 2, 1 << 27, 16, 32, 64, None, None) == 2
    # empty work is a no-op that succeeds without a launch
    assert lib.kvq_append(ctypes.byref(s), 0, 5, None, None, None, None, None) == 0
    assert lib.kvq_append(ctypes.byref(s), 2, 0, None, None, None, None, None) == 0
    # decode: bad group size, scale and null pointers are rejected before any launch
    assert lib.kvq_decode_attn(ctypes.byref(s), None, 2, 3, 16, 32, 0.1, 64, 128, 1 << 20, None, None) == 1
    assert lib.kvq_decode_attn(ctypes.byref(s), None, 2, 4, 16, 32, -1.0, 64, 128, 1 << 20, None, None) == 1
    assert lib.kvq_decode_attn(ctypes.byref(s), None, 2, 4, None, 32, 0.1, 64, 128, 1 << 20, None, None) == 1
    assert lib.kvq_dequant(ctypes.byref(s), 2, 16, 8, 5, 32, 64, None, None) == 1
