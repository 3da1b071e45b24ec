"""The bounded-wait path of the decode kernel, exercised on the GPU without a
fault or a hang: the kernel's work waits (a consumer waiting for a stage to
land, the producer waiting for a free stage) are shortened to 1 ns through
kvq_test_set_wait_limit_ns, so they give up at once.  The call must return,
raise KVQ_FLAG_TIMEOUT, and leave the context usable: the next call with the
default limit reproduces the result taken before, bit for bit.  (The
producer always drains the copies it issued with the fixed limit, so no copy
lands in the shared memory of a retired CTA.)
"""
import math

import pytest
import torch

from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import build_fp4, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    return ensure_built()


@pytest.mark.parametrize("fused,context", [(False, 65536), (True, 65536), (True, 8192)])
def test_short_wait_limit_times_out_and_returns(lib, fused, context):
    # 65536 positions: about 36 chunks per CTA range, so every producer reaches
    # its fourth stage and waits for the consumers to free one, and
    # kvq_append_decode_attn fuses the append into the decode kernel.  8192
    # positions: about 9 chunks per range, under the capacity at which it
    # fuses, so it launches the append kernel and the decode as its
    # programmatic dependent
    w = workloads.scaled(workloads.WORKLOADS["long_context"], batch=8, context=context, k_outlier_channels=())
    lens = [context] * 8
    built = build_fp4(w, lens, seed=11, reserve=1, keep_kv=False)
    q = workloads.queries(w, seed=11, device="cuda")
    scale = 1.0 / math.sqrt(w.head_dim)
    kn, vn = workloads.step_tokens(w, 1, seed=11, device="cuda")
    kn, vn = kn[:, 0].contiguous(), vn[:, 0].contiguous()
    lens_dev = built.lens_dev

    def call(err):
        if fused:
            return kvq.append_decode_attn(built.cache, lens_dev, kn, vn, q, scale, err=err)
        return kvq.decode_attn(built.cache, lens_dev, q, scale, err=err)

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = call(err)
    torch.cuda.synchronize()
    assert err.item() == 0
    try:
        lib.kvq_test_set_wait_limit_ns(1)
        err_t = torch.zeros(1, dtype=torch.int32, device="cuda")
        call(err_t)
        torch.cuda.synchronize()  # the call returned
        assert err_t.item() & kvq.FLAG_TIMEOUT
    finally:
        lib.kvq_test_set_wait_limit_ns(0)
    err2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    again = call(err2)
    torch.cuda.synchronize()
    assert err2.item() == 0
    assert torch.equal(again, ref)
