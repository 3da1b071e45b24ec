"""The decode grid chosen from the cache's capacity: three CTAs per SM, or two
when three per SM would get fewer than 8 chunks each.  The same sequences
decoded from two caches whose page-table rows differ only in length (so the
capacity, not the content, differs) on either side of that threshold: both
outputs within the decode tolerance of the oracle, and close to each other.

How close: the split points differ, so each CTA's softmax reference (its
running max) differs, and P = 2^(S - m) is rounded to f16 against a
different reference.  A relative rounding u = 2^-11 of every weight moves a
normalised average by at most 2u/(1 - u) of max|V^|, so two evaluations
differ by at most about 2^-9 max|V^| (the fp32 accumulation adds far less),
with max|V^| <= 1.0625 max|V| (the largest E2M1 rounding of a block's
maximum)."""
import math

import pytest
import torch

from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import build_fp4, check_units, ensure_built, host_kv_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def test_two_and_three_ctas_per_sm_agree():
    w = workloads.scaled(workloads.WORKLOADS["gqa_outliers"], batch=8, paged=True)
    lens = [4096, 3000, 4096, 1, 4000, 2048, 4096, 129]
    props = torch.cuda.get_device_properties(0)
    ctas3 = 3 * props.multi_processor_count
    units = w.batch * w.num_kv_heads
    # capacities in chunks of 128 positions per unit: below 8 per range at
    # three per SM, and well above it
    small_pos = 4096 + 1
    assert units * -(-small_pos // 128) < 8 * ctas3
    large_pos = -(-16 * ctas3 // units) * 128
    built_small = build_fp4(w, lens, seed=21, reserve=small_pos - max(lens), keep_kv=True)
    built_large = build_fp4(w, lens, seed=21, reserve=large_pos - max(lens), keep_kv=False)
    assert built_large.cache.max_pages_per_seq > built_small.cache.max_pages_per_seq
    q = workloads.queries(w, seed=21, device="cuda")
    scale = 1.0 / math.sqrt(w.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o_small = kvq.decode_attn(built_small.cache, built_small.lens_dev, q, scale, err=err)
    o_large = kvq.decode_attn(built_large.cache, built_large.lens_dev, q, scale, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    G = w.num_q_heads // w.num_kv_heads
    units_all = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    kv_of = host_kv_of(built_small)
    check_units(o_small, q, units_all, kv_of, G, scale)
    check_units(o_large, q, units_all, kv_of, G, scale)
    vmax = max(float(v.abs().max()) for v in built_small.seq_v if v.numel())
    assert (o_small - o_large).abs().max().item() <= 2.0 ** -9 * 1.0625 * vmax * 1.01
