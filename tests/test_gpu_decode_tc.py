"""kvq_decode_attn_tc (head_dim 128, both products on the tensor-memory MMA)
against fp64 attention over the oracle's dequantised cache, with the bound of
kvq_decode_attn: max |err| <= 2e-3 * max |V^| per (sequence, kv head) unit.

It shares the workspace, partials and merge of kvq_decode_attn and differs in
the decode kernel only, so the cases cover what that kernel decides: group
sizes (the 16-row query tile padded from G rows), page sizes (pool groups per
128-token stage), ragged and empty sequences (masked tokens of a partial
stage), ranges that start and end inside units (three pipelines per CTA, each
its own range), extreme query magnitudes (the per-row power-of-two prescale),
the FP8 window and the long-context benchmark shape.
"""
import math

import numpy as np
import pytest
import torch

from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import build_fp4, check_units, ensure_built, host_kv_of
from tests.test_gpu_swa import run_loop

pytestmark = pytest.mark.gpu

BASE = workloads.WORKLOADS["gqa_outliers"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def run_tc(w, lens, seed=0, units=None, q=None, scale=None):
    built = build_fp4(w, lens, seed=seed)
    if q is None:
        q = workloads.queries(w, seed=seed, device="cuda")
    scale = scale if scale is not None else 1.0 / math.sqrt(w.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvq.decode_attn(built.cache, built.lens_dev, q, scale, err=err, kernel="tcgen05")
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.isfinite(out).all()
    if units is None:
        units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    return check_units(out, q, units, host_kv_of(built), w.group, scale)


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_group_sizes(g):
    w = workloads.scaled(BASE, batch=3, num_kv_heads=2, num_q_heads=2 * g)
    run_tc(w, [300, 1, 77], seed=g)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
def test_page_sizes(page_size):
    w = workloads.scaled(BASE, batch=4, num_kv_heads=2, num_q_heads=8, page_size=page_size, paged=True)
    run_tc(w, [1000, 15, 64, 129], seed=page_size)


def test_ragged_tails_and_empty_sequences():
    w = workloads.scaled(BASE, batch=9, num_kv_heads=3, num_q_heads=12, paged=True)
    run_tc(w, [0, 1, 2, 15, 16, 17, 63, 65, 0], seed=5)


def test_one_long_sequence_over_many_pipelines():
    w = workloads.scaled(BASE, batch=1, num_kv_heads=1, num_q_heads=8, k_outlier_channels=())
    run_tc(w, [200_000], seed=7)


def test_many_short_sequences():
    w = workloads.scaled(BASE, batch=300, num_kv_heads=2, num_q_heads=8, paged=True)
    lens = [int(x) for x in np.random.default_rng(1).integers(1, 200, size=300)]
    run_tc(w, lens, seed=6, units=[(b, h) for b in range(0, 300, 7) for h in range(2)])


def test_query_dynamic_range():
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8, k_outlier_channels=())
    q = workloads.queries(w, seed=8, device="cuda").float()
    q[0] *= 1e-12
    q[1, :4] *= 3e3
    q[1, 4:, :64] *= 1e-20
    run_tc(w, [500, 700], seed=8, q=q.to(torch.bfloat16), scale=0.02)


def test_with_fp8_window():
    w = workloads.scaled(workloads.WORKLOADS["swa_append"], batch=3, num_kv_heads=2, num_q_heads=16,
                         context=300, window=128)
    every = lambda s: [(b, h) for b in range(3) for h in range(2)]  # noqa: E731
    run_loop(w, [300] * 3, steps=3, check_steps={1, 3}, units_of_step=every, kernel="tcgen05")


def test_long_context_full_size_sampled():
    w = workloads.WORKLOADS["long_context"]
    lens = workloads.lengths(w)
    rng = np.random.default_rng(0)
    units = [(int(b), int(rng.integers(0, w.num_kv_heads))) for b in (0, 13, w.batch - 1)]
    run_tc(w, lens, units=units)


def test_head_dim_64_is_refused():
    w = workloads.scaled(BASE, batch=1, num_kv_heads=1, num_q_heads=8, head_dim=64,
                         k_outlier_channels=(3, 17, 40))
    built = build_fp4(w, [100])
    q = workloads.queries(w, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attn(built.cache, built.lens_dev, q, kernel="tcgen05")
    assert e.value.status == 2  # KVQ_ERR_UNSUPPORTED
