"""kvq_decode_attn against fp64 attention over the oracle's own dequantised
cache: max |err| <= 2e-3 * max |V^| for every (sequence, kv head) unit.

Small cases cover every head_dim (64, 128), group size (1, 2, 4, 8), page
size (16 .. 256), contiguous and paged layouts, ragged tails shorter than a
warp's 16-token slice, empty sequences, a single long sequence spread over
many CTAs and many short sequences packed into one CTA.  The tiny and
gqa_outliers workloads are checked in full; long_context and paged_ragged at
full size on sampled units, in the launch configuration the benchmark times.
"""
import math

import numpy as np
import pytest
import torch

from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import build_fp4, check_units, ensure_built, host_kv_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def run_case(w, lens, seed=0, units=None, q=None, scale=None):
    built = build_fp4(w, lens, seed=seed)
    if q is None:
        q = workloads.queries(w, seed=seed, device="cuda")
    scale = scale if scale is not None else 1.0 / math.sqrt(w.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvq.decode_attn(built.cache, built.lens_dev, q, scale, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.isfinite(out).all()
    if units is None:
        units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    worst = check_units(out, q, units, host_kv_of(built), w.group, scale)
    return built, out, worst


BASE = workloads.WORKLOADS["gqa_outliers"]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_group_sizes_and_head_dims(d, g):
    w = workloads.scaled(BASE, batch=3, num_kv_heads=2, num_q_heads=2 * g, head_dim=d,
                         k_outlier_channels=(3, 17, 40) if d == 64 else (3, 17, 64, 101))
    run_case(w, [300, 1, 77], seed=g + d)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("paged", [False, True])
def test_page_sizes_and_layouts(page_size, paged):
    w = workloads.scaled(BASE, batch=4, num_kv_heads=2, num_q_heads=8, page_size=page_size, paged=paged)
    run_case(w, [1000, 15, 64, 129], seed=page_size)


def test_ragged_tails_and_empty_sequences():
    w = workloads.scaled(BASE, batch=9, num_kv_heads=3, num_q_heads=12, paged=True)
    lens = [0, 1, 2, 15, 16, 17, 63, 65, 0]
    run_case(w, lens, seed=5)


def test_many_short_sequences_share_ctas():
    w = workloads.scaled(BASE, batch=300, num_kv_heads=2, num_q_heads=8, paged=True)
    lens = [int(x) for x in np.random.default_rng(1).integers(1, 200, size=300)]
    run_case(w, lens, seed=6, units=[(b, h) for b in range(0, 300, 7) for h in range(2)])


def test_one_long_sequence_over_many_ctas():
    w = workloads.scaled(BASE, batch=1, num_kv_heads=1, num_q_heads=8, k_outlier_channels=())
    run_case(w, [200_000], seed=7)


def test_query_dynamic_range():
    """bf16 queries far outside f16's range are pre-scaled by a power of two."""
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8, k_outlier_channels=())
    q = workloads.queries(w, seed=8, device="cuda").float()
    q[0] *= 1e-12
    q[1, :4] *= 3e3
    q[1, 4:, :64] *= 1e-20
    run_case(w, [500, 700], seed=8, q=q.to(torch.bfloat16), scale=0.02)


def test_softmax_scales():
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8)
    for scale in (1e-3, 0.5, 2.0):
        run_case(w, [300, 100], seed=9, scale=scale)


def test_tiny_workload_in_full():
    w = workloads.WORKLOADS["tiny"]
    run_case(w, workloads.lengths(w))


def test_gqa_outliers_workload_in_full():
    w = workloads.WORKLOADS["gqa_outliers"]
    run_case(w, workloads.lengths(w))


def _sampled_units(w, lens, n=6, seed=0):
    rng = np.random.default_rng(seed)
    bs = sorted({0, w.batch - 1, *rng.integers(0, w.batch, size=n).tolist()})
    return [(int(b), int(rng.integers(0, w.num_kv_heads))) for b in bs if lens[b] > 0]


def test_long_context_full_size_sampled():
    w = workloads.WORKLOADS["long_context"]
    lens = workloads.lengths(w)
    run_case(w, lens, units=_sampled_units(w, lens, n=4))


def test_paged_ragged_full_size_sampled():
    w = workloads.WORKLOADS["paged_ragged"]
    lens = workloads.lengths(w)
    run_case(w, lens, units=_sampled_units(w, lens, n=4, seed=1))


def test_out_of_range_page_sets_flag_without_fault():
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8, paged=True)
    built = build_fp4(w, [256, 256], seed=10)
    bad = built.table.clone()
    bad[1, 2] = 10_000_000  # page id beyond the pool
    built.cache.page_table = bad
    q = workloads.queries(w, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvq.decode_attn(built.cache, built.lens_dev, q, err=err)
    torch.cuda.synchronize()
    assert err.item() & kvq.FLAG_PAGE_OOB
    assert torch.isfinite(out).all()
    # sequence 0 does not touch the bad page and is still exact
    check_units(out, q, [(0, 0), (0, 1)], host_kv_of(built), w.group, 1.0 / math.sqrt(w.head_dim))


def test_negative_length_flag():
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8)
    built = build_fp4(w, [64, 64], seed=11)
    lens = torch.tensor([64, -5], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvq.decode_attn(built.cache, lens, workloads.queries(w, device="cuda"), err=err)
    torch.cuda.synchronize()
    assert err.item() & kvq.FLAG_BAD_LENGTH
    assert not out[1].any()


def test_workspace_too_small_is_refused():
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8)
    built = build_fp4(w, [64, 64], seed=12)
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attn(built.cache, built.lens_dev, workloads.queries(w, device="cuda"), workspace=ws)
    assert e.value.status == 3


def test_decode_replays_from_a_cuda_graph():
    """kvq_decode_attn enqueues only kernels on the caller's stream (no
    allocation, no synchronisation), so it can be captured in a CUDA graph; a
    replay gives the eager result bit for bit, and a replay after the captured
    query is changed in place computes with the new values."""
    w = workloads.scaled(BASE, batch=3, num_kv_heads=2, num_q_heads=8)
    lens = [700, 129, 64]
    built = build_fp4(w, lens, seed=11)
    q = workloads.queries(w, seed=11, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(kvq.decode_workspace_bytes(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim), 16),
                     dtype=torch.uint8, device="cuda")
    eager = kvq.decode_attn(built.cache, built.lens_dev, q, workspace=ws, err=err).clone()
    out = torch.empty_like(eager)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            kvq.decode_attn(built.cache, built.lens_dev, q, out=out, workspace=ws, err=err)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    q2 = workloads.queries(w, seed=12, device="cuda")
    q.copy_(q2)
    eager2 = kvq.decode_attn(built.cache, built.lens_dev, q2, workspace=ws, err=err).clone()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager2) and not torch.equal(eager2, eager)
    assert err.item() == 0
