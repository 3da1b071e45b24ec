"""Global FP4 cache + FP8 sliding window, with appends between decode steps.

Each step appends one token per sequence to both caches (FP4 at position T,
FP8 ring slot T mod W), then decodes: positions [0, T - W') come from the FP4
cache, the last W' = min(W, T) from the FP8 window, one softmax over the
union ("Week 6 -- FP4 KV Caches and Bounded Replay": global KV ~4-bit, SWA
KV FP8).  The FP8 per-head scales are set once from the initial window and
checked against the oracle; the oracle then quantises everything itself.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import build_fp4, check_units, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def run_loop(w, lens, steps, check_steps, units_of_step, seed=0, kernel="mma"):
    W = w.window
    built = build_fp4(w, lens, seed=seed, reserve=steps + 1)
    B, Hkv, d, G = w.batch, w.num_kv_heads, w.head_dim, w.group
    swa = kvq.Fp8WindowCache(B, Hkv, d, W)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # initial window: the last min(W, T) prefill positions of every sequence
    T0 = min(lens)
    assert all(n == T0 for n in lens)
    w0 = min(W, T0)
    if w0 > 0:
        kw = torch.stack([built.seq_k[b][T0 - w0:] for b in range(B)]).contiguous()
        vw = torch.stack([built.seq_v[b][T0 - w0:] for b in range(B)]).contiguous()
        kvq.fp8_set_scales(swa, kw, vw, err=err)
        kvq.append(swa, torch.full((B,), T0 - w0, dtype=torch.int32, device="cuda"), kw, vw, err=err)
        sk = [oracle.fp8_head_scale(kw[:, :, h].float().cpu().numpy()) for h in range(Hkv)]
        sv = [oracle.fp8_head_scale(vw[:, :, h].float().cpu().numpy()) for h in range(Hkv)]
        torch.cuda.synchronize()
        assert swa.k_scales.cpu().numpy().tolist() == sk
        assert swa.v_scales.cpu().numpy().tolist() == sv
    else:
        sk = sv = [1.0] * Hkv
    host_k = [built.seq_k[b].float().cpu() for b in range(B)]
    host_v = [built.seq_v[b].float().cpu() for b in range(B)]
    scale = 1.0 / math.sqrt(d)
    worst = 0.0
    T = T0
    for step in range(1, steps + 1):
        kn, vn = workloads.step_tokens(w, step, seed=seed, device="cuda")
        pos = torch.full((B,), T, dtype=torch.int32, device="cuda")
        kvq.append(built.cache, pos, kn, vn, err=err)
        kvq.append(swa, pos, kn, vn, err=err)
        T += 1
        lens_dev = torch.full((B,), T, dtype=torch.int32, device="cuda")
        q = workloads.queries(w, seed=seed, step=step, device="cuda")
        out = kvq.decode_attn(built.cache, lens_dev, q, scale, swa=swa, err=err, kernel=kernel)
        for b in range(B):
            host_k[b] = torch.cat([host_k[b], kn[b, :1].float().cpu()])
            host_v[b] = torch.cat([host_v[b], vn[b, :1].float().cpu()])
        if step in check_steps:
            torch.cuda.synchronize()
            assert err.item() == 0
            worst = max(worst, check_units(
                out, q, units_of_step(step), lambda b, h: (host_k[b][:, h].numpy(), host_v[b][:, h].numpy()),
                G, scale, window=W, swa_scales_of=lambda h: (sk[h], sv[h])))
    return worst


@pytest.mark.parametrize("T0", [0, 1, 50, 127, 128, 300])
def test_window_boundaries(T0):
    w = workloads.scaled(workloads.WORKLOADS["swa_append"], batch=3, num_kv_heads=2, num_q_heads=8,
                         context=T0, window=128)
    every = lambda s: [(b, h) for b in range(3) for h in range(2)]  # noqa: E731
    run_loop(w, [T0] * 3, steps=3, check_steps={1, 2, 3}, units_of_step=every)


def test_small_window_many_steps():
    w = workloads.scaled(workloads.WORKLOADS["swa_append"], batch=2, num_kv_heads=2, num_q_heads=4,
                         context=40, window=16, head_dim=64)
    every = lambda s: [(b, h) for b in range(2) for h in range(2)]  # noqa: E731
    run_loop(w, [40] * 2, steps=40, check_steps=set(range(1, 41, 3)), units_of_step=every)


@pytest.mark.parametrize("W,T0", [(1024, 1500), (1024, 700), (200, 450)])
def test_large_and_odd_windows(W, T0):
    """Windows spanning several 128-token V tiles (a ragged last tile), the
    largest window the library takes, and a window still filling up."""
    w = workloads.scaled(workloads.WORKLOADS["swa_append"], batch=2, num_kv_heads=2, num_q_heads=16,
                         context=T0, window=W)
    every = lambda s: [(b, h) for b in range(2) for h in range(2)]  # noqa: E731
    run_loop(w, [T0] * 2, steps=2, check_steps={1, 2}, units_of_step=every)


def test_swa_append_workload_full_size_sampled():
    w = workloads.WORKLOADS["swa_append"]
    rng = np.random.default_rng(3)

    def units(step):
        return [(int(rng.integers(0, w.batch)), int(rng.integers(0, w.num_kv_heads))) for _ in range(2)]

    run_loop(w, workloads.lengths(w), steps=32, check_steps={1, 2, 3, 4, 32}, units_of_step=units)
