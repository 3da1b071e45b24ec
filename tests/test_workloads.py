"""The seeded synthetic inputs follow their stated recipe (shapes, length
mix, page tables, outlier structure, distributions), and have the properties
the parity tests rely on (each sequence redrawn on its own; a replay
position's input independent of the range drawn).  CPU only; small draws."""
import math

import numpy as np
import pytest
import torch

from fp4_kv_cache_kvq_gb300 import workloads

W = workloads.WORKLOADS


def _fp4_bytes_per_token(w):
    return 2 * w.num_kv_heads * (w.head_dim // 2 + w.head_dim // 16)


@pytest.mark.parametrize("name,shape", [
    ("tiny", (1, 2, 2, 64, 256)),
    ("gqa_outliers", (8, 8, 32, 128, 4096)),
    ("long_context", (32, 8, 64, 128, 32768)),
    ("swa_append", (16, 8, 64, 128, 65536)),
    ("prefill", (16, 8, 8, 128, 16384)),
    ("prefill_b1", (1, 8, 8, 128, 16384)),
    ("prefill_attn", (4, 8, 64, 128, 16384)),
])
def test_shapes(name, shape):
    w = W[name]
    assert (w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim, w.context) == shape
    assert w.num_q_heads % w.num_kv_heads == 0


def test_cache_sizes_of_the_decode_configurations():
    # FP4 codes + E4M3 scales: 2 (K, V) x (d/2 + d/16) bytes per kv head and position
    assert _fp4_bytes_per_token(W["tiny"]) * 256 == 36_864
    assert _fp4_bytes_per_token(W["gqa_outliers"]) * 8 * 4096 == 37_748_736
    assert _fp4_bytes_per_token(W["long_context"]) * 32 * 32768 == 1_207_959_552
    assert _fp4_bytes_per_token(W["swa_append"]) * 16 * 65536 == 1_207_959_552
    w = W["swa_append"]
    assert w.window == 128 and w.batch * w.num_kv_heads * w.window * w.head_dim * 2 == 4_194_304  # FP8 K and V
    assert W["prefill_attn"].chunk == 1024


def test_paged_ragged_lengths_and_page_tables():
    w = W["paged_ragged"]
    assert (w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim, w.page_size) == (64, 8, 32, 128, 64)
    lens = workloads.lengths(w)
    assert len(lens) == 64 and all(1024 <= n <= 131072 for n in lens)
    assert lens == workloads.lengths(w)  # seeded
    assert lens != workloads.lengths(w, seed=1)
    # about 64 x the mean of U[1024, 131072] positions
    assert 0.6 * 64 * 66048 < sum(lens) < 1.4 * 64 * 66048
    table, pool, max_pages = workloads.page_layout(w, lens)
    need = [-(-n // 64) for n in lens]
    assert pool == sum(need) and max_pages == max(need)
    used = np.concatenate([table[b, :need[b]].numpy() for b in range(64)])
    # one permutation of the pool, cut into consecutive slices in sequence order
    assert np.array_equal(np.sort(used), np.arange(pool))
    assert all((table[b, need[b]:] == -1).all() for b in range(64))
    # contiguous layout: no table
    t2, pool2, mp2 = workloads.page_layout(W["long_context"], workloads.lengths(W["long_context"]))
    assert t2 is None and mp2 == 512 and pool2 == 32 * 512


def test_bf16_normal_draws_and_sequence_independence():
    w = W["long_context"]
    k, v = workloads.sequence_kv(w, 3, 2048, seed=0)
    assert k.dtype == torch.bfloat16 and k.shape == (2048, 8, 128) and v.shape == k.shape
    for x in (k.float(), v.float()):
        assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    # sequence b's draws depend only on (seed, b, length): K is drawn first,
    # so its first n tokens are a prefix of a longer draw (V follows all of K)
    k1, v1 = workloads.sequence_kv(w, 3, 2048, seed=0)
    assert torch.equal(k1, k) and torch.equal(v1, v)
    k2, _ = workloads.sequence_kv(w, 3, 4096, seed=0)
    assert torch.equal(k2[:2048], k)
    k3, _ = workloads.sequence_kv(w, 4, 2048, seed=0)
    assert not torch.equal(k3, k)
    q = workloads.queries(w, seed=0, step=1)
    assert q.shape == (32, 64, 128) and q.dtype == torch.bfloat16
    assert not torch.equal(q, workloads.queries(w, seed=0, step=2))


def test_fixed_outlier_channels():
    w = W["gqa_outliers"]
    assert w.k_outlier_channels == (3, 17, 64, 101) and w.k_outlier_factor == 20.0
    # the outliers fall in 16-channel blocks 0, 1, 4 and 6 of 8
    assert sorted({c // 16 for c in w.k_outlier_channels}) == [0, 1, 4, 6]
    k, v = workloads.sequence_kv(w, 0, 2048, seed=0)
    ka = k.float().abs().mean(dim=(0, 1))
    hot = list(w.k_outlier_channels)
    cold = [c for c in range(128) if c not in hot]
    ratio = ka[hot].mean() / ka[cold].mean()
    assert 19.0 < float(ratio) < 21.0
    va = v.float().abs().mean(dim=(0, 1))
    assert float(va[hot].mean() / va[cold].mean()) < 1.1  # values untouched
    kn, vn = workloads.step_tokens(w, 1)
    assert kn.shape == (8, 1, 8, 128)


def test_iid_outlier_entries():
    w = W["paged_ragged"]
    assert w.k_outlier_prob == 0.02 and w.k_outlier_prob_factor == 30.0
    k, v = workloads.sequence_kv(w, 0, 4096, seed=0)
    # |30 x| > 6 for |x| > 0.2 (probability ~0.84); an N(0,1) entry passes 6
    # with probability ~2e-9
    frac = float((k.float().abs() > 6.0).float().mean())
    expect = 0.02 * math.erfc(0.2 / math.sqrt(2.0))
    assert abs(frac - expect) < 0.1 * expect
    assert float((v.float().abs() > 6.0).float().mean()) < 1e-6


def test_replay_inputs_do_not_depend_on_the_range_drawn():
    """Position p's input row is the same whichever range it is drawn in, which
    is what lets a replay from a later start see the same inputs as the full
    forward pass."""
    d = 64
    full = workloads.replay_inputs(0, 3000, d, seed=2)
    part = workloads.replay_inputs(1234, 1500, d, seed=2)
    assert torch.equal(part, full[1234:2734])
    assert abs(float(full.mean())) < 0.01 and abs(float(full.std()) - 1.0) < 0.01
    net = workloads.replay_net(3, d, seed=2)
    assert net.shape == (3, 4, d, d)
    assert abs(float(net.std()) * math.sqrt(d) - 1.0) < 0.02
    R = workloads.REPLAY
    assert (R["layers"], R["d"], R["n_win"], R["T"]) == (8, 128, 512, 65536)
