"""kvq_swa_replay (the toy sliding-window network and its replays) against
the fp64 oracle, plus the properties the replay rests on, checked on the GPU
output itself:

  * every layer's window state and the last layer's output match the oracle
    within 2e-5 * max|ref| per layer (fp32 against fp64: d-term dot products,
    an expf per score and a residual stream that grows with depth stay far
    inside it);
  * a replay from the exact start reproduces a forward over the whole range
    bit for bit (the kernels' arithmetic for a position depends only on its
    window, in a fixed order);
  * with one layer the bounded replay is exact;
  * window 1 and window = range edge cases, and the largest window (4096)."""
import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import ensure_built

pytestmark = pytest.mark.gpu

TOL = 2e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _close(got: torch.Tensor, ref: np.ndarray, what: str) -> float:
    got = got.double().cpu().numpy()
    scale = float(np.abs(ref).max())
    err = float(np.abs(got - ref).max())
    assert err <= TOL * scale, (what, err, scale)
    return err / scale


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L,n_win,n", [(1, 7, 150), (3, 1, 40), (3, 64, 150), (2, 33, 33)])
def test_matches_oracle(d, L, n_win, n):
    w = workloads.replay_net(L, d, seed=d + L)
    e = workloads.replay_inputs(500, n, d, seed=n_win)
    states, hidden = kvq.swa_replay(w.cuda(), e.cuda(), n_win)
    torch.cuda.synchronize()
    ref_h, ref_s = oracle.swa_forward(w.numpy(), e.numpy(), n_win)
    for l in range(L):
        _close(states[l], ref_s[l], f"state {l}")
    _close(hidden, ref_h, "hidden")


def test_matches_oracle_wide_window():
    L, d, n_win, n = 2, 128, 512, 600
    w = workloads.replay_net(L, d, seed=9)
    e = workloads.replay_inputs(0, n, d, seed=9)
    states, hidden = kvq.swa_replay(w.cuda(), e.cuda(), n_win)
    torch.cuda.synchronize()
    ref_h, ref_s = oracle.swa_forward(w.numpy(), e.numpy(), n_win)
    for l in range(L):
        _close(states[l], ref_s[l], f"state {l}")
    _close(hidden, ref_h, "hidden")


@pytest.mark.parametrize("d,L,n_win,T", [(128, 4, 64, 700), (64, 3, 17, 300), (128, 2, 4096, 8200)])
def test_exact_replay_is_bit_exact(d, L, n_win, T):
    w = workloads.replay_net(L, d, seed=T).cuda()
    e = workloads.replay_inputs(0, T, d, seed=T).cuda()
    full, _ = kvq.swa_replay(w, e, n_win, want_hidden=False)
    t0 = oracle.exact_replay_start(T, L, n_win)
    assert t0 > 0
    rep, _ = kvq.swa_replay(w, e[t0:].contiguous(), n_win, want_hidden=False)
    torch.cuda.synchronize()
    assert torch.equal(rep, full)
    # a bounded replay keeps the first layer exact and differs above it
    tb = oracle.bounded_replay_start(T, n_win)
    bnd, _ = kvq.swa_replay(w, e[tb:].contiguous(), n_win, want_hidden=False)
    torch.cuda.synchronize()
    assert torch.equal(bnd[0], full[0])
    assert not torch.equal(bnd[L - 1], full[L - 1])


def test_one_layer_bounded_replay_is_exact():
    d, n_win, T = 128, 100, 1000
    w = workloads.replay_net(1, d, seed=3).cuda()
    e = workloads.replay_inputs(0, T, d, seed=3).cuda()
    full, _ = kvq.swa_replay(w, e, n_win, want_hidden=False)
    rep, _ = kvq.swa_replay(w, e[T - n_win:].contiguous(), n_win, want_hidden=False)
    torch.cuda.synchronize()
    assert torch.equal(rep, full)


def test_benchmark_configuration():
    """The benchmark's toy (L8, d128, window 512, state after 65536
    positions): the exact replay (4089 positions) equals a forward over all
    65536 positions bit for bit, and the bounded replay matches the oracle."""
    R = workloads.REPLAY
    L, d, nw, T = R["layers"], R["d"], R["n_win"], R["T"]
    w = workloads.replay_net(L, d, seed=0).cuda()
    e = workloads.replay_inputs(0, T, d, seed=0).cuda()
    full, _ = kvq.swa_replay(w, e, nw, want_hidden=False)
    t0 = oracle.exact_replay_start(T, L, nw)
    assert T - t0 == 4089
    rep, _ = kvq.swa_replay(w, e[t0:].contiguous(), nw, want_hidden=False)
    bnd, hid = kvq.swa_replay(w, e[T - nw:].contiguous(), nw)
    torch.cuda.synchronize()
    assert torch.equal(rep, full)
    ref_h, ref_s = oracle.swa_forward(w.cpu().numpy(), e[T - nw:].cpu().numpy(), nw)
    for l in range(L):
        _close(bnd[l], ref_s[l], f"state {l}")
    _close(hid, ref_h, "hidden")
