"""Pins for the oracle's toy sliding-window network and its replays ("Week 6
-- FP4 KV Caches and Bounded Replay", Core Concepts "Bounded replay", Lab).

Each pin checks the oracle against something other than its own code:
  * the receptive-field argument: starting n_win - 1 positions further back
    per layer reproduces the full forward's window state exactly, and one
    position later no longer does;
  * one layer: the window state depends only on the last n_win inputs, so a
    bounded replay is exact;
  * a window covering the whole range is plain causal attention, written here
    in matrix form with a mask (a textbook routine);
  * n_win = 1: each position attends only itself (closed form);
  * RMS normalisation: scaling any position's input leaves its K, V and q
    unchanged, so the layer output moves by exactly the scaled input."""
import numpy as np
import pytest

import oracle


def _net(L, d, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((L, 4, d, d)) / np.sqrt(d)


def _emb(n, d, seed):
    return np.random.default_rng(seed + 1000).standard_normal((n, d))


@pytest.mark.parametrize("L,d,n_win,T", [(3, 8, 4, 40), (2, 16, 5, 23), (4, 8, 3, 17)])
def test_exact_replay_start_reproduces_full_forward(L, d, n_win, T):
    w, e = _net(L, d, T), _emb(T, d, T)
    _, full = oracle.swa_forward(w, e, n_win)
    t0 = oracle.exact_replay_start(T, L, n_win)
    assert t0 == T - L * n_win + L - 1 and t0 > 0
    _, rep = oracle.swa_forward(w, e[t0:], n_win)
    assert np.array_equal(rep, full)
    # one position later the top layer's window is no longer exact
    _, late = oracle.swa_forward(w, e[t0 + 1:], n_win)
    assert np.array_equal(late[0], full[0])          # the first layer still is
    assert not np.array_equal(late[L - 1], full[L - 1])


def test_one_layer_bounded_replay_is_exact():
    w, e = _net(1, 16, 3), _emb(50, 16, 3)
    _, full = oracle.swa_forward(w, e, 7)
    t0 = oracle.bounded_replay_start(50, 7)
    _, rep = oracle.swa_forward(w, e[t0:], 7)
    assert np.array_equal(rep, full)


def _rms(x):
    return x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6)


def test_full_window_is_causal_attention():
    d, n = 16, 12
    w, e = _net(1, d, 5), _emb(n, d, 5)
    hidden, states = oracle.swa_forward(w, e, n)
    U = _rms(e)
    Q, K, V = U @ w[0, 0].T, U @ w[0, 1].T, U @ w[0, 2].T
    S = Q @ K.T / np.sqrt(d)
    S[np.triu_indices(n, 1)] = -np.inf
    P = np.exp(S - S.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    ref = e + (P @ V) @ w[0, 3].T
    assert np.abs(hidden - ref).max() < 1e-12
    assert np.abs(states[0, 0] - K).max() < 1e-12 and np.abs(states[0, 1] - V).max() < 1e-12


def test_window_of_one_attends_itself():
    d, n = 8, 9
    w, e = _net(1, d, 6), _emb(n, d, 6)
    hidden, states = oracle.swa_forward(w, e, 1)
    U = _rms(e)
    ref = e + (U @ w[0, 2].T) @ w[0, 3].T
    assert np.abs(hidden - ref).max() < 1e-12
    assert np.abs(states[0, 1, 0] - U[-1] @ w[0, 2].T).max() < 1e-12


def test_rms_normalisation_scale_invariance():
    """Inputs near 1000 make the normalisation's 1e-6 epsilon negligible
    (relative 1e-12), so the invariance must hold to rounding."""
    d, n = 8, 10
    w, e = _net(1, d, 7), 1000.0 * _emb(n, d, 7)
    c = np.linspace(0.25, 4.0, n)[:, None]
    h1, s1 = oracle.swa_forward(w, e, 4)
    h2, s2 = oracle.swa_forward(w, e * c, 4)
    assert np.abs(s2 - s1).max() < 1e-9
    assert np.abs((h2 - c * e) - (h1 - e)).max() < 1e-8
