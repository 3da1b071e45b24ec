"""Pins for the oracle's fp64 attention and its per-unit decode (CPU only).

"Quantising the KV cache", section "Code": the quantised K and V replace the
real ones ahead of an otherwise unchanged attention.  The attention is
therefore plain softmax(scale * q.k) v, pinned here against:
  * torch float64 softmax attention (a library routine) on the same inputs;
  * closed forms: one position returns its value row; identical keys return
    the mean of the values; m + log(l) equals torch.logsumexp of the scores;
  * invariance under a permutation of the positions;
  * decode_unit with a sliding window reads FP8 values for exactly the last
    min(W, T) positions and FP4 values for the rest.
"""
import numpy as np
import torch

import oracle


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16).float().numpy()


def test_attend_vs_torch_float64():
    for (G, T, d, seed) in [(1, 7, 16, 0), (8, 300, 128, 1), (4, 33, 64, 2)]:
        q, k, v = _rand((G, d), seed), _rand((T, d), seed + 10, 3.0), _rand((T, d), seed + 20)
        scale = 1.0 / np.sqrt(d)
        out, m, l = oracle.attend(q, k, v, scale)
        qt, kt, vt = (torch.from_numpy(a).double() for a in (q, k, v))
        s = (qt @ kt.T) * scale
        want = torch.softmax(s, dim=-1) @ vt
        assert np.allclose(out, want.numpy(), rtol=1e-12, atol=1e-12)
        lse = torch.logsumexp(s, dim=-1).numpy()
        assert np.allclose(m + np.log(l), lse, rtol=1e-12, atol=1e-12)
        assert np.allclose(m, s.max(dim=-1).values.numpy(), rtol=0, atol=0)


def test_attend_closed_forms():
    q, v = _rand((3, 32), 5), _rand((1, 32), 6)
    out, _, l = oracle.attend(q, _rand((1, 32), 7), v, 0.3)
    assert np.array_equal(out, np.repeat(v.astype(np.float64), 3, axis=0)) and np.all(l == 1.0)
    k = np.repeat(_rand((1, 32), 8), 50, axis=0)
    v = _rand((50, 32), 9)
    out, _, _ = oracle.attend(q, k, v, 0.3)
    assert np.allclose(out, np.repeat(v.astype(np.float64).mean(axis=0, keepdims=True), 3, axis=0),
                       rtol=1e-13, atol=1e-13)
    out, _, _ = oracle.attend(q, np.zeros((0, 32)), np.zeros((0, 32)), 0.3)
    assert np.all(out == 0)


def test_attend_permutation_invariance():
    q, k, v = _rand((4, 64), 11), _rand((97, 64), 12), _rand((97, 64), 13)
    perm = np.random.default_rng(0).permutation(97)
    a, _, _ = oracle.attend(q, k, v, 0.125)
    b, _, _ = oracle.attend(q, k[perm], v[perm], 0.125)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14)


def test_decode_unit_window_split():
    G, d = 4, 64
    q = _rand((G, d), 21)
    for T, W in [(300, 128), (100, 128), (128, 128), (1, 128), (129, 128), (50, 0)]:
        k, v = _rand((T, d), 22), _rand((T, d), 23)
        sk = oracle.fp8_head_scale(k[max(0, T - W):]) if W else 1.0
        sv = oracle.fp8_head_scale(v[max(0, T - W):]) if W else 1.0
        out, vmax = oracle.decode_unit(q, k, v, 0.125, window=W, swa_scales=(sk, sv))
        w = min(W, T) if W else 0
        kc, ks, _ = oracle.quantize_rows(k[: T - w])
        vc, vs, _ = oracle.quantize_rows(v[: T - w])
        kh = [oracle.dequantize_rows(kc, ks)]
        vh = [oracle.dequantize_rows(vc, vs)]
        if w:
            # FP8 window values: fp32 product of the E4M3 code and the head scale
            k8 = torch.from_numpy((k[T - w:] / np.float32(sk)).astype(np.float32)).clamp(-448, 448)
            v8 = torch.from_numpy((v[T - w:] / np.float32(sv)).astype(np.float32)).clamp(-448, 448)
            kh.append((k8.to(torch.float8_e4m3fn).float() * sk).double().numpy())
            vh.append((v8.to(torch.float8_e4m3fn).float() * sv).double().numpy())
        kh, vh = np.concatenate(kh), np.concatenate(vh)
        qt, kt, vt = (torch.from_numpy(np.asarray(a, np.float64)) for a in (q, kh, vh))
        want = torch.softmax((qt @ kt.T) * 0.125, dim=-1) @ vt
        assert np.allclose(out, want.numpy(), rtol=1e-12, atol=1e-12), (T, W)
        assert vmax == np.abs(vh).max()
