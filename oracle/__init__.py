"""CPU oracle for the FP4 KV cache and its decode attention.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product path never does and must fail loudly if its CUDA library is missing.

The arithmetic lives in ``kvq_oracle.c`` (plain C, fp32 where the method fixes
fp32, fp64 attention).  This module builds it with gcc on first use, loads it
with ctypes, and composes its primitives into the per-unit computations the
tests compare against:

  * ``quantize_rows`` / ``dequantize_rows`` -- the per-16-channel block
    quantiser of "Quantising the KV cache", section "Code".
  * ``fp8_head_scale`` / ``fp8_quantize`` / ``fp8_dequantize`` -- the FP8 E4M3
    sliding-window KV ("Week 6 -- FP4 KV Caches and Bounded Replay",
    "Overview": SWA KV stays FP8) with one fp32 scale per head.
  * ``attend`` -- fp64 softmax attention over dequantised K/V ("Quantising the
    KV cache", section "Code": the quantised K and V replace the real ones
    ahead of an unchanged attention).
  * ``nvfp4_global_scale`` / ``nvfp4_quantize_rows`` /
    ``nvfp4_dequantize_rows`` -- NVFP4: the FP4 block quantiser over x / S
    with one fp32 second-level scale S ("KV Cache Quantisation": FP8 or
    NVFP4 with the scales handled at read time).
  * ``fp16_encode`` / ``int_quantize`` / ``int_dequantize`` -- the
    symmetric INT-b quantisers with one FP16 scale per token or per channel
    of the bit-width sweep ("Quantising the KV cache", table and section
    "Per token or per channel?").
  * ``decode_unit`` -- one (sequence, kv head) decode: FP4 for positions
    [0, T - W'), FP8 for the last W' = min(W, T) positions, one softmax over
    the union.
  * ``swa_forward`` / ``exact_replay_start`` / ``bounded_replay_start`` -- a
    toy multilayer sliding-window network and the two replays of its window
    state ("Week 6 -- FP4 KV Caches and Bounded Replay", Core Concepts
    "Bounded replay" and Lab: exact replay ~ L n_win tokens, bounded replay
    the last n_win).

Parity pins live in ``tests/test_oracle_*.py``.  Functions without a pin:
none (see the tests' module docstrings).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB = os.path.join(_HERE, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i8p = ctypes.POINTER(ctypes.c_int8)


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into libkvq_oracle.so with gcc (no fast-math,
    no FMA contraction) and return its path."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            L.oq_e2m1_value.restype = ctypes.c_double
            L.oq_e2m1_value.argtypes = [ctypes.c_uint8]
            L.oq_e4m3_value.restype = ctypes.c_double
            L.oq_e4m3_value.argtypes = [ctypes.c_uint8]
            for name in ("oq_e2m1_encode", "oq_e4m3_encode", "oq_e2m1_encode_brute",
                         "oq_e4m3_encode_brute"):
                getattr(L, name).restype = ctypes.c_uint8
                getattr(L, name).argtypes = [ctypes.c_float]
            for name in ("oq_e2m1_encode_array", "oq_e4m3_encode_array"):
                getattr(L, name).restype = None
                getattr(L, name).argtypes = [_f32p, ctypes.c_int64, _u8p, ctypes.c_int]
            L.oq_quantize_block.restype = ctypes.c_int
            L.oq_quantize_block.argtypes = [_f32p, _u8p, _u8p]
            L.oq_quantize_rows.restype = ctypes.c_int64
            L.oq_quantize_rows.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int, _u8p, _u8p]
            L.oq_dequantize_rows.restype = None
            L.oq_dequantize_rows.argtypes = [_u8p, _u8p, ctypes.c_int64, ctypes.c_int, _f64p]
            L.oq_fp8_head_scale.restype = ctypes.c_float
            L.oq_fp8_head_scale.argtypes = [_f32p, ctypes.c_int64]
            L.oq_fp8_quantize.restype = ctypes.c_int64
            L.oq_fp8_quantize.argtypes = [_f32p, ctypes.c_int64, ctypes.c_float, _u8p]
            L.oq_fp8_dequantize.restype = None
            L.oq_fp8_dequantize.argtypes = [_u8p, ctypes.c_int64, ctypes.c_float, _f64p]
            L.oq_nvfp4_global_scale.restype = ctypes.c_float
            L.oq_nvfp4_global_scale.argtypes = [_f32p, ctypes.c_int64]
            L.oq_nvfp4_quantize_rows.restype = ctypes.c_int64
            L.oq_nvfp4_quantize_rows.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, _u8p, _u8p]
            L.oq_nvfp4_dequantize_rows.restype = None
            L.oq_nvfp4_dequantize_rows.argtypes = [_u8p, _u8p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, _f64p]
            L.oq_fp16_value.restype = ctypes.c_double
            L.oq_fp16_value.argtypes = [ctypes.c_uint16]
            L.oq_fp16_encode.restype = ctypes.c_uint16
            L.oq_fp16_encode.argtypes = [ctypes.c_float]
            L.oq_fp16_encode_array.restype = None
            L.oq_fp16_encode_array.argtypes = [_f32p, ctypes.c_int64, _u16p]
            L.oq_int_quantize_group.restype = ctypes.c_int64
            L.oq_int_quantize_group.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _i8p, _u16p]
            for name in ("oq_int_quantize_per_token", "oq_int_quantize_per_channel"):
                getattr(L, name).restype = ctypes.c_int64
                getattr(L, name).argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int, _i8p, _u16p]
            L.oq_swa_forward.restype = None
            L.oq_swa_forward.argtypes = [_f64p, ctypes.c_int, ctypes.c_int, _f64p, ctypes.c_int64, ctypes.c_int,
                                         _f64p, _f64p, _f64p, _f64p, _f64p, _f64p]
            L.oq_attend.restype = None
            L.oq_attend.argtypes = [_f64p, _f64p, _f64p, ctypes.c_int, ctypes.c_int64,
                                    ctypes.c_int, ctypes.c_double, _f64p, _f64p, _f64p, _f64p]
            _lib = L
    return _lib


def _p(a: np.ndarray, ty):
    return a.ctypes.data_as(ty)


def _f32(x) -> np.ndarray:
    """Inputs arrive as numpy float32 or as torch tensors (bf16 or fp32);
    bf16 -> fp32 widening is exact."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------- formats
def e2m1_value(nibble: int) -> float:
    return lib().oq_e2m1_value(int(nibble) & 0xF)


def e4m3_value(byte: int) -> float:
    return lib().oq_e4m3_value(int(byte) & 0xFF)


def e2m1_encode(y, brute: bool = False) -> np.ndarray:
    y = _f32(y).ravel()
    out = np.empty(y.size, np.uint8)
    lib().oq_e2m1_encode_array(_p(y, _f32p), y.size, _p(out, _u8p), int(brute))
    return out


def e4m3_encode(t, brute: bool = False) -> np.ndarray:
    t = _f32(t).ravel()
    out = np.empty(t.size, np.uint8)
    lib().oq_e4m3_encode_array(_p(t, _f32p), t.size, _p(out, _u8p), int(brute))
    return out


# ---------------------------------------------------------------- FP4 block quantiser
def quantize_rows(x):
    """x: (..., d) values, d % 16 == 0.  Returns (codes uint8 (..., d/2),
    scales uint8 (..., d/16), number of blocks holding a non-finite value)."""
    x = _f32(x)
    d = x.shape[-1]
    assert d % 16 == 0
    n = x.size // d
    codes = np.empty(x.shape[:-1] + (d // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (d // 16,), np.uint8)
    bad = lib().oq_quantize_rows(_p(x, _f32p), n, d, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales, int(bad)


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    d = codes.shape[-1] * 2
    n = codes.size // (d // 2)
    out = np.empty(codes.shape[:-1] + (d,), np.float64)
    lib().oq_dequantize_rows(_p(codes, _u8p), _p(scales, _u8p), n, d, _p(out, _f64p))
    return out


# ---------------------------------------------------------------- FP8 SWA
def fp8_head_scale(x) -> float:
    x = _f32(x).ravel()
    return float(lib().oq_fp8_head_scale(_p(x, _f32p), x.size))


def fp8_quantize(x, s: float):
    x = _f32(x)
    out = np.empty(x.shape, np.uint8)
    bad = lib().oq_fp8_quantize(_p(x, _f32p), x.size, ctypes.c_float(s), _p(out, _u8p))
    return out, int(bad)


def fp8_dequantize(c: np.ndarray, s: float) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().oq_fp8_dequantize(_p(c, _u8p), c.size, ctypes.c_float(s), _p(out, _f64p))
    return out


# ---------------------------------------------------------------- NVFP4
def nvfp4_global_scale(x) -> float:
    """S = amax / (6 * 448) in fp32 over every value (1 when amax == 0)."""
    x = _f32(x).ravel()
    return float(lib().oq_nvfp4_global_scale(_p(x, _f32p), x.size))


def nvfp4_quantize_rows(x, S: float):
    """The FP4 block quantiser over x / S (fp32 division): (codes, scales,
    non-finite block count), shaped like quantize_rows."""
    x = _f32(x)
    d = x.shape[-1]
    n = x.size // d
    codes = np.empty(x.shape[:-1] + (d // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (d // 16,), np.uint8)
    bad = lib().oq_nvfp4_quantize_rows(_p(x, _f32p), n, d, ctypes.c_float(S), _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales, int(bad)


def nvfp4_dequantize_rows(codes: np.ndarray, scales: np.ndarray, S: float) -> np.ndarray:
    """fp32(fp32(e2m1 * e4m3) * S), widened to fp64."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    d = codes.shape[-1] * 2
    n = codes.size // (d // 2)
    out = np.empty(codes.shape[:-1] + (d,), np.float64)
    lib().oq_nvfp4_dequantize_rows(_p(codes, _u8p), _p(scales, _u8p), n, d, ctypes.c_float(S), _p(out, _f64p))
    return out


# ---------------------------------------------------------------- bit-width sweep
def fp16_value(bits: int) -> float:
    return lib().oq_fp16_value(int(bits) & 0xFFFF)


def fp16_encode(x) -> np.ndarray:
    """binary16 bit patterns, RNE, saturating at 65504 (NaN -> 0x7E00)."""
    x = _f32(x).ravel()
    out = np.empty(x.size, np.uint16)
    lib().oq_fp16_encode_array(_p(x, _f32p), x.size, _p(out, _u16p))
    return out


def int_quantize_group(x, bits: int):
    """One group: (codes int8 (n,), fp16 scale bits, non-finite count)."""
    x = _f32(x).ravel()
    codes = np.empty(x.size, np.int8)
    sb = np.zeros(1, np.uint16)
    bad = lib().oq_int_quantize_group(_p(x, _f32p), x.size, 1, int(bits), _p(codes, _i8p), _p(sb, _u16p))
    return codes, int(sb[0]), int(bad)


def int_quantize(x, bits: int, per: str):
    """x: (batch, tokens, heads, d).  per == "token": one FP16 scale per
    (b, t, head); per == "channel": one per (b, head, channel) over the
    tokens.  Returns (codes int8 like x, scale bits uint16, non-finite
    count)."""
    x = _f32(x)
    B, T, H, d = x.shape
    codes = np.empty(x.shape, np.int8)
    if per == "token":
        scales = np.empty((B, T, H), np.uint16)
        fn = lib().oq_int_quantize_per_token
    elif per == "channel":
        scales = np.empty((B, H, d), np.uint16)
        fn = lib().oq_int_quantize_per_channel
    else:
        raise ValueError(per)
    bad = fn(_p(x, _f32p), B, T, H, d, int(bits), _p(codes, _i8p), _p(scales, _u16p))
    return codes, scales, int(bad)


def int_dequantize(codes: np.ndarray, scales: np.ndarray, per: str) -> np.ndarray:
    """Values code * s (exact), fp64, shaped like codes."""
    s = np.vectorize(fp16_value, otypes=[np.float64])(scales)
    if per == "token":
        return codes.astype(np.float64) * s[..., None]
    B, T, H, d = codes.shape
    return codes.astype(np.float64) * s[:, None, :, :]


# ---------------------------------------------------------------- attention
def attend(q, k, v, scale: float):
    """q: (G, d), k, v: (T, d), any float dtype (widened to fp64).
    Returns (out (G, d), m (G,), l (G,)) in fp64; m, l are the max score and
    the softmax denominator relative to it (natural-log units)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    G, d = q.shape
    T = k.shape[0]
    out = np.empty((G, d), np.float64)
    m = np.empty(G, np.float64)
    l = np.empty(G, np.float64)
    tmp = np.empty(max(T, 1), np.float64)
    lib().oq_attend(_p(q, _f64p), _p(k, _f64p), _p(v, _f64p), G, T, d, float(scale),
                    _p(out, _f64p), _p(m, _f64p), _p(l, _f64p), _p(tmp, _f64p))
    return out, m, l


def decode_unit(q, k, v, scale: float, window: int = 0, swa_scales=None, nvfp4_scales=None):
    """One (sequence, kv head) decode step over T cached positions.

    q: (G, d) query rows of the group; k, v: (T, d) the unquantised cached
    keys/values in position order.  With window == 0 every position is read
    from the FP4 cache.  With window W > 0 the last W' = min(W, T) positions
    are read from the FP8 cache with per-head scales swa_scales = (s_k, s_v)
    and the rest from the FP4 cache.  nvfp4_scales = (S_k, S_v) reads the
    global positions as NVFP4 (second-level scales) instead of plain FP4.
    Returns (out (G, d) fp64, vmax) where
    vmax = max |V^| over the attended dequantised values.
    """
    k = _f32(k)
    v = _f32(v)
    T, d = k.shape
    w = min(window, T) if window > 0 else 0
    n4 = T - w
    if nvfp4_scales is None:
        kc, ks, _ = quantize_rows(k[:n4])
        vc, vs, _ = quantize_rows(v[:n4])
        kh = dequantize_rows(kc, ks)
        vh = dequantize_rows(vc, vs)
    else:
        Sk, Sv = nvfp4_scales
        kc, ks, _ = nvfp4_quantize_rows(k[:n4], Sk)
        vc, vs, _ = nvfp4_quantize_rows(v[:n4], Sv)
        kh = nvfp4_dequantize_rows(kc, ks, Sk)
        vh = nvfp4_dequantize_rows(vc, vs, Sv)
    if w > 0:
        sk, sv = swa_scales
        k8, _ = fp8_quantize(k[n4:], sk)
        v8, _ = fp8_quantize(v[n4:], sv)
        kh = np.concatenate([kh, fp8_dequantize(k8, sk)], axis=0)
        vh = np.concatenate([vh, fp8_dequantize(v8, sv)], axis=0)
    out, _, _ = attend(_f32(q), kh, vh, scale)
    vmax = float(np.abs(vh).max()) if T > 0 else 0.0
    return out, vmax


# ---------------------------------------------------------------- replay
def swa_forward(w, emb, n_win: int):
    """Toy sliding-window network over the replayed positions (fp64).

    w: (L, 4, d, d) -- Wq, Wk, Wv, Wo per layer; emb: (n, d), the inputs of
    the n >= n_win replayed positions in order (position i of the replay
    attends positions max(0, i - n_win + 1) .. i).  Returns (hidden (n, d),
    states (L, 2, n_win, d)): the last layer's output and each layer's K and
    V rows of the last n_win positions -- the window state a decoder keeps.
    """
    w = np.ascontiguousarray(w, dtype=np.float64)
    emb = np.ascontiguousarray(emb, dtype=np.float64)
    L, four, d, d2 = w.shape
    assert four == 4 and d == d2
    n = emb.shape[0]
    assert emb.shape == (n, d) and 1 <= n_win <= n
    hidden = np.empty((n, d), np.float64)
    states = np.empty((L, 2, n_win, d), np.float64)
    x = np.empty((n, d), np.float64)
    kb = np.empty((n, d), np.float64)
    vb = np.empty((n, d), np.float64)
    tmp = np.empty(3 * d + n_win, np.float64)
    lib().oq_swa_forward(_p(w, _f64p), L, d, _p(emb, _f64p), n, int(n_win), _p(hidden, _f64p),
                         _p(states, _f64p), _p(x, _f64p), _p(kb, _f64p), _p(vb, _f64p), _p(tmp, _f64p))
    return hidden, states


def exact_replay_start(T: int, layers: int, n_win: int) -> int:
    """First position an exact replay of the window state after T positions
    must start from: the top layer's window [T - n_win, T) reaches back
    n_win - 1 positions per layer below it."""
    return max(0, T - n_win - (layers - 1) * (n_win - 1))


def bounded_replay_start(T: int, n_win: int) -> int:
    """Bounded replay starts at the window: only the last n_win positions."""
    return max(0, T - n_win)
