"""Thin Python binding of libkvq (the C ABI declared in include/kvq.h).

Argument marshalling only: every step of the path runs in the CUDA kernels of
libkvq.so.  PyTorch is used for device memory and streams.  There is no CPU
fallback -- if libkvq.so is missing, ``load()`` raises.

Names follow the header: ``append`` (kvq_append), ``fp8_set_scales``
(kvq_fp8_set_scales), ``decode_attn`` (kvq_decode_attn), ``dequant``
(kvq_dequant), ``decode_workspace_bytes`` (kvq_decode_workspace_bytes).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

FORMAT_FP4 = 1
FORMAT_FP8 = 2
FORMAT_NVFP4 = 3
FLAG_NONFINITE = 0x1
FLAG_PAGE_OOB = 0x2
FLAG_TIMEOUT = 0x4
FLAG_BAD_LENGTH = 0x8
LAYOUT_FP8_TENSOR = 1
LAYOUT_INT_PER_TOKEN = 2
LAYOUT_INT_PER_CHANNEL = 3
LAYOUT_FP4_G16 = 4

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_status_string(status)} (status {status})")
        self.status = status


class KvqCacheStruct(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("max_pages_per_seq", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
        ("data", ctypes.c_void_p),
        ("v_data", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
    ]


_P = ctypes.c_void_p
_CP = ctypes.POINTER(KvqCacheStruct)


def load() -> ctypes.CDLL:
    """Load libkvq.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m fp4_kv_cache_kvq_gb300.build` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            L.kvq_append.restype = ctypes.c_int
            L.kvq_append.argtypes = [_CP, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P]
            L.kvq_fp8_set_scales.restype = ctypes.c_int
            L.kvq_fp8_set_scales.argtypes = [_CP, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]
            L.kvq_decode_workspace_bytes.restype = ctypes.c_size_t
            L.kvq_decode_workspace_bytes.argtypes = [ctypes.c_int32] * 4
            L.kvq_decode_attn.restype = ctypes.c_int
            L.kvq_decode_attn.argtypes = [_CP, _CP, ctypes.c_int32, ctypes.c_int32, _P, _P, ctypes.c_float,
                                          _P, _P, ctypes.c_size_t, _P, _P]
            L.kvq_decode_attn_tc.restype = ctypes.c_int
            L.kvq_decode_attn_tc.argtypes = L.kvq_decode_attn.argtypes
            L.kvq_test_set_wait_limit_ns.restype = None
            L.kvq_test_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.kvq_append_decode_attn.restype = ctypes.c_int
            L.kvq_append_decode_attn.argtypes = [_CP, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, ctypes.c_float,
                                                 _P, _P, ctypes.c_size_t, _P, _P]
            L.kvq_dequant.restype = ctypes.c_int
            L.kvq_dequant.argtypes = [_CP, ctypes.c_int32, _P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]
            L.kvq_status_string.restype = ctypes.c_char_p
            L.kvq_status_string.argtypes = [ctypes.c_int]
            L.kvq_version.restype = ctypes.c_int32
            L.kvq_version.argtypes = []
            L.kvq_prefill_attn.restype = ctypes.c_int
            L.kvq_prefill_attn.argtypes = [_CP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                           ctypes.c_float, _P, _P, _P]
            L.kvq_fake_quant.restype = ctypes.c_int
            L.kvq_fake_quant.argtypes = [ctypes.c_int32] * 6 + [_P] * 6
            L.kvq_attn_dense.restype = ctypes.c_int
            L.kvq_attn_dense.argtypes = [ctypes.c_int32] * 5 + [_P, _P, _P, ctypes.c_float, _P, _P, _P]
            L.kvq_swa_replay_workspace_bytes.restype = ctypes.c_size_t
            L.kvq_swa_replay_workspace_bytes.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32]
            L.kvq_swa_replay.restype = ctypes.c_int
            L.kvq_swa_replay.argtypes = [_P, ctypes.c_int32, ctypes.c_int32, _P, ctypes.c_int64, ctypes.c_int32,
                                         _P, _P, _P, ctypes.c_size_t, _P]
            L.kvq_fp4_pool_bytes.restype = ctypes.c_size_t
            L.kvq_fp4_pool_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
            _lib = L
    return _lib


def _status_string(status: int) -> str:
    try:
        return load().kvq_status_string(status).decode()
    except Exception:  # pragma: no cover
        return "unknown"


def _check(status: int, what: str) -> None:
    if status != 0:
        raise KvqError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t: torch.Tensor, dtype: torch.dtype, name: str) -> None:
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of dtype {dtype}")


class Fp4Cache:
    """FP4 (E2M1 codes, E4M3 scale per 16 channels) paged cache for K and V.

    pool  uint8 [num_pages][num_kv_heads][page_size / G][G * 9 * head_dim / 8],
          G = min(page_size, 128): one contiguous block per group of G tokens
          of one kv head (K codes, K scales, V codes in token pairs, V scales;
          the byte layout is documented in include/kvq.h).
    page_table int32 [batch][max_pages_per_seq] or None (contiguous).
    nvfp4=True adds one fp32 second-level scale per kv head for K and for V
    (k_gscale, v_gscale: float [num_kv_heads], 1 until set by fp8_set_scales).
    """

    def __init__(self, num_kv_heads: int, head_dim: int, page_size: int, num_pages: int,
                 max_pages_per_seq: int, page_table: Optional[torch.Tensor] = None, device="cuda",
                 nvfp4: bool = False):
        self.num_kv_heads, self.head_dim, self.page_size = num_kv_heads, head_dim, page_size
        self.num_pages, self.max_pages_per_seq = num_pages, max_pages_per_seq
        self.group = min(page_size, 128)
        nbytes = load().kvq_fp4_pool_bytes(num_pages, num_kv_heads, page_size, head_dim)
        if nbytes == 0:
            raise ValueError("invalid FP4 cache geometry (head_dim 64/128/256, page_size 16..256)")
        shape = (num_pages, num_kv_heads, page_size // self.group, self.group * 9 * head_dim // 8)
        self.pool = torch.zeros(shape, dtype=torch.uint8, device=device)
        assert self.pool.numel() == nbytes
        if page_table is not None:
            _need(page_table, torch.int32, "page_table")
        self.page_table = page_table
        self.nvfp4 = nvfp4
        self.k_gscale = torch.ones(num_kv_heads, dtype=torch.float32, device=device) if nvfp4 else None
        self.v_gscale = torch.ones(num_kv_heads, dtype=torch.float32, device=device) if nvfp4 else None

    def struct(self, page_table: Optional[torch.Tensor] = None) -> KvqCacheStruct:
        """The kvq_cache description (kept between calls while the tensors it
        points at are the same objects; a page_table argument overrides the
        cache's own for one call)."""
        pt = self.page_table if page_table is None else page_table
        key = (id(self.pool), id(pt), id(self.k_gscale), id(self.v_gscale))
        cached = self.__dict__.get("_struct")
        if cached is not None and cached[0] == key:
            return cached[1]
        s = KvqCacheStruct(FORMAT_NVFP4 if self.nvfp4 else FORMAT_FP4, self.num_kv_heads, self.head_dim,
                           self.page_size, self.num_pages, self.max_pages_per_seq, 0, _ptr(pt), _ptr(self.pool),
                           None, _ptr(self.k_gscale), _ptr(self.v_gscale))
        if page_table is None:
            self._struct = (key, s)
        return s

    @property
    def nbytes(self) -> int:
        return self.pool.numel()


class Fp8WindowCache:
    """FP8 E4M3 sliding-window cache: one ring of `window` slots per sequence,
    one fp32 scale per kv head (K and V apart).

    codes  uint8 [num_seqs][num_kv_heads][window][head_dim]
    scales float32 [num_kv_heads]
    """

    def __init__(self, num_seqs: int, num_kv_heads: int, head_dim: int, window: int, device="cuda"):
        self.num_seqs, self.num_kv_heads, self.head_dim, self.window = num_seqs, num_kv_heads, head_dim, window
        shape = (num_seqs, num_kv_heads, window, head_dim)
        self.k_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
        self.v_codes = torch.zeros_like(self.k_codes)
        self.k_scales = torch.ones(num_kv_heads, dtype=torch.float32, device=device)
        self.v_scales = torch.ones_like(self.k_scales)

    def struct(self) -> KvqCacheStruct:
        """The kvq_cache description (kept while the tensors are the same objects)."""
        key = (id(self.k_codes), id(self.v_codes), id(self.k_scales), id(self.v_scales))
        cached = self.__dict__.get("_struct")
        if cached is not None and cached[0] == key:
            return cached[1]
        s = KvqCacheStruct(FORMAT_FP8, self.num_kv_heads, self.head_dim, self.window, self.num_seqs, 0, 0,
                           None, _ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_scales), _ptr(self.v_scales))
        self._struct = (key, s)
        return s



def append(cache, start_pos: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
           err: Optional[torch.Tensor] = None, stream=None, page_table: Optional[torch.Tensor] = None) -> None:
    """kvq_append: k, v bf16 [batch][n_new][Hkv][head_dim]; start_pos int32 [batch]."""
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v")
    _need(start_pos, torch.int32, "start_pos")
    if k.dim() != 4 or k.shape != v.shape:
        raise ValueError("k and v must have shape [batch, n_new, num_kv_heads, head_dim]")
    s = cache.struct(page_table) if isinstance(cache, Fp4Cache) else cache.struct()
    st = load().kvq_append(ctypes.byref(s), k.shape[0], k.shape[1], _ptr(start_pos), _ptr(k), _ptr(v),
                           _ptr(err), _stream(stream))
    _check(st, "kvq_append")


def fp8_set_scales(cache, k: torch.Tensor, v: torch.Tensor,
                   err: Optional[torch.Tensor] = None, stream=None) -> None:
    """kvq_fp8_set_scales over k, v bf16 [batch][n][Hkv][D]: an FP8 window
    cache gets s_h = amax/448 per head, an NVFP4 cache its second-level
    scales S_h = amax/(6*448)."""
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v")
    s = cache.struct()
    st = load().kvq_fp8_set_scales(ctypes.byref(s), k.shape[0], k.shape[1], _ptr(k), _ptr(v), _ptr(err),
                                   _stream(stream))
    _check(st, "kvq_fp8_set_scales")


def decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load().kvq_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim))


def decode_attn(cache: Fp4Cache, seq_lens: torch.Tensor, q: torch.Tensor, softmax_scale: Optional[float] = None,
                swa: Optional[Fp8WindowCache] = None, out: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
                stream=None, kernel: str = "mma") -> torch.Tensor:
    """kvq_decode_attn: q bf16 [batch][Hq][head_dim] -> out float32 [batch][Hq][head_dim].
    kernel="tcgen05" calls kvq_decode_attn_tc instead (head_dim 128: both
    products on the tensor-memory MMA; a measured, slower alternative)."""
    if kernel not in ("mma", "tcgen05"):
        raise ValueError(f"unknown decode kernel {kernel!r}")
    _need(q, torch.bfloat16, "q")
    _need(seq_lens, torch.int32, "seq_lens")
    batch, hq, d = q.shape
    if out is None:
        out = torch.empty((batch, hq, d), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out")
    if workspace is None:  # a caller's workspace is size-checked by the library
        need = decode_workspace_bytes(batch, hq, cache.num_kv_heads, d)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    g = cache.struct()
    w = swa.struct() if swa is not None else None
    fn = load().kvq_decode_attn_tc if kernel == "tcgen05" else load().kvq_decode_attn
    st = fn(ctypes.byref(g), ctypes.byref(w) if w is not None else None, batch, hq, _ptr(seq_lens), _ptr(q),
            float(softmax_scale), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(err), _stream(stream))
    _check(st, "kvq_decode_attn_tc" if kernel == "tcgen05" else "kvq_decode_attn")
    return out


def append_decode_attn(cache: Fp4Cache, seq_lens: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                       q: torch.Tensor, softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None,
                       stream=None) -> torch.Tensor:
    """kvq_append_decode_attn: append k_new/v_new bf16 [batch][Hkv][head_dim] at
    position seq_lens[b] - 1, then decode attention over seq_lens[b] positions."""
    _need(q, torch.bfloat16, "q")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    batch, hq, d = q.shape
    if out is None:
        out = torch.empty((batch, hq, d), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out")
    if workspace is None:
        need = decode_workspace_bytes(batch, hq, cache.num_kv_heads, d)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    g = cache.struct()
    st = load().kvq_append_decode_attn(ctypes.byref(g), batch, hq, _ptr(seq_lens), _ptr(k_new), _ptr(v_new), _ptr(q),
                                       float(softmax_scale), _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream))
    _check(st, "kvq_append_decode_attn")
    return out


def prefill_attn(cache: Fp4Cache, seq_lens: torch.Tensor, q: torch.Tensor, softmax_scale: Optional[float] = None,
                 out: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """kvq_prefill_attn: q bf16 [batch][chunk][Hq][head_dim] (their keys and
    values already appended) -> out float32, same shape; causal over the cache."""
    _need(q, torch.bfloat16, "q")
    _need(seq_lens, torch.int32, "seq_lens")
    batch, chunk, hq, d = q.shape
    if out is None:
        out = torch.empty((batch, chunk, hq, d), dtype=torch.float32, device=q.device)
    _need(out, torch.float32, "out")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    c = cache.struct()
    st = load().kvq_prefill_attn(ctypes.byref(c), batch, hq, chunk, _ptr(seq_lens), _ptr(q), float(softmax_scale),
                                 _ptr(out), _ptr(err), _stream(stream))
    _check(st, "kvq_prefill_attn")
    return out


def swa_replay(w: torch.Tensor, emb: torch.Tensor, n_win: int, want_hidden: bool = True,
               workspace: Optional[torch.Tensor] = None, states: Optional[torch.Tensor] = None, stream=None):
    """kvq_swa_replay: the toy sliding-window network over the positions whose
    inputs are emb (float32 [n][d]) with weights w (float32 [L][4][d][d]:
    Wq, Wk, Wv, Wo).  Returns (states float32 [L][2][n_win][d] -- each
    layer's K then V rows of the last n_win positions --, hidden float32
    [n][d] or None)."""
    _need(w, torch.float32, "w")
    _need(emb, torch.float32, "emb")
    L, four, d, _ = w.shape
    n = emb.shape[0]
    if states is None:
        states = torch.empty((L, 2, n_win, d), dtype=torch.float32, device=emb.device)
    _need(states, torch.float32, "states")
    hidden = torch.empty((n, d), dtype=torch.float32, device=emb.device) if want_hidden else None
    need = load().kvq_swa_replay_workspace_bytes(L, n, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=emb.device)
    st = load().kvq_swa_replay(_ptr(w), L, d, _ptr(emb), n, int(n_win), _ptr(states), _ptr(hidden), _ptr(workspace),
                               workspace.numel(), _stream(stream))
    _check(st, "kvq_swa_replay")
    return states, hidden


def dequant(cache, seq_lens: Optional[torch.Tensor], max_len: int, dtype: torch.dtype = torch.float32,
            err: Optional[torch.Tensor] = None, stream=None):
    """kvq_dequant: dense K, V [batch][max_len][Hkv][head_dim] (FP8: max_len == window, slot order)."""
    if isinstance(cache, Fp4Cache):
        batch = seq_lens.shape[0]
        s = cache.struct()
        device = cache.pool.device
    else:
        batch = cache.num_seqs
        s = cache.struct()
        device = cache.k_codes.device
    code = {torch.float32: 0, torch.bfloat16: 1}[dtype]
    shape = (batch, max_len, cache.num_kv_heads, cache.head_dim)
    k = torch.empty(shape, dtype=dtype, device=device)
    v = torch.empty(shape, dtype=dtype, device=device)
    st = load().kvq_dequant(ctypes.byref(s), batch, _ptr(seq_lens), max_len, code, _ptr(k), _ptr(v), _ptr(err),
                            _stream(stream))
    _check(st, "kvq_dequant")
    return k, v


# ---------------------------------------------------------------- bit-width sweep
def fake_quant(x: torch.Tensor, layout: int, bits: int, want_codes: bool = False,
               err: Optional[torch.Tensor] = None, stream=None):
    """kvq_fake_quant: x bf16 [batch][tokens][heads][head_dim] -> (x_hat float
    like x, codes int8 like x or None, scales or None).  Scales: FP8 tensor ->
    float[2] (s in [1]); INT per token -> uint16-as-int16 [batch][tokens][heads];
    INT per channel -> [batch][heads][head_dim]; FP4 -> uint8 [numel/16]."""
    _need(x, torch.bfloat16, "x")
    B, T, H, d = x.shape
    xh = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    codes = torch.empty(x.shape, dtype=torch.int8, device=x.device) if want_codes else None
    if layout == LAYOUT_FP8_TENSOR:
        scales = torch.empty(2, dtype=torch.float32, device=x.device)
    elif layout == LAYOUT_INT_PER_TOKEN:
        scales = torch.empty((B, T, H), dtype=torch.int16, device=x.device)
    elif layout == LAYOUT_INT_PER_CHANNEL:
        scales = torch.empty((B, H, d), dtype=torch.int16, device=x.device)
    else:
        scales = torch.empty(x.numel() // 16, dtype=torch.uint8, device=x.device)
    st = load().kvq_fake_quant(layout, bits, B, T, H, d, _ptr(x), _ptr(xh), _ptr(codes), _ptr(scales), _ptr(err),
                               _stream(stream))
    _check(st, "kvq_fake_quant")
    return xh, codes, scales


def attn_dense(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, softmax_scale: Optional[float] = None,
               want_top: bool = False, stream=None):
    """kvq_attn_dense: q bf16 [batch][Hq][d], k, v float [batch][T][Hkv][d] ->
    (out float [batch][Hq][d], top int32 [batch][Hq] or None)."""
    _need(q, torch.bfloat16, "q")
    _need(k, torch.float32, "k")
    _need(v, torch.float32, "v")
    B, Hq, d = q.shape
    T, Hkv = k.shape[1], k.shape[2]
    out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    top = torch.empty((B, Hq), dtype=torch.int32, device=q.device) if want_top else None
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else softmax_scale
    st = load().kvq_attn_dense(B, T, Hq, Hkv, d, _ptr(q), _ptr(k), _ptr(v), float(scale), _ptr(out), _ptr(top),
                               _stream(stream))
    _check(st, "kvq_attn_dense")
    return out, top
