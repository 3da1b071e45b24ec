"""Seeded synthetic inputs for the FP4 KV cache workloads.

Holds none of the method's arithmetic: it only draws queries, keys and values
(fp32 normal draws, outlier scaling in fp32, one cast to bf16), sequence
lengths and page tables.  The tests, the smoke check and the benchmark feed
the same tensors to the CUDA library and (as host copies) to the CPU oracle.

Workloads (one layer each):
  tiny           B1, Hkv2, Hq2 (G1), d64, T256, N(0,1).
  gqa_outliers   B8, Hkv8, Hq32 (G4), d128, T4096, N(0,1); in every head K
                 channels {3, 17, 64, 101} are scaled x20 (fixed outlier
                 channels, the "Quantising the KV cache" lesson that a few key
                 channels carry very large magnitudes).
  long_context   B32, Hkv8, Hq64 (G8), d128, T32768, N(0,1).
  paged_ragged   B64, Hkv8, Hq32 (G4), d128, page 64, T_b ~ U[1024, 131072]
                 inclusive, page tables from one random permutation of a shared
                 pool (sequence b takes a consecutive slice), 2% of K entries
                 i.i.d. scaled x30.
  swa_append     B16, Hkv8, Hq64 (G8), d128, FP4 context 65536 plus an FP8
                 window of 128; each step appends one N(0,1) token per sequence.
  prefill        B16 x 16384 new tokens, Hkv8, d128 (append throughput).
  prefill_attn   B4, Hkv8, Hq64 (G8), d128: the last 1024 of 16384 cached
                 positions are a chunk of new queries attending causally.

Toy sliding-window network for the replay experiment (``replay_net`` /
``replay_inputs``): L layers of four d x d matrices drawn N(0, 1/d) (weights of
unit gain on RMS-normalised inputs), position inputs N(0, 1).  ``REPLAY`` is
the benchmark's configuration: L = 8, d = 128, window 512, state after 65536
positions.

Draw order per sequence b: K then V (then the i.i.d. outlier mask), from a
generator seeded with (seed, b), so any subset of sequences can be redrawn.
Queries and per-step tokens use their own seeded generators.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    context: int = 0                       # equal sequence length (0 when ragged)
    ragged: Optional[Tuple[int, int]] = None  # inclusive length range
    page_size: int = 64
    paged: bool = False                    # random page tables over a shared pool
    k_outlier_channels: Tuple[int, ...] = ()
    k_outlier_factor: float = 1.0
    k_outlier_prob: float = 0.0
    k_outlier_prob_factor: float = 1.0
    window: int = 0                        # FP8 sliding window (0 = none)
    chunk: int = 0                         # chunked prefill: new query tokens per sequence
    description: str = field(default="", compare=False)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 2, 64, context=256,
                     description="B1 Hkv2 Hq2 d64 T256 N(0,1)"),
    "gqa_outliers": Workload("gqa_outliers", 8, 8, 32, 128, context=4096, k_outlier_channels=(3, 17, 64, 101),
                             k_outlier_factor=20.0,
                             description="B8 Hkv8 Hq32 d128 T4096, K channels {3,17,64,101} x20"),
    "long_context": Workload("long_context", 32, 8, 64, 128, context=32768,
                             description="B32 Hkv8 Hq64 d128 T32768 N(0,1)"),
    "paged_ragged": Workload("paged_ragged", 64, 8, 32, 128, ragged=(1024, 131072), paged=True,
                             k_outlier_prob=0.02, k_outlier_prob_factor=30.0,
                             description="B64 Hkv8 Hq32 d128 page64 T~U[1024,131072], 2% of K x30"),
    "swa_append": Workload("swa_append", 16, 8, 64, 128, context=65536, window=128,
                           description="B16 Hkv8 Hq64 d128 FP4 T65536 + FP8 window 128, append 1/step"),
    "prefill": Workload("prefill", 16, 8, 8, 128, context=16384,
                        description="B16 x 16384-token bf16 prefill, Hkv8 d128"),
    "prefill_b1": Workload("prefill_b1", 1, 8, 8, 128, context=16384,
                           description="B1 x 16384-token bf16 prefill, Hkv8 d128"),
    "prefill_attn": Workload("prefill_attn", 4, 8, 64, 128, context=16384, chunk=1024,
                             description="B4 Hkv8 Hq64 d128: a 1024-token chunk attending causally over a "
                                         "16384-position FP4 cache (the chunk's own tokens included)"),
}

_MIX = 1_000_003


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def lengths(w: Workload, seed: int = 0) -> List[int]:
    if w.ragged is None:
        return [w.context] * w.batch
    lo, hi = w.ragged
    g = _gen("cpu", seed * _MIX + 17)
    return torch.randint(lo, hi + 1, (w.batch,), generator=g).tolist()


def page_layout(w: Workload, lens: List[int], reserve: int = 0, seed: int = 0):
    """Pages for each sequence's first len_b + reserve positions.
    Returns (page_table int32 [B][max_pages] or None, num_pages, max_pages)."""
    P = w.page_size
    need = [(n + reserve + P - 1) // P for n in lens]
    max_pages = max(max(need), 1)
    if not w.paged:
        return None, w.batch * max_pages, max_pages
    pool = sum(need)
    perm = torch.randperm(pool, generator=_gen("cpu", seed * _MIX + 29)).to(torch.int32)
    table = torch.full((w.batch, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return table, pool, max_pages


def sequence_kv(w: Workload, b: int, n_tokens: int, seed: int = 0, device="cpu"):
    """Keys and values of sequence b's first n_tokens positions, bf16
    [n_tokens][Hkv][d] each."""
    g = _gen(device, seed * _MIX + 1000 + b)
    shape = (n_tokens, w.num_kv_heads, w.head_dim)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if w.k_outlier_channels:
        idx = torch.tensor(w.k_outlier_channels, device=device)
        k[..., idx] *= w.k_outlier_factor
    if w.k_outlier_prob > 0.0:
        mask = torch.rand(shape, generator=g, device=device) < w.k_outlier_prob
        k = torch.where(mask, k * w.k_outlier_prob_factor, k)
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def queries(w: Workload, seed: int = 0, step: int = 0, device="cpu") -> torch.Tensor:
    """bf16 [B][Hq][d]."""
    g = _gen(device, seed * _MIX + 7 + 7919 * step)
    return torch.randn((w.batch, w.num_q_heads, w.head_dim), generator=g, device=device).to(torch.bfloat16)


def step_tokens(w: Workload, step: int, seed: int = 0, device="cpu"):
    """One new token per sequence for decode step `step`: k, v bf16 [B][1][Hkv][d]."""
    g = _gen(device, seed * _MIX + 500_000 + step)
    shape = (w.batch, 1, w.num_kv_heads, w.head_dim)
    k = torch.randn(shape, generator=g, device=device)
    v = torch.randn(shape, generator=g, device=device)
    if w.k_outlier_channels:
        idx = torch.tensor(w.k_outlier_channels, device=device)
        k[..., idx] *= w.k_outlier_factor
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def scaled(w: Workload, **changes) -> Workload:
    """A copy with some fields changed (smaller parity cases of a workload)."""
    d = dict(w.__dict__)
    d.update(changes)
    return Workload(**d)


# ------------------------------------------------------------ replay toy
REPLAY = {"layers": 8, "d": 128, "n_win": 512, "T": 65536}


def replay_net(layers: int, d: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Weights of the toy network: float32 [layers][4][d][d] (Wq, Wk, Wv, Wo),
    N(0, 1/d)."""
    g = _gen(device, seed * _MIX + 31)
    return torch.randn((layers, 4, d, d), generator=g, device=device) * (1.0 / d ** 0.5)


def replay_inputs(first: int, n: int, d: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Inputs of positions first .. first + n - 1 of one synthetic sequence:
    float32 [n][d], N(0, 1); position p's row does not depend on the range
    drawn (each row from its own seeded generator chunk of 1024 positions)."""
    out = torch.empty((n, d), dtype=torch.float32, device=device)
    p = first
    while p < first + n:
        blk = p // 1024
        g = _gen(device, (seed * _MIX + 47) * 1_000_003 + blk)
        rows = torch.randn((1024, d), generator=g, device=device)
        lo = p - blk * 1024
        take = min(1024 - lo, first + n - p)
        out[p - first:p - first + take] = rows[lo:lo + take]
        p += take
    return out
