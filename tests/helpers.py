"""Host-side helpers for the parity tests: build caches through the C ABI from
the seeded workloads, and compare against the CPU oracle.

Nothing here computes the method: quantisation, dequantisation and attention
on the reference side all come from ``oracle``; on the device side from
libkvq through the binding.  The helpers only move tensors, slice units and
gather bytes by page table (index arithmetic).
"""
from __future__ import annotations

import concurrent.futures as cf
import math
import os
from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

import oracle
from fp4_kv_cache_kvq_gb300 import kvq, workloads

TOL = 2e-3  # max |err| <= TOL * max |V^| over the unit's attended values

_POOL = cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))


@dataclass
class Built:
    w: workloads.Workload
    cache: kvq.Fp4Cache
    lens: List[int]
    lens_dev: torch.Tensor
    table: Optional[torch.Tensor]       # device page table used for decode (None = contiguous)
    seq_k: List[torch.Tensor]           # per sequence, device bf16 [T_b][Hkv][d]
    seq_v: List[torch.Tensor]
    err: torch.Tensor


def ensure_built():
    from fp4_kv_cache_kvq_gb300 import build
    build.build()
    return kvq.load()


def build_fp4(w: workloads.Workload, lens: List[int], seed: int = 0, device="cuda", reserve: int = 0,
              keep_kv: bool = True) -> Built:
    """Allocate an FP4 cache for `lens` (+reserve positions per sequence) and
    append every sequence's keys/values through kvq_append, one call per
    sequence (page-table row b; contiguous caches get an explicit identity row
    for the append and are decoded with page_table == NULL)."""
    table_cpu, num_pages, max_pages = workloads.page_layout(w, lens, reserve=reserve, seed=seed)
    table = table_cpu.to(device) if table_cpu is not None else None
    cache = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, w.page_size, num_pages, max_pages, page_table=table,
                         device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    zero = torch.zeros(1, dtype=torch.int32, device=device)
    seq_k, seq_v = [], []
    for b, n in enumerate(lens):
        k, v = workloads.sequence_kv(w, b, n, seed=seed, device=device)
        if n > 0:
            row = table[b:b + 1] if table is not None else torch.arange(
                b * max_pages, (b + 1) * max_pages, dtype=torch.int32, device=device)[None]
            kvq.append(cache, zero, k[None], v[None], err=err, page_table=row)
        if keep_kv:
            seq_k.append(k)
            seq_v.append(v)
    lens_dev = torch.tensor(lens, dtype=torch.int32, device=device)
    return Built(w, cache, list(lens), lens_dev, table, seq_k, seq_v, err)


def oracle_unit(q_rows, k_rows, v_rows, scale, window=0, swa_scales=None):
    return oracle.decode_unit(q_rows, k_rows, v_rows, scale, window=window, swa_scales=swa_scales)


def check_units(out: torch.Tensor, q: torch.Tensor, units, kv_of, G: int, scale: float, window: int = 0,
                swa_scales_of=None, tol: float = TOL):
    """Compare decode output rows of each (b, h) unit with the oracle.
    kv_of(b, h) -> (k [T][d], v [T][d]) host tensors.  Returns the worst
    err / max|V^| ratio seen."""
    out_h = out.detach().cpu().double().numpy()
    q_h = q.detach().cpu().float().numpy()

    def one(bh):
        b, h = bh
        k, v = kv_of(b, h)
        sc = swa_scales_of(h) if swa_scales_of else None
        ref, vmax = oracle.decode_unit(q_h[b, h * G:(h + 1) * G], k, v, scale, window=window, swa_scales=sc)
        got = out_h[b, h * G:(h + 1) * G]
        if k.shape[0] == 0:
            return b, h, float(np.abs(got).max()), 0.0
        return b, h, float(np.abs(got - ref).max()), vmax

    worst = 0.0
    for b, h, err, vmax in _POOL.map(one, list(units)):
        if vmax == 0.0:
            assert err == 0.0, (b, h, err)
            continue
        ratio = err / vmax
        worst = max(worst, ratio)
        assert ratio <= tol, f"unit (b={b}, h={h}): max|err| {err:.3e} > {tol} * max|V^| ({vmax:.3e})"
    return worst


def host_kv_of(built: Built):
    def kv_of(b, h):
        k = built.seq_k[b][:, h].float().cpu()
        v = built.seq_v[b][:, h].float().cpu()
        return k.numpy(), v.numpy()

    return kv_of


def unpack_pool_rows(cache: kvq.Fp4Cache, phys_pages, h: int, n: int):
    """Positions 0..n-1 of one kv head, read from the listed physical pages of
    the FP4 pool and rearranged (byte indexing only) into per-token rows:
    (k_codes [n][D/2], k_scales [n][D/16], v_codes [n][D/2], v_scales [n][D/16])
    with byte k of a code row holding channel 2k (low nibble) and 2k+1 (high
    nibble), as the oracle's quantiser writes them."""
    D, G = cache.head_dim, cache.group
    nb = D // 16
    idx = torch.as_tensor(np.asarray(phys_pages), dtype=torch.long, device=cache.pool.device)
    blocks = cache.pool.index_select(0, idx)[:, h].reshape(-1, cache.pool.shape[-1]).cpu().numpy()
    ng = blocks.shape[0]
    kc = blocks[:, :G * D // 2].reshape(ng * G, D // 2)
    ks = blocks[:, G * D // 2:G * (D // 2 + nb)].reshape(ng * G, nb)
    vrows = blocks[:, G * (D // 2 + nb):G * (D + nb)].reshape(ng * G // 2, D)
    vs = blocks[:, G * (D + nb):].reshape(ng * G // 2, nb, 2).transpose(0, 2, 1).reshape(ng * G, nb)
    # undo the per-row chunk permutation of the pair rows
    i = np.arange(vrows.shape[0])[:, None] % (G // 2)
    if D == 64:
        chunks = vrows.reshape(-1, 8, 8)
        u = np.arange(8)[None, :] ^ (((i >> 1) & 1) << 2)
    else:
        chunks = vrows.reshape(-1, D // 16, 16)
        u = np.arange(D // 16)[None, :] ^ ((i & 3) << 1)
    logical = np.take_along_axis(chunks, u[:, :, None], axis=1).reshape(-1, D)
    nib = np.stack([logical & 0x0F, logical >> 4], axis=1).reshape(-1, D)  # token 2i, then 2i+1
    vc = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return kc[:n], ks[:n], vc[:n], vs[:n]


def gather_unit_bytes(cache: kvq.Fp4Cache, table_row: Optional[np.ndarray], b: int, h: int, n: int):
    """Codes and scales of positions 0..n-1 of sequence b, kv head h (see
    unpack_pool_rows)."""
    P = cache.page_size
    pages = max(1, (n + P - 1) // P)
    if table_row is None:
        phys = np.arange(b * cache.max_pages_per_seq, b * cache.max_pages_per_seq + pages)
    else:
        phys = np.asarray(table_row[:pages])
    return unpack_pool_rows(cache, phys, h, n)


def softmax_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
