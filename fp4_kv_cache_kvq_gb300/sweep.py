"""Bit-width / layout sweep: what each KV-cache format of the results table on
"Quantising the KV cache" does to decode attention, on synthetic keys and
values (the page measures logit drift in a tiny trained model whose weights
and prompts are not available; here the measure is the attention output
itself, against fp64-accumulated attention over the unquantised values).

Every format runs through ``kvq_fake_quant`` (quantise, then dequantise) and
the outputs through ``kvq_attn_dense``, both CUDA kernels of libkvq.  Cases:
N(0,1) keys and values; four fixed K outlier channels x20 (the GQA workload);
one K channel x100 (the week's "an outlier channel destroying a group").

    python -m fp4_kv_cache_kvq_gb300.sweep [--batch 8 --tokens 4096 ...] [--json FILE]

Columns: bits per number (b + s/g, section "Maths"); max |err| / max|V| over
the (sequence, query head) rows; RMS error relative to the RMS output; the
share of rows whose most attended position is unchanged.
"""
from __future__ import annotations

import argparse
import json
import math
from typing import Dict, List

import torch

from . import build, kvq, workloads

_LAYOUT = {"fp8": kvq.LAYOUT_FP8_TENSOR, "tok": kvq.LAYOUT_INT_PER_TOKEN,
           "chan": kvq.LAYOUT_INT_PER_CHANNEL, "fp4": kvq.LAYOUT_FP4_G16}

CASES: Dict[str, dict] = {
    "N(0,1)": {},
    "K channels {3,17,64,101} x20": {"k_outlier_channels": (3, 17, 64, 101), "k_outlier_factor": 20.0},
    "K channel 3 x100": {"k_outlier_channels": (3,), "k_outlier_factor": 100.0},
}


def formats(bit_widths=(8, 6, 4, 3, 2)):
    """(name, (K layout, bits), (V layout, bits))."""
    out = [("FP8 E4M3, one scale per tensor", ("fp8", 8), ("fp8", 8))]
    out += [(f"INT{b} per token", ("tok", b), ("tok", b)) for b in bit_widths]
    out += [(f"INT{b}, K per channel, V per token", ("chan", b), ("tok", b)) for b in bit_widths]
    out.append(("FP4 E2M1, E4M3 scale per 16", ("fp4", 4), ("fp4", 4)))
    return out


def bits_per_number(kind: str, b: int, tokens: int, head_dim: int) -> float:
    """b + s/g: an FP16 scale per head_dim channels (per token) or per
    `tokens` positions (per channel); FP4 pays an E4M3 byte per 16 values;
    FP8's single fp32 scale per tensor rounds to nothing."""
    if kind == "fp8":
        return 8.0
    if kind == "fp4":
        return 4.0 + 8.0 / 16.0
    return b + 16.0 / (head_dim if kind == "tok" else tokens)


def _kv(w: workloads.Workload, seed: int, device) -> tuple:
    ks, vs = [], []
    for b in range(w.batch):
        k, v = workloads.sequence_kv(w, b, w.context, seed=seed, device=device)
        ks.append(k)
        vs.append(v)
    return torch.stack(ks).contiguous(), torch.stack(vs).contiguous()


def run(batch=8, tokens=4096, kv_heads=8, q_heads=32, head_dim=128, seed=0, device="cuda",
        bit_widths=(8, 6, 4, 3, 2)) -> List[dict]:
    rows = []
    for case, changes in CASES.items():
        w = workloads.Workload("sweep", batch, kv_heads, q_heads, head_dim, context=tokens, **changes)
        K, V = _kv(w, seed, device)
        q = workloads.queries(w, seed=seed, device=device)
        scale = 1.0 / math.sqrt(head_dim)
        ref, top_ref = kvq.attn_dense(q, K.float(), V.float(), scale, want_top=True)
        G = q_heads // kv_heads
        vmax = V.float().abs().amax(dim=(1, 3)).repeat_interleave(G, dim=1)  # [B][Hq]
        rms_ref = ref.pow(2).mean().sqrt()
        rows.append({"case": case, "format": "BF16 (unquantised)", "bits": 16.0, "max_err_rel": 0.0,
                     "rms_err_rel": 0.0, "top1_unchanged": 1.0})
        for name, (kk, kb), (vk, vb) in formats(bit_widths):
            kh, _, _ = kvq.fake_quant(K, _LAYOUT[kk], kb)
            vh, _, _ = kvq.fake_quant(V, _LAYOUT[vk], vb)
            out, top = kvq.attn_dense(q, kh, vh, scale, want_top=True)
            err = (out - ref).abs()
            rows.append({
                "case": case, "format": name,
                "bits": 0.5 * (bits_per_number(kk, kb, tokens, head_dim) + bits_per_number(vk, vb, tokens, head_dim)),
                "max_err_rel": float((err.amax(dim=2) / vmax).max()),
                "rms_err_rel": float((out - ref).pow(2).mean().sqrt() / rms_ref),
                "top1_unchanged": float((top == top_ref).float().mean()),
            })
    return rows


def markdown(rows: List[dict]) -> str:
    lines = []
    for case in dict.fromkeys(r["case"] for r in rows):
        lines += [f"**{case}**", "", "| format | bits/number | max err / max abs V | RMS err / RMS out | top position unchanged |",
                  "|---|---|---|---|---|"]
        for r in rows:
            if r["case"] == case:
                lines.append(f"| {r['format']} | {r['bits']:.4g} | {r['max_err_rel']:.3g} | {r['rms_err_rel']:.3g} | "
                             f"{100 * r['top1_unchanged']:.1f}% |")
        lines.append("")
    return "\n".join(lines)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--kv-heads", type=int, default=8)
    ap.add_argument("--q-heads", type=int, default=32)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--json", default=None, help="also write the rows as JSON to this file")
    a = ap.parse_args(argv)
    build.build()
    rows = run(a.batch, a.tokens, a.kv_heads, a.q_heads, a.head_dim, a.seed)
    print(markdown(rows))
    if a.json:
        with open(a.json, "w") as f:
            json.dump({"config": vars(a), "rows": rows}, f, indent=1)


if __name__ == "__main__":
    main()
