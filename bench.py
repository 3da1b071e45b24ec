#!/usr/bin/env python3
"""Decode-attention throughput on the FP4 KV cache (one JSON line on rank 0).

A step is one pass of the hot path over the long_context workload (B32,
Hkv8, Hq64, d128, context 32768, one layer): append one new bf16 token per
sequence into the FP4 cache (quantise-on-append), then split-K decode
attention of 64 query heads per sequence over the cache (dequantised in the
kernel) and the cross-split merge.  The appended position cycles through the
64 slots after the prefilled context, so every step attends 32769..32832
positions.  `value` is KV-tokens/s (one KV-token = one cached position of one
sequence across all kv heads, K and V) over the timed steps; inputs are
resident in HBM and the 1.2 GB cache is far larger than L2.

--impl reference times the CPU oracle (plain C, fp64 attention over the
dequantised cache) on the host cores on a bounded sample of the same step.
Under torchrun every rank runs an independent replica (weak scaling, no
data-path collective); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from fp4_kv_cache_kvq_gb300 import workloads  # noqa: E402

METRIC = "decode-attn KV-tokens/s and achieved HBM GB/s (% of ~8 TB/s) on FP4 cache, 1xGB300"
UNIT = "KV-tokens/s"
PREROLL_US = 2000   # GPU-side wait queued ahead of a timed region
CYCLE = 64          # appended positions cycle through this many slots after the context
NQ = 8              # distinct query sets cycled through the steps
FALLBACK_HBM_GBS = 6800.0
_CSRC = os.path.join(ROOT, "fp4_kv_cache_kvq_gb300", "csrc")
# the sources a committed capture's kernel is compiled from (hashed together)
DECODE_SRC = tuple(os.path.join(_CSRC, f) for f in ("kvq_decode_kernel.cuh", "kvq_decode.cu", "kvq_append.cuh",
                                                    "kvq_common.cuh"))
PROFILE = os.path.join(ROOT, "profiles", "decode_fp4_long_context.md")
APPEND_SRC = tuple(os.path.join(_CSRC, f) for f in ("kvq_append.cu", "kvq_append.cuh", "kvq_common.cuh"))
APPEND_PROFILE = os.path.join(ROOT, "profiles", "append_fp4_prefill.md")
PREFILL_SRC = tuple(os.path.join(_CSRC, f) for f in ("kvq_prefill.cu", "kvq_tc.cuh", "kvq_common.cuh"))
PREFILL_PROFILE = os.path.join(ROOT, "profiles", "prefill_fp4_prefill_attn.md")


# ----------------------------------------------------------------- distributed plumbing
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def _dev(self):
        return torch.device("cuda", self.local) if (self.pg and self.pg.get_backend() == "nccl") else "cpu"

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def reduce(self, x: float, op: str) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=self._dev())
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def combine_ranks(dist: Dist, units: float, seconds: float):
    """Whole-job throughput: units summed over ranks / max time over ranks."""
    total_units = dist.reduce(units, "sum")
    max_s = dist.reduce(seconds, "max")
    return total_units / max_s, max_s


# ----------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        exe = shutil.which("nvidia-smi")
        if exe is None:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.proc = subprocess.Popen([exe, f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                      "-i", str(device_index), "-lms", "200"],
                                     stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [r.split(",") for r in open(self.path).read().strip().splitlines() if r.strip()]
        os.unlink(self.path)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for i, n in enumerate(names):
                    if r[5 + i].strip().lower().startswith("active"):
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- helpers
def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_sha256(src) -> str:
    """sha256 of a kernel's source: one file, or several files' bytes in order."""
    h = hashlib.sha256()
    for f in ((src,) if isinstance(src, str) else src):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(profile=PROFILE, src=DECODE_SRC, key="traffic_bytes_per_launch"):
    """DRAM bytes per launch (the summary's line `key`) from a committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    try:
        text = open(profile).read()
        sha = source_sha256(src)
        fields = dict(line.split(":", 1) for line in text.splitlines() if line.startswith(("traffic_", "source_")))
        if fields.get("source_sha256", "").strip() != sha:
            return None
        return int(float(fields[key].strip()))
    except Exception:
        return None


def flush_l2(buf, i: int):
    """Evict L2 before a timed step: write `buf` (2 x L2) and then read it
    back, so that L2 holds clean lines of an unrelated buffer (as after a
    flush and invalidate) rather than dirty ones whose write-back would land
    inside the next timed launch."""
    buf.fill_(i & 0xFF)
    buf.view(torch.int32).max()


def fp4_bytes_per_token(w) -> int:
    """FP4 cache bytes of one KV-token: K and V, all kv heads, codes + scales."""
    return 2 * w.num_kv_heads * (w.head_dim // 2 + w.head_dim // 16)


class Setup:
    """The resident FP4 cache of a workload plus the per-step inputs."""

    def __init__(self, w, seed: int, device, layers: int = 1, nvfp4: bool = False, kernel: str = "mma",
                 fused: bool = True):
        from fp4_kv_cache_kvq_gb300 import kvq
        self.w = w
        self.kernel = kernel
        # the append fused into the decode launch (kvq_append_decode_attn):
        # caches without an FP8 window, decoded by the default kernel
        self.fused = fused and w.window == 0 and kernel == "mma"
        self.layers = layers
        self.kvq = kvq
        self.lens0 = workloads.lengths(w, seed)
        table, num_pages, max_pages = workloads.page_layout(w, self.lens0, reserve=CYCLE, seed=seed)
        self.table = table.to(device) if table is not None else None
        self.cache = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, w.page_size, num_pages, max_pages,
                                  page_table=self.table, device=device, nvfp4=nvfp4)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        if nvfp4:  # second-level scales from the first sequence's prefill (calibration)
            k0, v0 = workloads.sequence_kv(w, 0, min(self.lens0[0], 8192), seed=seed, device=device)
            kvq.fp8_set_scales(self.cache, k0[None], v0[None], err=self.err)
            del k0, v0
        zero = torch.zeros(1, dtype=torch.int32, device=device)
        for b, n in enumerate(self.lens0):
            k, v = workloads.sequence_kv(w, b, n, seed=seed, device=device)
            row = self.table[b:b + 1] if self.table is not None else torch.arange(
                b * max_pages, (b + 1) * max_pages, dtype=torch.int32, device=device)[None]
            kvq.append(self.cache, zero, k[None], v[None], err=self.err, page_table=row)
            del k, v
        self.swa = None
        if w.window > 0:
            # FP8 window beside the FP4 cache: scales from the prefill's last W
            # positions of every sequence, then those positions into the rings
            W = w.window
            tails_k, tails_v = [], []
            for b, n in enumerate(self.lens0):
                k, v = workloads.sequence_kv(w, b, n, seed=seed, device=device)
                tails_k.append(k[n - W:])
                tails_v.append(v[n - W:])
                del k, v
            kw, vw = torch.stack(tails_k).contiguous(), torch.stack(tails_v).contiguous()
            self.swa = kvq.Fp8WindowCache(w.batch, w.num_kv_heads, w.head_dim, W, device=device)
            kvq.fp8_set_scales(self.swa, kw, vw, err=self.err)
            start = torch.tensor([n - W for n in self.lens0], dtype=torch.int32, device=device)
            kvq.append(self.swa, start, kw, vw, err=self.err)
            del kw, vw, tails_k, tails_v
        # further layers: their own copies of the cache (same contents)
        self.caches = [self.cache]
        self.swas = [self.swa]
        for _ in range(1, layers):
            c = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, w.page_size, num_pages, max_pages,
                             page_table=self.table, device=device, nvfp4=nvfp4)
            c.pool.copy_(self.cache.pool)
            if nvfp4:
                c.k_gscale.copy_(self.cache.k_gscale)
                c.v_gscale.copy_(self.cache.v_gscale)
            self.caches.append(c)
            if self.swa is not None:
                sw = kvq.Fp8WindowCache(w.batch, w.num_kv_heads, w.head_dim, w.window, device=device)
                for dst, src in ((sw.k_codes, self.swa.k_codes), (sw.v_codes, self.swa.v_codes),
                                 (sw.k_scales, self.swa.k_scales), (sw.v_scales, self.swa.v_scales)):
                    dst.copy_(src)
                self.swas.append(sw)
            else:
                self.swas.append(None)
        toks = [workloads.step_tokens(w, i, seed=seed, device=device) for i in range(CYCLE)]
        self.k_new = [t[0] for t in toks]
        self.v_new = [t[1] for t in toks]
        self.k_row = [k[:, 0] for k in self.k_new]  # [B][Hkv][d] views for the fused call
        self.v_row = [v[:, 0] for v in self.v_new]
        self.q = [workloads.queries(w, seed=seed, step=i, device=device) for i in range(NQ)]
        base = torch.tensor(self.lens0, dtype=torch.int32, device=device)
        self.pos = [base + i for i in range(CYCLE)]
        self.lens = [base + i + 1 for i in range(CYCLE)]
        self.kv_tokens = [sum(self.lens0) + (i + 1) * w.batch for i in range(CYCLE)]
        self.scale = 1.0 / math.sqrt(w.head_dim)
        B, Hq, D = w.batch, w.num_q_heads, w.head_dim
        self.outs = [torch.empty((B, Hq, D), dtype=torch.float32, device=device) for _ in range(layers)]
        self.out = self.outs[-1]
        nbytes = kvq.decode_workspace_bytes(B, Hq, w.num_kv_heads, D)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

    def step(self, i: int, q=None, k=None, v=None, ev=None, outs=None):
        """One decode step: append the new token to every layer's caches,
        then decode attention for every layer (the same token and query per
        layer).  Returns the KV-tokens attended (all layers)."""
        s = i % CYCLE
        kvq = self.kvq
        kk = self.k_new[s] if k is None else k
        vv = self.v_new[s] if v is None else v
        qq = self.q[i % NQ] if q is None else q
        if self.fused:
            if ev is not None:
                ev[0].record()
            kr = self.k_row[s] if k is None else kk[:, 0]
            vr = self.v_row[s] if v is None else vv[:, 0]
            for cache, out in zip(self.caches, self.outs if outs is None else outs):
                kvq.append_decode_attn(cache, self.lens[s], kr, vr, qq, self.scale, out=out, workspace=self.ws,
                                       err=self.err)
            if ev is not None:
                ev[1].record()
            return self.kv_tokens[s] * self.layers
        for cache, swa in zip(self.caches, self.swas):
            kvq.append(cache, self.pos[s], kk, vv, err=self.err)
            if swa is not None:
                kvq.append(swa, self.pos[s], kk, vv, err=self.err)
        if ev is not None:
            ev[0].record()
        for cache, swa, out in zip(self.caches, self.swas, self.outs if outs is None else outs):
            kvq.decode_attn(cache, self.lens[s], qq, self.scale, swa=swa, out=out, workspace=self.ws, err=self.err,
                            kernel=self.kernel)
        if ev is not None:
            ev[1].record()
        return self.kv_tokens[s] * self.layers

    def capture_graphs(self):
        """One CUDA graph per step of the cycle for the appends and one for the
        decode calls (the same launches as step(), replayed without host
        launch gaps); the decode-only events go between the two replays."""
        self.graphs = []
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i in range(CYCLE):
                s = i % CYCLE
                ga, gd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.graph(ga, stream=side):
                    for cache, swa in zip(self.caches, self.swas):
                        self.kvq.append(cache, self.pos[s], self.k_new[s], self.v_new[s], err=self.err)
                        if swa is not None:
                            self.kvq.append(swa, self.pos[s], self.k_new[s], self.v_new[s], err=self.err)
                with torch.cuda.graph(gd, stream=side):
                    for cache, swa, out in zip(self.caches, self.swas, self.outs):
                        self.kvq.decode_attn(cache, self.lens[s], self.q[i % NQ], self.scale, swa=swa, out=out,
                                             workspace=self.ws, err=self.err, kernel=self.kernel)
                self.graphs.append((ga, gd))
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()

    def step_graph(self, i: int, ev=None):
        """step(i) replayed from the captured graphs (i % CYCLE == the cycle
        slot, and CYCLE is a multiple of NQ, so slot and query set match)."""
        ga, gd = self.graphs[i % CYCLE]
        ga.replay()
        if ev is not None:
            ev[0].record()
        gd.replay()
        if ev is not None:
            ev[1].record()
        return self.kv_tokens[i % CYCLE] * self.layers

    def decode_algorithmic_bytes(self, i: int) -> int:
        """Algorithmic bytes of one layer's decode call at step i."""
        w = self.w
        s = i % CYCLE
        win = min(w.window, min(self.lens0) + s + 1) if w.window else 0
        b = (self.kv_tokens[s] - win * w.batch) * fp4_bytes_per_token(w)
        b += win * w.batch * 2 * w.num_kv_heads * w.head_dim  # FP8 window codes (K and V)
        b += w.batch * w.num_q_heads * w.head_dim * (2 + 4)  # q in, out
        b += w.batch * 4                                      # lengths
        if self.table is not None:
            b += sum(-(-(n + s + 1) // w.page_size) for n in self.lens0) * 4
        return b


# ----------------------------------------------------------------- GPU arm
def run_gpu(args, dist: Dist):
    device = torch.device("cuda", dist.local)
    torch.cuda.set_device(device)
    from fp4_kv_cache_kvq_gb300 import build
    build.build()
    w = workloads.WORKLOADS[args.workload]
    L = args.layers
    st = Setup(w, args.seed, device, layers=L, nvfp4=args.format == "nvfp4", kernel=args.decode_kernel,
               fused=args.fused_append)
    K, Wm = args.steps, args.warmup
    for i in range(Wm):
        st.step(i)
    torch.cuda.synchronize()
    if st.err.item() != 0:
        raise RuntimeError(f"device error flag {st.err.item()} during warm-up")
    if args.graphs:
        st.capture_graphs()
        for i in range(Wm):
            st.step_graph(Wm + i)
        torch.cuda.synchronize()

    # ---- device-resident timing.  A cache smaller than twice L2 would stay
    # in L2 from step to step: then every step is timed on its own, after a
    # write of a 2 x L2 buffer that evicts it, and the warm-L2 rate is
    # reported beside it.
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size
    small = st.cache.nbytes < 2 * l2_bytes
    flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=device) if small else None

    def run_step(i, ev=None):
        return st.step_graph(i, ev=ev) if args.graphs else st.step(i, ev=ev)

    def preroll():
        """Queue a GPU-side wait of about PREROLL_US before the first timed
        event, so that the stream is busy while the host enqueues the first
        step: the start event then marks the GPU reaching the steps, not the
        host's latency from an idle stream.  After the first step the host
        stays ahead by itself (a step's enqueue takes a fraction of its GPU
        time), so this only removes the start-up gap."""
        torch.cuda._sleep(int(PREROLL_US * 1e-6 * sm_hz))

    sm_hz = torch.cuda.get_device_properties(device).clock_rate * 1e3 if hasattr(
        torch.cuda.get_device_properties(device), "clock_rate") else 2.0e9

    def timed(flushed: bool):
        """K steps.  Back to back (events only at the two ends: a timing event
        between two kernels keeps the second from starting while the first
        drains), or, after an L2 flush, each step on its own events."""
        steps = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(device.index)
        dist.barrier()
        torch.cuda.synchronize()
        preroll()
        t0.record()
        tokens = 0
        for i in range(K):
            if flushed:
                flush_l2(flush, i)
                steps[i][0].record()
            tokens += run_step(Wm + i)
            if flushed:
                steps[i][1].record()
        t1.record()
        torch.cuda.synchronize()
        dist.barrier()
        clk = clocks.stop()
        if flushed:
            elapsed = sum(a.elapsed_time(b) for a, b in steps) / 1e3
        else:
            elapsed = t0.elapsed_time(t1) / 1e3
        return tokens, elapsed, clk

    def decode_call_ms(flushed: bool):
        """The decode calls' own duration (events around the decode part of
        each step), for the roofline: the same steps, timed again."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        torch.cuda.synchronize()
        preroll()
        for i in range(K):
            if flushed:
                flush_l2(flush, i)
            run_step(Wm + i, ev=evs[i])
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    warm_value = None
    if small:
        wt, we, _ = timed(False)
        warm_value, _ = combine_ranks(dist, wt, we)
    tokens, elapsed_s, clk = timed(small)
    decode_ms = decode_call_ms(small)
    if st.err.item() != 0:
        raise RuntimeError(f"device error flag {st.err.item()} during the timed steps")
    value, max_s = combine_ranks(dist, tokens, elapsed_s)
    dec_bytes = statistics.mean(st.decode_algorithmic_bytes(Wm + i) for i in range(K))
    dec_s = statistics.mean(decode_ms) / 1e3 / L  # one layer's decode call
    achieved = dec_bytes / dec_s / 1e9
    peak, peak_src = measured_hbm_peak()
    # append: read the new bf16 K and V, write their codes and scales
    append_bytes = w.batch * (2 * w.num_kv_heads * w.head_dim * 2 + fp4_bytes_per_token(w))
    step_bytes = L * (dec_bytes + append_bytes)

    # ---- end to end through the public API with pinned host buffers.  Every
    # step copies its query and new token in from pinned host memory and its
    # output back.  For caches larger than L2 the copies run on a second
    # stream, double-buffered, so that step i + 1's inputs upload and step
    # i - 1's output downloads while step i computes (events order each
    # buffer's reuse).
    Ke = min(K, max(50, K // 4))
    q_host = [q.cpu().pin_memory() for q in st.q]
    k_host = [k.cpu().pin_memory() for k in st.k_new]
    v_host = [v.cpu().pin_memory() for v in st.v_new]
    outs_host = [[torch.empty(st.out.shape, dtype=torch.float32).pin_memory() for _ in range(L)] for _ in range(2)]
    bufs = [(torch.empty_like(st.q[0]), torch.empty_like(st.k_new[0]), torch.empty_like(st.v_new[0]),
             [torch.empty_like(st.out) for _ in range(L)]) for _ in range(2)]
    q_dev, k_dev, v_dev = bufs[0][0], bufs[0][1], bufs[0][2]
    compute = torch.cuda.current_stream()
    copier = torch.cuda.Stream()
    loaded = [torch.cuda.Event() for _ in range(2)]    # inputs of a buffer set uploaded
    consumed = [torch.cuda.Event() for _ in range(2)]  # step done with a buffer set's inputs and outputs
    fetched = [torch.cuda.Event() for _ in range(2)]   # a buffer set's outputs downloaded
    torch.cuda.synchronize()
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    preroll()  # as for the device-resident timing: the host's first enqueue is not timed as GPU idle
    e0.record()
    copier.wait_stream(compute)

    def upload(i):
        qd, kd, vd, _ = bufs[i % 2]
        with torch.cuda.stream(copier):
            if i >= 2:
                copier.wait_event(consumed[i % 2])
            s_ = (Wm + i) % CYCLE
            qd.copy_(q_host[(Wm + i) % NQ], non_blocking=True)
            kd.copy_(k_host[s_], non_blocking=True)
            vd.copy_(v_host[s_], non_blocking=True)
            loaded[i % 2].record(copier)

    e2e_tokens = 0
    if small:
        # steps of a few tens of microseconds: the host's event calls would
        # cost more than the copies they hide, so the copies go in line on the
        # compute stream
        qd, kd, vd, od = bufs[0]
        for i in range(Ke):
            s_ = (Wm + i) % CYCLE
            qd.copy_(q_host[(Wm + i) % NQ], non_blocking=True)
            kd.copy_(k_host[s_], non_blocking=True)
            vd.copy_(v_host[s_], non_blocking=True)
            e2e_tokens += st.step(Wm + i, q=qd, k=kd, v=vd, outs=od)
            for oh, o in zip(outs_host[0], od):
                oh.copy_(o, non_blocking=True)
    else:
        upload(0)
        for i in range(Ke):
            if i + 1 < Ke:
                upload(i + 1)
            qd, kd, vd, od = bufs[i % 2]
            compute.wait_event(loaded[i % 2])
            if i >= 2:
                compute.wait_event(fetched[i % 2])  # its outputs of step i - 2 are on the host
            e2e_tokens += st.step(Wm + i, q=qd, k=kd, v=vd, outs=od)
            consumed[i % 2].record(compute)
            with torch.cuda.stream(copier):
                copier.wait_event(consumed[i % 2])
                for oh, o in zip(outs_host[i % 2], od):
                    oh.copy_(o, non_blocking=True)
                fetched[i % 2].record(copier)
    compute.wait_stream(copier)
    e1.record()
    torch.cuda.synchronize()
    dist.barrier()
    e2e_value, _ = combine_ranks(dist, e2e_tokens, e0.elapsed_time(e1) / 1e3)
    h2d = q_dev.numel() * 2 + k_dev.numel() * 2 + v_dev.numel() * 2
    d2h = sum(oh.numel() for oh in outs_host[0]) * 4

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": K, "warmup": Wm,
        "ms_per_step": max_s * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}; step = append 1 token/seq + decode attention"
                   + (f", {L} layers" if L > 1 else "") + (", NVFP4 cache" if args.format == "nvfp4" else ""),
                   "layers": L, "format": args.format,
                   "batch": w.batch, "kv_heads": w.num_kv_heads, "q_heads": w.num_q_heads,
                   "head_dim": w.head_dim, "context": w.context, "page_size": w.page_size,
                   "cache_bytes": st.cache.nbytes * L,
                   "l2": (f"cache smaller than 2 x L2: {2 * l2_bytes} B written and read back before every step, "
                          f"steps timed "
                          f"one by one (warm-L2 rate without the flush: {warm_value:.4g} {UNIT})") if small
                   else f"inputs larger than L2 (FP4 cache {st.cache.nbytes} B vs {l2_bytes} B L2), no flush",
                   "launch": "CUDA graphs (one per step of the cycle: appends, then decode)" if args.graphs
                   else "eager launches",
                   "timing": f"a {PREROLL_US} us GPU-side wait is queued before the start events (the "
                             "device-resident steps, the per-call events and the end-to-end steps), so the "
                             "host's enqueue of the first step from an idle stream is not timed",
                   "parallelism": f"replicas x{dist.world}",
                   "decode_kernel": "kvq_decode_attn_tc (tcgen05)" if args.decode_kernel == "tcgen05"
                   else "kvq_append_decode_attn (append fused into the mma.sync decode)" if st.fused
                   else "kvq_decode_attn (mma.sync)"},
        "value_l2_warm": warm_value,
        "hbm_gbs_step": step_bytes * K / elapsed_s / 1e9,
        "hbm_gbs_decode": achieved,
        "hbm_pct_of_8tbs_decode": 100.0 * achieved / 8000.0,
        "roofline": {"bound": "hbm", "kernel": ("kvq_append_decode_attn (append fused into the split-K decode, "
                                                "+ merge launch)" if st.fused
                                                else "kvq_decode_attn (split-K decode + merge launches)")
                     + (", FP8 window folded into the merge" if w.window else ""),
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src,
                     "traffic": profiled_traffic() if w.name == "long_context" and args.decode_kernel == "mma"
                     else None,
                     "algorithmic_bytes_per_launch": dec_bytes, "avg_launch_ms": dec_s * 1e3,
                     "median_launch_ms": statistics.median(decode_ms) / L,
                     "min_launch_ms": min(decode_ms) / L},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": Ke},
        "gpu_launches": L * (4 if w.window else 2 if st.fused else 3) * K,
    }
    if clk is not None:
        result["clocks"] = clk
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.seed, st, budget_s=args.cpu_budget,
                                              nvfp4=args.format == "nvfp4")
    return result


# ----------------------------------------------------------------- append throughput (prefill)
PREFILL_METRIC = "append (quantise-on-append) tokens/s and HBM GB/s into the FP4 cache, 1xGB300"


class AppendOracleSample:
    """The oracle's quantise-on-append of prefill tokens: the K and V of
    sequence 0's first `n_tok` tokens, every kv head, through the CPU block
    quantiser (NVFP4: with each head's second-level scale set from the
    sample beforehand, outside the timing), 256 tokens of one head per task
    on the host's threads (the oracle's C calls release the interpreter
    lock).  One token = one position of one sequence across all kv heads,
    K and V."""

    CHUNK = 256

    def __init__(self, w, seed: int, n_tok: int, nvfp4: bool, cores: int):
        import numpy as np

        import oracle
        self.oracle, self.nvfp4, self.cores = oracle, nvfp4, cores
        self.n_tok = max(self.CHUNK, n_tok // self.CHUNK * self.CHUNK)
        k, v = workloads.sequence_kv(w, 0, self.n_tok, seed=seed, device="cpu")
        # [Hkv][n][d], contiguous per head
        self.k = np.ascontiguousarray(k.float().numpy().transpose(1, 0, 2))
        self.v = np.ascontiguousarray(v.float().numpy().transpose(1, 0, 2))
        self.hkv = self.k.shape[0]
        self.Sk = [oracle.nvfp4_global_scale(self.k[h]) for h in range(self.hkv)] if nvfp4 else None
        self.Sv = [oracle.nvfp4_global_scale(self.v[h]) for h in range(self.hkv)] if nvfp4 else None

    def _task(self, h: int, t0: int):
        o, c = self.oracle, self.CHUNK
        if self.nvfp4:
            o.nvfp4_quantize_rows(self.k[h, t0:t0 + c], self.Sk[h])
            o.nvfp4_quantize_rows(self.v[h, t0:t0 + c], self.Sv[h])
        else:
            o.quantize_rows(self.k[h, t0:t0 + c])
            o.quantize_rows(self.v[h, t0:t0 + c])

    def run(self, pool):
        """Quantise the whole sample once: (tokens, seconds)."""
        t = time.perf_counter()
        futs = [pool.submit(self._task, h, t0) for t0 in range(0, self.n_tok, self.CHUNK) for h in range(self.hkv)]
        for f in futs:
            f.result()
        return self.n_tok, time.perf_counter() - t

    def describe(self, rounds: int, secs: float) -> str:
        return (f"{self.n_tok} tokens x {self.hkv} kv heads (K and V) of one prefill sequence through the CPU "
                f"{'NVFP4' if self.nvfp4 else 'FP4'} quantiser, {rounds} pass(es), {self.cores} threads, {secs:.1f} s")


def append_oracle_sample(w, seed: int, budget_s: float, nvfp4: bool = False):
    """cpu_baseline of the append workload: AppendOracleSample passes until
    about budget_s of host time is spent."""
    cores = os.cpu_count() or 1
    sample = AppendOracleSample(w, seed, 4096, nvfp4, cores)
    toks, secs, rounds = 0, 0.0, 0
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        while secs < budget_s:
            n, dt = sample.run(pool)
            toks += n
            secs += dt
            rounds += 1
    return {"value": toks / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample.describe(rounds, secs)}


def run_prefill(args, dist: Dist):
    """A step appends a whole prefill (B16 x 16384 tokens, or B1 x 16384 for
    prefill_b1; Hkv8, d128, bf16 K and V) into the FP4 cache; value = appended
    tokens/s (one token = one position of one sequence across all kv heads, K
    and V).  The B16 step reads 1.07 GB (past L2); the B1 step's 67 MB would
    sit in L2, so that run writes a 2 x L2 buffer before every step and times
    each append alone with events on its own stream position."""
    from fp4_kv_cache_kvq_gb300 import build, kvq
    device = torch.device("cuda", dist.local)
    torch.cuda.set_device(device)
    build.build()
    w = workloads.WORKLOADS[args.workload]
    B, T = w.batch, w.context
    max_pages = -(-T // w.page_size)
    nv = args.format == "nvfp4"
    cache = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, w.page_size, B * max_pages, max_pages, device=device, nvfp4=nv)
    k = torch.empty((B, T, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    for b in range(B):
        k[b], v[b] = workloads.sequence_kv(w, b, T, seed=args.seed, device=device)
    start = torch.zeros(B, dtype=torch.int32, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    if nv:  # second-level scales from the whole prefill (calibration, outside the timed region)
        kvq.fp8_set_scales(cache, k, v, err=err)
    K, Wm = args.steps, args.warmup
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=device) if 2 * k.nbytes < 2 * l2 else None
    for i in range(Wm):
        if flush is not None:
            flush_l2(flush, i)
        kvq.append(cache, start, k, v, err=err)
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index)
    dist.barrier()
    if flush is None:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(K):
            kvq.append(cache, start, k, v, err=err)
        t1.record()
        torch.cuda.synchronize()
        secs = t0.elapsed_time(t1) / 1e3
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush_l2(flush, i)
            evs[i][0].record()
            kvq.append(cache, start, k, v, err=err)
            evs[i][1].record()
        torch.cuda.synchronize()
        secs = sum(a.elapsed_time(b) for a, b in evs) / 1e3
    dist.barrier()
    clk = clocks.stop()
    if err.item() != 0:
        raise RuntimeError(f"device error flag {err.item()}")
    tokens = B * T
    value, max_s = combine_ranks(dist, tokens * K, secs)
    nbytes = 2 * k.numel() * 2 + tokens * fp4_bytes_per_token(w)
    achieved = nbytes * K / secs / 1e9
    peak, peak_src = measured_hbm_peak()
    # end to end: host K/V (pinned) copied in every step, the error word copied back
    Ke = min(K, 10)
    kh, vh = k.cpu().pin_memory(), v.cpu().pin_memory()
    errh = torch.empty(1, dtype=torch.int32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(Ke):
        k.copy_(kh, non_blocking=True)
        v.copy_(vh, non_blocking=True)
        kvq.append(cache, start, k, v, err=err)
        errh.copy_(err, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e, _ = combine_ranks(dist, tokens * Ke, e0.elapsed_time(e1) / 1e3)
    res = {
        "metric": PREFILL_METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world, "steps": K,
        "warmup": Wm, "ms_per_step": max_s * 1e3 / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}" + (", NVFP4 cache" if nv else ""), "format": args.format,
                   "batch": B, "tokens": T, "kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "page_size": w.page_size,
                   "l2": (f"inputs larger than L2 ({2 * k.nbytes / 1e9:.2f} GB of bf16 per step), no flush"
                          if flush is None else
                          f"L2 flushed before every step (a {2 * l2 >> 20} MiB buffer written and read back); "
                          f"each append timed alone"),
                   "parallelism": f"replicas x{dist.world}"},
        "roofline": {"bound": "hbm", "kernel": "append_fp4_kernel", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_src,
                     "traffic": profiled_traffic(APPEND_PROFILE, APPEND_SRC,
                                                 "traffic_bytes_per_launch" + ("_b1" if B == 1 else "")
                                                 + ("_nvfp4" if nv else "")),
                     "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": secs * 1e3 / K},
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": 2 * k.numel() * 2, "d2h_bytes_per_step": 4,
                "steps": Ke},
        "gpu_launches": K,
    }
    if clk is not None:
        res["clocks"] = clk
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = append_oracle_sample(w, args.seed, budget_s=min(20.0, args.cpu_budget), nvfp4=nv)
    return res


PREFILL_ATTN_METRIC = "chunked-prefill attention over the FP4 cache: query tokens/s (tensor-core TFLOP/s), 1xGB300"


def measured_tensor_peak():
    """Dense bf16 (= f16) tensor peak in TFLOP/s: the measured burst figure,
    else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "MEASURED_PEAKS.json bf16_tflops (burst), of measured"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s bf16 burst"


def run_prefill_attn(args, dist: Dist):
    """A step is one kvq_prefill_attn call: B4 x 1024 query tokens (Hq64, d128)
    attending causally over 16384 cached FP4 positions each.  value = query
    tokens/s; the roofline counts the causally attended multiply-adds
    (4 flop per query head, position and channel: QK^T and PV)."""
    from fp4_kv_cache_kvq_gb300 import build, kvq
    device = torch.device("cuda", dist.local)
    torch.cuda.set_device(device)
    build.build()
    w = workloads.WORKLOADS["prefill_attn"]
    B, T, C = w.batch, w.context, w.chunk
    max_pages = -(-T // w.page_size)
    nv = args.format == "nvfp4"
    cache = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, w.page_size, B * max_pages, max_pages, device=device, nvfp4=nv)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    k = torch.empty((B, T, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    for b in range(B):
        k[b], v[b] = workloads.sequence_kv(w, b, T, seed=args.seed, device=device)
    if nv:
        kvq.fp8_set_scales(cache, k, v, err=err)
    kvq.append(cache, torch.zeros(B, dtype=torch.int32, device=device), k, v, err=err)
    del k, v
    g = torch.Generator(device=device)
    g.manual_seed(args.seed * 1_000_003 + 4242)
    q = torch.randn((B, C, w.num_q_heads, w.head_dim), generator=g, device=device).to(torch.bfloat16)
    lens = torch.full((B,), T, dtype=torch.int32, device=device)
    out = torch.empty((B, C, w.num_q_heads, w.head_dim), dtype=torch.float32, device=device)
    K, Wm = args.steps, args.warmup
    for _ in range(Wm):
        kvq.prefill_attn(cache, lens, q, out=out, err=err)
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    t0.record()
    for _ in range(K):
        kvq.prefill_attn(cache, lens, q, out=out, err=err)
    t1.record()
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    if err.item() != 0:
        raise RuntimeError(f"device error flag {err.item()}")
    secs = t0.elapsed_time(t1) / 1e3
    tokens = B * C
    value, max_s = combine_ranks(dist, tokens * K, secs)
    positions = B * w.num_q_heads * sum(T - C + i + 1 for i in range(C))  # causally attended (row, position)
    flops = 4 * positions * w.head_dim
    achieved = flops * K / secs / 1e12
    peak, peak_src = measured_tensor_peak()
    # end to end: the chunk's queries in from pinned host memory, the output back
    qh = q.cpu().pin_memory()
    oh = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    Ke = min(K, 10)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(Ke):
        q.copy_(qh, non_blocking=True)
        kvq.prefill_attn(cache, lens, q, out=out, err=err)
        oh.copy_(out, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e, _ = combine_ranks(dist, tokens * Ke, e0.elapsed_time(e1) / 1e3)
    res = {
        "metric": PREFILL_ATTN_METRIC, "value": value, "unit": "query tokens/s", "n_gpus": dist.world, "steps": K,
        "warmup": Wm, "ms_per_step": max_s * 1e3 / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"prefill_attn: {w.description}" + (", NVFP4 cache" if nv else ""),
                   "format": args.format, "batch": B, "context": T, "chunk": C, "kv_heads": w.num_kv_heads,
                   "q_heads": w.num_q_heads, "head_dim": w.head_dim, "page_size": w.page_size,
                   "l2": "each kv head's cache (2.36 MB) is read by the 32 query-block CTAs of its chunk; no flush",
                   "parallelism": f"replicas x{dist.world}"},
        "roofline": {"bound": "tensor", "kernel": "prefill_fp4_kernel (tcgen05.mma f16, TMEM accumulators)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": peak_src,
                     "traffic": profiled_traffic(PREFILL_PROFILE, PREFILL_SRC) if not nv else None,
                     "algorithmic_flops_per_launch": flops,
                     "avg_launch_ms": secs * 1e3 / K},
        "e2e": {"value": e2e, "unit": "query tokens/s", "h2d_bytes_per_step": q.numel() * 2,
                "d2h_bytes_per_step": out.numel() * 4, "steps": Ke},
        "gpu_launches": K,
    }
    if clk is not None:
        res["clocks"] = clk
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = prefill_oracle_sample(w, args.seed, q, budget_s=min(20.0, args.cpu_budget))
    return res


def prefill_oracle_sample(w, seed: int, q, budget_s: float):
    """The oracle's prefill of sampled query tokens: for one (sequence, kv
    head) unit, the FP4 cache dequantised once (resident state), then fp64
    attention of each sampled token's G query rows over its causal prefix,
    tokens taken from the end of the chunk until the budget is spent.  Value
    in query tokens/s of the whole head group (Hq rows per token)."""
    import numpy as np

    import oracle
    T, C, G, d = w.context, w.chunk, w.group, w.head_dim
    k, v = workloads.sequence_kv(w, 0, T, seed=seed, device="cpu")
    kc, ks, _ = oracle.quantize_rows(k[:, 0].float().numpy())
    vc, vs, _ = oracle.quantize_rows(v[:, 0].float().numpy())
    kh, vh = oracle.dequantize_rows(kc, ks), oracle.dequantize_rows(vc, vs)
    qh = q[0, :, :G].float().cpu().numpy()
    scale = 1.0 / math.sqrt(d)
    t = time.perf_counter()
    rows = 0
    for i in range(C - 1, -1, -1):
        oracle.attend(qh[i], kh[:T - C + i + 1], vh[:T - C + i + 1], scale)
        rows += G
        if time.perf_counter() - t > budget_s:
            break
    dt = time.perf_counter() - t
    return {"value": rows / w.num_q_heads / dt, "unit": "query tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows // G} tokens x G={G} query rows of one kv head over ~{T} positions "
                      f"(fp64 C attention, one thread, {dt:.1f} s), scaled to Hq={w.num_q_heads} rows per token"}


SWA_REPLAY_METRIC = ("bounded SWA replay of a toy 8-layer sliding-window network (d 128, window 512): "
                     "replayed layer-positions/s, 1xGB300")


def run_swa_replay(args, dist: Dist):
    """A step is one bounded replay: the last n_win = 512 positions before
    position T = 65536 through all 8 layers of the toy sliding-window network
    (d 128), rebuilding every layer's window state.  value = layers x
    positions replayed per second.  The exact replay (from the receptive-field
    start, 4089 positions) is timed beside it, and the bounded replay's error
    against it is reported: each layer's state, and the output at position T
    computed from each state."""
    from fp4_kv_cache_kvq_gb300 import build, kvq
    device = torch.device("cuda", dist.local)
    torch.cuda.set_device(device)
    build.build()
    R = workloads.REPLAY
    L, d, nw, T = R["layers"], R["d"], R["n_win"], R["T"]
    t_exact = max(0, T - nw - (L - 1) * (nw - 1))
    t_bound = T - nw
    w = workloads.replay_net(L, d, seed=args.seed).to(device)
    emb = workloads.replay_inputs(t_exact, T + 1 - t_exact, d, seed=args.seed).to(device)  # through position T
    e_x = emb[:T - t_exact].contiguous()
    e_b = emb[t_bound - t_exact:T - t_exact].contiguous()
    ws = torch.empty(kvq.load().kvq_swa_replay_workspace_bytes(L, T + 1 - t_exact, d), dtype=torch.uint8,
                     device=device)
    states = torch.empty((L, 2, nw, d), dtype=torch.float32, device=device)
    # quality of the bounded state against the exact one
    sx, _ = kvq.swa_replay(w, e_x, nw, want_hidden=False, workspace=ws)
    sx = sx.clone()
    sb, _ = kvq.swa_replay(w, e_b, nw, want_hidden=False, workspace=ws)
    sb = sb.clone()
    _, hx = kvq.swa_replay(w, emb, nw, workspace=ws)
    hx = hx[-1].clone()
    _, hb = kvq.swa_replay(w, emb[t_bound - t_exact:].contiguous(), nw, workspace=ws)
    hb = hb[-1].clone()
    torch.cuda.synchronize()
    state_err = [float((sb[l] - sx[l]).abs().max() / sx[l].abs().max()) for l in range(L)]
    next_err = float((hb - hx).norm() / hx.norm())
    K, Wm = args.steps, args.warmup
    # quality against compute: replays that start m positions before the
    # window, from bounded (m = 0) up to exact (m = (L - 1)(n_win - 1))
    curve = []
    for m in sorted({0, nw // 4, nw // 2, nw, 2 * nw, 4 * nw, (L - 1) * (nw - 1)}):
        if m > (L - 1) * (nw - 1):
            continue
        t0 = T - nw - m
        sm, _ = kvq.swa_replay(w, emb[t0 - t_exact:T - t_exact].contiguous(), nw, want_hidden=False, workspace=ws)
        top = float((sm[L - 1] - sx[L - 1]).abs().max() / sx[L - 1].abs().max())
        _, hm = kvq.swa_replay(w, emb[t0 - t_exact:].contiguous(), nw, workspace=ws)
        nxt = float((hm[-1] - hx).norm() / hx.norm())
        e_m = emb[t0 - t_exact:T - t_exact].contiguous()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(10):
            kvq.swa_replay(w, e_m, nw, want_hidden=False, workspace=ws, states=states)
        b.record()
        torch.cuda.synchronize()
        curve.append({"replayed_positions": nw + m, "ms": a.elapsed_time(b) / 10,
                      "top_state_rel_err": top, "next_output_rel_err": nxt})

    def timed(e, n_steps):
        for _ in range(Wm):
            kvq.swa_replay(w, e, nw, want_hidden=False, workspace=ws, states=states)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # the same GPU-side wait as the decode workloads: the host enqueues
        # the first replays while the stream is busy
        sm_hz = getattr(torch.cuda.get_device_properties(device), "clock_rate", 2.0e6) * 1e3
        torch.cuda._sleep(int(PREROLL_US * 1e-6 * sm_hz))
        a.record()
        for _ in range(n_steps):
            kvq.swa_replay(w, e, nw, want_hidden=False, workspace=ws, states=states)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3

    ke = min(K, 50)
    secs_exact = timed(e_x, ke)
    clocks = ClockSampler(device.index)
    dist.barrier()
    secs = timed(e_b, K)
    dist.barrier()
    clk = clocks.stop()
    value, max_s = combine_ranks(dist, L * nw * K, secs)
    # algorithmic fp32 work of one bounded replay: 4 d x d projections per
    # position and layer (2 d^2 flop each), 4 d flop per (position, window
    # position) for the scores and the weighted sum
    attended = sum(min(i + 1, nw) for i in range(nw))
    flops = L * (nw * 4 * 2 * d * d + attended * 4 * d)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    max_mhz = (clk or {}).get("sm_max_mhz") or 2070.0
    peak = sms * 128 * 2 * max_mhz * 1e6 / 1e12  # fp32 FMA lanes x 2 flop x clock
    achieved = flops * K / secs / 1e12
    # end to end: the window's inputs in from pinned host memory, the state back
    eh = e_b.cpu().pin_memory()
    sh = torch.empty(states.shape, dtype=torch.float32).pin_memory()
    Ke = min(K, 20)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(Ke):
        e_b.copy_(eh, non_blocking=True)
        kvq.swa_replay(w, e_b, nw, want_hidden=False, workspace=ws, states=states)
        sh.copy_(states, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    e2e, _ = combine_ranks(dist, L * nw * Ke, a.elapsed_time(b) / 1e3)
    res = {
        "metric": SWA_REPLAY_METRIC, "value": value, "unit": "layer-positions/s", "n_gpus": dist.world, "steps": K,
        "warmup": Wm, "ms_per_step": max_s * 1e3 / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"swa_replay: toy network L{L} d{d}, window {nw}, state after {T} positions; "
                               f"bounded replay {nw} positions, exact replay {T - t_exact}",
                   "layers": L, "d": d, "n_win": nw, "T": T,
                   "exact_replay_ms": secs_exact * 1e3 / ke,
                   "bounded_replay_ms": secs * 1e3 / K,
                   "compute_saved": (secs_exact / ke) / (secs / K),
                   "bounded_state_rel_err_per_layer": state_err,
                   "bounded_next_output_rel_err": next_err,
                   "quality_vs_replay_length": curve,
                   "l2": "all operands (under 10 MB) stay in L2; no flush (latency-bound toy)",
                   "parallelism": f"replicas x{dist.world}"},
        "roofline": {"bound": "alu", "kernel": "one kvq_swa_replay call (swa_proj_kernel + swa_attn_kernel per layer)",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"fp32 FMA: {sms} SMs x 128 lanes x 2 flop x {max_mhz:.0f} MHz (derived)",
                     "traffic": None, "algorithmic_flops_per_launch": flops},
        "e2e": {"value": e2e, "unit": "layer-positions/s", "h2d_bytes_per_step": e_b.numel() * 4,
                "d2h_bytes_per_step": states.numel() * 4, "steps": Ke},
        "gpu_launches": K * (1 + 2 * L),
    }
    if clk is not None:
        res["clocks"] = clk
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        import oracle
        wn, en = w.cpu().double().numpy(), e_b.cpu().double().numpy()
        t = time.perf_counter()
        oracle.swa_forward(wn, en, nw)
        dt = time.perf_counter() - t
        res["cpu_baseline"] = {"value": L * nw / dt, "unit": "layer-positions/s", "cores": 1, "kind": "oracle",
                               "sample": f"one bounded replay ({nw} positions x {L} layers), fp64 C, one thread"}
    return res


# ----------------------------------------------------------------- CPU oracle (baseline / reference arm)
class OracleSample:
    """Host copies of some (sequence, kv head) units of the workload, already
    quantised by the oracle (the cache is resident state, not step work)."""

    def __init__(self, w, seed: int, n_units: int, max_tokens=None, device="cpu", nvfp4: bool = False):
        import numpy as np

        import oracle
        self.o = oracle
        self.w = w
        self.nvfp4 = nvfp4
        rng = np.random.default_rng(seed + 99)
        lens = workloads.lengths(w, seed)
        self.units = []
        for _ in range(n_units):
            b = int(rng.integers(0, w.batch))
            h = int(rng.integers(0, w.num_kv_heads))
            T = lens[b] if max_tokens is None else min(lens[b], max_tokens)
            k, v = workloads.sequence_kv(w, b, lens[b], seed=seed, device=device)
            kh = k[:T, h].float().cpu().numpy()
            vh = v[:T, h].float().cpu().numpy()
            q = workloads.queries(w, seed=seed, device=device)[b, h * w.group:(h + 1) * w.group].float().cpu()
            sk = oracle.nvfp4_global_scale(kh) if nvfp4 else 1.0
            sv = oracle.nvfp4_global_scale(vh) if nvfp4 else 1.0
            kc, ks, _ = oracle.nvfp4_quantize_rows(kh, sk) if nvfp4 else oracle.quantize_rows(kh)
            vc, vs, _ = oracle.nvfp4_quantize_rows(vh, sv) if nvfp4 else oracle.quantize_rows(vh)
            self.units.append((q.numpy(), kc, ks, vc, vs, kh[-1:].copy(), vh[-1:].copy(), T, sk, sv))

    def run_unit(self, u):
        q, kc, ks, vc, vs, knew, vnew, T, sk, sv = u
        o = self.o
        if self.nvfp4:  # the step's append of this unit's new token, then the cache read back
            o.nvfp4_quantize_rows(knew, sk)
            o.nvfp4_quantize_rows(vnew, sv)
            kd = o.nvfp4_dequantize_rows(kc, ks, sk)
            vd = o.nvfp4_dequantize_rows(vc, vs, sv)
        else:
            o.quantize_rows(knew)
            o.quantize_rows(vnew)
            kd = o.dequantize_rows(kc, ks)
            vd = o.dequantize_rows(vc, vs)
        o.attend(q, kd, vd, 1.0 / math.sqrt(self.w.head_dim))
        return T

    def run(self, pool):
        t = time.perf_counter()
        toks = sum(pool.map(self.run_unit, self.units))
        return toks / self.w.num_kv_heads, time.perf_counter() - t


def cpu_baseline(w, seed, st=None, budget_s=20.0, nvfp4=False):
    cores = os.cpu_count() or 1
    n_units = max(cores, 8)
    sample = OracleSample(w, seed, n_units, device="cuda" if torch.cuda.is_available() else "cpu", nvfp4=nvfp4)
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        kv, secs = sample.run(pool)
        reps = 1
        while secs < budget_s / 2 and reps < 200:
            k2, s2 = sample.run(pool)
            kv += k2
            secs += s2
            reps += 1
    return {"value": kv / secs, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_units} (sequence, kv head) units of one {w.name} step x{reps}: append quantise + "
                      f"dequantise + fp64 attention, {cores} threads, {secs:.1f} s"}


def run_reference_replay(args):
    """The oracle's bounded replay of the swa_replay workload, one per step
    (about a second each in fp64 C), capped at 5 timed steps."""
    import oracle
    R = workloads.REPLAY
    L, d, nw, T = R["layers"], R["d"], R["n_win"], R["T"]
    wn = workloads.replay_net(L, d, seed=args.seed).double().numpy()
    en = workloads.replay_inputs(T - nw, nw, d, seed=args.seed).double().numpy()
    steps = min(args.steps, 5)
    for _ in range(min(args.warmup, 3)):
        oracle.swa_forward(wn, en, nw)
    t = time.perf_counter()
    for _ in range(steps):
        oracle.swa_forward(wn, en, nw)
    secs = time.perf_counter() - t
    value = L * nw * steps / secs
    unit = "layer-positions/s"
    return {
        "impl": "reference", "metric": SWA_REPLAY_METRIC, "value": value, "unit": unit, "n_gpus": 1,
        "steps": steps, "warmup": min(args.warmup, 3), "ms_per_step": secs * 1e3 / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"swa_replay: toy network L{L} d{d}, window {nw}; bounded replay of {nw} positions",
                   "parallelism": "one host thread"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": f"one bounded replay ({nw} positions x {L} layers) per step, fp64 C"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def reference_budget_s(args) -> float:
    """Host seconds the whole reference run (warm-up and timed steps) is sized
    for: three times --cpu-budget, a minute by default."""
    return 3.0 * args.cpu_budget


def _reference_line(args, metric: str, unit: str, value: float, secs: float, dtype: str, config: dict,
                    cores: int, sample: str):
    return {
        "impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_prefill(args):
    """The oracle's quantise-on-append of the prefill workload: each step one
    pass of an AppendOracleSample sized so that the whole run takes about
    reference_budget_s of host time."""
    w = workloads.WORKLOADS[args.workload]
    nv = args.format == "nvfp4"
    cores = os.cpu_count() or 1
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        probe = AppendOracleSample(w, args.seed, 4096, nv, cores)
        n, dt = probe.run(pool)
        budget_per_step = reference_budget_s(args) / max(1, args.steps + args.warmup)
        n_tok = int(min(w.context, max(AppendOracleSample.CHUNK, budget_per_step * n / dt)))
        sample = AppendOracleSample(w, args.seed, n_tok, nv, cores)
        for _ in range(args.warmup):
            sample.run(pool)
        toks, secs = 0, 0.0
        for _ in range(args.steps):
            n, dt = sample.run(pool)
            toks += n
            secs += dt
    config = {"workload": f"{w.name}: {w.description}" + (", NVFP4 cache" if nv else ""), "format": args.format,
              "batch": w.batch, "tokens": w.context, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
              "page_size": w.page_size, "parallelism": "host threads"}
    return _reference_line(args, PREFILL_METRIC, "tokens/s", toks / secs, secs, "f32", config, cores,
                           sample.describe(args.steps, secs) + " per step")


def run_reference_prefill_attn(args):
    """The oracle's chunked prefill of the prefill_attn workload: fp64
    attention of the chunk's query tokens (from its end) over the dequantised
    FP4 cache of one (sequence, kv head) unit, each step a bounded sample
    sized so that the whole run takes about reference_budget_s; value in query
    tokens/s of the whole head group (Hq rows per token)."""
    import oracle
    w = workloads.WORKLOADS["prefill_attn"]
    T, C, G, d = w.context, w.chunk, w.group, w.head_dim
    k, v = workloads.sequence_kv(w, 0, T, seed=args.seed, device="cpu")
    kc, ks, _ = oracle.quantize_rows(k[:, 0].float().numpy())
    vc, vs, _ = oracle.quantize_rows(v[:, 0].float().numpy())
    kh, vh = oracle.dequantize_rows(kc, ks), oracle.dequantize_rows(vc, vs)
    g = torch.Generator()
    g.manual_seed(args.seed * 1_000_003 + 4242)
    qh = torch.randn((C, G, d), generator=g).to(torch.bfloat16).float().numpy()
    scale = 1.0 / math.sqrt(d)
    budget_per_step = reference_budget_s(args) / max(1, args.steps + args.warmup)

    def step():
        t = time.perf_counter()
        rows = 0
        for i in range(C - 1, -1, -1):
            oracle.attend(qh[i], kh[:T - C + i + 1], vh[:T - C + i + 1], scale)
            rows += G
            if time.perf_counter() - t > budget_per_step:
                break
        return rows, time.perf_counter() - t

    for _ in range(args.warmup):
        step()
    rows, secs = 0, 0.0
    for _ in range(args.steps):
        r, dt = step()
        rows += r
        secs += dt
    value = rows / w.num_q_heads / secs
    config = {"workload": f"prefill_attn: {w.description}", "format": "fp4", "batch": w.batch, "context": T,
              "chunk": C, "kv_heads": w.num_kv_heads, "q_heads": w.num_q_heads, "head_dim": d,
              "page_size": w.page_size, "parallelism": "one host thread"}
    return _reference_line(args, PREFILL_ATTN_METRIC, "query tokens/s", value, secs, "f64", config, 1,
                           f"{rows // G} tokens x G={G} query rows of one kv head over ~{T} positions in all "
                           f"(fp64 C attention, one thread, about {budget_per_step:.2f} s per step), scaled to "
                           f"Hq={w.num_q_heads} rows per token")


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return None
    if args.workload == "swa_replay":
        return run_reference_replay(args)
    if args.workload in ("prefill", "prefill_b1"):
        return run_reference_prefill(args)
    if args.workload == "prefill_attn":
        return run_reference_prefill_attn(args)
    w = workloads.WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    # size each step so the whole warm-up + timed run stays around reference_budget_s
    nv = args.format == "nvfp4"
    probe = OracleSample(w, args.seed, 1, max_tokens=4096, device=dev, nvfp4=nv)
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        _, t_probe = probe.run(pool)
        per_token_s = t_probe / 4096
        budget_per_step = reference_budget_s(args) / max(1, args.steps + args.warmup)
        max_tokens = int(min(w.context or 131072, max(64, budget_per_step * cores / per_token_s)))
        sample = OracleSample(w, args.seed, cores, max_tokens=max_tokens, device=dev, nvfp4=nv)
        for _ in range(args.warmup):
            sample.run(pool)
        kv, secs = 0.0, 0.0
        for _ in range(args.steps):
            k2, s2 = sample.run(pool)
            kv += k2
            secs += s2
    value = kv / secs
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}; step = append 1 token/seq + decode attention"
                   + (f", {args.layers} layers" if args.layers > 1 else "")
                   + (", NVFP4 cache" if args.format == "nvfp4" else ""), "layers": args.layers, "format": args.format,
                   "batch": w.batch, "kv_heads": w.num_kv_heads, "q_heads": w.num_q_heads,
                   "head_dim": w.head_dim, "context": w.context, "page_size": w.page_size,
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{cores} units x {max_tokens} positions per step (CPU oracle)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--workload", default="long_context",
                    choices=["long_context", "gqa_outliers", "paged_ragged", "swa_append", "tiny", "prefill",
                             "prefill_b1", "prefill_attn", "swa_replay"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--format", choices=["fp4", "nvfp4"], default="fp4",
                    help="cache format: FP4 (E4M3 scale per 16) or NVFP4 (plus an fp32 scale per kv head)")
    ap.add_argument("--layers", type=int, default=1,
                    help="layers per step, each with its own cache (long_context at 4 layers: 4.84 GB)")
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="host seconds for the CPU-oracle baseline; the reference arm's whole run is sized "
                         "for three times this")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-kernel", choices=["mma", "tcgen05"], default="mma",
                    help="decode kernel: mma (kvq_decode_attn, the default) or tcgen05 (kvq_decode_attn_tc, "
                         "head_dim 128 only, a measured slower alternative)")
    ap.add_argument("--fused-append", action=argparse.BooleanOptionalAction, default=True,
                    help="each step as one kvq_append_decode_attn call (the append fused into the decode launch; "
                         "workloads without an FP8 window) instead of kvq_append then kvq_decode_attn")
    ap.add_argument("--graphs", action=argparse.BooleanOptionalAction, default=False,
                    help="replay each step's appends and decode from CUDA graphs (decode workloads)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist()
    try:
        if args.impl == "reference":
            res = run_reference(args, dist)
        elif args.workload in ("prefill", "prefill_b1"):
            res = run_prefill(args, dist)
        elif args.workload == "prefill_attn":
            res = run_prefill_attn(args, dist)
        elif args.workload == "swa_replay":
            res = run_swa_replay(args, dist)
        else:
            res = run_gpu(args, dist)
        if dist.rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
