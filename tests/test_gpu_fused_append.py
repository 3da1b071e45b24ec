"""kvq_append_decode_attn (the decode step with its append fused into the
decode launch) against the two calls it replaces: kvq_append of one token
per sequence at position T_b - 1, then kvq_decode_attn over T_b positions.

Both paths start from copies of the same cache.  The pool bytes must be
identical after the step: the same quantiser writes the same codes and scale
bytes to the same places, including the read-modify-write of a token pair's
shared V bytes.

The outputs are compared with the oracle (fp64 attention over the
quantised-then-dequantised K and V, as in the decode parity tests) and with
the separate calls' output.  When the append is fused, the decode kernel adds
a stage's PV products straight into its fp32 O accumulator instead of
summing them apart and adding the sum: the same products, reassociated.  Each
stage adds at most three roundings of 2^-24 relative to the running sum,
whose magnitude is at most l * max|V^|, so after n <= T/128 stages of one
range the normalised outputs differ by at most about 3 n 2^-24 max|V^|:
below 1e-4 max|V^| for any T up to 2^20 (asserted with max|V^| bounded by
1.0625 max|V|, the largest E2M1 rounding of a block's maximum).  When the
kernel does not fuse (below), the two outputs are equal bit for bit.

The library fuses the append into the decode kernel when the cache's
capacity (max_pages_per_seq * page_size, known on the host) gives every CTA
range at least 16 chunks, and otherwise launches the append kernel first;
the cases run both ways (`fused_kernel`: capacity reserved past that bound).

Cases: head_dim 64 and 128; page sizes 16..256, contiguous and paged; new
tokens at even and odd positions (the first or second token of a V pair),
in the first slot of a page and of a 128-token chunk; empty sequences (no
append); several steps in a row; many units per range; NVFP4 caches;
non-finite inputs; the long-context benchmark shape.
"""
import math

import pytest
import torch

from fp4_kv_cache_kvq_gb300 import kvq, workloads
from tests.helpers import build_fp4, check_units, ensure_built

pytestmark = pytest.mark.gpu

BASE = workloads.WORKLOADS["gqa_outliers"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _twin(cache):
    c = kvq.Fp4Cache(cache.num_kv_heads, cache.head_dim, cache.page_size, cache.num_pages, cache.max_pages_per_seq,
                     page_table=cache.page_table, nvfp4=cache.nvfp4)
    c.pool.copy_(cache.pool)
    if cache.nvfp4:
        c.k_gscale.copy_(cache.k_gscale)
        c.v_gscale.copy_(cache.v_gscale)
    return c


def _step_both(a, b, lens, k_new, v_new, q, scale=None):
    """Separate calls on cache a, the fused call on cache b; returns both
    outputs and both device flags."""
    ea = torch.zeros(1, dtype=torch.int32, device="cuda")
    eb = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens_dev = torch.tensor(lens, dtype=torch.int32, device="cuda")
    pos = (lens_dev - 1).clamp(min=0)
    # kvq_append has no "skip this sequence": give empty sequences a position
    # the test never reads (they append nothing in the fused call), so compare
    # only non-empty batches through kvq_append
    assert all(n > 0 for n in lens)
    kvq.append(a, pos, k_new[:, None].contiguous(), v_new[:, None].contiguous(), err=ea)
    oa = kvq.decode_attn(a, lens_dev, q, scale, err=ea)
    ob = kvq.append_decode_attn(b, lens_dev, k_new, v_new, q, scale, err=eb)
    torch.cuda.synchronize()
    return oa, ob, ea.item(), eb.item()


REASSOC = 1e-4  # |fused - separate| <= REASSOC * max|V^| (fp32 reassociation, see above)


def _assert_outputs(oa, ob, vmax_raw, fused_kernel):
    if fused_kernel:
        assert (oa - ob).abs().max().item() <= REASSOC * 1.0625 * vmax_raw
    else:
        assert torch.equal(oa, ob)


def _reserve(w, n_seq, fused_kernel, steps):
    """Positions to reserve per sequence: past the fusing bound (16 chunks per
    range over 3 x 152 ranges, with margin) or just the steps."""
    if not fused_kernel:
        return steps + 1
    return -(-16 * 3 * 160 // (n_seq * w.num_kv_heads)) * 128 + steps + 1


def _run(w, lens0, steps=1, seed=0, fused_kernel=False, oracle_units=None):
    """`oracle_units`: the (b, h) units checked against the oracle after each
    step (None: all of them)."""
    reserve = _reserve(w, len(lens0), fused_kernel, steps)
    built = build_fp4(w, lens0, seed=seed, reserve=reserve, keep_kv=True)
    a = built.cache
    b = _twin(a)
    lens = list(lens0)
    G = w.num_q_heads // w.num_kv_heads
    units = oracle_units if oracle_units is not None else [(i, h) for i in range(w.batch)
                                                          for h in range(w.num_kv_heads)]
    # host K and V rows of the checked units only, and max|V| over everything
    kv = {(i, h): (built.seq_k[i][:, h].float().cpu(), built.seq_v[i][:, h].float().cpu()) for i, h in units}
    vmax = max((float(v.abs().max()) for v in built.seq_v if v.numel()), default=0.0)
    built.seq_k.clear()
    built.seq_v.clear()
    for step in range(1, steps + 1):
        lens = [n + 1 for n in lens]
        kn, vn = workloads.step_tokens(w, step, seed=seed, device="cuda")
        q = workloads.queries(w, seed=seed, step=step, device="cuda")
        oa, ob, ea, eb = _step_both(a, b, lens, kn[:, 0].contiguous(), vn[:, 0].contiguous(), q)
        assert ea == 0 and eb == 0
        assert torch.equal(a.pool, b.pool), f"pool bytes differ at step {step}"
        kv = {(i, h): (torch.cat([k, kn[i, :, h].float().cpu()]), torch.cat([v, vn[i, :, h].float().cpu()]))
              for (i, h), (k, v) in kv.items()}
        vmax = max(vmax, float(vn.abs().max()))
        _assert_outputs(oa, ob, vmax, fused_kernel)
        check_units(ob, q, units, lambda i, h: (kv[(i, h)][0].numpy(), kv[(i, h)][1].numpy()), G,
                    1.0 / math.sqrt(w.head_dim))


@pytest.mark.parametrize("fused_kernel", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("page_size,paged", [(16, True), (32, False), (64, True), (128, True), (256, False)])
def test_matches_separate_calls(d, page_size, paged, fused_kernel):
    w = workloads.scaled(BASE, batch=5, num_kv_heads=2, num_q_heads=8, head_dim=d, page_size=page_size, paged=paged,
                         k_outlier_channels=(3, 17, 40) if d == 64 else (3, 17, 64, 101))
    # new tokens at odd and even positions, the first slot of a page / chunk
    _run(w, [300, 127, 128, 255, 1000], steps=2, seed=d + page_size, fused_kernel=fused_kernel)


@pytest.mark.parametrize("fused_kernel", [False, True])
def test_many_steps_and_short_sequences(fused_kernel):
    w = workloads.scaled(BASE, batch=7, num_kv_heads=3, num_q_heads=12, paged=True)
    _run(w, [1, 2, 15, 16, 63, 64, 200], steps=5, seed=3, fused_kernel=fused_kernel)


@pytest.mark.parametrize("fused_kernel", [False, True])
def test_many_units_per_range(fused_kernel):
    w = workloads.scaled(BASE, batch=300, num_kv_heads=2, num_q_heads=8, paged=True)
    lens = [1 + (7 * b) % 150 for b in range(300)]
    _run(w, lens, steps=2, seed=4, fused_kernel=fused_kernel)


@pytest.mark.parametrize("fused_kernel", [False, True])
def test_empty_sequences_append_nothing(fused_kernel):
    """T_b == 0 appends nothing and gives a zero row; the other sequences of the
    batch match kvq_append (called for them alone) + kvq_decode_attn."""
    w = workloads.scaled(BASE, batch=3, num_kv_heads=2, num_q_heads=8, paged=True)
    built = build_fp4(w, [100, 0, 50], seed=5, reserve=_reserve(w, 3, fused_kernel, 1), keep_kv=True)
    a = built.cache
    b = _twin(a)
    kn, vn = workloads.step_tokens(w, 1, seed=5, device="cuda")
    q = workloads.queries(w, seed=5, device="cuda")
    ea = torch.zeros(1, dtype=torch.int32, device="cuda")
    eb = torch.zeros(1, dtype=torch.int32, device="cuda")
    lens = torch.tensor([101, 0, 51], dtype=torch.int32, device="cuda")
    for s in (0, 2):
        kvq.append(a, lens[s:s + 1] - 1, kn[s:s + 1].contiguous(), vn[s:s + 1].contiguous(), err=ea,
                   page_table=a.page_table[s:s + 1])
    oa = kvq.decode_attn(a, lens, q, err=ea)
    ob = kvq.append_decode_attn(b, lens, kn[:, 0].contiguous(), vn[:, 0].contiguous(), q, err=eb)
    torch.cuda.synchronize()
    assert ea.item() == 0 and eb.item() == 0
    assert torch.equal(a.pool, b.pool)
    _assert_outputs(oa, ob, max(float(vn.abs().max()), max(float(v.abs().max()) for v in built.seq_v if v.numel())),
                    fused_kernel)
    assert torch.count_nonzero(ob[1]).item() == 0


@pytest.mark.parametrize("fused_kernel", [False, True])
@pytest.mark.parametrize("mag", [1.0, 1e-6, 3e3])
def test_nvfp4(mag, fused_kernel):
    w = workloads.scaled(BASE, batch=3, num_kv_heads=2, num_q_heads=8)
    B, T = w.batch, 300
    ks, vs = [], []
    for b in range(B):
        k, v = workloads.sequence_kv(w, b, T, seed=6, device="cuda")
        ks.append((k.float() * mag).to(torch.bfloat16))
        vs.append((v.float() * mag).to(torch.bfloat16))
    K, V = torch.stack(ks).contiguous(), torch.stack(vs).contiguous()
    max_pages = -(-(T + _reserve(w, B, fused_kernel, 3)) // w.page_size)
    a = kvq.Fp4Cache(w.num_kv_heads, w.head_dim, w.page_size, B * max_pages, max_pages, nvfp4=True)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.fp8_set_scales(a, K, V, err=err)
    kvq.append(a, torch.zeros(B, dtype=torch.int32, device="cuda"), K, V, err=err)
    b = _twin(a)
    lens = [T] * B
    for step in range(1, 3):
        lens = [n + 1 for n in lens]
        kn, vn = workloads.step_tokens(w, step, seed=6, device="cuda")
        kn = (kn.float() * mag).to(torch.bfloat16)[:, 0].contiguous()
        vn = (vn.float() * mag).to(torch.bfloat16)[:, 0].contiguous()
        q = workloads.queries(w, seed=6, step=step, device="cuda")
        oa, ob, ea, eb = _step_both(a, b, lens, kn, vn, q)
        assert ea == 0 and eb == 0
        assert torch.equal(a.pool, b.pool)
        _assert_outputs(oa, ob, max(float(V.abs().max()), float(vn.abs().max())), fused_kernel)


@pytest.mark.parametrize("fused_kernel", [False, True])
def test_non_finite_input_flags_like_append(fused_kernel):
    w = workloads.scaled(BASE, batch=2, num_kv_heads=2, num_q_heads=8, k_outlier_channels=())
    built = build_fp4(w, [70, 91], seed=7, reserve=_reserve(w, 2, fused_kernel, 1), keep_kv=False)
    a = built.cache
    b = _twin(a)
    kn, vn = workloads.step_tokens(w, 1, seed=7, device="cuda")
    kn = kn[:, 0].contiguous()
    vn = vn[:, 0].contiguous()
    kn[0, 1, 5] = float("inf")
    vn[1, 0, 40] = float("nan")
    q = workloads.queries(w, seed=7, device="cuda")
    oa, ob, ea, eb = _step_both(a, b, [71, 92], kn, vn, q)
    assert ea == eb and ea & kvq.FLAG_NONFINITE
    assert torch.equal(a.pool, b.pool)


def test_long_context_shape():
    """The benchmark's shape (the fused kernel: its capacity passes the bound);
    eight units checked against the oracle."""
    w = workloads.WORKLOADS["long_context"]
    _run(w, workloads.lengths(w), steps=1, seed=0, fused_kernel=True,
         oracle_units=[(0, 0), (3, 7), (9, 2), (15, 5), (16, 1), (22, 6), (28, 3), (31, 4)])


def test_needs_both_new_rows():
    w = workloads.scaled(BASE, batch=1, num_kv_heads=1, num_q_heads=8)
    built = build_fp4(w, [10], reserve=1, keep_kv=False)
    q = workloads.queries(w, device="cuda")
    g = built.cache.struct()
    lib = kvq.load()
    out = torch.empty((1, 8, w.head_dim), dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.decode_workspace_bytes(1, 8, 1, w.head_dim), dtype=torch.uint8, device="cuda")
    import ctypes
    st = lib.kvq_append_decode_attn(ctypes.byref(g), 1, 8, built.lens_dev.data_ptr(), q.data_ptr(), None,
                                    q.data_ptr(), 0.1, out.data_ptr(), ws.data_ptr(), ws.numel(), None,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == 1  # KVQ_ERR_INVALID_ARGUMENT
