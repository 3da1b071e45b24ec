"""The bit-width sweep kernels through the C ABI against the oracle: codes and
scales bit for bit, dequantised values exactly, for every layout the results
table of "Quantising the KV cache" compares; the fp64 dense attention against
the oracle's fp64 attention."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_kvq_gb300 import kvq
from tests.helpers import ensure_built
from tests.test_oracle_formats import all_bf16_as_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _bf16(x: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.from_numpy(np.asarray(x, np.float32)))  # inputs are bf16 values
    return t.cuda()


def _kv(shape, seed, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape).astype(np.float32)
    if outliers:
        x[..., 3] *= 20.0
        x[..., shape[-1] - 5] *= -35.0
    x[0, 0, 0, :4] = [0.0, -0.0, 1e-30, -3e-38]  # zeros and tiny values
    return torch.from_numpy(x).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("per,layout", [("token", kvq.LAYOUT_INT_PER_TOKEN), ("channel", kvq.LAYOUT_INT_PER_CHANNEL)])
@pytest.mark.parametrize("bits", [2, 3, 4, 6, 8])
def test_int_layouts_bit_exact(per, layout, bits):
    x = _kv((3, 37, 4, 64), seed=bits + len(per))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xh, codes, scales = kvq.fake_quant(_bf16(x), layout, bits, want_codes=True, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    oc, os_, bad = oracle.int_quantize(x, bits, per)
    assert bad == 0
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), os_)
    assert np.array_equal(xh.cpu().numpy().astype(np.float64), oracle.int_dequantize(oc, os_, per))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_int_every_bf16_value_under_many_scales(bits):
    """Groups of 64: the group's first value sets the amax (64 amaxes spread
    over the bf16 exponent range), the other 63 run through every finite bf16
    value no larger than it."""
    allv = all_bf16_as_f32()
    allv = allv[np.isfinite(allv)]
    rng = np.random.default_rng(bits)
    groups = []
    for amax in np.sort(np.abs(rng.choice(allv[np.abs(allv) > 1e-35], 64))):
        v = allv[np.abs(allv) <= amax]
        pad = (-v.size) % 63
        v = np.concatenate([v, np.zeros(pad, np.float32)]).reshape(-1, 63)
        g = np.empty((v.shape[0], 64), np.float32)
        g[:, 0] = amax
        g[:, 1:] = v
        groups.append(g)
    x = np.concatenate(groups).reshape(1, -1, 1, 64)
    xh, codes, scales = kvq.fake_quant(_bf16(x), kvq.LAYOUT_INT_PER_TOKEN, bits, want_codes=True)
    oc, os_, _ = oracle.int_quantize(x, bits, "token")
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), os_)


def test_int_specials_and_flag():
    x = np.zeros((1, 4, 1, 32), np.float32)
    x[0, 1, 0, :3] = [np.inf, 1.0, -2.0]          # amax inf: scale saturates at 65504
    x[0, 2, 0, :3] = [np.nan, 1.0, -2.0]          # NaN: code 0, ignored by the amax
    x[0, 3, 0, :2] = [3.0e38, -1.0]               # amax / qmax above FP16's range
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    xh, codes, scales = kvq.fake_quant(xt, kvq.LAYOUT_INT_PER_TOKEN, 4, want_codes=True, err=err)
    torch.cuda.synchronize()
    assert err.item() & kvq.FLAG_NONFINITE
    oc, os_, bad = oracle.int_quantize(xt.float().cpu().numpy(), 4, "token")
    assert bad == 2
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), os_)
    assert os_[0, 0, 0] == 1 and os_[0, 1, 0] == 0x7BFF and os_[0, 3, 0] == 0x7BFF


def test_fp8_tensor_bit_exact():
    x = _kv((2, 50, 3, 128), seed=7)
    xh, codes, scales = kvq.fake_quant(_bf16(x), kvq.LAYOUT_FP8_TENSOR, 8, want_codes=True)
    s = oracle.fp8_head_scale(x)
    assert scales.cpu().numpy()[1] == np.float32(s)
    oc, _ = oracle.fp8_quantize(x, s)
    assert np.array_equal(codes.cpu().numpy().view(np.uint8), oc)
    assert np.array_equal(xh.cpu().numpy().astype(np.float64), oracle.fp8_dequantize(oc, s))


def test_fp4_blocks_bit_exact():
    x = _kv((2, 30, 2, 64), seed=8)
    xh, codes, scales = kvq.fake_quant(_bf16(x), kvq.LAYOUT_FP4_G16, 4, want_codes=True)
    oc, os_, _ = oracle.quantize_rows(x.reshape(-1, 64))
    assert np.array_equal(scales.cpu().numpy(), os_.ravel())
    nib = codes.cpu().numpy().view(np.uint8).reshape(-1, 64)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(packed, oc)
    assert np.array_equal(xh.cpu().numpy().reshape(-1, 64).astype(np.float64), oracle.dequantize_rows(oc, os_))


def test_bad_arguments_are_refused():
    x = torch.zeros((1, 2, 1, 64), dtype=torch.bfloat16, device="cuda")
    for layout, bits in [(kvq.LAYOUT_FP8_TENSOR, 4), (kvq.LAYOUT_INT_PER_TOKEN, 1), (kvq.LAYOUT_INT_PER_CHANNEL, 9),
                         (kvq.LAYOUT_FP4_G16, 8), (9, 4)]:
        with pytest.raises(kvq.KvqError) as e:
            kvq.fake_quant(x, layout, bits)
        assert e.value.status == 1


@pytest.mark.parametrize("T,G", [(1, 1), (77, 4), (1000, 8)])
def test_attn_dense_against_oracle(T, G):
    rng = np.random.default_rng(T)
    B, Hkv, d = 2, 2, 64
    q = torch.from_numpy(rng.standard_normal((B, Hkv * G, d)).astype(np.float32)).to(torch.bfloat16).cuda()
    k = torch.from_numpy(rng.standard_normal((B, T, Hkv, d)).astype(np.float32) * 2).cuda()
    v = torch.from_numpy(rng.standard_normal((B, T, Hkv, d)).astype(np.float32)).cuda()
    scale = 1.0 / math.sqrt(d)
    out, top = kvq.attn_dense(q, k, v, scale, want_top=True)
    qh, kh, vh = q.float().cpu().numpy(), k.cpu().numpy(), v.cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            ref, _, _ = oracle.attend(qh[b, h * G:(h + 1) * G], kh[b, :, h], vh[b, :, h], scale)
            got = out[b, h * G:(h + 1) * G].cpu().numpy()
            assert np.abs(got - ref).max() <= 1e-6 * max(1.0, np.abs(ref).max())
            sc = qh[b, h * G:(h + 1) * G].astype(np.float64) @ kh[b, :, h].astype(np.float64).T
            assert np.array_equal(top[b, h * G:(h + 1) * G].cpu().numpy(), sc.argmax(axis=1))


def test_attn_dense_empty_and_too_long():
    q = torch.zeros((1, 2, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 0, 1, 64), dtype=torch.float32, device="cuda")
    out, top = kvq.attn_dense(q, k, k, 0.1, want_top=True)
    assert not out.any() and (top == -1).all()
    with pytest.raises(kvq.KvqError) as e:
        big = torch.zeros((1, 16385, 1, 64), dtype=torch.float32, device="cuda")
        kvq.attn_dense(q, big, big, 0.1)
    assert e.value.status == 2


def test_sweep_orders_the_formats():
    """A small sweep.  N(0,1): the error falls with every extra bit, FP8 beats
    INT4, FP4/16 lands between INT6 and INT3.  With K outlier channels the
    per-channel K layout beats per-token K at 8 and 6 bits (the page's "Per
    token or per channel?").  Every unquantised row is exact."""
    from fp4_kv_cache_kvq_gb300 import sweep
    rows = sweep.run(batch=2, tokens=512, kv_heads=2, q_heads=8, head_dim=128, seed=1)
    by = {(r["case"], r["format"]): r for r in rows}
    for case in sweep.CASES:
        assert by[(case, "BF16 (unquantised)")]["max_err_rel"] == 0.0
    e = lambda f: by[("N(0,1)", f)]["max_err_rel"]  # noqa: E731
    chain = [e(f"INT{b} per token") for b in (8, 6, 4, 3, 2)]
    assert chain == sorted(chain) and len(set(chain)) == 5
    assert e("FP8 E4M3, one scale per tensor") < e("INT4 per token")
    assert e("INT6 per token") < e("FP4 E2M1, E4M3 scale per 16") < e("INT3 per token")
    out_case = "K channels {3,17,64,101} x20"
    for b in (8, 6):
        assert by[(out_case, f"INT{b}, K per channel, V per token")]["rms_err_rel"] < \
            by[(out_case, f"INT{b} per token")]["rms_err_rel"]
