"""The append's division-free quotients rely on y * RN(1/s) plus one fused
residual correction being exactly the IEEE fp32 y / s for the divisors and
dividends it meets:
  * an E4M3 block scale (and the divisor 6 of amax/6) with any fp32 dividend,
    the NVFP4 value already divided by the kv head's scale included;
  * the NVFP4 kv head's fp32 second-level scale with a bf16 input value,
    over the scale range [2^-90, 2^126] the append uses it for.
For the FP4 codes (bf16 values over an E4M3 block scale) the reciprocal
need not be RN(1/s): any r within two ulps of it gives the same E2M1 code
after the correction, which lets the kernel take the hardware's approximate
reciprocal.  This runs the host check of these identities (all 2^23 fp32 significands
against the eight E4M3 significands; all 2^7 bf16 significands against all
2^23 fp32 significands; every finite bf16 value against sampled scales at
both ends of that range, where tiny values and overflow meet) in IEEE fp32
with fused multiply-adds, as the GPU computes them."""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))


def test_reciprocal_quotient_is_the_ieee_quotient():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "quotient_check")
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-o", exe,
                        os.path.join(HERE, "native", "quotient_check.c"), "-lm"], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout
    assert "e4m3 divisors: checked 67108864, mismatches 0" in r.stdout
    assert "fp32 divisors, bf16 dividends: checked 1073741824, mismatches 0" in r.stdout
    assert "second-level scale range ends: checked 267248132, mismatches 0" in r.stdout
    assert "approximate reciprocals, e2m1 codes: checked 21260610, mismatches 0" in r.stdout
