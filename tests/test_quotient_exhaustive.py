"""The append's division-free quotient for NVFP4 blocks (the value already
divided by the kv head's fp32 scale, then by the block's E4M3 scale) relies on
y * RN(1/s) plus one fused residual correction being exactly the IEEE fp32
y / s.  This runs the exhaustive host check of that identity (all 2^23
significands of y against the eight E4M3 significands) in IEEE fp32 with
fused multiply-adds, as the GPU computes it."""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))


def test_reciprocal_quotient_is_the_ieee_quotient_for_e4m3_divisors():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "quotient_check")
        subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-o", exe,
                        os.path.join(HERE, "native", "quotient_check.c"), "-lm"], check=True)
        r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
    assert "mismatches 0" in r.stdout
