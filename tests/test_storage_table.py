"""The storage columns of the results table on "Quantising the KV cache"
(golden file tests/golden/storage_table.txt, copied from the page) against the
b + s/g formula of its section "Maths" and, for the FP4 row, against the bytes
the oracle's quantiser actually writes (8 code bytes + 1 scale byte per 16)."""
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "storage_table.txt")


def _rows():
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, bits, pct, b, s, g = [c.strip() for c in line.split("|")]
        yield name, float(bits), float(pct), int(b), int(s), int(g)


def test_storage_table_from_formula():
    rows = list(_rows())
    assert len(rows) == 8
    for name, bits, pct, b, s, g in rows:
        assert b + s / g == bits, name
        assert round(100.0 * bits / 16.0, 1) == pct, name


def test_fp4_row_matches_written_bytes():
    row = [r for r in _rows() if r[0].startswith("FP4")][0]
    x = np.random.default_rng(0).standard_normal((10, 128)).astype(np.float32)
    codes, scales, _ = oracle.quantize_rows(x)
    assert 8 * (codes.nbytes + scales.nbytes) / x.size == row[1]
