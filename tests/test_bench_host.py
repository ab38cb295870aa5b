"""Host logic of bench.py that needs no GPU: the end-to-end leg's bucket split."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import WORKLOADS  # noqa: E402


def _layout(shapes):
    offs, tot = [], 0
    for a, b in shapes:
        offs.append(tot)
        tot += -(-(a * b) // 128) * 128
    return offs, tot


def test_e2e_buckets_cover_the_set_in_order():
    for key in ("mmdit-15b", "mmdit-1.3b", "bf16-64x1536sq", "fp32-256x1024"):
        shapes = [(m.rows, m.cols) for m in WORKLOADS[key].matrices]
        offs, tot = _layout(shapes)
        for nb in (1, 2, 3, 8, 10_000):
            bk = bench.e2e_buckets(offs, tot, nb)
            assert 1 <= len(bk) <= min(nb, len(shapes))
            assert bk[0][:1] == (0,) and bk[-1][1] == len(shapes)
            assert bk[0][2] == 0 and bk[-1][3] == tot
            for (a0, b0, s0, e0), (a1, b1, s1, e1) in zip(bk, bk[1:]):
                assert b0 == a1 and e0 == s1 and b0 > a0
            for a, b, s, e in bk:
                assert s == offs[a] and e == (offs[b] if b < len(offs) else tot)


def test_e2e_buckets_balance_bytes():
    shapes = [(m.rows, m.cols) for m in WORKLOADS["mmdit-15b"].matrices]
    offs, tot = _layout(shapes)
    bk = bench.e2e_buckets(offs, tot, 8)
    assert len(bk) == 8
    biggest = max((offs[j + 1] if j + 1 < len(offs) else tot) - offs[j] for j in range(len(offs)))
    for a, b, s, e in bk:
        assert abs((e - s) - tot / 8) <= biggest
