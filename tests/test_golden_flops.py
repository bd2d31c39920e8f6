"""The FLOP rule bench.py reports TFLOPS with, pinned to the pages' own tables:
each printed (latency, TFLOPS) pair of the L20 rows must follow from the rule
(tests/golden/more_benchmark_l20.txt, with its citation)."""
import os

import pytest

from bench import attention_flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "more_benchmark_l20.txt")


def rows():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            ps, case, nq, nkv, bh, causal, ms, tf = line.split()
            out.append((ps, case, int(nq), int(nkv), int(bh), causal == "1", float(ms), float(tf)))
    return out


@pytest.mark.parametrize("row", rows(), ids=lambda r: f"{r[0]}-{r[1]}")
def test_rule_reproduces_printed_tflops(row):
    ps, case, nq, nkv, bh, causal, ms, tflops = row
    got = attention_flops(nq, nkv, 512, bh, causal=causal, backward=(ps == "bwd")) / (ms * 1e-3) / 1e12
    # both printed numbers are rounded: TFLOPS to a whole unit (two decimals
    # below 1) and the latency to 0.01 ms, which is up to 0.65% at 0.77 ms
    tol = (0.5 if tflops >= 1 else 0.005) + 0.005 / ms * got
    assert abs(got - tflops) <= tol, (got, tflops)


def test_rule_counts_causal_half_and_backward_ten():
    assert attention_flops(8, 8, 64, 1, causal=True) == attention_flops(8, 8, 64, 1) / 2
    assert attention_flops(8, 8, 64, 1, backward=True) == 2.5 * attention_flops(8, 8, 64, 1)
