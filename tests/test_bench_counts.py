"""The bench's flop counts: the pair counts behind the dense definition, against
brute-force counts of the visible (query, key) pairs (CPU only)."""
import importlib
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


@pytest.fixture()
def bench():
    b = importlib.import_module("bench")
    saved = (b.CAUSAL, b.WINDOW)
    yield b
    b.CAUSAL, b.WINDOW = saved


def visible_pairs(N, causal, W=0):
    i, j = np.meshgrid(np.arange(N), np.arange(N), indexing="ij")
    m = np.ones((N, N), bool) if not causal else (j <= i)
    if causal and W:
        m &= j > i - W
    return int(m.sum())


@pytest.mark.parametrize("N,W", [(64, 1), (100, 17), (300, 64), (300, 299), (257, 128)])
def test_window_pairs_are_the_visible_pairs(bench, N, W):
    bench.CAUSAL, bench.WINDOW = True, W
    assert bench.pairs(N) == visible_pairs(N, True, W)


def test_causal_and_full_counts(bench):
    # The dense definition halves N^2 under the causal mask (N (N + 1) / 2 pairs are
    # visible; the diagonal's N / 2 is not counted), and counts N^2 without it.
    bench.CAUSAL, bench.WINDOW = True, 0
    N = 512
    assert bench.pairs(N) == N * N / 2 and abs(bench.pairs(N) - visible_pairs(N, True)) == N / 2
    bench.CAUSAL = False
    assert bench.pairs(N) == visible_pairs(N, False)
    bench.CAUSAL, bench.WINDOW = True, N + 5  # a window past N is the causal mask
    assert bench.pairs(N) == N * N / 2
