"""Pins for the Winograd oracle (``oracle/winograd.py``), CPU only.

The oracle builds its transforms from interpolation points, so what is pinned
here is the construction: exact agreement with direct correlation in rational
arithmetic, the worked example and the transform properties the pages state
("im2col Expansion, FFT Convolution, and Winograd Transforms", Winograd
section), and agreement of the 2-D tiled convolution with the direct C oracle.
"""
import os
import random
from fractions import Fraction

import numpy as np
import pytest

from oracle import ref
from oracle import winograd as wg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _direct_1d(d, g, m):
    return [sum(d[i + k] * g[k] for k in range(len(g))) for i in range(m)]


def test_worked_example_f23():
    # The page's F(2,3) example: input tile [1, 2, 3, 4], filter [2, 0, -1]
    # (the same fixture pins the direct path).
    with open(os.path.join(ROOT, "tests", "golden", "winograd_f23_worked_example.txt")) as f:
        rows = [[int(v) for v in line.split()] for line in f if line.strip() and not line.startswith("#")]
    d, g, want = rows
    assert wg.correlate_1d(d, g, 2, 3) == want
    assert _direct_1d(d, g, 2) == want


@pytest.mark.parametrize("m,r", [(2, 3), (4, 3), (3, 2), (2, 5), (6, 3), (3, 3)])
def test_exact_against_direct_correlation(m, r):
    rng = random.Random(m * 100 + r)
    n = m + r - 1
    for _ in range(200):
        d = [Fraction(rng.randint(-99, 99), rng.randint(1, 9)) for _ in range(n)]
        g = [Fraction(rng.randint(-99, 99), rng.randint(1, 9)) for _ in range(r)]
        assert wg.correlate_1d(d, g, m, r) == _direct_1d(d, g, m)


def test_multiplication_counts():
    # F(2,3): 4 multiplications for 2 outputs (direct: 6); F(4,3): 6 for 4
    # (direct: 12); 2-D F(2x2,3x3): 16 for 4 (direct: 36).
    for m, r, mults in [(2, 3, 4), (4, 3, 6)]:
        at, g, bt = wg.transforms(m, r)
        assert len(g) == len(bt) == mults and len(at) == m
        assert len(at[0]) == mults and len(g[0]) == r
    assert len(wg.transforms(2, 3)[1]) ** 2 == 16


def test_transform_entries_as_the_pages_describe():
    # Integer input and output transforms; the fractions sit in the filter
    # transform.  F(4,3): factors 1/6 and 1/24 in G, integer coefficients as
    # large as 5 (input) and 8 (output).
    for m, r in [(2, 3), (4, 3)]:
        at, g, bt = wg.transforms(m, r)
        assert all(v.denominator == 1 for row in at + bt for v in row)
    at, g, bt = wg.transforms(4, 3)
    dens = {v.denominator for row in g for v in row}
    assert 6 in dens and 24 in dens
    assert max(abs(v) for row in bt for v in row) == 5
    assert max(abs(v) for row in at for v in row) == 8


def test_points_must_be_valid():
    with pytest.raises(ValueError):
        wg.transforms(2, 3, [Fraction(0), Fraction(1), Fraction(2), Fraction(3)])    # no infinity
    with pytest.raises(ValueError):
        wg.transforms(2, 3, [Fraction(0), Fraction(1), None])                        # too few points


@pytest.mark.parametrize("shape", [(1, 1, 4, 4, 1, 0), (2, 3, 7, 9, 4, 1), (1, 5, 11, 6, 3, 2), (2, 2, 3, 3, 2, 1),
                                   (1, 4, 16, 16, 8, 1)])
@pytest.mark.parametrize("m", [2, 4])
def test_conv2d_matches_direct_oracle(shape, m):
    N, Ci, H, W, Co, p = shape
    rng = np.random.default_rng(sum(shape) * 7 + m)
    x = rng.standard_normal((N, Ci, H, W))
    w = rng.standard_normal((Co, Ci, 3, 3))
    Y, S = ref.conv2d(x, w, 1, p)
    Yw = wg.conv2d_winograd(x, w, p, m=m)
    assert Yw.shape == Y.shape
    assert np.max(np.abs(Yw - Y) / np.maximum(S, 1e-300)) <= 1e-12


def test_conv2d_catches_a_flipped_filter():
    # Convolution instead of correlation (the filter flipped) must not pass.
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 2, 6, 6))
    w = rng.standard_normal((2, 2, 3, 3))
    Y, _ = ref.conv2d(x, w, 1, 1)
    Yf = wg.conv2d_winograd(x, w[:, :, ::-1, ::-1].copy(), 1)
    assert np.max(np.abs(Yf - Y)) > 1e-3
