"""Pins for the oracle's drafter K/V projector ("VFlash-FM" project page,
"How VFlash-FM works": the drafter reads the target's cached hidden states
through a linear projector).

The oracle is a plain sum of products; the pins fix it by closed forms that a
slip in the indexing (a transposed weight, a wrong row or column) would break:
a selection weight returns the chosen hidden columns exactly, a one-hot row
returns the matching weight column, and the projection is linear in the
hidden states (exactly, for integer-valued inputs).
"""
import numpy as np

import oracle


def test_selection_weight_returns_hidden_columns():
    rng = np.random.default_rng(1)
    N, Hd, Dout = 7, 11, 5
    h = rng.standard_normal((N, Hd))
    cols = np.array([3, 0, 10, 3, 7])
    w = np.zeros((Dout, Hd))
    w[np.arange(Dout), cols] = 1.0
    assert np.array_equal(oracle.project_rows(h, w), h[:, cols])


def test_one_hot_hidden_row_returns_weight_column():
    rng = np.random.default_rng(2)
    Hd, Dout = 9, 6
    w = rng.standard_normal((Dout, Hd))
    h = np.zeros((Hd, Hd))
    h[np.arange(Hd), np.arange(Hd)] = 1.0
    out = oracle.project_rows(h, w)            # row k = w[:, k]
    assert np.array_equal(out, w.T)


def test_linear_and_row_selection_exact_on_integers():
    rng = np.random.default_rng(3)
    N, Hd, Dout = 12, 16, 8
    h1 = rng.integers(-8, 8, (N, Hd)).astype(np.float64)
    h2 = rng.integers(-8, 8, (N, Hd)).astype(np.float64)
    w = rng.integers(-8, 8, (Dout, Hd)).astype(np.float64)
    a, b = oracle.project_rows(h1, w), oracle.project_rows(h2, w)
    assert np.array_equal(oracle.project_rows(h1 + h2, w), a + b)
    rows = [11, 0, 5]
    assert np.array_equal(oracle.project_rows(h1, w, rows=rows), a[rows])
    # a hand-computed entry
    assert a[4, 2] == sum(h1[4, k] * w[2, k] for k in range(Hd))
