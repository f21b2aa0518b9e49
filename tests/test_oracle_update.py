"""Pins of the oracle's prediction update (no GPU).

"Module Design: Training Core" s.6 step 7 and "Gradient boosted trees (spec
model)", Forward pass: after a tree is built every row's prediction moves by
learning_rate times the value of the leaf the row reached,
pred_i <- pred_i + (lr * w[leaf(i)]), with the product rounded to FP64 before
the addition (no fused multiply-add).

The expected values are worked out here without the oracle: by hand for exact
binary fractions, and with exact rational arithmetic (fractions.Fraction,
rounded to the nearest double once per operation) where the rounding order
matters.
"""
from fractions import Fraction

import numpy as np

import oracle


def _round(x: Fraction) -> float:
    """The double nearest to the exact rational x (Python rounds ties to even)."""
    return float(x)


def _update_exact(p: float, lr: float, w: float) -> float:
    step = _round(Fraction(lr) * Fraction(w))  # the product, rounded once
    return _round(Fraction(p) + Fraction(step))  # the sum, rounded once


def test_hand_values_exact_fractions(o=oracle):
    # lr = 3/8; every product and sum below is exact in binary, worked by hand:
    #   row 0: leaf 2 (w =  1/4):  1/2  + 3/32 =  19/32 =  0.59375
    #   row 1: leaf 0 (w =  1  ): -5/4  + 3/8  =  -7/8  = -0.875
    #   row 2: leaf 1 (w = -1/2):  2    - 3/16 =  29/16 =  1.8125
    #   row 3: leaf 3 (w =  3  ):  0    + 9/8  =   9/8  =  1.125
    #   row 4: leaf 2 (w =  1/4): -3/32 + 3/32 =   0
    pred = np.array([0.5, -1.25, 2.0, 0.0, -0.09375])
    leaf_value = np.array([1.0, -0.5, 0.25, 3.0, 7.0])
    node_of_row = np.array([2, 0, 1, 3, 2])
    got = o.update_predictions(pred, leaf_value, node_of_row, 0.375)
    assert np.array_equal(got, np.array([0.59375, -0.875, 1.8125, 1.125, 0.0]))


def test_product_rounded_before_the_sum(o=oracle):
    # lr = 0.37 is not a binary fraction.  Rows are chosen (by a seeded search) so that rounding the
    # product first gives a different double than one rounding of pred + lr * w (a fused multiply-add):
    # a mistake in the rounding order, the sign, the learning rate or the leaf index changes them.
    rng = np.random.default_rng(7)
    lr = 0.37
    rows = []
    while len(rows) < 16:
        p, w = float(rng.normal() * 3.0), float(rng.normal())
        once = _round(Fraction(p) + Fraction(lr) * Fraction(w))
        if _update_exact(p, lr, w) != once:
            rows.append((p, w))
    n_leaves = 24
    leaf_value = rng.normal(size=n_leaves)
    node_of_row = rng.permutation(n_leaves)[: len(rows)]
    for i, (_, w) in enumerate(rows):
        leaf_value[node_of_row[i]] = w
    pred = np.array([p for p, _ in rows])
    want = np.array([_update_exact(p, lr, w) for p, w in rows])
    got = o.update_predictions(pred, leaf_value, node_of_row, lr)
    assert np.array_equal(got, want)


def test_zero_rate_and_no_rows(o=oracle):
    pred = np.array([1.5, -2.0, 0.0])
    assert np.array_equal(o.update_predictions(pred, np.array([4.0, -4.0]), np.array([1, 0, 1]), 0.0), pred)
    assert o.update_predictions(np.zeros(0), np.array([1.0]), np.zeros(0, np.int32), 0.1).shape == (0,)
