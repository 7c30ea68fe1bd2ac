"""Pins of the oracle's LM head (z = h W^T) against closed forms.

* one-hot hidden states: row r with h = e_k gives z[r, v] = W[v, k] -- the
  k-th weight column, a transposed operand or a wrong contraction axis fails;
* a hand-computed 2 x 3 case;
* linearity: z(a h1 + b h2) = a z(h1) + b z(h2), and a scaled weight scales
  the logits;
* batched shapes: [B, M, H] hidden states give [B, M, V] logits, row by row.
"""
import numpy as np

from oracle import oracle_lm_head


def test_one_hot_rows_select_weight_columns():
    rng = np.random.default_rng(1)
    H, V = 6, 9
    W = rng.normal(size=(V, H))
    h = np.eye(H)
    z = oracle_lm_head(h, W)
    assert z.shape == (H, V)
    for k in range(H):
        assert np.array_equal(z[k], W[:, k])


def test_hand_computed_case():
    h = np.array([[1.0, 2.0], [-1.0, 0.5]])
    W = np.array([[3.0, 0.0], [1.0, 1.0], [0.0, -2.0]])
    # row 0: [1*3 + 2*0, 1*1 + 2*1, 1*0 + 2*(-2)] = [3, 3, -4]
    # row 1: [-3, -1 + 0.5, -1] = [-3, -0.5, -1]
    assert np.array_equal(oracle_lm_head(h, W), np.array([[3.0, 3.0, -4.0], [-3.0, -0.5, -1.0]]))


def test_linearity_and_scaling():
    rng = np.random.default_rng(2)
    H, V = 16, 40
    W = rng.normal(size=(V, H))
    h1, h2 = rng.normal(size=(3, H)), rng.normal(size=(3, H))
    lhs = oracle_lm_head(2.0 * h1 - 0.5 * h2, W)
    rhs = 2.0 * oracle_lm_head(h1, W) - 0.5 * oracle_lm_head(h2, W)
    assert np.allclose(lhs, rhs, rtol=1e-13, atol=1e-12)
    assert np.allclose(oracle_lm_head(h1, 4.0 * W), 4.0 * oracle_lm_head(h1, W), rtol=1e-14)


def test_batched_rows():
    rng = np.random.default_rng(3)
    B, M, H, V = 2, 3, 8, 5
    W = rng.normal(size=(V, H))
    h = rng.normal(size=(B, M, H))
    z = oracle_lm_head(h, W)
    assert z.shape == (B, M, V)
    for b in range(B):
        for m in range(M):
            assert np.allclose(z[b, m], oracle_lm_head(h[b, m][None], W)[0], rtol=1e-14)
