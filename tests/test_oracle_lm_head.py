"""Pins of the oracle's LM-head logits (CPU).

The target's logits of the verify rows come from its final hidden states and
the LM head that the drafter shares with it ("LongSpec: Long-Context Lossless
Speculative Decoding with Efficient Drafting and Verification", section 2.1),
z[r][v] = sum_k H[r][k] W[v][k] with W stored one vocabulary entry per row.

Pinned by: a product worked out by hand (distinct sizes, so a transposed
operand cannot pass), one-hot rows of W selecting columns of H and one-hot
hidden states selecting columns of W, exact integer products (bf16-sized
integers, computed with Python integers), and additivity in H.
"""
import numpy as np

import oracle


def test_hand_worked_example():
    # rows = 2, hidden = 3, V = 4
    H = np.array([[1, 2, 3], [-1, 0, 2]], np.float32)
    W = np.array([[1, 0, 0], [0, 1, 1], [2, -1, 0.5], [0, 0, 0]], np.float32)
    z = oracle.lm_head_logits(H, W)
    # row 0: [1, 2+3, 2-2+1.5, 0]; row 1: [-1, 0+2, -2+0+1, 0]
    assert z.shape == (2, 4)
    assert z.tolist() == [[1.0, 5.0, 1.5, 0.0], [-1.0, 2.0, -1.0, 0.0]]


def test_one_hot_rows_select_columns():
    rng = np.random.default_rng(0)
    H = rng.standard_normal((5, 7)).astype(np.float32)
    W = np.zeros((9, 7), np.float32)
    cols = [3, 0, 6, 6, 1, 2, 5, 4, 0]
    for v, k in enumerate(cols):
        W[v, k] = 1.0
    z = oracle.lm_head_logits(H, W)
    assert np.array_equal(z, H[:, cols].astype(np.float64))
    # one-hot hidden states pick columns of W (entry k of every vocabulary row)
    W2 = rng.standard_normal((11, 7)).astype(np.float32)
    E = np.eye(7, dtype=np.float32)[[2, 5]]
    z2 = oracle.lm_head_logits(E, W2)
    assert np.array_equal(z2, W2[:, [2, 5]].T.astype(np.float64))


def test_exact_on_integers():
    rng = np.random.default_rng(1)
    rows, hd, V = 3, 64, 50
    H = rng.integers(-128, 128, size=(rows, hd))
    W = rng.integers(-128, 128, size=(V, hd))
    z = oracle.lm_head_logits(H.astype(np.float32), W.astype(np.float32))
    for r in range(rows):
        for v in range(V):
            exact = sum(int(H[r, k]) * int(W[v, k]) for k in range(hd))
            assert z[r, v] == exact


def test_additive_in_hidden():
    rng = np.random.default_rng(2)
    A = rng.integers(-8, 8, size=(4, 32)).astype(np.float32)
    B = rng.integers(-8, 8, size=(4, 32)).astype(np.float32)
    W = rng.integers(-8, 8, size=(20, 32)).astype(np.float32)
    za, zb, zab = (oracle.lm_head_logits(x, W) for x in (A, B, A + B))
    assert np.array_equal(za + zb, zab)
