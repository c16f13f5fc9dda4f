"""The output law of the tree acceptance rule, against a closed form derived
independently of the oracle (CPU).

The pages define the token tree only through its attention mask ("LongSpec:
Long-Context Lossless Speculative Decoding with Efficient Drafting and
Verification", section 2.3); the acceptance over a tree is this library's
stated reading: every root-to-leaf path is checked by the ratio test of
"RAPID: Long-Context Inference with Retrieval-Augmented Speculative
Decoding", section 2.1, the path with the most accepted nodes wins (ties to
the smallest leaf id), and the next token comes from the residual of the last
accepted node's row.  For a root with m leaf children drafted independently
from q, at eta = 0 (p_hat = p), the first emitted token then has the law

    P(x) = min(p, q)(x) * sum_{k<m} (1 - beta)^k + (1 - beta)^(m-1) * max(p - q, 0)(x),
    beta = sum_x min(p, q)(x):

child k wins iff it is the first accepted one (each accepts with total
probability beta, token x with probability q(x) min(1, p(x)/q(x)) =
min(p, q)(x)), and if none is accepted the residual max(p - q, 0) / (1 - beta)
is drawn.  For m = 1 this is p (standard speculative sampling); for m >= 2 it
differs from p: the reading is not distribution-preserving on branching
trees.  These tests pin the oracle's tree rule to that law by sampling, and
check that the difference from p is real.
"""
import numpy as np
import pytest

import oracle


def star_law(p, q, m):
    mn = np.minimum(p, q)
    beta = mn.sum()
    geo = sum((1.0 - beta) ** k for k in range(m))
    return mn * geo + (1.0 - beta) ** (m - 1) * np.maximum(p - q, 0.0)


def _sample_first_tokens(z_row, q_row, m, n, seed):
    V = z_row.shape[0]
    n_q = m + 1
    z = np.broadcast_to(z_row, (n, n_q, V)).astype(np.float32)
    q = np.broadcast_to(q_row, (n, n_q, V)).astype(np.float32)
    parent = np.zeros((n, n_q), np.int32)
    parent[:, 0] = -1
    rng = np.random.default_rng(seed)
    qd = q_row.astype(np.float64) / q_row.astype(np.float64).sum()
    tok = np.zeros((n, n_q), np.int32)
    tok[:, 1:] = rng.choice(V, size=(n, m), p=qd)
    r = oracle.accept(z, q, tok, parent, T=1.0, eta=0.0, seed=seed, clamp=True)
    first = np.where(r["n_accepted"] >= 1, tok[np.arange(n), np.maximum(r["path"][:, 0], 0)],
                     r["next_token"])
    return np.bincount(first, minlength=V) / n


CASES = {
    # p and q far apart: beta = 0.55
    "far": (np.array([0.5, 0.3, 0.15, 0.05]), np.array([0.1, 0.2, 0.3, 0.4])),
    # close: beta = 0.9
    "close": (np.array([0.4, 0.3, 0.2, 0.1]), np.array([0.35, 0.3, 0.2, 0.15])),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("m", [1, 2, 3])
def test_star_tree_first_token_law(case, m):
    p, q = CASES[case]
    z_row = np.log(p).astype(np.float32)
    q_row = q.astype(np.float32)
    p64 = np.exp(z_row.astype(np.float64))
    p64 /= p64.sum()
    law = star_law(p64, q_row.astype(np.float64), m)
    assert abs(law.sum() - 1.0) < 1e-12
    n = 400_000
    freq = _sample_first_tokens(z_row, q_row, m, n, seed=0x7EE0 + m)
    sigma = np.sqrt(law * (1 - law) / n)
    assert (np.abs(freq - law) < 5 * sigma + 1e-12).all(), (freq, law)
    tv = 0.5 * np.abs(law - p64).sum()
    if m == 1:
        assert tv < 1e-12                      # a chain step is exact
    elif case == "far":
        assert tv > 0.05                       # the branching bias is real ...
        assert (np.abs(freq - p64) > 10 * sigma).any()   # ... and visible in the samples


def test_star_law_formula_by_enumeration():
    # the closed form against a direct enumeration of the rule over the
    # children's tokens and accept / reject outcomes (m = 2, V = 3)
    p = np.array([0.6, 0.3, 0.1])
    q = np.array([0.2, 0.5, 0.3])
    a = np.minimum(1.0, p / q)
    res = np.maximum(p - q, 0.0)
    res /= res.sum()
    out = np.zeros(3)
    for t1 in range(3):
        for t2 in range(3):
            w = q[t1] * q[t2]
            out[t1] += w * a[t1]                       # child 1 accepted: it wins the tie
            out[t2] += w * (1 - a[t1]) * a[t2]         # only child 2 accepted
            out += w * (1 - a[t1]) * (1 - a[t2]) * res  # none: the residual of the root
    np.testing.assert_allclose(out, star_law(p, q, 2), rtol=0, atol=1e-15)
