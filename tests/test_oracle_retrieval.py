"""Pins of the oracle's retrieval step (CPU).

"RAPID: Long-Context Inference with Retrieval-Augmented Speculative Decoding",
section 3.1 (RAG settings): 512-token chunks, cosine similarity with the query
embedding, chunks below 0.3 dropped, the retrieved context within at least
4096 tokens and 1/24 of the input (reading: budget = max(4096, n / 24), chunks
taken greedily by descending score, ties to the lower index, a chunk that does
not fit the remaining budget skipped, kept chunks returned in document order).

Scores are pinned by closed forms (parallel, antiparallel, orthogonal, scale
invariance, zero vectors, a 45-degree pair).  The selection is pinned by the
budget arithmetic of the pages' example sizes, by invariants on random scores
and by brute force over every subset on tiny inputs.
"""
import itertools

import numpy as np
import pytest

import oracle


def test_score_closed_forms():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 64)).astype(np.float32)
    orth = rng.standard_normal(64).astype(np.float32)
    orth -= q[0] * (orth @ q[0]) / (q[0] @ q[0])
    c = np.stack([q[0] * 3.0, -q[0] * 0.5, orth, np.zeros(64, np.float32)])[None].astype(np.float32)
    s = oracle.retrieval_scores(q, c)
    assert s[0, 0] == pytest.approx(1.0, abs=1e-12)
    assert s[0, 1] == pytest.approx(-1.0, abs=1e-12)
    assert abs(s[0, 2]) < 1e-6               # orthogonal up to the float32 rounding of orth
    assert s[0, 3] == 0.0                     # zero vector scores 0
    # 45 degrees: q = e0, c = e0 + e1
    q2 = np.zeros((1, 8), np.float32); q2[0, 0] = 1
    c2 = np.zeros((1, 1, 8), np.float32); c2[0, 0, :2] = 1
    assert oracle.retrieval_scores(q2, c2)[0, 0] == pytest.approx(np.sqrt(0.5), abs=1e-15)
    # the query's scale does not matter (a power of two: exact in float32)
    s_scaled = oracle.retrieval_scores(q * 4.0, c)
    assert np.allclose(s, s_scaled, atol=1e-12)


def test_budget_of_the_pages_sizes():
    # 120K context: max(4096, 122880 / 24 = 5120) -> 10 chunks of 512
    n = 122880
    scores = np.full((1, 240), 0.9, np.float32)
    sel, ns, ts = oracle.retrieval_select(scores, np.array([n]))
    assert ns[0] == 10 and ts[0] == 5120 and sel[0, :10].tolist() == list(range(10))
    # 32K context: the 4096-token floor -> 8 chunks
    sel, ns, ts = oracle.retrieval_select(np.full((1, 64), 0.9, np.float32), np.array([32768]))
    assert ns[0] == 8 and ts[0] == 4096


def test_threshold_and_order():
    scores = np.array([[0.1, 0.8, 0.29999, 0.3, 0.95, 0.5]], np.float32)
    sel, ns, ts = oracle.retrieval_select(scores, np.array([6 * 512]), min_tokens=3 * 512)
    # budget 3 chunks: 0.95 (4), 0.8 (1), 0.5 (5); ids in document order
    assert sel[0, :3].tolist() == [1, 4, 5] and ns[0] == 3
    sel, ns, ts = oracle.retrieval_select(scores, np.array([6 * 512]), min_tokens=100 * 512)
    # everything at or above 0.3: 0.95, 0.8, 0.5, 0.3
    assert sel[0, :4].tolist() == [1, 3, 4, 5] and ns[0] == 4
    assert oracle.retrieval_select(np.full((1, 4), 0.2, np.float32), np.array([2048]))[1][0] == 0


def test_short_last_chunk_fills_the_rest():
    # 5 chunks, the last one 100 tokens; budget 4 x 512 - 400 = 1648 tokens
    n = 4 * 512 + 100
    scores = np.array([[0.9, 0.8, 0.7, 0.6, 0.5]], np.float32)
    sel, ns, ts = oracle.retrieval_select(scores, np.array([n]), min_tokens=1648)
    # 3 full chunks (1536) fit, the 4th (512) does not and is skipped, the short one (100) fits
    assert sel[0, :4].tolist() == [0, 1, 2, 4] and ts[0] == 1636


def _greedy_reference(s, lens, budget, thr):
    """The same rule by brute force: the kept set is the one the greedy visit
    reaches, checked against every subset for the defining properties."""
    best = None
    nc = len(s)
    order = sorted(range(nc), key=lambda j: (-s[j], j))
    for r in range(nc + 1):
        for sub in itertools.combinations(range(nc), r):
            if sum(lens[j] for j in sub) > budget or any(s[j] < thr for j in sub):
                continue
            # greedy property: every chunk visited before the first below-threshold
            # chunk is either kept or did not fit what the better-ranked kept
            # chunks had left
            ok = True
            used = 0
            for j in order:
                if s[j] < thr:
                    break
                if j in sub:
                    used += lens[j]
                elif used + lens[j] <= budget:
                    ok = False
                    break
            if ok:
                assert best is None, "the greedy set must be unique"
                best = sorted(sub)
    return best


@pytest.mark.parametrize("seed", range(8))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    nc = int(rng.integers(1, 8))
    chunk = 4
    n = (nc - 1) * chunk + int(rng.integers(1, chunk + 1))
    scores = rng.choice(np.array([0.1, 0.3, 0.5, 0.5, 0.7, 0.9], np.float32), size=nc)[None]
    budget = int(rng.integers(0, n + 3))
    sel, ns, ts = oracle.retrieval_select(scores, np.array([n]), chunk=chunk, min_tokens=budget,
                                          ratio=10 ** 6)
    lens = [min(chunk, n - j * chunk) for j in range(nc)]
    ref = _greedy_reference(scores[0].tolist(), lens, budget, np.float32(0.3))
    assert sel[0, :ns[0]].tolist() == ref
    assert ts[0] == sum(lens[j] for j in ref) <= budget


def test_invariants_random():
    rng = np.random.default_rng(9)
    B, N = 6, 300
    scores = rng.uniform(-0.2, 0.9, size=(B, N)).astype(np.float32)
    n = rng.integers(1, N * 512, size=B)
    sel, ns, ts = oracle.retrieval_select(scores, n)
    for b in range(B):
        nc = -(-int(n[b]) // 512)
        ids = sel[b, :ns[b]]
        assert np.all(np.diff(ids) > 0) and np.all(ids < nc)
        assert np.all(scores[b, ids] >= np.float32(0.3))
        assert ts[b] <= max(4096, int(n[b]) // 24)
        lens = np.minimum(512, int(n[b]) - np.arange(nc) * 512)
        assert ts[b] == lens[ids].sum()
        assert np.all(sel[b, ns[b]:] == -1)
