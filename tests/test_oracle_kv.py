"""Pins of the oracle's KV commit (CPU).

The commit is the step after acceptance: the accepted path's speculative rows
(node i of a verify step sits at cache row P + i, node 0 the root; "LongSpec:
Long-Context Lossless Speculative Decoding with Efficient Drafting and
Verification", section 2.3) join the history right after the root, in path
order, and the history grows by 1 + n_accepted.

What pins it, beyond its own statement: a chain is already in place; rows
outside the committed window never change; the committed cache gives the next
step's attention exactly what a cache built from scratch by appending the
accepted tokens does (through the independent attention oracle); invalid
inputs leave the cache untouched.
"""
import numpy as np
import pytest

import oracle


def _caches(rng, layers=2, B=3, Hkv=2, cap=64, d=8):
    K = rng.standard_normal((layers, B, Hkv, cap, d)).astype(np.float32)
    V = rng.standard_normal((layers, B, Hkv, cap, d)).astype(np.float32)
    return K, V


def _tree_path(rng, n_q, depth):
    """Node ids of a root-to-leaf prefix of a random tree (strictly increasing)."""
    nodes = sorted(rng.choice(np.arange(1, n_q), size=depth, replace=False).tolist())
    return nodes


def test_chain_path_is_already_in_place():
    rng = np.random.default_rng(1)
    K, V = _caches(rng)
    K0, V0 = K.copy(), V.copy()
    n_q = 9
    path = np.full((3, n_q), -1, np.int32)
    n_acc = np.array([0, 3, 8], np.int32)
    for b in range(3):
        path[b, :n_acc[b]] = np.arange(1, n_acc[b] + 1)
    assert oracle.kv_commit(K, V, np.array([0, 10, 40], np.int32), path, n_acc) == 0
    assert np.array_equal(K, K0) and np.array_equal(V, V0)


@pytest.mark.parametrize("seed", [2, 3, 4])
def test_tree_path_moves_rows_and_nothing_else(seed):
    rng = np.random.default_rng(seed)
    layers, B, Hkv, cap, d, n_q = 3, 4, 2, 80, 16, 16
    K, V = _caches(rng, layers, B, Hkv, cap, d)
    K0, V0 = K.copy(), V.copy()
    P = rng.integers(0, cap - n_q, size=B).astype(np.int32)
    path = np.full((B, n_q), -1, np.int32)
    n_acc = rng.integers(0, n_q, size=B).astype(np.int32)
    for b in range(B):
        path[b, :n_acc[b]] = _tree_path(rng, n_q, int(n_acc[b]))
    assert oracle.kv_commit(K, V, P, path, n_acc) == 0
    for b in range(B):
        n = int(n_acc[b])
        win = np.zeros(cap, bool)
        win[P[b] + 1:P[b] + 1 + n] = True
        for C, C0 in ((K, K0), (V, V0)):
            # every row outside the committed window is unchanged
            assert np.array_equal(C[:, b][:, :, ~win], C0[:, b][:, :, ~win])
            for k in range(n):
                assert np.array_equal(C[:, b, :, P[b] + 1 + k], C0[:, b, :, P[b] + path[b, k]])


def test_shift_by_one_overlap():
    # path 2, 3, 4: every destination is the source of the previous entry
    rng = np.random.default_rng(5)
    K, V = _caches(rng, 1, 1, 1, 32, 4)
    K0 = K.copy()
    path = np.array([[2, 3, 4, -1, -1, -1]], np.int32)
    assert oracle.kv_commit(K, V, np.array([10], np.int32), path, np.array([3], np.int32)) == 0
    assert np.array_equal(K[0, 0, 0, 11:14], K0[0, 0, 0, 12:15])
    assert np.array_equal(K[0, 0, 0, 14:], K0[0, 0, 0, 14:])


def test_next_step_attention_matches_a_cache_built_by_appending():
    # Commit + advance, then the next verify step's queries attend over the
    # new history; a cache assembled from scratch (history, root, accepted
    # rows, in order) must give the same output and LSE, bit for bit.
    rng = np.random.default_rng(6)
    B, Hkv, G, d, n_q, cap = 2, 2, 2, 16, 8, 96
    Hq = Hkv * G
    P = np.array([30, 47], np.int32)
    K = rng.standard_normal((1, B, Hkv, cap, d)).astype(np.float32)
    V = rng.standard_normal((1, B, Hkv, cap, d)).astype(np.float32)
    path = np.full((B, n_q), -1, np.int32)
    path[0, :3] = [1, 3, 6]
    path[1, :2] = [2, 5]
    n_acc = np.array([3, 2], np.int32)
    # the rows the next step must see after the history: root, then the path
    Kref = np.zeros((B, Hkv, cap, d), np.float32)
    Vref = np.zeros((B, Hkv, cap, d), np.float32)
    for b in range(B):
        keep = list(range(P[b] + 1)) + [P[b] + j for j in path[b, :n_acc[b]]]
        Kref[b, :, :len(keep)] = K[0, b][:, keep]
        Vref[b, :, :len(keep)] = V[0, b][:, keep]
    K_before, V_before = K[0].copy(), V[0].copy()
    assert oracle.kv_commit(K, V, P, path, n_acc) == 0
    P2 = oracle.kv_advance(P, n_acc)
    assert P2.tolist() == [34, 50]
    # next step: n_q2 new speculative rows after the new history, same in both caches
    n_q2 = 4
    spec_k = rng.standard_normal((B, Hkv, n_q2, d)).astype(np.float32)
    spec_v = rng.standard_normal((B, Hkv, n_q2, d)).astype(np.float32)
    Kc, Vc = K[0].copy(), V[0].copy()
    for b in range(B):
        Kc[b, :, P2[b]:P2[b] + n_q2] = spec_k[b]
        Vc[b, :, P2[b]:P2[b] + n_q2] = spec_v[b]
        Kref[b, :, P2[b]:P2[b] + n_q2] = spec_k[b]
        Vref[b, :, P2[b]:P2[b] + n_q2] = spec_v[b]
    Q = rng.standard_normal((B, Hq, n_q2, d)).astype(np.float32)
    O1, L1 = oracle.verify_attn(Q, Kc, Vc, P2)
    O2, L2 = oracle.verify_attn(Q, Kref, Vref, P2)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    # without the commit the new history would hold the rejected rows
    for b in range(B):
        K_before[b, :, P2[b]:P2[b] + n_q2] = spec_k[b]
        V_before[b, :, P2[b]:P2[b] + n_q2] = spec_v[b]
    O3, _ = oracle.verify_attn(Q, K_before, V_before, P2)
    assert not np.array_equal(O1, O3)


@pytest.mark.parametrize("case", ["decreasing", "too_far", "too_many", "overflow", "zero_node"])
def test_invalid_inputs_leave_the_cache_alone(case):
    rng = np.random.default_rng(7)
    K, V = _caches(rng, 1, 2, 1, 40, 4)
    K0 = K.copy()
    n_q = 8
    P = np.array([5, 5], np.int32)
    path = np.full((2, n_q), -1, np.int32)
    n_acc = np.array([2, 2], np.int32)
    path[0, :2] = [1, 3]
    path[1, :2] = [1, 3]
    if case == "decreasing":
        path[1, :2] = [4, 3]
    elif case == "too_far":
        path[1, :2] = [1, 8]
    elif case == "too_many":
        n_acc[1] = n_q
    elif case == "overflow":
        P[1] = 40 - n_q + 1
    elif case == "zero_node":
        path[1, :2] = [0, 3]
    assert oracle.kv_commit(K, V, P, path, n_acc) == 1
    assert np.array_equal(K[0, 1], K0[0, 1])            # sequence 1 untouched
    assert np.array_equal(K[0, 0, 0, 7], K0[0, 0, 0, 8])  # sequence 0 committed
