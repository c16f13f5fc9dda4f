"""Pins of the oracle's verify attention (CPU only).

What fixes the values here:
 * hand-computed attention of a 3-row example (exact weights 1/5, 3/5, 1/5);
 * closed forms: all keys equal (or scale 0) gives the mean of the visible V
   rows and LSE = s + ln(n_visible); an empty history leaves the masked
   speculative rows only; a dominating key returns its V row;
 * invariants of attention: linear in V, invariant to permuting the
   speculative rows together with the mask, the chain equals the explicit
   lower-triangular mask, query head h reads KV head h // (Hq / Hkv);
 * the hybrid form of "LongSpec: Long-Context Lossless Speculative Decoding
   with Efficient Drafting and Verification", section 2.3 (history pieces
   without a mask + speculative piece with a mask, merged by log-sum-exp)
   equals the unsplit definition for any cut of the history, empty pieces
   included.
"""
import math

import numpy as np
import pytest

import oracle
from long_context_speculative_gb300 import workloads as wl


def _rand(B, Hq, Hkv, d, n_q, cap, seed, qs=1.0):
    rng = np.random.default_rng(seed)
    Q = (rng.standard_normal((B, Hq, n_q, d)) * qs).astype(np.float32)
    K = rng.standard_normal((B, Hkv, cap, d)).astype(np.float32)
    V = rng.standard_normal((B, Hkv, cap, d)).astype(np.float32)
    return Q, K, V


def test_hand_computed_three_rows():
    d = 2
    s = 1.0 / math.sqrt(d)
    Q = np.array([[[[math.sqrt(2) * math.log(3.0), 0.0]]]], np.float32)  # [1,1,1,2]
    K = np.zeros((1, 1, 4, d), np.float32)
    K[0, 0, 1] = [1.0, 0.0]          # score ln 3; rows 0 and 2 score 0
    V = np.zeros((1, 1, 4, d), np.float32)
    V[0, 0, 0] = [1.0, 0.0]
    V[0, 0, 1] = [0.0, 1.0]
    V[0, 0, 2] = [2.0, 2.0]          # the query's own speculative row
    V[0, 0, 3] = [100.0, 100.0]      # beyond prefix + n_q: never visible
    O, L = oracle.verify_attn(Q, K, V, np.array([2], np.int32), scale=s)
    # weights (1, 3, 1) / 5; Q is float32-rounded, so ln 3 is exact to ~1e-7
    np.testing.assert_allclose(O[0, 0, 0], [0.2 * 1 + 0.2 * 2, 0.6 + 0.2 * 2], rtol=1e-6)
    np.testing.assert_allclose(L[0, 0, 0], math.log(5.0), rtol=1e-6)


def test_uniform_keys_give_mean_of_visible_rows():
    B, Hq, Hkv, d, n_q, cap = 2, 4, 2, 64, 5, 80
    Q, K, V = _rand(B, Hq, Hkv, d, n_q, cap, 1)
    K[:] = K[:, :, :1, :]                     # every key row equal
    pl = np.array([40, 0], np.int32)
    O, L = oracle.verify_attn(Q, K, V, pl)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for i in range(n_q):
                vis = list(range(pl[b])) + [pl[b] + j for j in range(i + 1)]
                np.testing.assert_allclose(O[b, h, i], V[b, g, vis].astype(np.float64).mean(0),
                                           rtol=1e-10, atol=1e-12)
                s = float(Q[b, h, i].astype(np.float64) @ K[b, g, 0].astype(np.float64)) / 8.0
                np.testing.assert_allclose(L[b, h, i], s + math.log(len(vis)), rtol=1e-10)


def test_scale_zero_is_plain_average():
    Q, K, V = _rand(1, 2, 1, 64, 3, 20, 2)
    O, L = oracle.verify_attn(Q, K, V, np.array([10], np.int32), scale=0.0)
    for i in range(3):
        n = 10 + i + 1
        np.testing.assert_allclose(O[0, :, i], np.broadcast_to(V[0, 0, :n].astype(np.float64).mean(0), (2, 64)),
                                   rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(L[0, :, i], math.log(n), rtol=1e-12)


def test_empty_history_and_first_query_sees_itself_only():
    Q, K, V = _rand(1, 2, 2, 64, 4, 16, 3)
    O, L = oracle.verify_attn(Q, K, V, np.array([0], np.int32))
    for h in range(2):
        np.testing.assert_allclose(O[0, h, 0], V[0, h, 0], rtol=1e-12)
        s = float(Q[0, h, 0].astype(np.float64) @ K[0, h, 0].astype(np.float64)) / 8.0
        np.testing.assert_allclose(L[0, h, 0], s, rtol=1e-12)


def test_dominating_key_returns_its_value_row():
    Q, K, V = _rand(1, 1, 1, 64, 1, 64, 4, qs=0.05)
    K[0, 0, 17] = Q[0, 0, 0] * 3000.0
    O, L = oracle.verify_attn(Q, K, V, np.array([60], np.int32))
    np.testing.assert_allclose(O[0, 0, 0], V[0, 0, 17], rtol=1e-9, atol=1e-9)


def test_linear_in_values():
    Q, K, V1 = _rand(1, 4, 2, 64, 3, 50, 5)
    _, _, V2 = _rand(1, 4, 2, 64, 3, 50, 6)
    pl = np.array([30], np.int32)
    O1, L1 = oracle.verify_attn(Q, K, V1, pl)
    O2, _ = oracle.verify_attn(Q, K, V2, pl)
    O3, L3 = oracle.verify_attn(Q, K, (V1.astype(np.float64) + V2).astype(np.float32), pl)
    np.testing.assert_allclose(O3, O1 + O2, atol=1e-6)
    np.testing.assert_array_equal(L1, L3)


def test_chain_equals_lower_triangular_mask():
    Q, K, V = _rand(2, 4, 1, 64, 6, 40, 7)
    pl = np.array([20, 34], np.int32)
    tri = np.tril(np.ones((6, 6), np.uint8))[None].repeat(2, 0)
    a = oracle.verify_attn(Q, K, V, pl)
    b = oracle.verify_attn(Q, K, V, pl, mask=tri)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_permuting_speculative_rows_with_mask():
    rng = np.random.default_rng(8)
    n_q, P = 8, 25
    par = wl.random_tree(n_q, 4, wl.gen(3))
    mask = wl.ancestor_mask(par).numpy()[None]
    Q, K, V = _rand(1, 2, 1, 64, n_q, 40, 9)
    pl = np.array([P], np.int32)
    O, L = oracle.verify_attn(Q, K, V, pl, mask=mask)
    perm = rng.permutation(n_q)        # new position of node j is perm[j]
    inv = np.argsort(perm)
    Q2 = Q[:, :, inv]
    K2, V2 = K.copy(), V.copy()
    K2[0, 0, P:P + n_q] = K[0, 0, P + inv]
    V2[0, 0, P:P + n_q] = V[0, 0, P + inv]
    m2 = mask[0][np.ix_(inv, inv)][None]
    O2, L2 = oracle.verify_attn(Q2, K2, V2, pl, mask=m2)
    np.testing.assert_allclose(O2, O[:, :, inv], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(L2, L[:, :, inv], rtol=1e-12)


def test_gqa_head_mapping():
    B, Hq, Hkv, d, n_q, cap = 1, 6, 3, 64, 2, 30
    Q, K, V = _rand(B, Hq, Hkv, d, n_q, cap, 10)
    for g in range(Hkv):
        V[0, g] = float(g + 1)          # KV head g holds the constant g+1
    O, _ = oracle.verify_attn(Q, K, V, np.array([20], np.int32))
    for h in range(Hq):
        np.testing.assert_allclose(O[0, h], h // 2 + 1.0, rtol=1e-12)


@pytest.mark.parametrize("cuts", [[], [0], [7, 7, 19], [1, 2, 3, 500], [32, 64, 96, 128]])
def test_lse_merge_of_history_pieces_equals_unsplit(cuts):
    B, Hq, Hkv, d, n_q, cap = 2, 4, 2, 64, 5, 160
    Q, K, V = _rand(B, Hq, Hkv, d, n_q, cap, 11, qs=0.5)
    pl = np.array([130, 3], np.int32)
    par = [wl.random_tree(n_q, 3, wl.gen(5)), wl.chain_parents(n_q)]
    mask = np.stack([wl.ancestor_mask(p).numpy() for p in par])
    for m in [None, mask]:
        O, L = oracle.verify_attn(Q, K, V, pl, mask=m)
        O2, L2 = oracle.verify_attn_split(Q, K, V, pl, cuts, mask=m)
        np.testing.assert_allclose(O2, O, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(L2, L, rtol=1e-12, atol=1e-12)


def test_bf16_input_decoding():
    import torch
    Q, K, V = _rand(1, 2, 1, 64, 3, 24, 12)
    tq, tk, tv = (torch.from_numpy(x).to(torch.bfloat16) for x in (Q, K, V))
    pl = np.array([16], np.int32)
    Ob, Lb = oracle.verify_attn(wl.bf16_bits(tq), wl.bf16_bits(tk), wl.bf16_bits(tv), pl,
                                dtype=oracle.DTYPE_BF16)
    Of, Lf = oracle.verify_attn(tq.float().numpy(), tk.float().numpy(), tv.float().numpy(), pl)
    np.testing.assert_array_equal(Ob, Of)
    np.testing.assert_array_equal(Lb, Lf)


def test_rows_entry_matches_full():
    Q, K, V = _rand(2, 4, 2, 64, 3, 40, 13)
    pl = np.array([30, 12], np.int32)
    O, L = oracle.verify_attn(Q, K, V, pl)
    rows = np.array([[0, 0, 0], [1, 3, 2], [1, 1, 1], [0, 2, 2]], np.int32)
    Or, Lr = oracle.verify_attn_rows(Q, K, V, pl, rows)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(Or[n], O[b, h, i])
        assert Lr[n] == L[b, h, i]


def _shards(K, V, pl, n_q, cuts):
    """Caches of the history pieces [cuts[k], cuts[k+1]) of every sequence,
    each followed by the sequence's n_q speculative rows (moved up after the
    piece); returns [(K_k, V_k, prefix_k)]."""
    B, Hkv, cap, d = K.shape
    out = []
    for k in range(len(cuts) - 1):
        Kk = np.zeros_like(K)
        Vk = np.zeros_like(V)
        pk = np.zeros(B, np.int32)
        for b in range(B):
            lo, hi = min(cuts[k], pl[b]), min(cuts[k + 1], pl[b])
            n = hi - lo
            Kk[b, :, :n] = K[b, :, lo:hi]
            Vk[b, :, :n] = V[b, :, lo:hi]
            Kk[b, :, n:n + n_q] = K[b, :, pl[b]:pl[b] + n_q]
            Vk[b, :, n:n + n_q] = V[b, :, pl[b]:pl[b] + n_q]
            pk[b] = n
        out.append((Kk, Vk, pk))
    return out


@pytest.mark.parametrize("tree", [False, True])
def test_lse_merge_of_key_shards_equals_unsplit(tree):
    # Shards of the history by key range (one of them empty), the speculative
    # rows visible only in the last shard (an all-zero mask hides them from
    # the others): merging the shards' (O, LSE) gives the unsplit attention.
    B, Hq, Hkv, d, n_q, cap = 2, 4, 2, 64, 6, 400
    Q, K, V = _rand(B, Hq, Hkv, d, n_q, cap, 31)
    pl = np.array([300, 170], np.int32)
    if tree:
        parents = [wl.random_tree(n_q, 3, wl.gen(40 + b)) for b in range(B)]
        mask = np.stack([wl.ancestor_mask(p).numpy() for p in parents])
    else:
        mask = np.stack([np.tril(np.ones((n_q, n_q), np.uint8))] * B)
    O_ref, L_ref = oracle.verify_attn(Q, K, V, pl, mask)
    cuts = [0, 100, 100, 230, 400]
    shards = _shards(K, V, pl, n_q, cuts)
    none = np.zeros_like(mask)
    parts = [oracle.verify_attn(Q, Kk, Vk, pk, mask if k == len(shards) - 1 else none)
             for k, (Kk, Vk, pk) in enumerate(shards)]
    # the empty piece of sequence 1 (rows 230..) and the repeated cut give
    # parts that saw no key: LSE -inf, O 0
    assert np.isneginf(parts[1][1]).all() and (parts[1][0] == 0).all()
    O, L = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(O, O_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, L_ref, rtol=0, atol=1e-12)


def test_lse_merge_closed_forms():
    rng = np.random.default_rng(4)
    O1 = rng.standard_normal((3, 5, 8))
    L1 = rng.standard_normal((3, 5))
    # one part: itself
    O, L = oracle.lse_merge(O1[None], L1[None])
    np.testing.assert_array_equal(O, O1)
    np.testing.assert_array_equal(L, L1)
    # the same part twice: the same O, LSE + ln 2
    O, L = oracle.lse_merge(np.stack([O1, O1]), np.stack([L1, L1]))
    np.testing.assert_allclose(O, O1, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(L, L1 + math.log(2.0), rtol=1e-14)
    # a part that saw no key adds nothing, whatever its O holds
    O, L = oracle.lse_merge(np.stack([O1, np.full_like(O1, 1e30)]),
                            np.stack([L1, np.full_like(L1, -np.inf)]))
    np.testing.assert_array_equal(O, O1)
    np.testing.assert_array_equal(L, L1)
    # no part at all: O = 0, LSE = -inf
    O, L = oracle.lse_merge(np.stack([O1, O1]), np.full((2, 3, 5), -np.inf))
    assert (O == 0).all() and np.isneginf(L).all()
    # two parts with LSE a and b: weights e^a / (e^a + e^b) and e^b / (e^a + e^b)
    a, b = 0.3, -1.2
    O, L = oracle.lse_merge(np.array([[[1.0, 0.0]], [[0.0, 1.0]]]), np.array([[a], [b]]))
    wa = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(O[0], [wa, 1.0 - wa], rtol=1e-14)
    np.testing.assert_allclose(L[0], a + math.log1p(math.exp(b - a)), rtol=1e-14)
