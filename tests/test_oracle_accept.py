"""Pins of the oracle's acceptance step (CPU only).

What fixes the values here (none of it re-types the oracle's own code):
 * "RAPID: Long-Context Inference with Retrieval-Augmented Speculative
   Decoding" (blog summary), section 2.1: at eta = 0 the step is standard
   speculative decoding -- ratio p/q, residual norm(max(p - q, 0)) -- and the
   emitted token is distributed exactly as p.
 * Section 2.4: p = softmax(z/T) (checked against scipy's softmax);
   p_hat = softmax(z/T + eta (q - p)) agrees with softmax(z_hat / T) for the
   distilled logit z_hat = z + eta T (q - p); Proposition 1 (gradient of
   T^2 KL(q || p) is T (p - q), by central differences); the tail rule.
 * Worked examples with values computed by hand (exact fractions).
 * At eta > 0 the first emitted token follows the closed form
   P_out = min(q, p_hat) + (1 - sum min(q, p_hat)) * w / W, with w the
   adjusted residual (derived from the acceptance rule; the page's claim that
   the output follows p exactly holds only where p >= min(q, p_hat)).
"""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import oracle
from long_context_speculative_gb300 import workloads as wl


def _rand_row(V, seed, z_std=3.0, noise=1.5, T=1.0):
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal(V) * z_std).astype(np.float32)
    q = sp_softmax(z.astype(np.float64) / T + rng.standard_normal(V) * noise).astype(np.float32)
    return z, q


@pytest.mark.parametrize("T", [0.6, 1.0, 2.5])
def test_p_is_softmax_of_z_over_T(T):
    z, q = _rand_row(500, 1, T=T)
    p, raw, ph = oracle.row_dists(z, q, T, 1.0)
    np.testing.assert_allclose(p, sp_softmax(z.astype(np.float64) / T), rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("eta", [0.5, 1.0, 5.0])
@pytest.mark.parametrize("T", [0.6, 1.0])
def test_phat_matches_library_softmax_and_distilled_logit(T, eta):
    z, q = _rand_row(700, 2, T=T)
    p_lib = sp_softmax(z.astype(np.float64) / T)
    expect = sp_softmax(z.astype(np.float64) / T + eta * (q.astype(np.float64) - p_lib))
    p, raw, _ = oracle.row_dists(z, q, T, eta, clamp=False)
    np.testing.assert_allclose(raw, expect, rtol=1e-10)
    # z_hat = z + eta T (q - p): softmax(z_hat / T) is the same distribution.
    zh = oracle.distilled_logits(z.astype(np.float64), q.astype(np.float64), T, eta)
    np.testing.assert_allclose(zh, z + eta * T * (q.astype(np.float64) - p_lib), rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(sp_softmax(zh / T), raw, rtol=1e-10)


@pytest.mark.parametrize("T", [0.6, 1.0, 2.0])
def test_proposition1_gradient_by_central_differences(T):
    rng = np.random.default_rng(3)
    V = 12
    z = rng.standard_normal(V) * 2.0
    q = sp_softmax(rng.standard_normal(V))
    g = oracle.kd_grad(z, q, T)
    h = 1e-6
    fd = np.zeros(V)
    for k in range(V):
        zp = z.copy(); zp[k] += h
        zm = z.copy(); zm[k] -= h
        fd[k] = (oracle.kd_loss(zp, q, T) - oracle.kd_loss(zm, q, T)) / (2 * h)
    np.testing.assert_allclose(fd, g, rtol=1e-6, atol=1e-9)
    # and the closed form itself: T (p - q) with p = softmax(z/T)
    np.testing.assert_allclose(g, T * (sp_softmax(z / T) - q), rtol=1e-12, atol=1e-15)


def test_eta_zero_reduces_to_standard_sd():
    z, q = _rand_row(300, 4)
    p, raw, ph = oracle.row_dists(z, q, 1.0, 0.0, clamp=True)
    assert np.array_equal(p, raw) and np.array_equal(p, ph)
    w = oracle.residual_weights(p, ph, q)
    np.testing.assert_array_equal(w, np.maximum(p - q.astype(np.float64), 0.0))


def test_q_equal_p_gives_phat_equal_p_and_accepts_everything():
    w = wl.Workload("t", B=2, Hq=1, Hkv=1, d=64, n_q=6, prefix=1, layers=1, V=64, dtype="f32",
                    z_std=2.0, q_noise_std=0.0, q_noise_uses_T=True, seed=9)
    inp = wl.accept_inputs(w)
    z = inp.z.numpy()
    q = sp_softmax(z.astype(np.float64), axis=-1).astype(np.float32)
    for eta in [0.0, 1.0, 10.0]:
        p, raw, ph = oracle.row_dists(z[0, 0], q[0, 0], 1.0, eta)
        np.testing.assert_allclose(raw, p, rtol=1e-6)
        res = oracle.accept(z, q, inp.tokens.numpy(), T=1.0, eta=eta, seed=77)
        # ratio = p_hat/q is 1 up to float32 rounding of q: r < 1 always accepts
        # unless the ratio rounds below r (probability ~1e-7 per node).
        assert (res["n_accepted"] == 5).all()
        assert (res["sample"][:, 1] == 0).all()   # bonus from p of the last row


def test_shift_invariance():
    z, q = _rand_row(400, 5)
    a = oracle.row_dists(z, q, 1.0, 2.0)
    b = oracle.row_dists((z.astype(np.float64) + 7.0).astype(np.float32), q, 1.0, 2.0)
    # +7 is exact in float32 for |z| < 2^20 only up to rounding of z + 7; compare loosely.
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-5)
    c = oracle.row_dists(z.astype(np.float32), q, 1.0, 2.0)
    for x, y in zip(a, c):
        assert np.array_equal(x, y)


def test_tail_rule():
    # Built so several entries sit below and above 0.1 * max(p_hat).
    z = np.log(np.array([50.0, 10.0, 6.0, 4.9, 5.1, 1.0, 0.5, 20.0])).astype(np.float32)
    q = np.array([0.3, 0.05, 0.1, 0.1, 0.05, 0.2, 0.1, 0.1], np.float32)
    for eta in [0.0, 0.7, 3.0]:
        p, raw, ph = oracle.row_dists(z, q, 1.0, eta, clamp=True)
        top = raw.max()
        low = raw < 0.1 * top
        assert low.any() and (~low).any()
        np.testing.assert_array_equal(ph[low], p[low])
        np.testing.assert_array_equal(ph[~low], raw[~low])
        _, raw2, ph2 = oracle.row_dists(z, q, 1.0, eta, clamp=False)
        np.testing.assert_array_equal(ph2, raw2)


def _first_token_worked_example(seed, expect_accept):
    # V = 3, T = 1: z = log(1, 2, 5) gives p = (1/8, 2/8, 5/8) exactly.
    # Draft row 0 proposes token 0 with q_0(0) = 1/2: ratio = (1/8)/(1/2) = 1/4.
    # Residual at eta = 0: max(p - q, 0) = (0, 0, 3/8) -> token 2 always.
    z = np.log(np.array([[1.0, 2.0, 5.0], [1.0, 1.0, 6.0]])).astype(np.float32)[None]
    q = np.array([[0.5, 0.25, 0.25], [0.2, 0.3, 0.5]], np.float32)[None]
    tokens = np.array([[0, 0]], np.int32)
    res = oracle.accept(z, q, tokens, T=1.0, eta=0.0, seed=seed)
    words1 = oracle.philox4x32_10([1, 0, 0, 0], [seed & 0xffffffff, seed >> 32])
    r1 = (int(words1[0]) >> 8) / 2.0 ** 24
    assert (r1 <= 0.25) == expect_accept
    np.testing.assert_allclose(res["diag"][0, 1, :4], [1 / 8, 1 / 8, 0.5, 0.25], rtol=1e-7)
    if not expect_accept:
        assert res["n_accepted"][0] == 0 and res["next_token"][0] == 2
    else:
        # bonus from row 1: p = (1/8, 1/8, 6/8); CDF boundaries 1/8, 2/8.
        words2 = oracle.philox4x32_10([2, 0, 0, 0], [seed & 0xffffffff, seed >> 32])
        u2 = (int(words2[1]) >> 8) / 2.0 ** 24
        expect_tok = 0 if u2 < 1 / 8 else (1 if u2 < 2 / 8 else 2)
        assert res["n_accepted"][0] == 1 and res["next_token"][0] == expect_tok


def test_worked_example_reject_and_accept():
    hits = {True: 0, False: 0}
    for seed in range(40):
        words = oracle.philox4x32_10([1, 0, 0, 0], [seed, 0])
        acc = ((int(words[0]) >> 8) / 2.0 ** 24) <= 0.25
        if hits[acc] < 3:
            _first_token_worked_example(seed, acc)
            hits[acc] += 1
    assert hits[True] == 3 and hits[False] == 3


def test_inverse_cdf_by_hand():
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    # W = 1: boundaries C = 0, .25, .25, .75, 1 -> smallest k with C_k > u.
    assert oracle.sample_inverse_cdf(w, 0.0) == 1
    assert oracle.sample_inverse_cdf(w, 0.2499) == 1
    assert oracle.sample_inverse_cdf(w, 0.25) == 3
    assert oracle.sample_inverse_cdf(w, 0.7) == 3
    assert oracle.sample_inverse_cdf(w, 0.75) == 4
    assert oracle.sample_inverse_cdf(w * 3.0, 0.999999) == 4


def _chi2_pvalue(hist, probs):
    from scipy.stats import chisquare
    n = hist.sum()
    mask = probs * n > 5
    f_exp = probs[mask] * n
    f_obs = hist[mask].astype(np.float64)
    # lump the rare cells into one
    if (~mask).any():
        f_exp = np.append(f_exp, probs[~mask].sum() * n)
        f_obs = np.append(f_obs, hist[~mask].sum())
    f_exp *= f_obs.sum() / f_exp.sum()
    return chisquare(f_obs, f_exp).pvalue


def _p_out(z, q, T, eta, clamp):
    p, raw, ph = oracle.row_dists(z, q, T, eta, clamp)
    qd = q.astype(np.float64)
    acc = np.minimum(qd, ph)
    w = np.maximum(np.maximum(p - ph, p - qd), 0.0)
    W = w.sum()
    if W <= 0:
        w, W = p, p.sum()
    return p, acc + (1.0 - acc.sum()) * w / W


@pytest.mark.parametrize("V,eta,T", [(8, 0.0, 1.0), (8, 0.0, 0.6), (1000, 0.0, 1.0),
                                     (8, 1.0, 1.0), (8, 10.0, 1.0), (1000, 1.0, 0.6),
                                     (8, 10.0, 0.6)])
def test_first_token_distribution_brute_force(V, eta, T):
    rng = np.random.default_rng(100 + V + int(eta * 10) + int(T * 10))
    z = (rng.standard_normal(V) * 2.0).astype(np.float32)
    q = sp_softmax(z.astype(np.float64) + rng.standard_normal(V)).astype(np.float32)
    n = 1_000_000
    hist = oracle.first_token_hist(z, q, T, eta, True, seed=0xABCD0000 + V, n_trials=n)
    assert hist.sum() == n
    p, pout = _p_out(z, q, T, eta, True)
    if eta == 0.0:
        # standard speculative decoding: output ~ p exactly
        np.testing.assert_allclose(pout, p, rtol=1e-9, atol=1e-15)
    pv = _chi2_pvalue(hist, pout)
    assert pv > 1e-4, pv
    tv = 0.5 * np.abs(hist / n - pout).sum()
    assert tv < (0.01 if V == 8 else 0.05)


def test_first_token_distribution_detects_wrong_target():
    # The same histogram is far from p once eta > 0 moves P_out away from p:
    # the test above has the power to see a wrong residual.
    V = 8
    rng = np.random.default_rng(7)
    z = (rng.standard_normal(V) * 2.0).astype(np.float32)
    q = sp_softmax(z.astype(np.float64) + rng.standard_normal(V) * 2).astype(np.float32)
    hist = oracle.first_token_hist(z, q, 1.0, 10.0, True, seed=5, n_trials=400_000)
    p, pout = _p_out(z, q, 1.0, 10.0, True)
    if 0.5 * np.abs(pout - p).sum() > 0.01:
        assert _chi2_pvalue(hist, p) < 1e-6


def test_tree_with_chain_parents_equals_chain():
    w = wl.Workload("t", B=3, Hq=1, Hkv=1, d=64, n_q=7, prefix=1, layers=1, V=300, dtype="f32",
                    z_std=2.0, q_noise_std=0.7, q_noise_uses_T=True, seed=21)
    inp = wl.accept_inputs(w)
    z, q, tok = inp.z.numpy(), inp.q.numpy(), inp.tokens.numpy()
    par = np.tile(np.arange(-1, 6, dtype=np.int32), (3, 1))
    for seed in range(20):
        a = oracle.accept(z, q, tok, None, T=1.0, eta=1.0, seed=seed)
        b = oracle.accept(z, q, tok, par, T=1.0, eta=1.0, seed=seed)
        for k in ["n_accepted", "next_token", "path"]:
            np.testing.assert_array_equal(a[k], b[k])


def test_chain_first_rejection_semantics():
    # n_accepted is the number of leading accepted drafts; the residual row is
    # the row before the first rejected draft; its uniform is u of that draft.
    w = wl.Workload("t", B=4, Hq=1, Hkv=1, d=64, n_q=9, prefix=1, layers=1, V=200, dtype="f32",
                    z_std=2.0, q_noise_std=1.2, q_noise_uses_T=True, seed=33)
    inp = wl.accept_inputs(w)
    z, q, tok = inp.z.numpy(), inp.q.numpy(), inp.tokens.numpy()
    seen = set()
    for seed in range(60):
        res = oracle.accept(z, q, tok, T=1.0, eta=1.0, seed=seed)
        for b in range(4):
            dg = res["diag"][b]
            acc = dg[1:, 4] <= np.minimum(1.0, dg[1:, 3])
            n = int(np.argmin(acc)) if not acc.all() else len(acc)
            assert res["n_accepted"][b] == n
            assert list(res["path"][b][:n]) == list(range(1, n + 1))
            e, kind = int(res["sample"][b, 0]), int(res["sample"][b, 1])
            assert e == n
            assert kind == (0 if n == 8 else 1)
            _, u = oracle.node_uniforms(seed, b, e + 1)
            assert res["sample"][b, 2] == u
            seen.add(n)
    assert len(seen) >= 4


def test_tree_selection_properties():
    w = wl.QWEN7B_TREE
    small = wl.Workload("tree", B=4, Hq=1, Hkv=1, d=64, n_q=12, prefix=1, layers=1, V=64,
                        dtype="f32", z_std=1.0, q_noise_std=0.8, q_noise_uses_T=True, tree=True,
                        tree_nodes_max_depth=4, seed=44)
    inp = wl.accept_inputs(small)
    z, q, tok, par = inp.z.numpy(), inp.q.numpy(), inp.tokens.numpy(), inp.parent.numpy()
    for seed in range(40):
        res = oracle.accept(z, q, tok, par, T=1.0, eta=1.0, seed=seed)
        for b in range(4):
            parent = par[b]
            acc = np.zeros(12, bool)
            dg = res["diag"][b]
            acc[1:] = dg[1:, 4] <= np.minimum(1.0, dg[1:, 3])
            children = [[i for i in range(1, 12) if parent[i] == j] for j in range(12)]
            # brute force over leaves: longest accepted prefix
            best = (-1, None)
            for leaf in range(12):
                if children[leaf]:
                    continue
                nodes = []
                v = leaf
                while v != 0:
                    nodes.append(v)
                    v = parent[v]
                nodes = nodes[::-1]
                L = 0
                while L < len(nodes) and acc[nodes[L]]:
                    L += 1
                if L > best[0]:
                    best = (L, nodes[:L])
            n = res["n_accepted"][b]
            assert n == best[0]
            assert list(res["path"][b][:n]) == best[1]
            assert (res["path"][b][n:] == -1).all()
            e = best[1][-1] if n > 0 else 0
            assert int(res["sample"][b, 0]) == e
            assert int(res["sample"][b, 1]) == (1 if children[e] else 0)
    assert w.tree


def test_single_query_row_is_bonus_draw():
    V = 50
    rng = np.random.default_rng(8)
    z = (rng.standard_normal((1, 1, V)) * 2).astype(np.float32)
    q = sp_softmax(rng.standard_normal((1, 1, V)), axis=-1).astype(np.float32)
    for seed in range(10):
        res = oracle.accept(z, q, np.zeros((1, 1), np.int32), T=0.8, eta=1.0, seed=seed)
        p, _, _ = oracle.row_dists(z[0, 0], q[0, 0], 0.8, 1.0)
        _, u = oracle.node_uniforms(seed, 0, 1)
        c = np.cumsum(p)
        expect = int(np.argmax(c > u * c[-1]))
        assert res["n_accepted"][0] == 0 and res["next_token"][0] == expect


def _garbage_padding(z, q, tok, n_nodes, rng):
    """Rows and tokens past each sequence's node count filled with values that
    would change any result they entered (NaN / inf logits, NaN
    probabilities, a token id far outside the vocabulary)."""
    z, q, tok = z.copy(), q.copy(), tok.copy()
    for b, n in enumerate(n_nodes):
        z[b, n:] = np.where(rng.random(z[b, n:].shape) < 0.5, np.nan, np.inf)
        q[b, n:] = np.nan
        tok[b, n:] = 1 << 30
    return z, q, tok


@pytest.mark.parametrize("tree", [False, True])
def test_ragged_drafts_equal_truncated_batches(tree):
    # Sequence b with n_nodes[b] nodes is the step on its first n_nodes[b]
    # nodes: for every count m, the sequences with m nodes give what a batch
    # with n_q = m gives (same sequence index b, so the same Philox blocks),
    # whatever sits in the padding.
    B, n_q = 6, 10
    w = wl.Workload("ragged", B=B, Hq=1, Hkv=1, d=64, n_q=n_q, prefix=1, layers=1, V=400,
                    dtype="f32", z_std=2.0, q_noise_std=1.0, q_noise_uses_T=True, tree=tree,
                    tree_nodes_max_depth=4, seed=51 if tree else 50)
    inp = wl.accept_inputs(w)
    z, q, tok = inp.z.numpy(), inp.q.numpy(), inp.tokens.numpy()
    par = None if inp.parent is None else inp.parent.numpy()
    n_nodes = np.array([4, n_q, 1, 4, 7, 2], np.int32)
    rng = np.random.default_rng(5)
    zg, qg, tg = _garbage_padding(z, q, tok, n_nodes, rng)
    pg = None
    if par is not None:   # padding parents out of range as well
        pg = par.copy()
        for b, n in enumerate(n_nodes):
            pg[b, n:] = -5
    for seed in range(12):
        res = oracle.accept(zg, qg, tg, pg, T=1.0, eta=1.0, seed=seed, n_nodes=n_nodes)
        for m in sorted(set(n_nodes.tolist())):
            ref = oracle.accept(z[:, :m], q[:, :m], tok[:, :m],
                                None if par is None else par[:, :m], T=1.0, eta=1.0, seed=seed)
            for b in np.nonzero(n_nodes == m)[0]:
                assert res["n_accepted"][b] == ref["n_accepted"][b]
                assert res["next_token"][b] == ref["next_token"][b]
                np.testing.assert_array_equal(res["path"][b, :m], ref["path"][b])
                assert (res["path"][b, m:] == -1).all()
                np.testing.assert_array_equal(res["diag"][b, :m], ref["diag"][b])
                assert (res["diag"][b, m:] == 0).all()
                np.testing.assert_array_equal(res["sample"][b], ref["sample"][b])


def test_ragged_fully_accepted_chain_ends_with_bonus_from_its_last_row():
    # q = p (eta = 0): every ratio is 1 and every draft is accepted, so a
    # chain of m nodes accepts m - 1 drafts and draws the bonus token from p of
    # row m - 1 with u_m, by inverse CDF (computed here with numpy).
    B, n_q, V, T = 4, 9, 60, 0.8
    rng = np.random.default_rng(12)
    z = (rng.standard_normal((B, n_q, V)) * 2).astype(np.float32)
    q = sp_softmax(z.astype(np.float64) / T, axis=-1).astype(np.float32)
    tok = rng.integers(0, V, size=(B, n_q)).astype(np.int32)
    n_nodes = np.array([3, 9, 1, 6], np.int32)
    zg, qg, tg = _garbage_padding(z, q, tok, n_nodes, rng)
    for seed in range(8):
        res = oracle.accept(zg, qg, tg, None, T=T, eta=0.0, seed=seed, n_nodes=n_nodes)
        for b, m in enumerate(n_nodes):
            assert res["n_accepted"][b] == m - 1
            assert list(res["path"][b][:m - 1]) == list(range(1, m))
            assert int(res["sample"][b, 0]) == m - 1 and int(res["sample"][b, 1]) == 0
            p = sp_softmax(z[b, m - 1].astype(np.float64) / T)
            _, u = oracle.node_uniforms(seed, b, m)
            c = np.cumsum(p)
            assert res["next_token"][b] == int(np.argmax(c > u * c[-1]))
