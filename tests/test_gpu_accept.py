"""Parity of the CUDA acceptance step with the oracle (GPU; calls the C ABI).

Probabilities within 1e-5 relative; decisions, paths and tokens bit-exact
except the counted near-boundary cases described in _parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_speculative_gb300 import rapid
from long_context_speculative_gb300 import workloads as wl

from _parity import check_accept

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(w, T, eta, seed, clamp=True, B=None, inp=None):
    if inp is None:
        inp = wl.accept_inputs(w, T=T, B=B)
    z, q, tok = inp.z, inp.q, inp.tokens
    par = inp.parent
    res = rapid.accept(z.to(DEV), q.to(DEV), tok.to(DEV), None if par is None else par.to(DEV),
                       T=T, eta=eta, seed=seed, tail_clamp=clamp)
    torch.cuda.synchronize()
    gpu = {k: (None if v is None else v.cpu().numpy()) for k, v in res.items()}
    zn, qn, tn = z.numpy(), q.numpy(), tok.numpy()
    pn = None if par is None else par.numpy()
    ref = oracle.accept(zn, qn, tn, pn, T=T, eta=eta, seed=seed, clamp=clamp)
    stats = check_accept(zn, qn, tn, pn, T, eta, seed, clamp, gpu, ref)
    assert rapid.rapid_device_error(True) == 0
    return stats, gpu, ref


@pytest.mark.parametrize("eta", [0.0, 1.0, 10.0])
def test_tiny_config_many_seeds(eta):
    w = wl.TINY
    inp = wl.accept_inputs(w, B=8)
    tot = dict(compared=0, ratio_exempt=0, cdf_exempt=0, clamp_exempt=0)
    seen_n = set()
    for seed in range(25):
        st, gpu, ref = _run(w, 1.0, eta, 0x5EED0000 + seed, inp=inp)
        for k in tot:
            tot[k] += st[k]
        seen_n.update(ref["n_accepted"].tolist())
    assert tot["compared"] >= 190
    assert len(seen_n) >= 2


@pytest.mark.parametrize("T,eta", [(1.0, 1.0), (0.6, 0.0), (0.6, 1.0), (1.0, 5.0)])
def test_llama_vocab_chain(T, eta):
    w = wl.LLAMA8B_LAYER_32K
    inp = wl.accept_inputs(w, T=T, B=2)
    for seed in range(3):
        _run(w, T, eta, 1000 + seed, inp=inp)


def test_eta_zero_gives_phat_equal_p_bitwise():
    w = wl.LLAMA8B_LAYER_32K
    _, gpu, _ = _run(w, 1.0, 0.0, 7, B=1)
    dg = gpu["diag"][0, 1:]
    assert np.array_equal(dg[:, 0], dg[:, 1])


def test_clamp_off():
    w = wl.TINY
    inp = wl.accept_inputs(w, B=4)
    for seed in range(10):
        _run(w, 1.0, 10.0, seed, clamp=False, inp=inp)


def test_tree_qwen_vocab():
    w = wl.QWEN7B_TREE
    inp = wl.accept_inputs(w)
    for seed in range(2):
        _run(w, 1.0, 1.0, 77 + seed, inp=inp)


@pytest.mark.parametrize("T,eta,clamp", [(0.6, 5.0, True), (1.0, 0.0, True), (1.3, 1.0, False)])
def test_tree_temperatures_and_strengths(T, eta, clamp):
    # the tree rule with a sharper and a flatter target, no knowledge transfer
    # (eta = 0: p_hat is p), a strong one, and the tail rule off
    w = wl.Workload("tree", B=4, Hq=1, Hkv=1, d=64, n_q=24, prefix=1, layers=1, V=50021,
                    dtype="f32", z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True, tree=True,
                    tree_nodes_max_depth=5, seed=9)
    inp = wl.accept_inputs(w, T=T)
    for seed in range(3):
        _run(w, T, eta, 300 + seed, clamp=clamp, inp=inp)


def test_small_tree_many_seeds():
    w = wl.Workload("tree", B=6, Hq=1, Hkv=1, d=64, n_q=20, prefix=1, layers=1, V=3001,
                    dtype="f32", z_std=1.5, q_noise_std=0.7, q_noise_uses_T=True, tree=True,
                    tree_nodes_max_depth=5, seed=5)
    inp = wl.accept_inputs(w)
    for seed in range(20):
        _run(w, 1.0, 1.0, seed, inp=inp)


@pytest.mark.parametrize("V", [1, 3, 7, 1000, 1023, 1025, 4097, 65537, 229376])
def test_vocab_sizes_and_unaligned_rows(V):
    w = wl.Workload("v", B=2, Hq=1, Hkv=1, d=64, n_q=4, prefix=1, layers=1, V=V, dtype="f32",
                    z_std=2.0, q_noise_std=1.0, q_noise_uses_T=True, seed=V)
    inp = wl.accept_inputs(w)
    for seed in range(4):
        _run(w, 1.0, 1.0, seed, inp=inp)


def test_single_row_bonus_only():
    w = wl.Workload("v", B=3, Hq=1, Hkv=1, d=64, n_q=1, prefix=1, layers=1, V=5000, dtype="f32",
                    z_std=2.0, q_noise_std=1.0, q_noise_uses_T=True, seed=3)
    st, gpu, ref = _run(w, 0.8, 1.0, 99)
    assert (gpu["n_accepted"] == 0).all()


def test_max_draft_tokens():
    w = wl.Workload("v", B=2, Hq=1, Hkv=1, d=64, n_q=64, prefix=1, layers=1, V=2048, dtype="f32",
                    z_std=1.0, q_noise_std=0.3, q_noise_uses_T=True, seed=4)
    for seed in range(3):
        _run(w, 1.0, 1.0, seed)


def test_batched_rows():
    w = wl.LLAMA8B_LAYER_32K
    _run(w, 1.0, 1.0, 5, B=16)


def test_c_abi_rejects_bad_arguments():
    L = rapid.lib()
    B, n_q, V = 1, 3, 100
    z = torch.zeros((B, n_q, V), device=DEV)
    tok = torch.zeros((B, n_q), dtype=torch.int32, device=DEV)
    o = torch.zeros(B, dtype=torch.int32, device=DEV)
    ws = torch.empty(rapid.rapid_accept_workspace_size(B, n_q, V), dtype=torch.uint8, device=DEV)
    p = lambda t: t.data_ptr()
    args = [p(z), p(z), p(tok), None, B, n_q, V, 1.0, 1.0, 0, 1, p(o), p(o), None, None, p(ws),
            ws.numel(), None]
    assert L.rapid_accept(*args) == 0
    torch.cuda.synchronize()
    for idx, val, code in [(7, 0.0, -1), (7, float("nan"), -1), (8, -1.0, -1), (5, 65, -1),
                           (6, 0, -1), (6, 229377, -1), (10, 2, -1), (16, 4, -3), (0, None, -1)]:
        bad = list(args)
        bad[idx] = val
        assert L.rapid_accept(*bad) == code, (idx, val)


def _garbage_padding(z, q, tok, n_nodes, seed):
    """Rows and tokens past each sequence's node count: NaN / inf logits, NaN
    probabilities and token ids outside the vocabulary (negative and huge)."""
    g = torch.Generator().manual_seed(seed)
    z, q, tok = z.clone(), q.clone(), tok.clone()
    for b, n in enumerate(n_nodes):
        pick = torch.rand(z[b, n:].shape, generator=g) < 0.5
        z[b, n:] = torch.where(pick, torch.tensor(float("nan")), torch.tensor(float("inf")))
        q[b, n:] = float("nan")
        tok[b, n:] = torch.where(torch.rand(tok[b, n:].shape, generator=g) < 0.5,
                                 torch.tensor(-7, dtype=torch.int32),
                                 torch.tensor(1 << 30, dtype=torch.int32))
    return z, q, tok


_RAGGED = {
    "chain": (wl.LLAMA8B_LAYER_32K, [11, 1, 5, 2, 11, 8]),
    "tree": (wl.QWEN7B_TREE, [32, 1, 17, 9]),
    # one real row per sequence: most clusters hold padding rows only
    "chain_roots_only": (wl.LLAMA8B_LAYER_32K, [1] * 20),
    # more rows than clusters, seeded lengths
    "chain_seeded_20": (wl.LLAMA8B_LAYER_32K,
                        np.random.default_rng(8).integers(1, 12, size=20).tolist()),
    # long runs of padding rows between a cluster's real rows: a warp group may
    # skip several padding rows while its first thread is still issuing the
    # previous row's copy (padding rows take no buffer phase)
    "sparse_40": (wl.LLAMA8B_LAYER_32K, ([1] * 9 + [11]) * 4),
}


@pytest.mark.parametrize("case", sorted(_RAGGED))
def test_ragged_drafts_through_rapid_accept_ex(case):
    # drafts of different lengths in one batch: the CUDA path with node counts
    # against the oracle with the same counts, padding full of garbage
    w, counts = _RAGGED[case]
    n_nodes = np.array(counts, np.int32)
    inp = wl.accept_inputs(w, T=1.0, B=len(n_nodes))
    z, q, tok = _garbage_padding(inp.z, inp.q, inp.tokens, n_nodes, seed=3)
    par = inp.parent
    if par is not None:   # padding parents out of range too
        par = par.clone()
        for b, n in enumerate(n_nodes):
            par[b, n:] = torch.tensor([-5, 1000], dtype=torch.int32).repeat(w.n_q)[:w.n_q - n]
    nn_d = torch.from_numpy(n_nodes).to(DEV)
    seen_bonus = 0
    for seed in (11, 12, 13):
        res = rapid.accept(z.to(DEV), q.to(DEV), tok.to(DEV),
                           None if par is None else par.to(DEV), T=1.0, eta=1.0, seed=seed,
                           n_nodes=nn_d)
        torch.cuda.synchronize()
        gpu = {k: v.cpu().numpy() for k, v in res.items()}
        zn, qn, tn = z.numpy(), q.numpy(), tok.numpy()
        pn = None if par is None else par.numpy()
        ref = oracle.accept(zn, qn, tn, pn, T=1.0, eta=1.0, seed=seed, n_nodes=n_nodes)
        stats = check_accept(zn, qn, tn, pn, 1.0, 1.0, seed, True, gpu, ref, n_nodes=n_nodes)
        assert stats["compared"] >= len(n_nodes) - 2
        seen_bonus += int((ref["sample"][:, 1] == 0).sum())
        # a single-node sequence draws its next token from p of the root row
        one = np.nonzero(n_nodes == 1)[0]
        assert (gpu["n_accepted"][one] == 0).all() and (gpu["path"][one] == -1).all()
    assert seen_bonus >= 3 * int((n_nodes == 1).sum())   # the single-node sequences at least
    assert rapid.rapid_device_error(True) == 0


def test_ragged_full_counts_equal_rapid_accept():
    # node counts of n_q everywhere give rapid_accept's results bit for bit
    w = wl.LLAMA8B_LAYER_32K
    inp = wl.accept_inputs(w, T=1.0, B=3)
    z, q, tok = inp.z.to(DEV), inp.q.to(DEV), inp.tokens.to(DEV)
    full = torch.full((3,), w.n_q, dtype=torch.int32, device=DEV)
    a = rapid.accept(z, q, tok, None, T=1.0, eta=1.0, seed=21)
    b = rapid.accept(z, q, tok, None, T=1.0, eta=1.0, seed=21, n_nodes=full)
    torch.cuda.synchronize()
    for k in ("n_accepted", "next_token", "path", "diag"):
        assert torch.equal(a[k], b[k]), k
