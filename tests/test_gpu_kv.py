"""Parity of the CUDA KV commit with the oracle (GPU; calls the C ABI).

Byte work, so the bar is bit-exact: after rapid_kv_commit every cache byte
equals the oracle's.  Accepted paths come from the oracle's acceptance on
seeded inputs (never from the CUDA path).
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_speculative_gb300 import rapid
from long_context_speculative_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _caches(layers, B, Hkv, cap, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    K = [torch.randn((B, Hkv, cap, d), generator=g).to(dtype) for _ in range(layers)]
    V = [torch.randn((B, Hkv, cap, d), generator=g).to(dtype) for _ in range(layers)]
    return K, V


def _np(ts):
    a = torch.stack(ts)
    if a.dtype == torch.bfloat16:
        return a.view(torch.int16).numpy().copy()
    return a.numpy().copy()


def _commit_both(K, V, P, path, n_acc, table=False):
    Kd = [k.to(DEV) for k in K]
    Vd = [v.to(DEV) for v in V]
    Pd = torch.as_tensor(P, dtype=torch.int32, device=DEV)
    pathd = torch.as_tensor(path, dtype=torch.int32, device=DEV)
    nd = torch.as_tensor(n_acc, dtype=torch.int32, device=DEV)
    if table:
        rapid.rapid_kv_commit(rapid.KVLayerTable(Kd, Vd), None, Pd, pathd, nd)
    else:
        rapid.rapid_kv_commit(Kd, Vd, Pd, pathd, nd)
    torch.cuda.synchronize()
    Ko, Vo = _np(K), _np(V)
    bad = oracle.kv_commit(Ko, Vo, np.asarray(P, np.int32), np.asarray(path, np.int32),
                           np.asarray(n_acc, np.int32))
    return _np([k.cpu() for k in Kd]), _np([v.cpu() for v in Vd]), Ko, Vo, bad


def _random_paths(rng, B, n_q, max_depth=6):
    """Accepted paths: a random tree per sequence, a random leaf, a random prefix of its path."""
    path = np.full((B, n_q), -1, np.int32)
    n_acc = np.zeros(B, np.int32)
    for b in range(B):
        par = wl.random_tree(n_q, max_depth, torch.Generator().manual_seed(int(rng.integers(1 << 30))))
        leaf = int(rng.integers(1, n_q))
        chain = []
        v = leaf
        while v != 0:
            chain.append(v)
            v = int(par[v])
        chain.reverse()
        n = int(rng.integers(0, len(chain) + 1))
        path[b, :n] = chain[:n]
        n_acc[b] = n
    return path, n_acc


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
def test_tree_paths_bit_exact(dtype, d):
    rng = np.random.default_rng(d + (1 if dtype == torch.float32 else 0))
    layers, B, Hkv, cap, n_q = 3, 5, 2, 400, 32
    K, V = _caches(layers, B, Hkv, cap, d, dtype, seed=d)
    P = rng.integers(0, cap - n_q + 1, size=B).astype(np.int32)
    P[0] = 0
    P[1] = cap - n_q            # the speculative rows end at the last cache row
    path, n_acc = _random_paths(rng, B, n_q)
    Kg, Vg, Ko, Vo, bad = _commit_both(K, V, P, path, n_acc, table=(d == 64))
    assert bad == 0
    assert np.array_equal(Kg, Ko) and np.array_equal(Vg, Vo)
    assert rapid.rapid_device_error(True) == 0


def test_chains_and_overlapping_shift():
    layers, B, Hkv, cap, d, n_q = 2, 3, 1, 64, 128, 11
    K, V = _caches(layers, B, Hkv, cap, d, torch.bfloat16, seed=3)
    path = np.full((B, n_q), -1, np.int32)
    path[0, :10] = np.arange(1, 11)          # full chain: nothing moves
    path[1, :3] = [2, 3, 4]                  # every destination is the previous source
    n_acc = np.array([10, 3, 0], np.int32)
    P = np.array([5, 20, 40], np.int32)
    Kg, Vg, Ko, Vo, bad = _commit_both(K, V, P, path, n_acc)
    assert bad == 0
    assert np.array_equal(Kg, Ko) and np.array_equal(Vg, Vo)
    assert np.array_equal(Kg[:, 0], _np(K)[:, 0])   # the chain is untouched


def test_path_from_acceptance():
    # the oracle's acceptance on a seeded tree batch picks the paths
    w = wl.Workload("t", B=4, Hq=8, Hkv=2, d=128, n_q=32, prefix=200, layers=2, V=512,
                    dtype="bf16", z_std=2, q_noise_std=0.5, q_noise_uses_T=True, tree=True,
                    tree_nodes_max_depth=6, seed=77)
    acc = wl.accept_inputs(w)
    ref = oracle.accept(acc.z.numpy(), acc.q.numpy(), acc.tokens.numpy(), acc.parent.numpy(),
                        T=w.T, eta=w.eta, seed=5)
    path = np.where(ref["path"] >= 0, ref["path"], -1).astype(np.int32)
    n_acc = ref["n_accepted"].astype(np.int32)
    K, V = _caches(w.layers, w.B, w.Hkv, 300, w.d, torch.bfloat16, seed=9)
    P = np.array([10, 100, 0, 268], np.int32)
    Kg, Vg, Ko, Vo, bad = _commit_both(K, V, P, path, n_acc)
    assert bad == 0
    assert np.array_equal(Kg, Ko) and np.array_equal(Vg, Vo)


def test_invalid_sequence_is_left_alone_and_flagged():
    layers, B, Hkv, cap, d, n_q = 1, 2, 1, 64, 64, 8
    K, V = _caches(layers, B, Hkv, cap, d, torch.float32, seed=4)
    path = np.full((B, n_q), -1, np.int32)
    path[0, :2] = [1, 3]
    path[1, :2] = [4, 3]                    # not increasing
    n_acc = np.array([2, 2], np.int32)
    P = np.array([5, 5], np.int32)
    rapid.rapid_device_error(True)
    Kg, Vg, Ko, Vo, bad = _commit_both(K, V, P, path, n_acc)
    assert bad == 1
    assert np.array_equal(Kg, Ko) and np.array_equal(Vg, Vo)
    assert rapid.rapid_device_error(True) & 2


def test_advance():
    P = torch.tensor([0, 10, 100, 5], dtype=torch.int32, device=DEV)
    n = torch.tensor([0, 3, 10, 7], dtype=torch.int32, device=DEV)
    rapid.rapid_device_error(True)
    rapid.rapid_kv_advance(P, n, n_q=11, kv_capacity=200)
    torch.cuda.synchronize()
    ref = oracle.kv_advance(np.array([0, 10, 100, 5], np.int32), np.array([0, 3, 10, 7], np.int32))
    assert P.cpu().numpy().tolist() == ref.tolist()
    assert rapid.rapid_device_error(True) == 0
    # n_accepted = n_q is invalid: the length stays, the error bit is set
    P2 = torch.tensor([4], dtype=torch.int32, device=DEV)
    rapid.rapid_kv_advance(P2, torch.tensor([11], dtype=torch.int32, device=DEV), n_q=11,
                           kv_capacity=200)
    torch.cuda.synchronize()
    assert P2.item() == 4
    assert rapid.rapid_device_error(True) & 2
