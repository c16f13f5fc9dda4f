"""Several verify steps in a row through the C ABI, each checked against the
oracle (GPU).

One step: the n_q speculative K/V rows of every layer are written after the
history, rapid_verify_attn runs on every layer ("LongSpec: Long-Context
Lossless Speculative Decoding with Efficient Drafting and Verification",
section 2.3), rapid_accept decides the accepted path ("RAPID: Long-Context
Inference with Retrieval-Augmented Speculative Decoding", sections 2.1 and
2.4), rapid_kv_commit moves the accepted rows next to the root and
rapid_kv_advance grows the histories.  The oracle runs the same steps on host
copies.  Attention is compared with the attention tolerances, acceptance with
the acceptance rules (counted near-boundary exemptions), and the caches and
history lengths bit for bit after every commit.  Both sides commit the
oracle's accepted path, so an exempted near-tie cannot make them drift apart.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_speculative_gb300 import rapid
from long_context_speculative_gb300 import workloads as wl

from _parity import check_accept, check_attn

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    return wl.bf16_bits(t)


@pytest.mark.parametrize("tree", [False, True])
def test_three_steps_through_the_abi(tree):
    B, Hq, Hkv, d, n_q, layers, V = 2, 8, 2, 128, 6, 2, 3000
    cap = 1600
    g = torch.Generator().manual_seed(2 if tree else 1)
    rng = np.random.default_rng(5 if tree else 4)
    K = [torch.randn((B, Hkv, cap, d), generator=g).to(torch.bfloat16) for _ in range(layers)]
    Vc = [torch.randn((B, Hkv, cap, d), generator=g).to(torch.bfloat16) for _ in range(layers)]
    Kd = [k.to(DEV) for k in K]
    Vd = [v.to(DEV) for v in Vc]
    Ko = np.stack([_bits(k) for k in K])            # the oracle's caches [layers, B, Hkv, cap, d]
    Vo = np.stack([_bits(v) for v in Vc])
    P = np.array([700, 1100], np.int32)
    if tree:
        parents = [wl.random_tree(n_q, 3, torch.Generator().manual_seed(30 + b)) for b in range(B)]
        par = np.array(parents, np.int32)
        par[:, 0] = -1
        mask = np.zeros((B, n_q, n_q), np.uint8)
        for b in range(B):
            for i in range(n_q):
                v = i
                while v >= 0:
                    mask[b, i, v] = 1
                    v = par[b, v] if v > 0 else -1
    else:
        par = None
        mask = None
    mask_d = None if mask is None else torch.from_numpy(mask).to(DEV)
    par_d = None if par is None else torch.from_numpy(par).to(DEV)
    Pd = torch.from_numpy(P.copy()).to(DEV)

    for step in range(3):
        # the step's speculative K/V rows, the same on both sides
        for layer in range(layers):
            for b in range(B):
                sk = torch.randn((Hkv, n_q, d), generator=g).to(torch.bfloat16)
                sv = torch.randn((Hkv, n_q, d), generator=g).to(torch.bfloat16)
                Kd[layer][b, :, P[b]:P[b] + n_q] = sk.to(DEV)
                Vd[layer][b, :, P[b]:P[b] + n_q] = sv.to(DEV)
                Ko[layer, b, :, P[b]:P[b] + n_q] = _bits(sk)
                Vo[layer, b, :, P[b]:P[b] + n_q] = _bits(sv)
        # attention on every layer
        for layer in range(layers):
            Q = torch.randn((B, Hq, n_q, d), generator=g).to(torch.bfloat16)
            O, L = rapid.verify_attn(Q.to(DEV), Kd[layer], Vd[layer], Pd, mask_d)
            torch.cuda.synchronize()
            Or, Lr = oracle.verify_attn(_bits(Q), Ko[layer], Vo[layer], P, mask,
                                        dtype=oracle.DTYPE_BF16)
            check_attn(O.float().cpu().numpy(), L.cpu().numpy(), Or, Lr)
        # acceptance on seeded logits of the step's rows
        z = (torch.randn((B, n_q, V), generator=g) * 2.0).numpy().astype(np.float32)
        x = z + rng.normal(0.0, 1.0, size=z.shape)
        q = np.exp(x - x.max(axis=2, keepdims=True))
        q = (q / q.sum(axis=2, keepdims=True)).astype(np.float32)
        tok = np.zeros((B, n_q), np.int32)
        for b in range(B):
            for i in range(1, n_q):
                j = (i - 1) if par is None else int(par[b, i])
                qj = q[b, j].astype(np.float64)
                tok[b, i] = rng.choice(V, p=qj / qj.sum())
        seed = 1000 + step
        res = rapid.accept(torch.from_numpy(z).to(DEV), torch.from_numpy(q).to(DEV),
                           torch.from_numpy(tok).to(DEV), par_d, T=1.0, eta=1.0, seed=seed)
        torch.cuda.synchronize()
        ref = oracle.accept(z, q, tok, par, T=1.0, eta=1.0, seed=seed)
        gpu = {k: v.cpu().numpy() for k, v in res.items()}
        check_accept(z, q, tok, par, 1.0, 1.0, seed, True, gpu, ref)
        # commit the oracle's path on both sides, then advance
        path = np.where(ref["path"] >= 0, ref["path"], -1).astype(np.int32)
        n_acc = ref["n_accepted"].astype(np.int32)
        rapid.rapid_kv_commit(Kd, Vd, Pd, torch.from_numpy(path).to(DEV),
                              torch.from_numpy(n_acc).to(DEV))
        rapid.rapid_kv_advance(Pd, torch.from_numpy(n_acc).to(DEV), n_q, cap)
        torch.cuda.synchronize()
        assert oracle.kv_commit(Ko, Vo, P, path, n_acc) == 0
        P = oracle.kv_advance(P, n_acc)
        assert np.array_equal(Pd.cpu().numpy(), P)
        for layer in range(layers):
            assert np.array_equal(_bits(Kd[layer]), Ko[layer])
            assert np.array_equal(_bits(Vd[layer]), Vo[layer])
        assert rapid.rapid_device_error(True) == 0
