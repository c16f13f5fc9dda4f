"""The log-sum-exp merge of separately computed attention parts, and verify
attention on shards of the key range (GPU; calls the C ABI).

"LongSpec: Long-Context Lossless Speculative Decoding with Efficient Drafting
and Verification", section 2.3: the parts of hybrid tree attention are
combined through their log-sum-exp.  rapid_attn_merge does that for any
number of parts computed elsewhere; merging the shards of a history split by
key range (the speculative rows visible in one shard only, hidden from the
others by an all-zero mask) must give the unsplit attention.  A query that
sees no key at all gets O = 0 and LSE = -inf, as the oracle's definition
gives.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_speculative_gb300 import rapid
from long_context_speculative_gb300 import workloads as wl

from _parity import check_attn

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bits(t):
    return wl.bf16_bits(t)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("n_parts", [1, 3, 11])
def test_merge_matches_oracle(dtype, d, n_parts):
    g = torch.Generator().manual_seed(7 * n_parts + d)
    rows = 333
    O_parts = torch.randn((n_parts, rows, d), generator=g).to(dtype)
    L_parts = torch.randn((n_parts, rows), generator=g) * 4.0
    L_parts[torch.rand((n_parts, rows), generator=g) < 0.3] = -float("inf")
    L_parts[:, 5] = -float("inf")                 # a row no part saw
    O_parts[:, 5] = float("nan")                  # whose O is never read
    O = torch.empty((rows, d), dtype=dtype, device=DEV)
    L = torch.empty(rows, dtype=torch.float32, device=DEV)
    rapid.rapid_attn_merge(O_parts.to(DEV), L_parts.to(DEV), O, L)
    torch.cuda.synchronize()
    Oref, Lref = oracle.lse_merge(O_parts.float().nan_to_num(0.0).numpy(), L_parts.numpy())
    Og, Lg = O.float().cpu().numpy(), L.cpu().numpy()
    fin = np.isfinite(Lref)
    assert (np.isneginf(Lg) == ~fin).all()
    assert np.abs(Lg[fin] - Lref[fin]).max() <= 1e-5
    # fp32: the fp32 sums; bf16: plus the output's rounding (2^-8 relative)
    tol = 1e-5 if dtype == torch.float32 else 1e-2
    assert np.isfinite(Og).all() and np.abs(Og - Oref).max() <= tol
    assert (Og[~fin] == 0).all()


def _shard_caches(K, V, P, n_q, cuts):
    """Per shard k: caches holding history rows [cuts[k], cuts[k+1]) of each
    sequence, then its n_q speculative rows; the shard's prefix lengths."""
    B = K.shape[0]
    out = []
    for k in range(len(cuts) - 1):
        Kk, Vk = torch.zeros_like(K), torch.zeros_like(V)
        pk = torch.zeros(B, dtype=torch.int32)
        for b in range(B):
            lo, hi = min(cuts[k], int(P[b])), min(cuts[k + 1], int(P[b]))
            n = hi - lo
            Kk[b, :, :n] = K[b, :, lo:hi]
            Vk[b, :, :n] = V[b, :, lo:hi]
            Kk[b, :, n:n + n_q] = K[b, :, int(P[b]):int(P[b]) + n_q]
            Vk[b, :, n:n + n_q] = V[b, :, int(P[b]):int(P[b]) + n_q]
            pk[b] = n
        out.append((Kk, Vk, pk))
    return out


@pytest.mark.parametrize("case", ["bf16_d128_chain", "bf16_d128_tree_wide", "bf16_d64_chain",
                                  "f32_d64_chain"])
def test_key_shards_merge_to_unsplit_attention(case):
    dtype = torch.bfloat16 if case.startswith("bf16") else torch.float32
    d = 128 if "d128" in case else 64
    tree = "tree" in case
    B, Hkv = 2, 2
    G, n_q = (4, 20) if "wide" in case else (4, 6)   # 80 or 24 group rows
    Hq, cap = G * Hkv, 3000
    g = torch.Generator().manual_seed({"bf16_d128_chain": 11, "bf16_d128_tree_wide": 12,
                                       "bf16_d64_chain": 14, "f32_d64_chain": 13}[case])
    Q = torch.randn((B, Hq, n_q, d), generator=g).to(dtype)
    K = torch.randn((B, Hkv, cap, d), generator=g).to(dtype)
    V = torch.randn((B, Hkv, cap, d), generator=g).to(dtype)
    P = torch.tensor([2500, 1210], dtype=torch.int32)
    if tree:
        parents = [wl.random_tree(n_q, 4, wl.gen(60 + b)) for b in range(B)]
        mask = torch.stack([wl.ancestor_mask(p) for p in parents])
    else:
        mask = torch.stack([torch.tril(torch.ones((n_q, n_q), dtype=torch.uint8))] * B)
    # shards: a long one, an empty one, one past sequence 1's history, the rest
    cuts = [0, 1300, 1300, 2000, cap]
    shards = _shard_caches(K, V, P, n_q, cuts)
    zero = torch.zeros_like(mask).to(DEV)
    Os, Ls = [], []
    for k, (Kk, Vk, pk) in enumerate(shards):
        m = mask.to(DEV) if k == len(shards) - 1 else zero
        O, L = rapid.verify_attn(Q.to(DEV), Kk.to(DEV), Vk.to(DEV), pk.to(DEV), m)
        Os.append(O)
        Ls.append(L)
    O = torch.empty_like(Os[0])
    L = torch.empty_like(Ls[0])
    rapid.rapid_attn_merge(torch.stack(Os), torch.stack(Ls), O, L)
    torch.cuda.synchronize()
    # the empty shard saw nothing
    assert torch.isneginf(Ls[1]).all() and (Os[1] == 0).all()
    if dtype == torch.bfloat16:
        Or, Lr = oracle.verify_attn(_bits(Q), _bits(K), _bits(V), P.numpy(), mask.numpy(),
                                    dtype=oracle.DTYPE_BF16)
    else:
        Or, Lr = oracle.verify_attn(Q.numpy(), K.numpy(), V.numpy(), P.numpy(), mask.numpy())
    check_attn(O.float().cpu().numpy(), L.cpu().numpy(), Or, Lr)
    assert rapid.rapid_device_error(True) == 0


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.bfloat16, 64),
                                     (torch.float32, 64)])
def test_query_that_sees_no_key(dtype, d):
    # empty history and mask rows that hide every speculative row from some
    # queries: those get O = 0 and LSE = -inf; the other rows match the oracle
    B, Hq, Hkv, n_q, cap = 2, 4, 2, 5, 64
    g = torch.Generator().manual_seed(3)
    Q = torch.randn((B, Hq, n_q, d), generator=g).to(dtype)
    K = torch.randn((B, Hkv, cap, d), generator=g).to(dtype)
    V = torch.randn((B, Hkv, cap, d), generator=g).to(dtype)
    P = torch.tensor([0, 17], dtype=torch.int32)
    mask = torch.stack([torch.tril(torch.ones((n_q, n_q), dtype=torch.uint8))] * B)
    mask[0, 1] = 0          # sequence 0, query 1: nothing visible at all
    mask[1, 2] = 0          # sequence 1, query 2: history only
    O, L = rapid.verify_attn(Q.to(DEV), K.to(DEV), V.to(DEV), P.to(DEV), mask.to(DEV))
    torch.cuda.synchronize()
    Og, Lg = O.float().cpu().numpy(), L.cpu().numpy()
    if dtype == torch.bfloat16:
        Or, Lr = oracle.verify_attn(_bits(Q), _bits(K), _bits(V), P.numpy(), mask.numpy(),
                                    dtype=oracle.DTYPE_BF16)
    else:
        Or, Lr = oracle.verify_attn(Q.numpy(), K.numpy(), V.numpy(), P.numpy(), mask.numpy())
    assert np.isneginf(Lr[0, :, 1]).all() and np.isneginf(Lg[0, :, 1]).all()
    assert (Og[0, :, 1] == 0).all()
    keep = np.ones(Lr.shape, bool)
    keep[0, :, 1] = False
    check_attn(Og[keep], Lg[keep], Or[keep], Lr[keep])
    assert rapid.rapid_device_error(True) == 0


def test_merge_rejects_bad_arguments():
    Lb = rapid.lib()
    O = torch.zeros((2, 4, 128), dtype=torch.bfloat16, device=DEV)
    L = torch.zeros((2, 4), dtype=torch.float32, device=DEV)
    out = torch.zeros((4, 128), dtype=torch.bfloat16, device=DEV)
    lo = torch.zeros(4, dtype=torch.float32, device=DEV)
    p = lambda t: t.data_ptr()
    good = [p(O), p(L), rapid.RAPID_DTYPE_BF16, 2, 4, 128, p(out), p(lo), None]
    assert Lb.rapid_attn_merge(*good) == rapid.RAPID_OK
    torch.cuda.synchronize()
    for idx, val in [(0, None), (1, None), (2, 7), (3, 0), (4, 0), (5, 96), (6, None),
                     (7, None), (0, p(O) + 8), (6, p(out) + 2)]:
        bad = list(good)
        bad[idx] = val
        assert Lb.rapid_attn_merge(*bad) == rapid.RAPID_EINVAL, (idx, val)
