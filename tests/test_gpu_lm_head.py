"""Parity of the CUDA LM-head logits and of the fused logits + acceptance step
with the oracle (GPU; calls the C ABI).

Logits: z = H W^T with bf16 H and W and fp32 accumulation on the tensor
cores.  The bound is the one of an fp32 dot product summed in blocks (16
products per MMA step, then 4096 / 16 accumulations): |z_gpu - z| <=
2e-5 * sum_k |H_k W_k| + 1e-6, checked element by element against the
oracle's double sums; the scale sum |H| |W| is the oracle's product of the
absolute values.

Fused step: the acceptance decisions on the GPU's own logits against the
oracle's acceptance on the oracle's logits (rounded to fp32).  The GPU's
logits deviate by dz (checked against the bound above); a softmax entry moves
by at most 2 dz / T relatively, so the probability tolerance and the
near-boundary bands of the acceptance tests widen to 1e-5 + 2 max|dz| / T.  The draft distribution q and the draft tokens are built
from the oracle's logits, never from the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_speculative_gb300 import rapid

from _parity import check_accept

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _weights(rows, hidden, V, seed, w_std=None):
    g = torch.Generator().manual_seed(seed)
    H = torch.randn((rows, hidden), generator=g).to(torch.bfloat16)
    std = w_std if w_std is not None else 3.0 / np.sqrt(hidden)
    W = (torch.randn((V, hidden), generator=g) * std).to(torch.bfloat16)
    return H, W


def _gpu_logits(H, W):
    z = torch.full((H.shape[0], W.shape[0]), float("nan"), dtype=torch.float32, device=DEV)
    rapid.rapid_lm_head(H.to(DEV), W.to(DEV), z)
    torch.cuda.synchronize()
    return z.cpu().numpy()


def _check_logits(z_gpu, Hf, Wf):
    ref = oracle.lm_head_logits(Hf, Wf)
    scale = oracle.lm_head_logits(np.abs(Hf), np.abs(Wf))
    assert np.isfinite(z_gpu).all()
    err = np.abs(z_gpu - ref)
    bound = 2e-5 * scale + 1e-6
    assert (err <= bound).all(), f"max err {err.max()} (bound there {bound.flat[err.argmax()]})"
    return err.max()


@pytest.mark.parametrize("rows", [1, 11, 16, 17, 40, 100, 176, 256])
def test_logits_row_counts(rows):
    # V = 1000: the last 128-entry tile is ragged (1000 = 7 x 128 + 104)
    H, W = _weights(rows, 256, 1000, seed=rows)
    z = _gpu_logits(H, W)
    _check_logits(z, H.float().numpy(), W.float().numpy())
    assert rapid.rapid_device_error(True) == 0


@pytest.mark.parametrize("hidden,V", [(64, 1), (64, 129), (4096, 513), (8192, 300), (1024, 40000)])
def test_logits_shapes(hidden, V):
    H, W = _weights(11, hidden, V, seed=hidden + V)
    z = _gpu_logits(H, W)
    _check_logits(z, H.float().numpy(), W.float().numpy())


def test_logits_full_llama_head_sampled():
    # 11 verify rows, hidden 4096, the 128256-entry vocabulary (1.05 GB of
    # bf16 weights on the device); the oracle checks a sample of entries.
    rows, hidden, V = 11, 4096, 128256
    g = torch.Generator(device=DEV).manual_seed(5)
    H = torch.randn((rows, hidden), generator=g, device=DEV).to(torch.bfloat16)
    W = (torch.randn((V, hidden), generator=g, device=DEV) * (3.0 / 64)).to(torch.bfloat16)
    z = torch.empty((rows, V), dtype=torch.float32, device=DEV)
    rapid.rapid_lm_head(H, W, z)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    idx = np.unique(np.concatenate([rng.choice(V, 2048, replace=False), np.arange(V - 128, V),
                                    np.arange(128)]))
    Hf = H.float().cpu().numpy()
    Wf = W[torch.from_numpy(idx).to(DEV)].float().cpu().numpy()
    _check_logits(z[:, torch.from_numpy(idx).to(DEV)].cpu().numpy(), Hf, Wf)
    del W
    torch.cuda.empty_cache()


def _draft_from_logits(z, parent, T, seed):
    """q = softmax(z / T + noise) per row; node i's token drawn from q of its parent."""
    B, n_q, V = z.shape
    rng = np.random.default_rng(seed)
    x = z / T + rng.normal(0.0, 1.5, size=z.shape)
    x -= x.max(axis=2, keepdims=True)
    q = np.exp(x)
    q /= q.sum(axis=2, keepdims=True)
    q = q.astype(np.float32)
    tokens = np.zeros((B, n_q), np.int32)
    for b in range(B):
        for i in range(1, n_q):
            j = (i - 1) if parent is None else int(parent[b, i])
            qj = q[b, j].astype(np.float64)
            tokens[b, i] = rng.choice(V, p=qj / qj.sum())
    return q, tokens


def _fused_case(B, n_q, hidden, V, parent, T, eta, seed, clamp=True, n_nodes=None,
                device_key=False):
    H, W = _weights(B * n_q, hidden, V, seed=seed)
    Hf, Wf = H.float().numpy(), W.float().numpy()
    z64 = oracle.lm_head_logits(Hf, Wf)
    z_ref = z64.reshape(B, n_q, V).astype(np.float32)
    q, tokens = _draft_from_logits(z_ref.astype(np.float64), parent, T, seed + 1)
    # the logits the fused call computes (the same product), within their
    # bound; their largest deviation sets how far the probabilities may move
    dz = _check_logits(_gpu_logits(H, W), Hf, Wf)
    band = 1e-5 + 2.0 * dz / T
    ref = oracle.accept(z_ref, q, tokens, parent, T=T, eta=eta, seed=seed + 2, clamp=clamp,
                        n_nodes=n_nodes)
    par_d = None if parent is None else torch.from_numpy(parent.astype(np.int32)).to(DEV)
    dev = lambda a: torch.from_numpy(a).to(DEV)
    if n_nodes is None and not device_key:
        out = rapid.lm_head_accept(H.to(DEV), W.to(DEV), dev(q), dev(tokens), par_d, T=T,
                                   eta=eta, seed=seed + 2, tail_clamp=clamp)
    else:
        out = dict(n_accepted=torch.empty(B, dtype=torch.int32, device=DEV),
                   next_token=torch.empty(B, dtype=torch.int32, device=DEV),
                   path=torch.empty((B, n_q), dtype=torch.int32, device=DEV),
                   diag=torch.empty((B, n_q, 5), dtype=torch.float32, device=DEV))
        ws = torch.empty(rapid.rapid_lm_head_accept_workspace_size(B, n_q, V),
                         dtype=torch.uint8, device=DEV)
        key = (torch.tensor([seed + 2], dtype=torch.int64, device=DEV) if device_key
               else seed + 2)
        rapid.rapid_lm_head_accept_ex(H.to(DEV), W.to(DEV), dev(q), dev(tokens), par_d,
                                      None if n_nodes is None else dev(n_nodes.astype(np.int32)),
                                      T, eta, key, rapid.RAPID_ACCEPT_TAIL_CLAMP if clamp else 0,
                                      out["n_accepted"], out["next_token"], out["path"],
                                      out["diag"], ws)
    torch.cuda.synchronize()
    gpu = {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items()}
    stats = check_accept(z_ref, q, tokens, parent, T, eta, seed + 2, clamp, gpu, ref,
                         prob_rtol=band, exempt=band, n_nodes=n_nodes)
    assert rapid.rapid_device_error(True) == 0
    return stats


def _random_tree(B, n_q, seed):
    rng = np.random.default_rng(seed)
    parent = np.zeros((B, n_q), np.int32)
    parent[:, 0] = -1
    for b in range(B):
        for i in range(1, n_q):
            parent[b, i] = rng.integers(0, i)
    return parent


# Up to 16 rows the fused call is one cooperative kernel: the product, then the
# acceptance step with z kept in shared memory.  Shapes: the Llama-3.1-8B
# vocabulary (one 11-row chain step), the Qwen2.5-7B vocabulary with a 16-node
# tree, a vocabulary smaller than one CTA per SM, eta above the bound of 32,
# the tail rule off, a single query row (bonus draw only).
@pytest.mark.parametrize("B,n_q,hidden,V,tree,T,eta,clamp", [
    (1, 11, 1024, 128256, False, 1.0, 1.0, True),
    (1, 16, 512, 152064, True, 1.0, 1.0, True),
    (2, 8, 512, 50000, False, 0.6, 5.0, True),
    (1, 11, 512, 32000, False, 1.0, 40.0, True),
    (4, 4, 256, 1000, True, 1.0, 1.0, True),
    (2, 6, 256, 20000, False, 1.0, 10.0, False),
    (1, 1, 1024, 128256, False, 1.0, 1.0, True),
    (3, 5, 256, 4100, True, 0.8, 0.0, True),
])
def test_fused_single_kernel_shapes(B, n_q, hidden, V, tree, T, eta, clamp):
    parent = _random_tree(B, n_q, seed=V + n_q) if tree else None
    tot = {}
    for k in range(3):
        st = _fused_case(B, n_q, hidden, V, parent, T, eta, seed=100 * k + B + V % 97,
                         clamp=clamp)
        for key, v in st.items():
            tot[key] = tot.get(key, 0) + v
    assert tot["compared"] >= 2 * B


def test_fused_single_kernel_ragged_and_device_key():
    B, n_q, V = 2, 8, 30000
    parent = _random_tree(B, n_q, seed=5)
    n_nodes = np.array([8, 3], np.int32)
    st = _fused_case(B, n_q, 512, V, parent, 1.0, 1.0, seed=55, n_nodes=n_nodes,
                     device_key=True)
    assert st["compared"] + st["ratio_exempt"] + st["clamp_exempt"] >= 1


@pytest.mark.parametrize("T,eta", [(1.0, 1.0), (0.6, 0.0), (1.0, 5.0)])
def test_fused_chain(T, eta):
    stats = _fused_case(1, 11, 4096, 32000, None, T, eta, seed=40)
    assert stats["compared"] + stats["ratio_exempt"] + stats["clamp_exempt"] >= 1


def test_fused_tree_batch():
    B, n_q = 4, 16
    rng = np.random.default_rng(3)
    parent = np.zeros((B, n_q), np.int32)
    parent[:, 0] = -1
    for b in range(B):
        for i in range(1, n_q):
            parent[b, i] = rng.integers(0, i)
    stats = _fused_case(B, n_q, 1024, 50000, parent, 1.0, 1.0, seed=70)
    assert stats["compared"] >= 2


def test_fused_equals_logits_then_accept():
    # the fused call is exactly rapid_lm_head followed by rapid_accept
    B, n_q, hidden, V = 2, 11, 512, 20000
    H, W = _weights(B * n_q, hidden, V, seed=9)
    Hd, Wd = H.to(DEV), W.to(DEV)
    z_ref = oracle.lm_head_logits(H.float().numpy(), W.float().numpy()).reshape(B, n_q, V)
    q, tokens = _draft_from_logits(z_ref, None, 1.0, 10)
    z = torch.empty((B * n_q, V), dtype=torch.float32, device=DEV)
    rapid.rapid_lm_head(Hd, Wd, z)
    qd, td = torch.from_numpy(q).to(DEV), torch.from_numpy(tokens).to(DEV)
    a = rapid.accept(z.view(B, n_q, V), qd, td, None, T=1.0, eta=1.0, seed=11)
    b = rapid.lm_head_accept(Hd, Wd, qd, td, None, T=1.0, eta=1.0, seed=11)
    torch.cuda.synchronize()
    for k in ("n_accepted", "next_token", "path", "diag"):
        assert torch.equal(a[k], b[k]), k


def test_fused_ex_equals_logits_then_accept_ex():
    # node counts and a device key through the fused call give what rapid_lm_head
    # followed by rapid_accept_ex gives, bit for bit
    B, n_q, hidden, V = 3, 11, 512, 20000
    H, W = _weights(B * n_q, hidden, V, seed=19)
    Hd, Wd = H.to(DEV), W.to(DEV)
    z_ref = oracle.lm_head_logits(H.float().numpy(), W.float().numpy()).reshape(B, n_q, V)
    q, tokens = _draft_from_logits(z_ref, None, 1.0, 20)
    qd, td = torch.from_numpy(q).to(DEV), torch.from_numpy(tokens).to(DEV)
    nn = torch.tensor([11, 4, 1], dtype=torch.int32, device=DEV)
    key = torch.tensor([0x0123_4567_89AB], dtype=torch.int64, device=DEV)
    z = torch.empty((B * n_q, V), dtype=torch.float32, device=DEV)
    rapid.rapid_lm_head(Hd, Wd, z)
    a = rapid.accept(z.view(B, n_q, V), qd, td, None, T=1.0, eta=1.0, seed=key, n_nodes=nn)
    outs = dict(n_accepted=torch.empty(B, dtype=torch.int32, device=DEV),
                next_token=torch.empty(B, dtype=torch.int32, device=DEV),
                path=torch.empty((B, n_q), dtype=torch.int32, device=DEV),
                diag=torch.empty((B, n_q, 5), dtype=torch.float32, device=DEV))
    ws = torch.empty(rapid.rapid_lm_head_accept_workspace_size(B, n_q, V), dtype=torch.uint8,
                     device=DEV)
    rapid.rapid_lm_head_accept_ex(Hd, Wd, qd, td, None, nn, 1.0, 1.0, key,
                                  rapid.RAPID_ACCEPT_TAIL_CLAMP, outs["n_accepted"],
                                  outs["next_token"], outs["path"], outs["diag"], ws)
    torch.cuda.synchronize()
    for k in ("n_accepted", "next_token", "path"):
        assert torch.equal(a[k], outs[k]), k
    real = torch.arange(n_q, device=DEV)[None, :] < nn[:, None]
    assert torch.equal(a["diag"][real], outs["diag"][real])
    assert rapid.rapid_device_error(True) == 0
