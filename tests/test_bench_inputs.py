"""CPU checks of the benchmark's input builders (no GPU).

The 128-sequence acceptance batch is generated on the device with the
distributions of workloads.accept_inputs; here the same builder runs on the
CPU and its output is checked for what the acceptance step assumes: q rows
are distributions, draft tokens are in the vocabulary, node 0 has no token,
tree parents point to earlier nodes and the root has none.
"""
import torch

import bench
from long_context_speculative_gb300 import workloads as wl


def _check(w, B):
    z, q, tok, par = bench._device_accept_inputs(w, B, "cpu")
    assert z.shape == q.shape == (B, w.n_q, w.V) and tok.shape == (B, w.n_q)
    assert torch.isfinite(z).all() and (q >= 0).all()
    torch.testing.assert_close(q.sum(-1).double(), torch.ones((B, w.n_q), dtype=torch.float64),
                               rtol=0, atol=1e-5)
    assert tok.dtype == torch.int32 and (tok[:, 0] == 0).all()
    assert ((tok >= 0) & (tok < w.V)).all()
    if w.tree:
        assert par is not None and par.dtype == torch.int32 and (par[:, 0] == -1).all()
        i = torch.arange(1, w.n_q)
        assert ((par[:, 1:] >= 0) & (par[:, 1:] < i)).all()
    else:
        assert par is None
    return z, q, tok


def test_chain_batch_on_cpu():
    w = wl.Workload("t", B=1, Hq=1, Hkv=1, d=64, n_q=11, prefix=1, layers=1, V=500, dtype="f32",
                    z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True, seed=5)
    z, q, tok = _check(w, 6)
    # each draft token is likely under its parent's q (drawn from it): its mean
    # probability is far above the uniform 1 / V
    picked = torch.gather(q[:, :-1], 2, tok[:, 1:, None].long()).mean()
    assert picked > 5.0 / w.V


def test_tree_batch_on_cpu():
    w = wl.Workload("t", B=1, Hq=1, Hkv=1, d=64, n_q=16, prefix=1, layers=1, V=300, dtype="f32",
                    z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True, tree=True,
                    tree_nodes_max_depth=4, seed=6)
    _check(w, 4)
