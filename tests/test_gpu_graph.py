"""A whole verify step captured once in a CUDA graph and replayed (GPU; calls
the C ABI).

Every quantity that changes from one verify step to the next lives in device
memory: the history lengths (grown in place by rapid_kv_advance), the accepted
paths and counts, the draft lengths, and, through rapid_accept_ex, the
Philox key.  One step — rapid_verify_attn on every layer, the acceptance step,
a bump of the key, rapid_kv_commit and rapid_kv_advance — can therefore be
captured once and replayed for every later step, with the step's new inputs
(including each sequence's draft length) written into the same buffers in
between.  The test runs three steps eagerly (host keys seed, seed + 1,
seed + 2) and three replays of one captured step from the same initial state
and inputs, and asks for identical results: O, LSE, the acceptance outputs,
the caches and the history lengths, bit for bit.  The eager path itself is
checked against the oracle by the decode-loop and acceptance tests.
"""
import pytest
import torch

from long_context_speculative_gb300 import rapid
from long_context_speculative_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"

B, HQ, HKV, D, NQ, LAYERS, V, CAP = 2, 8, 2, 128, 6, 2, 3000, 1600
STEPS = 3
SEED0 = 0x1234_5678_9ABC


def _problem(tree):
    g = torch.Generator().manual_seed(41 if tree else 40)
    K0 = [torch.randn((B, HKV, CAP, D), generator=g).to(torch.bfloat16) for _ in range(LAYERS)]
    V0 = [torch.randn((B, HKV, CAP, D), generator=g).to(torch.bfloat16) for _ in range(LAYERS)]
    P0 = torch.tensor([700, 1100], dtype=torch.int32)
    if tree:
        parents = [wl.random_tree(NQ, 3, g) for _ in range(B)]
    else:
        parents = [wl.chain_parents(NQ) for _ in range(B)]
    parent = torch.tensor(parents, dtype=torch.int32) if tree else None
    mask = torch.stack([wl.ancestor_mask(p) for p in parents]) if tree else None
    steps = []
    for _ in range(STEPS):
        s = dict(
            k=[torch.randn((B, HKV, NQ, D), generator=g).to(torch.bfloat16) for _ in range(LAYERS)],
            v=[torch.randn((B, HKV, NQ, D), generator=g).to(torch.bfloat16) for _ in range(LAYERS)],
            Q=[torch.randn((B, HQ, NQ, D), generator=g).to(torch.bfloat16) for _ in range(LAYERS)],
            z=torch.randn((B, NQ, V), generator=g) * 2.0)
        s["q"] = torch.softmax((s["z"] + torch.randn((B, NQ, V), generator=g)).double(), -1).float()
        tok = torch.zeros((B, NQ), dtype=torch.int32)
        for b in range(B):
            for i in range(1, NQ):
                tok[b, i] = int(torch.multinomial(s["q"][b, parents[b][i]].double(), 1,
                                                  generator=g))
        s["tok"] = tok
        steps.append(s)
    # draft lengths per step: full, then ragged
    counts = [[NQ, NQ], [NQ, 3], [2, NQ - 1]]
    for s, c in zip(steps, counts):
        s["n_nodes"] = torch.tensor(c, dtype=torch.int32)
    return K0, V0, P0, parent, mask, steps


def _write_spec_rows(K, Vc, P_host, s):
    # the step's speculative K/V rows after each history (the model's job)
    for layer in range(LAYERS):
        for b in range(B):
            p = int(P_host[b])
            K[layer][b, :, p:p + NQ] = s["k"][layer][b].to(DEV)
            Vc[layer][b, :, p:p + NQ] = s["v"][layer][b].to(DEV)


def _snapshot(O, L, out, K, Vc, P):
    return dict(O=[o.clone() for o in O], L=[x.clone() for x in L],
                acc={k: v.clone() for k, v in out.items()},
                K=[k.clone() for k in K], V=[v.clone() for v in Vc], P=P.clone())


@pytest.mark.parametrize("tree", [False, True])
def test_captured_step_replays_like_eager_steps(tree):
    K0, V0, P0, parent, mask, steps = _problem(tree)
    par_d = None if parent is None else parent.to(DEV)
    mask_d = None if mask is None else mask.to(DEV)
    flags = rapid.RAPID_ACCEPT_TAIL_CLAMP
    ws_attn = torch.empty(rapid.rapid_verify_attn_workspace_size(B, HQ, HKV, D, NQ, CAP,
                                                                 rapid.RAPID_DTYPE_BF16),
                          dtype=torch.uint8, device=DEV)
    ws_acc = torch.empty(rapid.rapid_accept_workspace_size(B, NQ, V), dtype=torch.uint8,
                         device=DEV)

    def state():
        return ([k.to(DEV) for k in K0], [v.to(DEV) for v in V0], P0.to(DEV))

    def buffers():
        Q = [torch.empty((B, HQ, NQ, D), dtype=torch.bfloat16, device=DEV) for _ in range(LAYERS)]
        O = [torch.empty_like(q) for q in Q]
        L = [torch.empty((B, HQ, NQ), dtype=torch.float32, device=DEV) for _ in range(LAYERS)]
        z = torch.empty((B, NQ, V), dtype=torch.float32, device=DEV)
        out = dict(n_accepted=torch.empty(B, dtype=torch.int32, device=DEV),
                   next_token=torch.empty(B, dtype=torch.int32, device=DEV),
                   path=torch.empty((B, NQ), dtype=torch.int32, device=DEV),
                   diag=torch.empty((B, NQ, 5), dtype=torch.float32, device=DEV))
        tok = torch.empty((B, NQ), dtype=torch.int32, device=DEV)
        nn = torch.empty(B, dtype=torch.int32, device=DEV)
        return Q, O, L, z, torch.empty_like(z), tok, nn, out

    def load_inputs(Q, z, q, tok, nn, s):
        for layer in range(LAYERS):
            Q[layer].copy_(s["Q"][layer])
        z.copy_(s["z"])
        q.copy_(s["q"])
        tok.copy_(s["tok"])
        nn.copy_(s["n_nodes"])

    # eager: three steps, host keys
    K, Vc, P = state()
    table = rapid.KVLayerTable(K, Vc)
    Q, O, L, z, q, tok, nn, out = buffers()
    eager, P_hosts = [], []
    for i, s in enumerate(steps):
        P_host = P.cpu()
        P_hosts.append(P_host)
        _write_spec_rows(K, Vc, P_host, s)
        load_inputs(Q, z, q, tok, nn, s)
        for layer in range(LAYERS):
            rapid.rapid_verify_attn(Q[layer], K[layer], Vc[layer], P, mask_d, 0.0, O[layer],
                                    L[layer], ws_attn)
        rapid.rapid_accept_ex(z, q, tok, par_d, nn, 1.0, 1.0, SEED0 + i, flags,
                              out["n_accepted"], out["next_token"], out["path"], out["diag"],
                              ws_acc)
        table.commit(P, out["path"], out["n_accepted"])
        rapid.rapid_kv_advance(P, out["n_accepted"], NQ, CAP)
        torch.cuda.synchronize()
        eager.append(_snapshot(O, L, out, K, Vc, P))
    assert rapid.rapid_device_error(True) == 0
    # the steps must move rows for the comparison to mean something
    assert sum(int(e["acc"]["n_accepted"].sum()) for e in eager) > 0

    # graph: the same three steps as replays of one capture, key in device memory
    K, Vc, P = state()
    table = rapid.KVLayerTable(K, Vc)
    Q, O, L, z, q, tok, nn, out = buffers()
    seed = torch.tensor([SEED0], dtype=torch.int64, device=DEV)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for layer in range(LAYERS):
            rapid.rapid_verify_attn(Q[layer], K[layer], Vc[layer], P, mask_d, 0.0, O[layer],
                                    L[layer], ws_attn)
        rapid.rapid_accept_ex(z, q, tok, par_d, nn, 1.0, 1.0, seed, flags, out["n_accepted"],
                              out["next_token"], out["path"], out["diag"], ws_acc)
        seed.add_(1)
        table.commit(P, out["path"], out["n_accepted"])
        rapid.rapid_kv_advance(P, out["n_accepted"], NQ, CAP)
    torch.cuda.synchronize()
    # capturing ran nothing
    assert torch.equal(P.cpu(), P0) and int(seed.item()) == SEED0
    for i, s in enumerate(steps):
        assert torch.equal(P.cpu(), P_hosts[i])
        _write_spec_rows(K, Vc, P_hosts[i], s)
        load_inputs(Q, z, q, tok, nn, s)
        graph.replay()
        torch.cuda.synchronize()
        got, want = _snapshot(O, L, out, K, Vc, P), eager[i]
        for layer in range(LAYERS):
            assert torch.equal(got["O"][layer], want["O"][layer]), (i, layer)
            assert torch.equal(got["L"][layer], want["L"][layer]), (i, layer)
            assert torch.equal(got["K"][layer], want["K"][layer]), (i, layer)
            assert torch.equal(got["V"][layer], want["V"][layer]), (i, layer)
        for k in ("n_accepted", "next_token", "path", "diag"):
            assert torch.equal(got["acc"][k], want["acc"][k]), (i, k)
        assert torch.equal(got["P"], want["P"]), i
    assert int(seed.item()) == SEED0 + STEPS
    assert rapid.rapid_device_error(True) == 0


@pytest.mark.parametrize("tree", [False, True])
def test_device_seed_matches_host_seed(tree):
    w = wl.Workload("devseed", B=3, Hq=1, Hkv=1, d=64, n_q=32 if tree else 11, prefix=1,
                    layers=1, V=50000, dtype="f32", z_std=3.0, q_noise_std=1.5,
                    q_noise_uses_T=True, tree=tree, seed=91 if tree else 90)
    inp = wl.accept_inputs(w, T=1.0)
    z, q, tok = inp.z.to(DEV), inp.q.to(DEV), inp.tokens.to(DEV)
    par = None if inp.parent is None else inp.parent.to(DEV)
    # keys with both 32-bit halves in use; the last has the sign bit of int64 set
    for key in (0x0000_0001_0000_0002, 0x7FFF_FFFF_FFFF_FFFF, 0x9E37_79B9_7F4A_7C15):
        host = rapid.accept(z, q, tok, par, T=1.0, eta=1.0, seed=key)
        signed = key - (1 << 64) if key >= (1 << 63) else key
        dev_key = torch.tensor([signed], dtype=torch.int64, device=DEV)
        dev = rapid.accept(z, q, tok, par, T=1.0, eta=1.0, seed=dev_key)
        torch.cuda.synchronize()
        for k in ("n_accepted", "next_token", "path", "diag"):
            assert torch.equal(host[k], dev[k]), (hex(key), k)
    assert rapid.rapid_device_error(True) == 0


def test_accept_ex_rejects_bad_pointers():
    L = rapid.lib()
    z = torch.zeros((1, 2, 100), dtype=torch.float32, device=DEV)
    tok = torch.zeros((1, 2), dtype=torch.int32, device=DEV)
    o = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(rapid.rapid_accept_workspace_size(1, 2, 100), dtype=torch.uint8, device=DEV)
    seed = torch.zeros(2, dtype=torch.int64, device=DEV)
    nn = torch.ones(2, dtype=torch.int32, device=DEV)

    def call(n_nodes, key_dev):
        return L.rapid_accept_ex(z.data_ptr(), z.data_ptr(), tok.data_ptr(), None, n_nodes, 1, 2,
                                 100, 1.0, 1.0, 5, key_dev, 1, o.data_ptr(), o.data_ptr(), None,
                                 None, ws.data_ptr(), ws.numel(), None)

    assert call(None, seed.data_ptr() + 4) == rapid.RAPID_EINVAL
    assert call(nn.data_ptr() + 2, None) == rapid.RAPID_EINVAL
    assert call(None, None) == rapid.RAPID_OK
    assert call(nn.data_ptr(), seed.data_ptr()) == rapid.RAPID_OK
    torch.cuda.synchronize()
    assert rapid.rapid_device_error(True) == 0
