"""Guard bands around every output and workspace (GPU; calls the C ABI).

Each buffer a call writes is carved out of a larger allocation whose bytes
before and after it hold a fill pattern; after the call (and a second call on
the same buffers) the pattern must be untouched, so that an index slip in a
kernel's stores -- a partial row written one slot too far, a vector store past
the end of a short output -- shows up here at the buffer that took it, not
later as a mismatch somewhere else.  The interiors are checked against the
oracle by the parity tests.
"""
import numpy as np
import pytest
import torch

from long_context_speculative_gb300 import rapid
from long_context_speculative_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096          # bytes on each side (keeps the buffer 256-byte aligned)
FILL = 0xA5


class Guarded:
    def __init__(self, shape, dtype):
        self.nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), FILL, dtype=torch.uint8, device=DEV)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == FILL).all()) and bool((tail == FILL).all())


def _check(*bufs):
    torch.cuda.synchronize()
    assert rapid.rapid_device_error(True) == 0
    for name, g in bufs:
        assert g.intact(), f"guard band of {name} overwritten"


@pytest.mark.parametrize("case", ["tc_chain", "tc_tree_pair", "tc_d64", "simt_f32", "decode"])
def test_verify_attn_outputs_and_workspace(case):
    cfg = {"tc_chain": dict(B=3, Hq=32, Hkv=8, d=128, n_q=11, dtype="bf16", tree=False),
           "tc_tree_pair": dict(B=3, Hq=14, Hkv=2, d=128, n_q=32, dtype="bf16", tree=True),
           "tc_d64": dict(B=2, Hq=32, Hkv=8, d=64, n_q=11, dtype="bf16", tree=False),
           "simt_f32": dict(B=2, Hq=6, Hkv=3, d=128, n_q=4, dtype="f32", tree=False),
           "decode": dict(B=3, Hq=32, Hkv=8, d=128, n_q=1, dtype="bf16", tree=False)}[case]
    w = wl.Workload("t", prefix=5000, prefix_lo=0, layers=1, V=10, z_std=1, q_noise_std=1,
                    q_noise_uses_T=True, tree_nodes_max_depth=6, seed=101, **cfg)
    a = wl.attn_inputs(w, device=DEV)
    B, Hq, n_q, d = a.Q.shape
    cap = a.K.shape[2]
    O = Guarded((B, Hq, n_q, d), a.Q.dtype)
    L = Guarded((B, Hq, n_q), torch.float32)
    nws = rapid.rapid_verify_attn_workspace_size(B, Hq, w.Hkv, d, n_q, cap,
                                                 rapid._dtype_code(a.Q))
    ws = Guarded((nws,), torch.uint8)
    for _ in range(2):
        rapid.rapid_verify_attn(a.Q, a.K, a.V, a.prefix_len, a.mask, 0.0, O.t, L.t, ws.t)
    _check(("O", O), ("LSE", L), ("workspace", ws))
    assert torch.isfinite(O.t.float()).all()


@pytest.mark.parametrize("case", ["chain", "tree", "ragged"])
def test_accept_outputs_and_workspace(case):
    w = wl.QWEN7B_TREE if case == "tree" else wl.LLAMA8B_LAYER_32K
    inp = wl.accept_inputs(w, B=5)
    z, q, tok = inp.z.to(DEV), inp.q.to(DEV), inp.tokens.to(DEV)
    par = None if inp.parent is None else inp.parent.to(DEV)
    B, n_q, V = z.shape
    na, nt = Guarded((B,), torch.int32), Guarded((B,), torch.int32)
    path, diag = Guarded((B, n_q), torch.int32), Guarded((B, n_q, 5), torch.float32)
    ws = Guarded((rapid.rapid_accept_workspace_size(B, n_q, V),), torch.uint8)
    nn = torch.tensor([n_q, 1, 5, 2, n_q], dtype=torch.int32, device=DEV) if case == "ragged" else None
    for seed in range(2):
        if nn is None:
            rapid.rapid_accept(z, q, tok, par, 1.0, 1.0, seed, rapid.RAPID_ACCEPT_TAIL_CLAMP,
                               na.t, nt.t, path.t, diag.t, ws.t)
        else:
            rapid.rapid_accept_ex(z, q, tok, par, nn, 1.0, 1.0, seed,
                                  rapid.RAPID_ACCEPT_TAIL_CLAMP, na.t, nt.t, path.t, diag.t, ws.t)
    _check(("n_accepted", na), ("next_token", nt), ("path", path), ("diag", diag),
           ("workspace", ws))


def test_accept_noalloc_outputs():
    w = wl.LLAMA8B_LAYER_32K
    inp = wl.accept_inputs(w, B=3)
    z, q, tok = inp.z.to(DEV), inp.q.to(DEV), inp.tokens.to(DEV)
    B, n_q, V = z.shape
    na, nt = Guarded((B,), torch.int32), Guarded((B,), torch.int32)
    path, diag = Guarded((B, n_q), torch.int32), Guarded((B, n_q, 5), torch.float32)
    rapid.rapid_accept_noalloc(z, q, tok, None, 1.0, 1.0, 3, rapid.RAPID_ACCEPT_TAIL_CLAMP,
                               na.t, nt.t, path.t, diag.t)
    _check(("n_accepted", na), ("next_token", nt), ("path", path), ("diag", diag))


@pytest.mark.parametrize("rows,V", [(11, 128256), (5, 1000), (200, 4099)])
def test_lm_head_logits(rows, V):
    g = torch.Generator(device=DEV).manual_seed(7)
    H = torch.randn((rows, 512), generator=g, device=DEV).to(torch.bfloat16)
    W = (torch.randn((V, 512), generator=g, device=DEV) / 8).to(torch.bfloat16)
    z = Guarded((rows, V), torch.float32)
    for _ in range(2):
        rapid.rapid_lm_head(H, W, z.t)
    _check(("z", z))


@pytest.mark.parametrize("B", [1, 2])   # 11 rows: the single fused kernel; 22: two launches
def test_lm_head_accept_workspace_and_outputs(B):
    w = wl.LLAMA8B_LAYER_32K
    inp = wl.accept_inputs(w, B=B)
    q, tok = inp.q.to(DEV), inp.tokens.to(DEV)
    B, n_q, V = q.shape
    g = torch.Generator(device=DEV).manual_seed(8)
    H = torch.randn((B * n_q, 256), generator=g, device=DEV).to(torch.bfloat16)
    W = (torch.randn((V, 256), generator=g, device=DEV) * (3 / 16)).to(torch.bfloat16)
    na, nt = Guarded((B,), torch.int32), Guarded((B,), torch.int32)
    path, diag = Guarded((B, n_q), torch.int32), Guarded((B, n_q, 5), torch.float32)
    ws = Guarded((rapid.rapid_lm_head_accept_workspace_size(B, n_q, V),), torch.uint8)
    for seed in range(2):
        rapid.rapid_lm_head_accept(H, W, q, tok, None, 1.0, 1.0, seed,
                                   rapid.RAPID_ACCEPT_TAIL_CLAMP, na.t, nt.t, path.t, diag.t, ws.t)
    _check(("n_accepted", na), ("next_token", nt), ("path", path), ("diag", diag),
           ("workspace", ws))


def test_attn_merge_outputs():
    parts, rows, d = 3, 37, 128
    g = torch.Generator(device=DEV).manual_seed(9)
    Op = torch.randn((parts, rows, d), generator=g, device=DEV).to(torch.bfloat16)
    Lp = torch.randn((parts, rows), generator=g, device=DEV)
    O, L = Guarded((rows, d), torch.bfloat16), Guarded((rows,), torch.float32)
    rapid.rapid_attn_merge(Op, Lp, O.t, L.t)
    _check(("O", O), ("LSE", L))


@pytest.mark.parametrize("B,N", [(1, 240), (3, 37), (2, 1000)])
def test_retrieval_outputs(B, N):
    g = torch.Generator(device=DEV).manual_seed(10)
    qe = torch.randn((B, 1024), generator=g, device=DEV).to(torch.bfloat16)
    ce = torch.randn((B, N, 1024), generator=g, device=DEV).to(torch.bfloat16)
    sc = Guarded((B, N), torch.float32)
    sel = Guarded((B, N), torch.int32)
    ns, ts = Guarded((B,), torch.int32), Guarded((B,), torch.int32)
    ctx = torch.full((B,), N * 512, dtype=torch.int32, device=DEV)
    rapid.rapid_retrieval_scores(qe, ce, sc.t)
    rapid.rapid_retrieval_select(sc.t, ctx, sel.t, ns.t, ts.t, threshold=-1.0)
    _check(("scores", sc), ("selected", sel), ("n_selected", ns), ("tokens_selected", ts))
