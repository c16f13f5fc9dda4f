"""Parity of the CUDA retrieval step with the oracle (GPU; calls the C ABI).

"RAPID: Long-Context Inference with Retrieval-Augmented Speculative Decoding",
section 3.1 (RAG settings).  Scores are floating point: within 2e-5 of the
oracle's double cosine (fp32 sums over at most a few thousand products of
unit-scale values).  The selection is integer work: bit-exact against the
oracle on the same seeded float32 scores (never scores the CUDA path made).
The end-to-end case builds embeddings whose cosines sit on a grid about 1e-3
apart and clear of the threshold, so that the scores' rounding cannot
change the ranking, and compares the kept ids exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from long_context_speculative_gb300 import rapid

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _embeddings(B, N, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, D), generator=g).to(dtype)
    c = torch.randn((B, N, D), generator=g).to(dtype)
    # a few chunks close to the query, one zero vector
    c[:, : min(N, 5)] = (q[:, None, :].float() * 2.0 + 0.1 * c[:, : min(N, 5)].float()).to(dtype)
    c[0, -1] = 0
    return q, c


def _gpu_scores(q, c):
    B, N, D = c.shape
    s = torch.full((B, N), float("nan"), dtype=torch.float32, device=DEV)
    rapid.rapid_retrieval_scores(q.to(DEV), c.to(DEV), s)
    torch.cuda.synchronize()
    return s.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,N,D", [(3, 240, 1024), (3, 301, 136), (3, 9, 8), (3, 1, 4096),
                                   (64, 240, 1024), (2, 1000, 8192)])
def test_scores(dtype, B, N, D):
    # the last two cases give every CTA several tiles, so shared-memory stages are reused
    q, c = _embeddings(B, N, D, dtype, seed=B + N + D)
    got = _gpu_scores(q, c)
    ref = oracle.retrieval_scores(q.float().numpy(), c.float().numpy())
    assert np.abs(got - ref).max() < 2e-5
    if N > 1:
        assert got[0, -1] == 0.0      # the zero vector scores 0


def _select_both(scores, ctx, **kw):
    B, N = scores.shape
    sel = torch.full((B, N), -7, dtype=torch.int32, device=DEV)
    ns = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    ts = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    kg = dict(kw)
    if "chunk" in kg:
        kg["chunk_tokens"] = kg.pop("chunk")
    rapid.rapid_retrieval_select(torch.from_numpy(scores).to(DEV),
                                 torch.from_numpy(ctx.astype(np.int32)).to(DEV), sel, ns, ts, **kg)
    torch.cuda.synchronize()
    ref = oracle.retrieval_select(scores, ctx, **kw)
    return (sel.cpu().numpy(), ns.cpu().numpy(), ts.cpu().numpy()), ref


def _assert_same(got, ref):
    for g, r in zip(got, ref):
        assert np.array_equal(g, r)


@pytest.mark.parametrize("N", [1, 7, 240, 1000, 8192])
def test_select_bit_exact_random(N):
    rng = np.random.default_rng(N)
    B = 6
    scores = rng.uniform(-0.3, 1.0, size=(B, N)).astype(np.float32)
    ctx = rng.integers(0, N * 512 + 1, size=B)
    ctx[0] = N * 512                  # every chunk full, the largest allowed context
    ctx[1] = 0                        # empty context
    ctx[2] = max(1, (N - 1) * 512 + 37)   # short last chunk
    rapid.rapid_device_error(True)
    got, ref = _select_both(scores, ctx)
    _assert_same(got, ref)
    assert rapid.rapid_device_error(True) == 0


@pytest.mark.parametrize("seed", range(4))
def test_select_ties_threshold_and_budgets(seed):
    rng = np.random.default_rng(100 + seed)
    B, N = 8, 600
    # few distinct levels: many exact ties, some exactly at the threshold, -0 and +0
    levels = np.array([-0.0, 0.0, 0.1, 0.29999998, 0.3, 0.3, 0.5, 0.5, 0.7, 0.9], np.float32)
    scores = rng.choice(levels, size=(B, N)).astype(np.float32)
    ctx = rng.integers(1, N * 64 + 1, size=B)
    for kw in (dict(chunk=64, min_tokens=2048, ratio=24, threshold=0.3),
               dict(chunk=64, min_tokens=0, ratio=3, threshold=0.0),
               dict(chunk=50, min_tokens=1000, ratio=1, threshold=-1.0),
               dict(chunk=1, min_tokens=123, ratio=7, threshold=0.5)):
        c = np.minimum(ctx, N * kw["chunk"])
        got, ref = _select_both(scores, c, **kw)
        _assert_same(got, ref)


def test_select_short_last_chunk_after_budget_runs_low():
    # budget 4 x 512 - 400: three full chunks fit, the fourth does not, the
    # 100-token last chunk still does (ranked last)
    scores = np.array([[0.9, 0.8, 0.7, 0.6, 0.5, 0.1]], np.float32)
    ctx = np.array([4 * 512 + 100])
    got, ref = _select_both(scores, ctx, min_tokens=1648)
    _assert_same(got, ref)
    assert got[0][0, :4].tolist() == [0, 1, 2, 4] and got[2][0] == 1636
    # the same with the last chunk below the threshold: not kept
    scores[0, 4] = 0.2
    got, ref = _select_both(scores, ctx, min_tokens=1648)
    _assert_same(got, ref)
    assert got[1][0] == 3


def test_pages_sizes_end_to_end():
    # 120K-token contexts (240 chunks of 512) with 1024-wide bf16 embeddings;
    # cosines placed on a grid about 1e-3 apart and clear of the threshold
    B, N, D = 4, 240, 1024
    rng = np.random.default_rng(11)
    q = rng.standard_normal((B, D))
    cos = np.empty((B, N))
    for b in range(B):
        grid = np.linspace(-0.2, 0.95, 4 * N)
        grid = grid[np.abs(grid - 0.3) > 1e-3]
        cos[b] = rng.permutation(rng.choice(grid, size=N, replace=False))
    u = rng.standard_normal((B, N, D))
    qh = q / np.linalg.norm(q, axis=1, keepdims=True)
    u -= np.einsum("bnd,bd->bn", u, qh)[..., None] * qh[:, None, :]
    u /= np.linalg.norm(u, axis=2, keepdims=True)
    c = cos[..., None] * qh[:, None, :] + np.sqrt(1 - cos**2)[..., None] * u
    c *= rng.uniform(0.5, 3.0, size=(B, N, 1))
    qt = torch.from_numpy(q).to(torch.bfloat16)
    ct = torch.from_numpy(c).to(torch.bfloat16)
    ref_scores = oracle.retrieval_scores(qt.float().numpy(), ct.float().numpy())
    srt = np.sort(ref_scores, axis=1)
    assert np.diff(srt, axis=1).min() > 5e-5 and np.abs(ref_scores - 0.3).min() > 5e-5
    ctx = np.array([122880, 100000, 32768, 5000])
    ref = oracle.retrieval_select(ref_scores.astype(np.float32), ctx)
    s = torch.empty((B, N), dtype=torch.float32, device=DEV)
    sel = torch.empty((B, N), dtype=torch.int32, device=DEV)
    ns = torch.empty((B,), dtype=torch.int32, device=DEV)
    ts = torch.empty((B,), dtype=torch.int32, device=DEV)
    rapid.rapid_retrieval_scores(qt.to(DEV), ct.to(DEV), s)
    rapid.rapid_retrieval_select(s, torch.from_numpy(ctx.astype(np.int32)).to(DEV), sel, ns, ts)
    torch.cuda.synchronize()
    _assert_same((sel.cpu().numpy(), ns.cpu().numpy(), ts.cpu().numpy()), ref)
    assert ts.cpu().numpy()[0] <= 5120


def test_invalid_context_is_flagged_and_selects_nothing():
    N = 16
    scores = np.full((3, N), 0.9, np.float32)
    ctx = torch.tensor([N * 512 + 1, -5, 1000], dtype=torch.int32, device=DEV)
    sel = torch.zeros((3, N), dtype=torch.int32, device=DEV)
    ns = torch.zeros(3, dtype=torch.int32, device=DEV)
    ts = torch.zeros(3, dtype=torch.int32, device=DEV)
    rapid.rapid_device_error(True)
    rapid.rapid_retrieval_select(torch.from_numpy(scores).to(DEV), ctx, sel, ns, ts)
    torch.cuda.synchronize()
    assert ns.cpu().tolist()[:2] == [0, 0] and ts.cpu().tolist()[:2] == [0, 0]
    assert (sel[:2] == -1).all().item()
    assert ns[2].item() == 2          # the valid sequence: both of its chunks fit
    assert rapid.rapid_device_error(True) & 2
