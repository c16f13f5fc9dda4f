"""Seeded synthetic inputs of the verification step (no method arithmetic here).

The shapes follow the model families the verification step is quoted on:
Llama-3.1-8B-shaped (32 query / 8 KV heads, head_dim 128, vocab 128256),
Llama-3.1-70B-shaped (64 / 8 heads, 80 layers), Qwen2.5-7B-shaped token trees
(28 / 4 heads, vocab 152064) and one tiny fp32 case small enough for the
double-precision oracle.  The 120K-token context with gamma = 10 drafts stands
in for the long-context efficiency workload of the RAPID experiments (about
120K input tokens, up to 1K generated; "RAPID: Long-Context Inference with
Retrieval-Augmented Speculative Decoding", section 3 / efficiency setup).

Only random draws and shapes live here.  The draft probabilities q are made
as softmax(z/T + noise), which is part of the input recipe, not of the method.
Both the CUDA path's tests and the oracle's tests take their inputs from this
module.
"""
from dataclasses import dataclass, field
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    n_q: int
    prefix: int               # history rows (for ragged batches: the upper end)
    layers: int
    V: int
    dtype: str                # "bf16" or "f32"
    z_std: float
    q_noise_std: float
    q_noise_uses_T: bool      # q = softmax(z/T + n) if True else softmax(z + n)
    T: float = 1.0
    eta: float = 1.0
    tree: bool = False
    tree_nodes_max_depth: int = 6
    prefix_lo: Optional[int] = None   # ragged prefixes U[prefix_lo, prefix]
    q_scale: float = 1.0      # Q ~ N(0, 1) * q_scale
    seed: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def capacity(self) -> int:
        # Room for the speculative rows behind the longest history, rounded up
        # to 16 rows so every head's slab stays 16-byte aligned for any d.
        need = self.prefix + self.n_q
        return (need + 15) // 16 * 16


TINY = Workload("tiny_1k_fp32", B=1, Hq=4, Hkv=1, d=64, n_q=5, prefix=1024, layers=1, V=1000,
                dtype="f32", z_std=2.0, q_noise_std=1.0, q_noise_uses_T=False, T=1.0, eta=1.0,
                q_scale=1.0 / 8.0, seed=1001)
LLAMA8B_LAYER_32K = Workload("llama3.1-8b_layer_32k", B=1, Hq=32, Hkv=8, d=128, n_q=11,
                             prefix=32768, layers=1, V=128256, dtype="bf16", z_std=3.0,
                             q_noise_std=1.5, q_noise_uses_T=True, T=1.0, eta=1.0, seed=1002)
LLAMA8B_120K = Workload("llama3.1-8b_32layers_120k", B=1, Hq=32, Hkv=8, d=128, n_q=11,
                        prefix=122880, layers=32, V=128256, dtype="bf16", z_std=3.0,
                        q_noise_std=1.5, q_noise_uses_T=True, T=1.0, eta=1.0, seed=1003)
LLAMA8B_1LAYER_120K = Workload("llama3.1-8b_1layer_120k", B=1, Hq=32, Hkv=8, d=128, n_q=11,
                               prefix=122880, layers=1, V=128256, dtype="bf16", z_std=3.0,
                               q_noise_std=1.5, q_noise_uses_T=True, T=1.0, eta=1.0, seed=1006)
LLAMA70B_128K = Workload("llama3.1-70b_80layers_128k", B=1, Hq=64, Hkv=8, d=128, n_q=11,
                         prefix=131072, layers=80, V=128256, dtype="bf16", z_std=3.0,
                         q_noise_std=1.5, q_noise_uses_T=True, T=1.0, eta=1.0, seed=1004)
QWEN7B_TREE = Workload("qwen2.5-7b_tree32_28layers", B=4, Hq=28, Hkv=4, d=128, n_q=32,
                       prefix=98304, prefix_lo=32768, layers=28, V=152064, dtype="bf16",
                       z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True, T=1.0, eta=1.0,
                       tree=True, seed=1005)

QWEN7B_TREE_1LAYER = Workload("qwen2.5-7b_tree32_1layer", B=4, Hq=28, Hkv=4, d=128, n_q=32,
                              prefix=98304, prefix_lo=32768, layers=1, V=152064, dtype="bf16",
                              z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True, T=1.0, eta=1.0,
                              tree=True, seed=1005)

# single-query decode attention over the same 120K cache (one query row per
# query head: the draft-side / plain decode shape of the split-KV pass)
LLAMA8B_DECODE_120K = Workload("llama3.1-8b_decode_32layers_120k", B=1, Hq=32, Hkv=8, d=128,
                               n_q=1, prefix=122880, layers=32, V=128256, dtype="bf16",
                               z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True, T=1.0, eta=1.0,
                               seed=1007)

# head dimension 64 (a Llama-3.2-1B-shaped target: 32 query / 8 KV heads, 16 layers)
LLAMA1B_D64_120K = Workload("llama3.2-1b_d64_16layers_120k", B=1, Hq=32, Hkv=8, d=64, n_q=11,
                            prefix=122880, layers=16, V=128256, dtype="bf16", z_std=3.0,
                            q_noise_std=1.5, q_noise_uses_T=True, T=1.0, eta=1.0, seed=1008)

ALL = [TINY, LLAMA8B_LAYER_32K, LLAMA8B_120K, LLAMA8B_1LAYER_120K, LLAMA70B_128K, QWEN7B_TREE,
       QWEN7B_TREE_1LAYER, LLAMA8B_DECODE_120K, LLAMA1B_D64_120K]


def gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def torch_dtype(name: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def prefix_lengths(w: Workload, seed: int) -> torch.Tensor:
    """int32 [B]: the history length of every sequence."""
    if w.prefix_lo is None:
        return torch.full((w.B,), w.prefix, dtype=torch.int32)
    g = gen(seed + 17)
    return torch.randint(w.prefix_lo, w.prefix + 1, (w.B,), generator=g, dtype=torch.int64).to(
        torch.int32)


def random_tree(n_nodes: int, max_depth: int, g: torch.Generator) -> List[int]:
    """Parent pointers of a random token tree: node 0 is the root (depth 1);
    node i >= 1 hangs under a uniformly drawn earlier node of depth < max_depth."""
    parent = [-1]
    depth = [1]
    for i in range(1, n_nodes):
        allowed = [j for j in range(i) if depth[j] < max_depth]
        pick = allowed[int(torch.randint(len(allowed), (1,), generator=g))]
        parent.append(pick)
        depth.append(depth[pick] + 1)
    return parent


def chain_parents(n_nodes: int) -> List[int]:
    return [-1] + list(range(n_nodes - 1))


def ancestor_mask(parent: List[int]) -> torch.Tensor:
    """uint8 [n, n]: mask[i][j] = 1 iff node j is node i or one of its ancestors."""
    n = len(parent)
    m = torch.zeros((n, n), dtype=torch.uint8)
    for i in range(n):
        v = i
        while v >= 0:
            m[i, v] = 1
            v = parent[v]
    return m


@dataclass
class AttnInputs:
    Q: torch.Tensor           # [B, Hq, n_q, d]
    K: torch.Tensor           # [B, Hkv, cap, d]
    V: torch.Tensor           # [B, Hkv, cap, d]
    prefix_len: torch.Tensor  # int32 [B]
    mask: Optional[torch.Tensor]  # uint8 [B, n_q, n_q] or None (chain)
    parents: List[List[int]] = field(default_factory=list)


def tile_signs(rows: int, seed: int, tile: int = 64) -> torch.Tensor:
    """float32 [rows]: +1 or -1 per run of ``tile`` consecutive cache rows, half
    of the runs of each sign in a seeded random order."""
    n = (rows + tile - 1) // tile
    s = torch.ones(n)
    s[torch.randperm(n, generator=gen(seed))[: n // 2]] = -1.0
    return s.repeat_interleave(tile)[:rows]


def attn_inputs(w: Workload, layer: int = 0, device="cpu", prefix_override=None,
                needle: bool = False, capacity: Optional[int] = None,
                v_offset: float = 0.0, needle_gain: float = 4.0) -> AttnInputs:
    """K, V ~ N(0,1); Q ~ N(0,1) * q_scale.  With ``needle`` 16 history rows of
    every KV head get K = needle_gain * (mean query direction of the group), so
    a handful of rows dominate the output (a gain of 8 keeps them dominant
    over a 120K-row history).  With ``v_offset`` = c every V row j gets
    c * s(j) added to all its entries, s(j) = +-1 per 64-row run of the cache
    (tile_signs): the output then carries about c / (history / 64) of every
    run, so a run of keys read twice or not at all moves it by that much."""
    seed = w.seed * 1000 + layer
    dt = torch_dtype(w.dtype)
    cap = capacity if capacity is not None else w.capacity
    if prefix_override is not None:
        pl = torch.as_tensor(prefix_override, dtype=torch.int32).reshape(w.B)
    else:
        pl = prefix_lengths(w, w.seed)
    gd = gen(seed, device)
    K = torch.randn((w.B, w.Hkv, cap, w.d), generator=gd, device=device, dtype=torch.float32)
    K = K.to(dt)
    V = torch.randn((w.B, w.Hkv, cap, w.d), generator=gd, device=device, dtype=torch.float32)
    if v_offset:
        V += (v_offset * tile_signs(cap, seed + 4)).to(device)[None, None, :, None]
    V = V.to(dt)
    gc = gen(seed + 1)
    Q = (torch.randn((w.B, w.Hq, w.n_q, w.d), generator=gc) * w.q_scale).to(dt).to(device)
    parents = []
    mask = None
    gt = gen(seed + 2)
    if w.tree:
        ms = []
        for _ in range(w.B):
            par = random_tree(w.n_q, w.tree_nodes_max_depth, gt)
            parents.append(par)
            ms.append(ancestor_mask(par))
        mask = torch.stack(ms).to(device)
    else:
        parents = [chain_parents(w.n_q) for _ in range(w.B)]
    if needle:
        gn = gen(seed + 3)
        for b in range(w.B):
            P = int(pl[b])
            for g_ in range(w.Hkv):
                qdir = Q[b, g_ * w.G:(g_ + 1) * w.G].float().mean(dim=(0, 1)).to(device)
                qdir = qdir / (qdir.norm() + 1e-6) * (w.d ** 0.5)
                rows = torch.randint(0, max(P, 1), (16,), generator=gn)
                if P > 0:
                    K[b, g_, rows.to(device)] = (needle_gain * qdir).to(dt)
    return AttnInputs(Q=Q, K=K, V=V, prefix_len=pl.to(device), mask=mask, parents=parents)


@dataclass
class AcceptInputs:
    z: torch.Tensor           # float32 [B, n_q, V]
    q: torch.Tensor           # float32 [B, n_q, V]
    tokens: torch.Tensor      # int32 [B, n_q]
    parent: Optional[torch.Tensor]  # int32 [B, n_q] or None (chain)


def accept_inputs(w: Workload, T: Optional[float] = None, seed_offset: int = 0, B=None,
                  parents: Optional[List[List[int]]] = None, device="cpu") -> AcceptInputs:
    """z ~ N(0, z_std^2); q = softmax(z/T + N(0, q_noise_std^2)) (or z + noise);
    draft token of node i drawn from q of its parent's row."""
    T = w.T if T is None else T
    B = w.B if B is None else B
    g = gen(w.seed * 7919 + 5 + seed_offset)
    z = torch.randn((B, w.n_q, w.V), generator=g) * w.z_std
    noise = torch.randn((B, w.n_q, w.V), generator=g) * w.q_noise_std
    base = z / T if w.q_noise_uses_T else z
    q = torch.softmax((base + noise).double(), dim=-1).float()
    if parents is None:
        if w.tree:
            gt = gen(w.seed * 7919 + 11 + seed_offset)
            parents = [random_tree(w.n_q, w.tree_nodes_max_depth, gt) for _ in range(B)]
        else:
            parents = [chain_parents(w.n_q) for _ in range(B)]
    tokens = torch.zeros((B, w.n_q), dtype=torch.int32)
    for b in range(B):
        for i in range(1, w.n_q):
            row = parents[b][i]
            tokens[b, i] = int(torch.multinomial(q[b, row].double(), 1, generator=g))
    parent = None
    if w.tree:
        parent = torch.tensor(parents, dtype=torch.int32)
        parent[:, 0] = -1
    return AcceptInputs(z=z.to(device), q=q.to(device), tokens=tokens.to(device),
                        parent=None if parent is None else parent.to(device))


def bf16_bits(t: torch.Tensor):
    """numpy uint16 bit patterns of a bf16 tensor (for the oracle's bf16 input)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
