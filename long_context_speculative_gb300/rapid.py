"""Thin Python binding of librapid.so (argument marshalling only).

Every step of the verification path runs in the CUDA kernels behind the C
ABI declared in include/rapid.h; this module only turns torch tensors into
device pointers, sizes workspaces and passes the current CUDA stream.  There
is no CPU or PyTorch fallback: if librapid.so is missing or cannot be loaded,
every call raises.
"""
import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "librapid.so")

RAPID_OK = 0
RAPID_EINVAL = -1
RAPID_ECUDA = -2
RAPID_ENOMEM = -3
RAPID_ETIMEOUT = -4
RAPID_EUNSUPPORTED = -5
RAPID_DTYPE_F32 = 0
RAPID_DTYPE_BF16 = 1
RAPID_ACCEPT_TAIL_CLAMP = 1
RAPID_MAX_NQ = 64
RAPID_MAX_VOCAB = 229376
RAPID_COMMIT_MAX_LAYERS = 128
RAPID_RETRIEVAL_MAX_CHUNKS = 8192
RAPID_LM_HEAD_MAX_ROWS = 256
RAPID_NOALLOC_MAX_NODES = 4096

_lib = None


class RapidError(RuntimeError):
    pass


def lib() -> ctypes.CDLL:
    """Load librapid.so (built by __graft_entry__.build()); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RapidError(f"librapid.so is not built ({LIB_PATH} missing); "
                         "run `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, u32, u64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                       ctypes.c_float, ctypes.c_uint32, ctypes.c_uint64,
                                       ctypes.c_size_t)
    L.rapid_verify_attn_workspace_size.argtypes = [i32, i32, i32, i32, i32, i64, i32]
    L.rapid_verify_attn_workspace_size.restype = sz
    L.rapid_verify_attn.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i64, vp, vp, f32,
                                    vp, vp, vp, sz, vp]
    L.rapid_verify_attn.restype = i32
    L.rapid_attn_merge.argtypes = [vp, vp, i32, i32, i64, i32, vp, vp, vp]
    L.rapid_attn_merge.restype = i32
    L.rapid_accept_workspace_size.argtypes = [i32, i32, i32]
    L.rapid_accept_workspace_size.restype = sz
    L.rapid_accept.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, f32, u64, u32, vp, vp, vp, vp,
                               vp, sz, vp]
    L.rapid_accept.restype = i32
    L.rapid_accept_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, f32, f32, u64, vp, u32, vp,
                                  vp, vp, vp, vp, sz, vp]
    L.rapid_accept_ex.restype = i32
    L.rapid_status_string.argtypes = [i32]
    L.rapid_status_string.restype = ctypes.c_char_p
    L.rapid_version.argtypes = []
    L.rapid_version.restype = i32
    L.rapid_device_error.argtypes = [i32]
    L.rapid_device_error.restype = i32
    L.rapid_device_error_info.argtypes = [vp, i32]
    L.rapid_device_error_info.restype = i32
    L.rapid_stream_status.argtypes = [vp, i32]
    L.rapid_stream_status.restype = i32
    L.rapid_wait_selftest.argtypes = [u64, vp]
    L.rapid_wait_selftest.restype = i32
    L.rapid_accept_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, f32, u64, u32, vp, vp,
                                       vp, vp, vp]
    L.rapid_accept_noalloc.restype = i32
    L.rapid_kv_commit.argtypes = [vp, vp, i32, i32, i32, i32, i32, i64, i32, vp, vp, vp, vp]
    L.rapid_kv_commit.restype = i32
    L.rapid_kv_advance.argtypes = [vp, vp, i32, i32, i64, vp]
    L.rapid_kv_advance.restype = i32
    L.rapid_retrieval_scores.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp]
    L.rapid_retrieval_scores.restype = i32
    L.rapid_retrieval_select.argtypes = [vp, vp, i32, i32, i32, f32, i32, i32, vp, vp, vp, vp]
    L.rapid_retrieval_select.restype = i32
    L.rapid_lm_head.argtypes = [vp, vp, i32, i32, i32, vp, vp]
    L.rapid_lm_head.restype = i32
    L.rapid_lm_head_accept_workspace_size.argtypes = [i32, i32, i32]
    L.rapid_lm_head_accept_workspace_size.restype = ctypes.c_size_t
    L.rapid_lm_head_accept.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, i32, f32, f32, u64, u32,
                                       vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    L.rapid_lm_head_accept.restype = i32
    L.rapid_lm_head_accept_ex.argtypes = [vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, f32, f32,
                                          u64, vp, u32, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    L.rapid_lm_head_accept_ex.restype = i32
    _lib = L
    return L


def _check(status: int, what: str):
    if status != RAPID_OK:
        msg = lib().rapid_status_string(status).decode()
        raise RapidError(f"{what} failed: {msg} ({status})")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise RapidError("librapid works on CUDA tensors only (no CPU path)")
        if t is not None and not t.is_contiguous():
            raise RapidError("librapid needs contiguous tensors")


def _need_same_device(*ts):
    """Every tensor on the current CUDA device (the launches go to it)."""
    cur = torch.cuda.current_device()
    for t in ts:
        if t is not None and t.device.index != cur:
            raise RapidError(f"tensor on {t.device}, but the current device is cuda:{cur}")


def _need(t, dtype, shape, name):
    if t is not None and (t.dtype != dtype or tuple(t.shape) != tuple(shape)):
        raise RapidError(f"{name} must be a {dtype} tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)}")


def _check_accept_tensors(z_target, q_draft, draft_tokens, parent, n_accepted, next_token, path,
                          diag, n_nodes=None):
    """The sizes the kernels will index by: z and q float32 [B, n_q, V]; tokens,
    parents and the path int32 [B, n_q]; counts int32 [B]; diag float32 [B, n_q, 5]."""
    if z_target is None or z_target.dim() != 3:
        raise RapidError("z_target must be a [B, n_q, V] tensor")
    B, n_q, V = z_target.shape
    _need(z_target, torch.float32, (B, n_q, V), "z_target")
    _need(q_draft, torch.float32, (B, n_q, V), "q_draft")
    _need(draft_tokens, torch.int32, (B, n_q), "draft_tokens")
    _need(parent, torch.int32, (B, n_q), "parent")
    _need(n_accepted, torch.int32, (B,), "n_accepted")
    _need(next_token, torch.int32, (B,), "next_token")
    _need(path, torch.int32, (B, n_q), "path")
    _need(diag, torch.float32, (B, n_q, 5), "diag")
    _need(n_nodes, torch.int32, (B,), "n_nodes")
    _need_same_device(z_target, q_draft, draft_tokens, parent, n_accepted, next_token, path, diag,
                      n_nodes)
    return B, n_q, V


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return RAPID_DTYPE_BF16
    if t.dtype == torch.float32:
        return RAPID_DTYPE_F32
    raise RapidError(f"unsupported dtype {t.dtype}")


# ---------------------------------------------------------------------------
# C-ABI mirrors (same names, same argument order; tensors in place of pointers)
# ---------------------------------------------------------------------------

def rapid_verify_attn_workspace_size(B, Hq, Hkv, d, n_q, kv_capacity, dtype) -> int:
    return int(lib().rapid_verify_attn_workspace_size(B, Hq, Hkv, d, n_q, kv_capacity, dtype))


def rapid_verify_attn(Q, Kcache, Vcache, prefix_len, spec_mask, softmax_scale, O, LSE,
                      workspace, stream=None):
    """Launch verify attention; shapes are read from the tensors."""
    _need_cuda(Q, Kcache, Vcache, prefix_len, spec_mask, O, LSE, workspace)
    B, Hq, n_q, d = Q.shape
    Hkv, cap = Kcache.shape[1], Kcache.shape[2]
    st = lib().rapid_verify_attn(_ptr(Q), _ptr(Kcache), _ptr(Vcache), _dtype_code(Q), B, Hq, Hkv,
                                 d, n_q, cap, _ptr(prefix_len), _ptr(spec_mask),
                                 float(softmax_scale), _ptr(O), _ptr(LSE), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "rapid_verify_attn")


def rapid_attn_merge(O_parts, LSE_parts, O, LSE, stream=None):
    """Log-sum-exp merge of n_parts attention results: O_parts [n_parts, ..., d] (bf16 or
    fp32), LSE_parts [n_parts, ...] float32 -> O [..., d], LSE [...]."""
    _need_cuda(O_parts, LSE_parts, O, LSE)
    n_parts, d = O_parts.shape[0], O_parts.shape[-1]
    rows = LSE_parts[0].numel()
    if (LSE_parts.dtype != torch.float32 or LSE.dtype != torch.float32 or O.dtype != O_parts.dtype
            or O_parts.numel() != n_parts * rows * d or O.numel() != rows * d
            or LSE.numel() != rows):
        raise RapidError("rapid_attn_merge: mismatched shapes or dtypes")
    st = lib().rapid_attn_merge(_ptr(O_parts), _ptr(LSE_parts), _dtype_code(O_parts), n_parts,
                                rows, d, _ptr(O), _ptr(LSE), _stream(stream))
    _check(st, "rapid_attn_merge")


def rapid_accept_workspace_size(B, n_q, V) -> int:
    return int(lib().rapid_accept_workspace_size(B, n_q, V))


def rapid_accept(z_target, q_draft, draft_tokens, parent, T, eta, philox_seed, flags,
                 n_accepted, next_token, path, diag, workspace, stream=None):
    _need_cuda(z_target, q_draft, draft_tokens, parent, n_accepted, next_token, path, diag,
               workspace)
    B, n_q, V = _check_accept_tensors(z_target, q_draft, draft_tokens, parent, n_accepted,
                                      next_token, path, diag)
    st = lib().rapid_accept(_ptr(z_target), _ptr(q_draft), _ptr(draft_tokens), _ptr(parent), B,
                            n_q, V, float(T), float(eta), int(philox_seed) & ((1 << 64) - 1),
                            int(flags), _ptr(n_accepted), _ptr(next_token), _ptr(path),
                            _ptr(diag), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "rapid_accept")


def rapid_accept_ex(z_target, q_draft, draft_tokens, parent, n_nodes, T, eta, philox_seed,
                    flags, n_accepted, next_token, path, diag, workspace, stream=None):
    """rapid_accept with optional per-sequence node counts n_nodes (int32 [B] CUDA tensor or
    None) and a Philox key that is either an int or a one-element 64-bit integer CUDA tensor
    read by the kernels when they run."""
    _need_cuda(z_target, q_draft, draft_tokens, parent, n_nodes, n_accepted, next_token, path,
               diag, workspace)
    B, n_q, V = _check_accept_tensors(z_target, q_draft, draft_tokens, parent, n_accepted,
                                      next_token, path, diag, n_nodes)
    if isinstance(philox_seed, torch.Tensor):
        _need_cuda(philox_seed)
        if philox_seed.dtype not in (torch.int64, torch.uint64) or philox_seed.numel() != 1:
            raise RapidError("a device philox_seed must be a one-element 64-bit integer tensor")
        key, key_dev = 0, _ptr(philox_seed)
    else:
        key, key_dev = int(philox_seed) & ((1 << 64) - 1), None
    st = lib().rapid_accept_ex(_ptr(z_target), _ptr(q_draft), _ptr(draft_tokens), _ptr(parent),
                               _ptr(n_nodes), B, n_q, V, float(T), float(eta), key, key_dev,
                               int(flags), _ptr(n_accepted), _ptr(next_token), _ptr(path),
                               _ptr(diag), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "rapid_accept_ex")


def rapid_accept_noalloc(z_target, q_draft, draft_tokens, parent, T, eta, philox_seed, flags,
                         n_accepted, next_token, path, diag, stream=None):
    """rapid_accept with the library's static scratch instead of a workspace."""
    _need_cuda(z_target, q_draft, draft_tokens, parent, n_accepted, next_token, path, diag)
    B, n_q, V = _check_accept_tensors(z_target, q_draft, draft_tokens, parent, n_accepted,
                                      next_token, path, diag)
    st = lib().rapid_accept_noalloc(_ptr(z_target), _ptr(q_draft), _ptr(draft_tokens),
                                    _ptr(parent), B, n_q, V, float(T), float(eta),
                                    int(philox_seed) & ((1 << 64) - 1), int(flags),
                                    _ptr(n_accepted), _ptr(next_token), _ptr(path), _ptr(diag),
                                    _stream(stream))
    _check(st, "rapid_accept_noalloc")


def rapid_lm_head(hidden, W_lm, z, stream=None):
    """Logits z [rows, V] (fp32) of hidden [rows, hidden_dim] against W_lm [V, hidden_dim] (bf16)."""
    _need_cuda(hidden, W_lm, z)
    rows, hd = hidden.shape
    V = W_lm.shape[0]
    _need(hidden, torch.bfloat16, (rows, hd), "hidden")
    _need(W_lm, torch.bfloat16, (V, hd), "W_lm")
    _need(z, torch.float32, (rows, V), "z")
    _need_same_device(hidden, W_lm, z)
    st = lib().rapid_lm_head(_ptr(hidden), _ptr(W_lm), rows, hd, V, _ptr(z), _stream(stream))
    _check(st, "rapid_lm_head")


def rapid_lm_head_accept_workspace_size(B, n_q, V):
    return int(lib().rapid_lm_head_accept_workspace_size(B, n_q, V))


def rapid_lm_head_accept(hidden, W_lm, q_draft, draft_tokens, parent, T, eta, philox_seed, flags,
                         n_accepted, next_token, path, diag, workspace, stream=None):
    """rapid_accept on the logits of hidden [B*n_q, hidden_dim] against W_lm [V, hidden_dim]."""
    _need_cuda(hidden, W_lm, q_draft, draft_tokens, parent, n_accepted, next_token, path, diag,
               workspace)
    B, n_q, V = _check_accept_tensors(q_draft, q_draft, draft_tokens, parent, n_accepted,
                                      next_token, path, diag)
    _need(hidden, torch.bfloat16, (B * n_q, hidden.shape[-1]), "hidden")
    _need(W_lm, torch.bfloat16, (V, hidden.shape[-1]), "W_lm")
    _need_same_device(hidden, W_lm, workspace)
    st = lib().rapid_lm_head_accept(_ptr(hidden), _ptr(W_lm), hidden.shape[1], _ptr(q_draft),
                                    _ptr(draft_tokens), _ptr(parent), B, n_q, V, float(T),
                                    float(eta), int(philox_seed) & ((1 << 64) - 1), int(flags),
                                    _ptr(n_accepted), _ptr(next_token), _ptr(path), _ptr(diag),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    _check(st, "rapid_lm_head_accept")


def rapid_lm_head_accept_ex(hidden, W_lm, q_draft, draft_tokens, parent, n_nodes, T, eta,
                            philox_seed, flags, n_accepted, next_token, path, diag, workspace,
                            stream=None):
    """rapid_lm_head_accept with rapid_accept_ex's node counts and device Philox key
    (philox_seed: an int, or a one-element 64-bit integer CUDA tensor)."""
    _need_cuda(hidden, W_lm, q_draft, draft_tokens, parent, n_nodes, n_accepted, next_token,
               path, diag, workspace)
    B, n_q, V = _check_accept_tensors(q_draft, q_draft, draft_tokens, parent, n_accepted,
                                      next_token, path, diag, n_nodes)
    _need(hidden, torch.bfloat16, (B * n_q, hidden.shape[-1]), "hidden")
    _need(W_lm, torch.bfloat16, (V, hidden.shape[-1]), "W_lm")
    _need_same_device(hidden, W_lm, workspace)
    if isinstance(philox_seed, torch.Tensor):
        _need_cuda(philox_seed)
        if philox_seed.dtype not in (torch.int64, torch.uint64) or philox_seed.numel() != 1:
            raise RapidError("a device philox_seed must be a one-element 64-bit integer tensor")
        key, key_dev = 0, _ptr(philox_seed)
    else:
        key, key_dev = int(philox_seed) & ((1 << 64) - 1), None
    st = lib().rapid_lm_head_accept_ex(_ptr(hidden), _ptr(W_lm), hidden.shape[1], _ptr(q_draft),
                                       _ptr(draft_tokens), _ptr(parent), _ptr(n_nodes), B, n_q,
                                       V, float(T), float(eta), key, key_dev, int(flags),
                                       _ptr(n_accepted), _ptr(next_token), _ptr(path),
                                       _ptr(diag), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    _check(st, "rapid_lm_head_accept_ex")


class KVLayerTable:
    """The device addresses of every layer's K and V cache, checked and packed
    once, for repeated rapid_kv_commit calls on the same caches (the per-call
    packing of a few dozen pointers otherwise costs tens of microseconds of
    host time)."""

    def __init__(self, K_layers, V_layers):
        if len(K_layers) != len(V_layers) or not K_layers:
            raise RapidError("rapid_kv_commit needs matching, non-empty K and V layer lists")
        if len(K_layers) > RAPID_COMMIT_MAX_LAYERS:
            raise RapidError(f"at most {RAPID_COMMIT_MAX_LAYERS} layers per call")
        _need_cuda(*K_layers, *V_layers)
        shape, dtype = tuple(K_layers[0].shape), K_layers[0].dtype
        for t in list(K_layers) + list(V_layers):
            if tuple(t.shape) != shape or t.dtype != dtype:
                raise RapidError("every layer's K and V cache needs the same shape and dtype")
        self.layers = len(K_layers)
        self.B, self.Hkv, self.cap, self.d = shape
        self.dtype = _dtype_code(K_layers[0])
        self._k = (ctypes.c_void_p * self.layers)(*[t.data_ptr() for t in K_layers])
        self._v = (ctypes.c_void_p * self.layers)(*[t.data_ptr() for t in V_layers])
        self._keep = (list(K_layers), list(V_layers))   # the caches outlive the table

    def commit(self, prefix_len, path, n_accepted, stream=None):
        st = lib().rapid_kv_commit(ctypes.cast(self._k, ctypes.c_void_p),
                                   ctypes.cast(self._v, ctypes.c_void_p), self.layers, self.dtype,
                                   self.B, self.Hkv, self.d, self.cap, path.shape[1],
                                   _ptr(prefix_len), _ptr(path), _ptr(n_accepted), _stream(stream))
        _check(st, "rapid_kv_commit")


def rapid_kv_commit(K_layers, V_layers, prefix_len, path, n_accepted, stream=None):
    """Move the accepted speculative K/V rows of every layer next to the root.

    K_layers, V_layers: sequences of [B, Hkv, kv_capacity, d] caches (one per
    layer), or K_layers a KVLayerTable and V_layers None; prefix_len [B],
    path [B, n_q], n_accepted [B] int32 on the device."""
    _need_cuda(prefix_len, path, n_accepted)
    table = K_layers if isinstance(K_layers, KVLayerTable) else KVLayerTable(K_layers, V_layers)
    table.commit(prefix_len, path, n_accepted, stream)


def rapid_kv_advance(prefix_len, n_accepted, n_q, kv_capacity, stream=None):
    """prefix_len += 1 + n_accepted (device, in place)."""
    _need_cuda(prefix_len, n_accepted)
    st = lib().rapid_kv_advance(_ptr(prefix_len), _ptr(n_accepted), prefix_len.shape[0], n_q,
                                kv_capacity, _stream(stream))
    _check(st, "rapid_kv_advance")


def rapid_retrieval_scores(query, chunks, scores, stream=None):
    """Cosine similarities scores [B, N] of chunks [B, N, D] with query [B, D]."""
    _need_cuda(query, chunks, scores)
    B, N, D = chunks.shape
    st = lib().rapid_retrieval_scores(_ptr(query), _ptr(chunks), _dtype_code(chunks), B, N, D,
                                      _ptr(scores), _stream(stream))
    _check(st, "rapid_retrieval_scores")


def rapid_retrieval_select(scores, context_tokens, selected, n_selected, tokens_selected,
                           chunk_tokens=512, threshold=0.3, min_tokens=4096, ratio=24, stream=None):
    """Kept chunk ids (ascending, then -1) per sequence under the RAG budget."""
    _need_cuda(scores, context_tokens, selected, n_selected, tokens_selected)
    B, N = scores.shape
    st = lib().rapid_retrieval_select(_ptr(scores), _ptr(context_tokens), B, N, chunk_tokens,
                                      float(threshold), min_tokens, ratio, _ptr(selected),
                                      _ptr(n_selected), _ptr(tokens_selected), _stream(stream))
    _check(st, "rapid_retrieval_select")


def rapid_device_error(clear: bool = True) -> int:
    return int(lib().rapid_device_error(1 if clear else 0))


def rapid_device_error_info(clear: bool = True):
    words = (ctypes.c_uint32 * 8)()
    if lib().rapid_device_error_info(ctypes.cast(words, ctypes.c_void_p), 1 if clear else 0) != 0:
        raise RapidError("could not read the device error record")
    return list(words)


def rapid_stream_status(stream=None, clear: bool = True) -> int:
    """Synchronise the stream and return RAPID_OK, RAPID_ETIMEOUT (a bounded wait
    inside a kernel gave up), RAPID_EINVAL (a bad device-side input) or RAPID_ECUDA."""
    return int(lib().rapid_stream_status(_stream(stream), 1 if clear else 0))


def rapid_wait_selftest(limit_ns: int, stream=None):
    """Launch the bounded-wait self-test kernel (its wait gives up after limit_ns)."""
    _check(lib().rapid_wait_selftest(int(limit_ns), _stream(stream)), "rapid_wait_selftest")


def rapid_version() -> int:
    return int(lib().rapid_version())


# ---------------------------------------------------------------------------
# Convenience wrappers that allocate outputs and workspaces with torch
# ---------------------------------------------------------------------------

def verify_attn(Q, K, V, prefix_len, spec_mask=None, softmax_scale=0.0, out=None, lse=None,
                workspace=None, stream=None):
    """O [B,Hq,n_q,d] (dtype of Q) and LSE [B,Hq,n_q] float32."""
    B, Hq, n_q, d = Q.shape
    Hkv, cap = K.shape[1], K.shape[2]
    if out is None:
        out = torch.empty_like(Q)
    if lse is None:
        lse = torch.empty((B, Hq, n_q), dtype=torch.float32, device=Q.device)
    if workspace is None:
        nbytes = rapid_verify_attn_workspace_size(B, Hq, Hkv, d, n_q, cap, _dtype_code(Q))
        if nbytes == 0:
            raise RapidError("unsupported verify_attn shape")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=Q.device)
    rapid_verify_attn(Q, K, V, prefix_len, spec_mask, softmax_scale, out, lse, workspace, stream)
    return out, lse


def accept(z, q, tokens, parent=None, T=1.0, eta=1.0, seed=0, tail_clamp=True, want_path=True,
           want_diag=True, workspace=None, stream=None, n_nodes=None):
    """Dict of device tensors n_accepted [B], next_token [B], path [B,n_q], diag [B,n_q,5].

    seed: the Philox key as an int, or a one-element int64 CUDA tensor that the kernels read
    when they run.  n_nodes: None, or int32 [B] node counts of drafts shorter than n_q.
    Either one goes through rapid_accept_ex."""
    B, n_q, V = z.shape
    dev = z.device
    n_acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, n_q), dtype=torch.int32, device=dev) if want_path else None
    diag = torch.empty((B, n_q, 5), dtype=torch.float32, device=dev) if want_diag else None
    if workspace is None:
        nbytes = rapid_accept_workspace_size(B, n_q, V)
        if nbytes == 0:
            raise RapidError("unsupported accept shape")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flags = RAPID_ACCEPT_TAIL_CLAMP if tail_clamp else 0
    if isinstance(seed, torch.Tensor) or n_nodes is not None:
        rapid_accept_ex(z, q, tokens, parent, n_nodes, T, eta, seed, flags, n_acc, nxt, path,
                        diag, workspace, stream)
    else:
        rapid_accept(z, q, tokens, parent, T, eta, seed, flags, n_acc, nxt, path, diag,
                     workspace, stream)
    return dict(n_accepted=n_acc, next_token=nxt, path=path, diag=diag)


def lm_head_accept(hidden, W_lm, q, tokens, parent=None, T=1.0, eta=1.0, seed=0, tail_clamp=True,
                   want_path=True, want_diag=True, workspace=None, stream=None):
    """accept() on the logits of the verify rows' hidden states [B*n_q, hidden_dim]."""
    B, n_q, V = q.shape
    dev = q.device
    n_acc = torch.empty(B, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    path = torch.empty((B, n_q), dtype=torch.int32, device=dev) if want_path else None
    diag = torch.empty((B, n_q, 5), dtype=torch.float32, device=dev) if want_diag else None
    if workspace is None:
        nbytes = rapid_lm_head_accept_workspace_size(B, n_q, V)
        if nbytes == 0:
            raise RapidError("unsupported lm_head_accept shape")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flags = RAPID_ACCEPT_TAIL_CLAMP if tail_clamp else 0
    rapid_lm_head_accept(hidden, W_lm, q, tokens, parent, T, eta, seed, flags, n_acc, nxt, path,
                         diag, workspace, stream)
    return dict(n_accepted=n_acc, next_token=nxt, path=path, diag=diag)
