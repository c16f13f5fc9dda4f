"""TEST INFRASTRUCTURE: Python face of the double-precision CPU oracle.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline and
reference legs may import this package.  The product library
(``long_context_speculative_gb300``) never imports it.

Every function here only marshals numpy arrays into ``liboracle.so`` (built
from ``rapid_oracle.cpp``); the arithmetic lives in that C++ file, which cites
the passages it follows:

* attention: "LongSpec: Long-Context Lossless Speculative Decoding with
  Efficient Drafting and Verification", section 2.3 (hybrid tree attention);
  ``verify_attn`` is the plain definition, ``verify_attn_split`` the
  history-pieces + speculative-piece form merged by log-sum-exp.
* acceptance: "RAPID: Long-Context Inference with Retrieval-Augmented
  Speculative Decoding" (blog summary), sections 2.1 and 2.4.
* random numbers: Philox4x32-10 (Salmon et al., SC'11).
* KV commit after acceptance: the accepted path's speculative rows join the
  history after the root, in path order (``kv_commit``, ``kv_advance``).
* retrieval for the draft's compressed context: "RAPID ..." section 3.1, RAG
  settings (``retrieval_scores``, ``retrieval_select``).
* target logits from the shared LM head: "LongSpec ..." section 2.1
  (``lm_head_logits``).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_vp = ctypes.c_void_p

DTYPE_F32 = 0
DTYPE_BF16 = 1


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_philox4x32_10.argtypes = [_u32p, _u32p, _u32p]
        L.orc_node_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, _dp, _dp]
        attn_common = [_vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                       ctypes.c_int, ctypes.c_int, ctypes.c_int64, _i32p, _u8p, ctypes.c_double]
        L.orc_verify_attn.argtypes = attn_common + [_dp, _dp, ctypes.c_int]
        L.orc_verify_attn_rows.argtypes = attn_common + [_i32p, ctypes.c_int, _dp, _dp, ctypes.c_int]
        L.orc_verify_attn_split.argtypes = attn_common + [_i64p, ctypes.c_int, _dp, _dp, ctypes.c_int]
        L.orc_row_dists.argtypes = [_fp, _fp, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                    ctypes.c_int, _dp, _dp, _dp]
        L.orc_residual_weights.argtypes = [_dp, _dp, _fp, ctypes.c_int, _dp]
        L.orc_sample_inverse_cdf.argtypes = [_dp, ctypes.c_int, ctypes.c_double]
        L.orc_sample_inverse_cdf.restype = ctypes.c_int
        L.orc_kd_loss.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_double]
        L.orc_kd_loss.restype = ctypes.c_double
        L.orc_kd_grad.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_double, _dp]
        L.orc_distilled_logits.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_double,
                                           ctypes.c_double, _dp]
        L.orc_lse_merge.argtypes = [_dp, _dp, ctypes.c_int, ctypes.c_int64, ctypes.c_int, _dp, _dp]
        L.orc_accept.argtypes = [_fp, _fp, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int,
                                 ctypes.c_double, ctypes.c_double, ctypes.c_uint64, ctypes.c_int,
                                 _i32p, _i32p, _i32p, _dp, _dp, ctypes.c_int]
        L.orc_kv_commit.argtypes = [_u8p, _u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i32p, _i32p, _i32p]
        L.orc_kv_commit.restype = ctypes.c_int
        L.orc_kv_advance.argtypes = [_i32p, _i32p, ctypes.c_int]
        L.orc_retrieval_scores.argtypes = [_fp, _fp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp]
        L.orc_retrieval_select.argtypes = [_fp, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_float, ctypes.c_int, ctypes.c_int, _i32p,
                                           _i32p, _i32p]
        L.orc_lm_head_logits.argtypes = [_fp, _fp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp,
                                          ctypes.c_int]
        L.orc_first_token_hist.argtypes = [_fp, _fp, ctypes.c_int, ctypes.c_double,
                                           ctypes.c_double, ctypes.c_int, ctypes.c_uint64,
                                           ctypes.c_int64, _i64p, ctypes.c_int]
        _lib = L
    return _lib


def _ptr(a, typ):
    return a.ctypes.data_as(typ)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Random numbers
# --------------------------------------------------------------------------

def philox4x32_10(ctr, key):
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_ptr(c, _u32p), _ptr(k, _u32p), _ptr(out, _u32p))
    return out


def node_uniforms(seed: int, b: int, i: int):
    r = ctypes.c_double()
    u = ctypes.c_double()
    lib().orc_node_uniforms(seed, b, i, ctypes.byref(r), ctypes.byref(u))
    return r.value, u.value


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def _kv_args(Q, K, V, dtype):
    """Q/K/V as raw buffers: float32 arrays, or bf16 bit patterns as uint16."""
    if dtype == DTYPE_F32:
        arrs = [_c(x, np.float32) for x in (Q, K, V)]
    else:
        arrs = [_c(x, np.uint16) for x in (Q, K, V)]
    return arrs


def verify_attn(Q, K, V, prefix_len, mask=None, scale=None, dtype=DTYPE_F32, nthreads=None):
    """O [B,Hq,n_q,d], LSE [B,Hq,n_q] (float64) by the definition of attention.

    Q [B,Hq,n_q,d], K/V [B,Hkv,cap,d]; dtype DTYPE_BF16 takes uint16 bit patterns.
    """
    B, Hq, n_q, d = Q.shape
    Hkv, cap = K.shape[1], K.shape[2]
    q, k, v = _kv_args(Q, K, V, dtype)
    pl = _c(prefix_len, np.int32)
    m = None if mask is None else _c(mask, np.uint8)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    O = np.zeros((B, Hq, n_q, d), np.float64)
    L = np.zeros((B, Hq, n_q), np.float64)
    lib().orc_verify_attn(q.ctypes.data, k.ctypes.data, v.ctypes.data, dtype, B, Hq, Hkv, d, n_q,
                          cap, _ptr(pl, _i32p), None if m is None else _ptr(m, _u8p), scale,
                          _ptr(O, _dp), _ptr(L, _dp), nthreads or default_threads())
    return O, L


def verify_attn_rows(Q, K, V, prefix_len, rows, mask=None, scale=None, dtype=DTYPE_F32,
                     nthreads=None):
    """Selected rows: ``rows`` is an int array [n, 3] of (b, h, i)."""
    B, Hq, n_q, d = Q.shape
    Hkv, cap = K.shape[1], K.shape[2]
    q, k, v = _kv_args(Q, K, V, dtype)
    pl = _c(prefix_len, np.int32)
    m = None if mask is None else _c(mask, np.uint8)
    bhi = _c(rows, np.int32).reshape(-1, 3)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    n = bhi.shape[0]
    O = np.zeros((n, d), np.float64)
    L = np.zeros((n,), np.float64)
    lib().orc_verify_attn_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dtype, B, Hq, Hkv, d,
                               n_q, cap, _ptr(pl, _i32p), None if m is None else _ptr(m, _u8p),
                               scale, _ptr(bhi, _i32p), n, _ptr(O, _dp), _ptr(L, _dp),
                               nthreads or default_threads())
    return O, L


def verify_attn_split(Q, K, V, prefix_len, cuts, mask=None, scale=None, dtype=DTYPE_F32,
                      nthreads=None):
    """Hybrid form: history pieces cut at ``cuts`` + speculative piece, LSE-merged."""
    B, Hq, n_q, d = Q.shape
    Hkv, cap = K.shape[1], K.shape[2]
    q, k, v = _kv_args(Q, K, V, dtype)
    pl = _c(prefix_len, np.int32)
    m = None if mask is None else _c(mask, np.uint8)
    c = _c(cuts, np.int64)
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    O = np.zeros((B, Hq, n_q, d), np.float64)
    L = np.zeros((B, Hq, n_q), np.float64)
    lib().orc_verify_attn_split(q.ctypes.data, k.ctypes.data, v.ctypes.data, dtype, B, Hq, Hkv, d,
                                n_q, cap, _ptr(pl, _i32p), None if m is None else _ptr(m, _u8p),
                                scale, _ptr(c, _i64p), len(c), _ptr(O, _dp), _ptr(L, _dp),
                                nthreads or default_threads())
    return O, L


# --------------------------------------------------------------------------
# Acceptance
# --------------------------------------------------------------------------

def lse_merge(O_parts, LSE_parts):
    """Log-sum-exp combine of attention parts: O_parts [P, ..., d], LSE_parts [P, ...]
    -> (O [..., d], LSE [...]) in double."""
    Op = _c(O_parts, np.float64)
    Lp = _c(LSE_parts, np.float64)
    P, d = Op.shape[0], Op.shape[-1]
    rows = Lp[0].size
    assert Op.size == P * rows * d and Lp.size == P * rows
    O = np.zeros(Lp.shape[1:] + (d,), np.float64)
    L = np.zeros(Lp.shape[1:], np.float64)
    lib().orc_lse_merge(_ptr(Op, _dp), _ptr(Lp, _dp), P, rows, d, _ptr(O, _dp), _ptr(L, _dp))
    return O, L


def row_dists(z, q, T, eta, clamp=True):
    """(p, p_hat unclamped, p_hat after the tail rule) of one vocabulary row."""
    z = _c(z, np.float32)
    q = _c(q, np.float32)
    V = z.shape[0]
    p = np.zeros(V)
    raw = np.zeros(V)
    ph = np.zeros(V)
    lib().orc_row_dists(_ptr(z, _fp), _ptr(q, _fp), V, T, eta, int(bool(clamp)), _ptr(p, _dp),
                        _ptr(raw, _dp), _ptr(ph, _dp))
    return p, raw, ph


def residual_weights(p, phat, q):
    p = _c(p, np.float64)
    phat = _c(phat, np.float64)
    q = _c(q, np.float32)
    w = np.zeros_like(p)
    lib().orc_residual_weights(_ptr(p, _dp), _ptr(phat, _dp), _ptr(q, _fp), p.shape[0],
                               _ptr(w, _dp))
    return w


def sample_inverse_cdf(w, u):
    w = _c(w, np.float64)
    return lib().orc_sample_inverse_cdf(_ptr(w, _dp), w.shape[0], float(u))


def kd_loss(z, q, T):
    z = _c(z, np.float64)
    q = _c(q, np.float64)
    return lib().orc_kd_loss(_ptr(z, _dp), _ptr(q, _dp), z.shape[0], T)


def kd_grad(z, q, T):
    z = _c(z, np.float64)
    q = _c(q, np.float64)
    g = np.zeros_like(z)
    lib().orc_kd_grad(_ptr(z, _dp), _ptr(q, _dp), z.shape[0], T, _ptr(g, _dp))
    return g


def distilled_logits(z, q, T, eta):
    z = _c(z, np.float64)
    q = _c(q, np.float64)
    out = np.zeros_like(z)
    lib().orc_distilled_logits(_ptr(z, _dp), _ptr(q, _dp), z.shape[0], T, eta, _ptr(out, _dp))
    return out


def accept(z, q, tokens, parent=None, T=1.0, eta=0.0, seed=0, clamp=True, nthreads=None,
           n_nodes=None):
    """Whole acceptance step.  z, q [B, n_q, V] float32; tokens/parent [B, n_q] int32.

    n_nodes: None, or [B] node counts in [1, n_q]; sequence b is then the same
    step on its first n_nodes[b] nodes (diag zero past them).

    Returns dict(n_accepted [B], next_token [B], path [B,n_q], diag [B,n_q,5],
    sample [B,6] = (row e, kind, u, W, u*W, token)).
    """
    z = _c(z, np.float32)
    q = _c(q, np.float32)
    B, n_q, V = z.shape
    tok = _c(tokens, np.int32)
    par = None if parent is None else _c(parent, np.int32)
    nn = None
    if n_nodes is not None:
        nn = _c(n_nodes, np.int32)
        assert nn.shape == (B,) and (nn >= 1).all() and (nn <= n_q).all()
    n_acc = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    path = np.zeros((B, n_q), np.int32)
    diag = np.zeros((B, n_q, 5), np.float64)
    info = np.zeros((B, 6), np.float64)
    lib().orc_accept(_ptr(z, _fp), _ptr(q, _fp), _ptr(tok, _i32p),
                     None if par is None else _ptr(par, _i32p),
                     None if nn is None else _ptr(nn, _i32p), B, n_q, V, float(T), float(eta),
                     int(seed), int(bool(clamp)), _ptr(n_acc, _i32p), _ptr(nxt, _i32p),
                     _ptr(path, _i32p), _ptr(diag, _dp), _ptr(info, _dp),
                     nthreads or default_threads())
    return dict(n_accepted=n_acc, next_token=nxt, path=path, diag=diag, sample=info)


def first_token_hist(z, q, T, eta, clamp, seed, n_trials, nthreads=None):
    """Counts of the first emitted token over n_trials single-draft steps (row 0 only)."""
    z = _c(z, np.float32)
    q = _c(q, np.float32)
    V = z.shape[0]
    hist = np.zeros(V, np.int64)
    lib().orc_first_token_hist(_ptr(z, _fp), _ptr(q, _fp), V, float(T), float(eta),
                               int(bool(clamp)), int(seed), int(n_trials), _ptr(hist, _i64p),
                               nthreads or default_threads())
    return hist


def kv_commit(K, V, prefix_len, path, n_accepted):
    """In place on numpy caches K, V [layers, B, Hkv, cap, d] (any dtype): row
    P_b + 1 + k of every (layer, b, head) takes the row of node path[b][k].
    Returns the number of sequences left untouched (invalid input)."""
    assert K.shape == V.shape and K.flags.c_contiguous and V.flags.c_contiguous
    layers, B, Hkv, cap = K.shape[:4]
    row_bytes = int(np.prod(K.shape[4:])) * K.itemsize
    n_q = path.shape[1]
    kb = K.view(np.uint8).reshape(-1)
    vb = V.view(np.uint8).reshape(-1)
    pl = _c(prefix_len, np.int32)
    pa = _c(path, np.int32)
    na = _c(n_accepted, np.int32)
    return int(lib().orc_kv_commit(_ptr(kb, _u8p), _ptr(vb, _u8p), layers, B, Hkv, cap, row_bytes,
                                   n_q, _ptr(pl, _i32p), _ptr(pa, _i32p), _ptr(na, _i32p)))


def kv_advance(prefix_len, n_accepted):
    """New history lengths: P_b + 1 + n_accepted[b]."""
    pl = _c(prefix_len, np.int32).copy()
    na = _c(n_accepted, np.int32)
    lib().orc_kv_advance(_ptr(pl, _i32p), _ptr(na, _i32p), pl.shape[0])
    return pl


def retrieval_scores(query, chunks):
    """Cosine similarities [B, N] (double) of chunks [B, N, D] with query [B, D] (float32)."""
    q = _c(query, np.float32)
    c = _c(chunks, np.float32)
    B, N, D = c.shape
    out = np.zeros((B, N), np.float64)
    lib().orc_retrieval_scores(_ptr(q, _fp), _ptr(c, _fp), B, N, D, _ptr(out, _dp))
    return out


def retrieval_select(scores, context_tokens, chunk=512, threshold=0.3, min_tokens=4096, ratio=24):
    """Kept chunk ids (ascending, -1 padded) [B, N], their count [B] and tokens [B]
    from float32 scores [B, N]."""
    s = _c(scores, np.float32)
    B, N = s.shape
    ct = _c(context_tokens, np.int32)
    sel = np.zeros((B, N), np.int32)
    ns = np.zeros(B, np.int32)
    ts = np.zeros(B, np.int32)
    lib().orc_retrieval_select(_ptr(s, _fp), _ptr(ct, _i32p), B, N, chunk, float(threshold),
                               min_tokens, ratio, _ptr(sel, _i32p), _ptr(ns, _i32p), _ptr(ts, _i32p))
    return sel, ns, ts


def lm_head_logits(hidden, W, nthreads=None):
    """Logits [rows, V] (double) of hidden states [rows, hidden_dim] against an LM
    head W [V, hidden_dim] (float32 arrays; bf16 values pass exactly)."""
    h = _c(hidden, np.float32)
    w = _c(W, np.float32)
    rows, hd = h.shape
    V, hd2 = w.shape
    if hd != hd2:
        raise ValueError("hidden sizes differ")
    out = np.zeros((rows, V), np.float64)
    lib().orc_lm_head_logits(_ptr(h, _fp), _ptr(w, _fp), rows, hd, V, _ptr(out, _dp),
                             nthreads or default_threads())
    return out
