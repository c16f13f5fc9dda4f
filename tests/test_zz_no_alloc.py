"""The allocation-free acceptance entry point (GPU; calls the C ABI).

rapid_accept_noalloc serves callers that cannot allocate device memory where
they run the acceptance step (a host framework that owns all device memory
and gives plug-ins no allocator, or a decode loop that must never call
cudaMalloc).  Its scratch is a static device array inside librapid.so.  This
file is collected last, so a run that stops at the first failure has already
run every other test; it passes alone in a fresh process and after the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

from long_context_speculative_gb300 import rapid
from long_context_speculative_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _outputs(B, n_q):
    return (torch.empty(B, dtype=torch.int32, device=DEV),
            torch.empty(B, dtype=torch.int32, device=DEV),
            torch.empty((B, n_q), dtype=torch.int32, device=DEV),
            torch.empty((B, n_q, 5), dtype=torch.float32, device=DEV))


def _run_both(w, seed, T=1.0, eta=1.0):
    inp = wl.accept_inputs(w, T=T)
    z, q, tok = inp.z.to(DEV), inp.q.to(DEV), inp.tokens.to(DEV)
    par = None if inp.parent is None else inp.parent.to(DEV)
    B, n_q, V = z.shape
    ref = rapid.accept(z, q, tok, par, T=T, eta=eta, seed=seed, tail_clamp=True)
    torch.cuda.synchronize()
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    for _ in range(2):   # two calls in a row share the static scratch
        n_acc, nxt, path, diag = _outputs(B, n_q)
        rapid.rapid_accept_noalloc(z, q, tok, par, T, eta, seed, rapid.RAPID_ACCEPT_TAIL_CLAMP,
                                   n_acc, nxt, path, diag)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(n_acc.cpu().numpy(), ref["n_accepted"])
        np.testing.assert_array_equal(nxt.cpu().numpy(), ref["next_token"])
        np.testing.assert_array_equal(path.cpu().numpy(), ref["path"])
        np.testing.assert_allclose(diag.cpu().numpy(), ref["diag"], rtol=1e-5, atol=0)
    assert rapid.rapid_device_error(True) == 0


def test_noalloc_matches_workspace_entry_point_chain():
    w = wl.Workload("noalloc", B=3, Hq=1, Hkv=1, d=64, n_q=11, prefix=1, layers=1, V=128256,
                    dtype="f32", z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True, seed=71)
    _run_both(w, seed=0x5EED0001)


def test_noalloc_matches_workspace_entry_point_tree():
    w = wl.Workload("noalloc_tree", B=4, Hq=1, Hkv=1, d=64, n_q=32, prefix=1, layers=1,
                    V=152064, dtype="f32", z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True,
                    tree=True, seed=72)
    _run_both(w, seed=0x5EED0002)


def test_noalloc_rejects_sizes_over_the_limit():
    L = rapid.lib()
    B, n_q, V = 65, 64, 16     # 4160 nodes > RAPID_NOALLOC_MAX_NODES = 4096
    z = torch.zeros((B, n_q, V), device=DEV)
    tok = torch.zeros((B, n_q), dtype=torch.int32, device=DEV)
    o = torch.zeros(B, dtype=torch.int32, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.rapid_accept_noalloc(p(z), p(z), p(tok), None, B, n_q, V, 1.0, 1.0, 0, 1, p(o), p(o),
                                None, None, None)
    assert st == rapid.RAPID_EUNSUPPORTED
    # sizes that no entry point accepts are invalid arguments, as for rapid_accept
    for b, n in ((0, 11), (1, 0), (1, 65)):
        st = L.rapid_accept_noalloc(p(z), p(z), p(tok), None, b, n, V, 1.0, 1.0, 0, 1, p(o),
                                    p(o), None, None, None)
        assert st == rapid.RAPID_EINVAL, (b, n)


def test_noalloc_allocates_nothing():
    # after a first call (which may load the library's device code), further
    # calls leave the device's free memory exactly where it was
    w = wl.Workload("noalloc_mem", B=2, Hq=1, Hkv=1, d=64, n_q=11, prefix=1, layers=1, V=32000,
                    dtype="f32", z_std=3.0, q_noise_std=1.5, q_noise_uses_T=True, seed=73)
    inp = wl.accept_inputs(w)
    z, q, tok = inp.z.to(DEV), inp.q.to(DEV), inp.tokens.to(DEV)
    n_acc, nxt, path, diag = _outputs(w.B, w.n_q)
    call = lambda s: rapid.rapid_accept_noalloc(z, q, tok, None, 1.0, 1.0, s,
                                                rapid.RAPID_ACCEPT_TAIL_CLAMP, n_acc, nxt, path,
                                                diag)
    call(0)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for s in range(50):
        call(s)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert rapid.rapid_device_error(True) == 0
