"""The C ABI's error paths on the GPU: bounded waits that give up, and
device-side inputs out of range (GPU; calls the C ABI).

No test here faults or hangs the GPU: the wait that runs out is the library's
own self-test kernel (a barrier phase nothing completes, with a short limit,
after which the kernel records the timeout, lets its copy land and returns),
and the bad inputs are values the kernels clamp or reject in bounds while
flagging them in the device error word.
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


def _clear():
    torch.cuda.synchronize()
    rapid.rapid_device_error(True)


def test_bounded_wait_gives_up_and_reports_timeout():
    _clear()
    assert rapid.rapid_stream_status() == rapid.RAPID_OK
    rapid.rapid_wait_selftest(2_000_000)            # 2 ms, then the wait gives up
    words = rapid.rapid_device_error_info(clear=False)
    assert words[0] & 1 and words[1] == 0xC7000001, [hex(x) for x in words]
    assert rapid.rapid_stream_status(clear=True) == rapid.RAPID_ETIMEOUT
    assert rapid.rapid_stream_status() == rapid.RAPID_OK   # cleared
    # the context stays usable: a verify call right after is still exact
    w = wl.Workload("t", B=2, Hq=8, Hkv=2, d=128, n_q=6, prefix=900, prefix_lo=300, layers=1,
                    V=10, dtype="bf16", z_std=1, q_noise_std=1, q_noise_uses_T=True, seed=91)
    a = wl.attn_inputs(w, device=DEV)
    O, L = rapid.verify_attn(a.Q, a.K, a.V, a.prefix_len, None)
    assert rapid.rapid_stream_status() == rapid.RAPID_OK
    Oo, Lo = oracle.verify_attn(wl.bf16_bits(a.Q), wl.bf16_bits(a.K), wl.bf16_bits(a.V),
                                a.prefix_len.cpu().numpy(), None, dtype=oracle.DTYPE_BF16)
    check_attn(O.float().cpu().numpy(), L.cpu().numpy(), Oo, Lo)


@pytest.mark.parametrize("d", [64, 128])
def test_history_length_out_of_range_is_flagged(d):
    # prefix_len + n_q > kv_capacity and a negative length: both clamped into
    # the cache (memory-safe) and reported as a bad device-side input
    _clear()
    w = wl.Workload("t", B=3, Hq=8, Hkv=2, d=d, n_q=5, prefix=500, layers=1, V=10,
                    dtype="bf16", z_std=1, q_noise_std=1, q_noise_uses_T=True, seed=92)
    a = wl.attn_inputs(w, device=DEV, prefix_override=[500, 10 ** 6, -3])
    rapid.verify_attn(a.Q, a.K, a.V, a.prefix_len, None)
    assert rapid.rapid_stream_status() == rapid.RAPID_EINVAL
    a = wl.attn_inputs(w, device=DEV, prefix_override=[500, 200, 0])
    rapid.verify_attn(a.Q, a.K, a.V, a.prefix_len, None)
    assert rapid.rapid_stream_status() == rapid.RAPID_OK


def _accept_inputs(tree):
    w = wl.QWEN7B_TREE if tree else wl.LLAMA8B_LAYER_32K
    inp = wl.accept_inputs(w, B=2)
    par = None if inp.parent is None else inp.parent.to(DEV)
    return inp.z.to(DEV), inp.q.to(DEV), inp.tokens.to(DEV), par


@pytest.mark.parametrize("what", ["token_negative", "token_past_vocab", "parent_self",
                                  "parent_negative", "n_nodes_zero", "n_nodes_too_many"])
def test_acceptance_device_inputs_out_of_range_are_flagged(what):
    _clear()
    tree = what.startswith("parent")
    z, q, tok, par = _accept_inputs(tree)
    B, n_q, V = z.shape
    res = rapid.accept(z, q, tok, par, seed=5)
    assert rapid.rapid_stream_status() == rapid.RAPID_OK
    tok2, par2, nn = tok.clone(), None if par is None else par.clone(), None
    if what == "token_negative":
        tok2[1, 3] = -1
    elif what == "token_past_vocab":
        tok2[0, 2] = V
    elif what == "parent_self":
        par2[1, 7] = 7
    elif what == "parent_negative":
        par2[0, 5] = -2
    elif what == "n_nodes_zero":
        nn = torch.tensor([n_q, 0], dtype=torch.int32, device=DEV)
    else:
        nn = torch.tensor([n_q + 1, 3], dtype=torch.int32, device=DEV)
    res = rapid.accept(z, q, tok2, par2, seed=5, n_nodes=nn)
    assert rapid.rapid_stream_status() == rapid.RAPID_EINVAL
    # memory-safe results: counts within the path, tokens inside the vocabulary
    n_acc = res["n_accepted"].cpu().numpy()
    nxt = res["next_token"].cpu().numpy()
    assert ((n_acc >= 0) & (n_acc < n_q)).all() and ((nxt >= 0) & (nxt < V)).all()
    assert rapid.rapid_stream_status() == rapid.RAPID_OK


def test_status_codes_and_strings():
    L = rapid.lib()
    codes = {rapid.RAPID_OK: b"ok", rapid.RAPID_EINVAL: b"invalid argument",
             rapid.RAPID_ETIMEOUT: b"a bounded wait inside a kernel gave up",
             rapid.RAPID_EUNSUPPORTED: b"unsupported shape"}
    for c, text in codes.items():
        assert L.rapid_status_string(c) == text
    assert len({rapid.RAPID_OK, rapid.RAPID_EINVAL, rapid.RAPID_ECUDA, rapid.RAPID_ENOMEM,
                rapid.RAPID_ETIMEOUT, rapid.RAPID_EUNSUPPORTED}) == 6
