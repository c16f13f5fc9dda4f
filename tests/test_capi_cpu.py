"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and rejects bad host-side arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from long_context_speculative_gb300 import build as lib_build
from long_context_speculative_gb300 import rapid

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(rapid_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return rapid.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "rapid_verify_attn" in names and "rapid_accept" in names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert lib.rapid_version() >= 100
    assert lib.rapid_status_string(0) == b"ok"
    assert lib.rapid_status_string(-1) == b"invalid argument"


def test_host_validation_without_gpu(lib):
    # NULL tensors are rejected before any CUDA call.
    assert lib.rapid_verify_attn(None, None, None, 1, 1, 4, 1, 128, 5, 64, None, None, 0.0, None,
                                 None, None, 0, None) == -1
    assert lib.rapid_accept(None, None, None, None, 1, 3, 100, 1.0, 1.0, 0, 1, None, None, None,
                            None, None, 0, None) == -1
    # rapid_accept_ex: misaligned node counts or key address, NULL tensors, bad sizes
    fake = ctypes.c_void_p(256)   # an aligned fake device address (never dereferenced)
    for nn, key in ((ctypes.c_void_p(258), None), (None, ctypes.c_void_p(260))):
        assert lib.rapid_accept_ex(fake, fake, fake, None, nn, 1, 3, 100, 1.0, 1.0, 0, key, 1,
                                   fake, fake, None, None, fake, 1 << 20, None) == -1
    assert lib.rapid_accept_ex(None, None, None, None, None, 1, 3, 100, 1.0, 1.0, 0, fake, 1,
                               None, None, None, None, None, 0, None) == -1
    assert lib.rapid_accept_ex(fake, fake, fake, None, fake, 1, 65, 100, 1.0, 1.0, 0, None, 1,
                               fake, fake, None, None, fake, 1 << 20, None) == -1
    # Sizes outside the supported range report a zero workspace.
    assert lib.rapid_verify_attn_workspace_size(1, 4, 1, 96, 5, 64, 1) == 0
    assert lib.rapid_verify_attn_workspace_size(1, 4, 1, 128, 65, 640, 1) == 0
    assert lib.rapid_verify_attn_workspace_size(1, 3, 2, 128, 5, 64, 1) == 0
    assert lib.rapid_verify_attn_workspace_size(8192, 8, 8, 128, 5, 64, 1) == 0   # B * Hkv
    assert lib.rapid_accept_workspace_size(1, 65, 100) == 0
    assert lib.rapid_accept_workspace_size(1, 5, 229377) == 0
    assert lib.rapid_accept_workspace_size(2, 11, 128256) > 0
    assert lib.rapid_verify_attn_workspace_size(1, 32, 8, 128, 11, 122896, 1) > 0


def test_kv_commit_host_validation_without_gpu(lib):
    arr = (ctypes.c_void_p * 1)(16)   # a fake, aligned device address (never dereferenced)
    good = [ctypes.cast(arr, ctypes.c_void_p), ctypes.cast(arr, ctypes.c_void_p), 1, 1, 2, 2, 128,
            4096, 8, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), None]
    for i, bad in [(0, None), (2, 0), (2, 129), (3, 5), (4, 0), (5, 0), (6, 96), (7, 0), (8, 0),
                   (8, 65), (9, None), (10, None), (11, None)]:
        args = list(good)
        args[i] = bad
        assert lib.rapid_kv_commit(*args) == -1, i
    unaligned = (ctypes.c_void_p * 1)(8)
    args = list(good)
    args[0] = ctypes.cast(unaligned, ctypes.c_void_p)
    assert lib.rapid_kv_commit(*args) == -1
    args = list(good)
    args[8] = 1   # n_q = 1: no draft node, nothing to launch
    assert lib.rapid_kv_commit(*args) == 0
    assert lib.rapid_kv_advance(None, ctypes.c_void_p(16), 1, 8, 4096, None) == -1
    assert lib.rapid_kv_advance(ctypes.c_void_p(16), ctypes.c_void_p(16), 0, 8, 4096, None) == -1
    assert lib.rapid_kv_advance(ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 65, 4096, None) == -1


def test_retrieval_host_validation_without_gpu(lib):
    p = ctypes.c_void_p(16)   # a fake, aligned device address (never dereferenced)
    good = [p, p, 1, 4, 240, 1024, p, None]
    for i, bad in [(0, None), (1, None), (2, 7), (3, 0), (4, 0), (5, 0), (5, 12), (5, 8200),
                   (6, None)]:
        args = list(good)
        args[i] = bad
        assert lib.rapid_retrieval_scores(*args) == -1, i
    args = list(good)
    args[1] = ctypes.c_void_p(24)   # not 16-byte aligned
    assert lib.rapid_retrieval_scores(*args) == -1
    good = [p, p, 4, 240, 512, ctypes.c_float(0.3), 4096, 24, p, p, p, None]
    for i, bad in [(0, None), (1, None), (2, 0), (3, 0), (3, 8193), (4, 0), (6, -1), (7, 0),
                   (8, None), (9, None), (10, None)]:
        args = list(good)
        args[i] = bad
        assert lib.rapid_retrieval_select(*args) == -1, i


def test_lm_head_host_validation_without_gpu(lib):
    p = ctypes.c_void_p(16)   # a fake, aligned device address (never dereferenced)
    good = [p, p, 11, 4096, 128256, p, None]
    for i, bad in [(0, None), (1, None), (2, 0), (2, 257), (3, 0), (3, 100), (3, 16448),
                   (4, 0), (4, (1 << 22) + 1), (5, None)]:
        args = list(good)
        args[i] = bad
        assert lib.rapid_lm_head(*args) == -1, i
    args = list(good)
    args[1] = ctypes.c_void_p(24)   # W not 16-byte aligned
    assert lib.rapid_lm_head(*args) == -1
    assert lib.rapid_lm_head_accept_workspace_size(1, 11, 128256) >= 11 * 128256 * 4
    assert lib.rapid_lm_head_accept_workspace_size(5, 64, 1000) == 0   # 320 rows > 256
    ws = lib.rapid_lm_head_accept_workspace_size(1, 11, 128256)
    good = [p, p, 4096, p, p, None, 1, 11, 128256, ctypes.c_float(1.0), ctypes.c_float(1.0), 7,
            1, p, p, None, None, p, ws, None]
    for i, bad in [(0, None), (1, None), (2, 96), (3, None), (4, None), (6, 0), (7, 65),
                   (8, 229377), (9, ctypes.c_float(0.0)), (10, ctypes.c_float(-1.0)), (12, 8),
                   (13, None), (14, None), (17, None)]:
        args = list(good)
        args[i] = bad
        assert lib.rapid_lm_head_accept(*args) == -1, i
    args = list(good)
    args[18] = ws - 1
    assert lib.rapid_lm_head_accept(*args) == -3   # workspace too small


def test_no_cpu_fallback_for_cpu_tensors(lib):
    import torch
    Q = torch.zeros((1, 4, 5, 128), dtype=torch.bfloat16)
    with pytest.raises(rapid.RapidError):
        rapid.verify_attn(Q, Q, Q, torch.zeros(1, dtype=torch.int32))


def test_binding_constants_match_the_header():
    # every RAPID_* constant the Python binding defines has the header's value
    text = open(os.path.join(ROOT, "include", "rapid.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    header = {}
    for name, expr in re.findall(r"\b(RAPID_[A-Z0-9_]+)\s*=\s*([^,}\n]+)", text):
        parts = [int(x.strip().rstrip("u")) for x in expr.split("<<")]   # literals and shifts
        header[name] = parts[0] << parts[1] if len(parts) == 2 else parts[0]
    ours = {k: v for k, v in vars(rapid).items() if k.startswith("RAPID_") and isinstance(v, int)}
    assert ours
    for k, v in ours.items():
        assert k in header, k
        assert header[k] == v, (k, header[k], v)
