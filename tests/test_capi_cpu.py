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
    # Sizes outside the supported range report a zero workspace.
    assert lib.rapid_verify_attn_workspace_size(1, 4, 1, 96, 5, 64, 1) == 0
    assert lib.rapid_verify_attn_workspace_size(1, 4, 1, 128, 65, 640, 1) == 0
    assert lib.rapid_verify_attn_workspace_size(1, 3, 2, 128, 5, 64, 1) == 0
    assert lib.rapid_accept_workspace_size(1, 65, 100) == 0
    assert lib.rapid_accept_workspace_size(1, 5, 229377) == 0
    assert lib.rapid_accept_workspace_size(2, 11, 128256) > 0
    assert lib.rapid_verify_attn_workspace_size(1, 32, 8, 128, 11, 122896, 1) > 0


def test_no_cpu_fallback_for_cpu_tensors(lib):
    import torch
    Q = torch.zeros((1, 4, 5, 128), dtype=torch.bfloat16)
    with pytest.raises(rapid.RapidError):
        rapid.verify_attn(Q, Q, Q, torch.zeros(1, dtype=torch.int32))
