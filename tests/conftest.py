import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and librapid.so")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when no GPU is present: run them with
    # -m gpu only on a GPU machine; the CPU suite deselects them with -m "not gpu".
    pass


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # The near-boundary cases the parity comparisons exempted (counted, not
    # failed) and, per attention comparison, the largest O error next to the
    # largest |O| of the expected output.
    mod = sys.modules.get("_parity")
    if mod is None:
        return
    tr = terminalreporter
    if mod.EXEMPTIONS:
        e = mod.EXEMPTIONS
        tr.write_line(
            "parity exemptions: "
            + ", ".join(f"{k}={e[k]}" for k in ("sequences", "compared", "ratio_exempt",
                                                  "cdf_exempt", "clamp_exempt")))
    if mod.ATTN_ERRORS:
        worst = max(mod.ATTN_ERRORS, key=lambda r: r[3])
        tr.write_line(f"attention comparisons: {len(mod.ATTN_ERRORS)}; largest "
                      f"max|dO|/max|O_ref| = {worst[3]:.3g} ({worst[0]}: max|dO| = {worst[1]:.3g}, "
                      f"max|O_ref| = {worst[2]:.3g})")
        for label, err_o, o_max, rel, err_l in mod.ATTN_ERRORS:
            if label:
                tr.write_line(f"  {label}: max|dO| {err_o:.3g}, max|O_ref| {o_max:.3g}, "
                              f"ratio {rel:.3g}, max|dLSE| {err_l:.3g}")
