import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")


def pytest_report_header(config):
    try:
        from lm_head_linear_tcgen05_gb300 import _build
        state = "up to date" if _build.up_to_date() else "missing or stale (compiled by the first test that needs it)"
        return f"liblp.so: sources {_build.source_hash()}, in-tree build {state}"
    except Exception as e:  # the header must never stop a run
        return f"liblp.so: build state unknown ({e})"


def pytest_terminal_summary(terminalreporter):
    try:
        from lm_head_linear_tcgen05_gb300 import _build
        for rec in _build.BUILDS.values():
            terminalreporter.write_line(f"liblp build used by this run: {rec}")
    except Exception:
        pass


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


# Every GPU test gets a time limit (pytest-timeout, where installed) so that a test that
# stalls ends with a failure instead of holding the GPU; the kernels' own waits are bounded
# at 2 s, so this only guards the host side.
GPU_TEST_TIMEOUT_S = 1200


def pytest_collection_modifyitems(config, items):
    has_timeout = config.pluginmanager.hasplugin("timeout")
    if _has_gpu():
        if has_timeout:
            for it in items:
                if "gpu" in it.keywords and it.get_closest_marker("timeout") is None:
                    it.add_marker(pytest.mark.timeout(GPU_TEST_TIMEOUT_S))
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
