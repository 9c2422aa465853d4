import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_sessionstart(session):
    # Build the CUDA library (a no-op while it is newer than its sources).
    import shutil
    if shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc"):
        from paged_kv_attention_prepare_gb300.builder import build
        build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    # the largest attention errors each check saw, when asked for
    path = os.environ.get("PA_ERROR_LOG")
    if path:
        import json
        from helpers import ERRORS
        with open(path, "w") as f:
            for e in ERRORS:
                f.write(json.dumps({"test": e[0], "dtype": e[1], "max_err_bound_1e-2": e[2],
                                    "max_err_coarse_outputs": e[3], "elements": e[4]}) + "\n")
