import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size oracle comparisons")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """Write the parity errors the GPU tests observed to $PEAGLE_PARITY_LOG (JSON)."""
    path = os.environ.get("PEAGLE_PARITY_LOG")
    if not path:
        return
    try:
        from pe_helpers import RECORD
    except Exception:  # pragma: no cover
        return
    rec = list(RECORD)
    mod = sys.modules.get("test_gpu_train_step")
    for case, name, worst in getattr(mod, "GRAD_RECORD", []):
        rec.append({"case": case, "gradient": name, "worst_bound_ratio": worst})
    import json
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
