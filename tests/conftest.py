import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_sessionstart(session):
    """Build the oracle (gcc) and the CUDA libraries (nvcc, sm_103a) if they are stale."""
    import oracle.build
    import invariant_bi_gemm_gb300.build
    oracle.build.build()
    invariant_bi_gemm_gb300.build.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    """GPU tests are skipped when no CUDA device is visible (the CPU-only dev box);
    on a GPU machine they run and fail loudly if the CUDA library is missing."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device visible")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def read_golden(name):
    """Parse a tests/golden fixture: 'key = values' lines, '#' comments."""
    out = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if "=" in line:
                k, v = line.split("=", 1)
                out[k.strip()] = v.strip()
            else:
                rows.append(line.split())
    if rows:
        out["_rows"] = rows
    return out
