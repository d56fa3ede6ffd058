import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size case, minutes of CPU oracle time")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """With MOE_PARITY_TABLE=<path>, write the parity margins the GPU tests
    measured (max|err| / RMS(oracle out) per case and path, and the share of
    the tolerance it uses) as a markdown table."""
    path = os.environ.get("MOE_PARITY_TABLE")
    if not path:
        return
    try:
        from gpu_cases import MARGINS
    except Exception:
        return
    if not MARGINS:
        return
    import json
    rows = ["| test | layer | n | cohort | path | out | tolerance (x RMS) | max abs err / RMS | share of tolerance |",
            "|---|---|---|---|---|---|---|---|---|"]
    for m in MARGINS:
        rows.append(f"| {m['test'].split('::')[-1]} | {m['shape']} | {m['n']} | {m['kind']} | {m['path']} | "
                    f"{m['out']} | {m['tol']:.0e} | {m['err_rel']:.3e} | {m['used']:.1%} |")
    with open(path, "w") as f:
        f.write("\n".join(rows) + "\n")
    with open(path + ".jsonl", "w") as f:
        for m in MARGINS:
            f.write(json.dumps(m) + "\n")
