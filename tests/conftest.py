import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this host")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """With GDN_ERR_LOG set, list the largest recorded error of each (test, label): the
    measured max|err| / RMS(ref) against the oracle, beside the bar the test applies."""
    import json
    path = os.environ.get("GDN_ERR_LOG")
    if not path or not os.path.exists(path):
        return
    worst = {}
    for line in open(path):
        try:
            r = json.loads(line)
        except ValueError:
            continue
        key = (r["test"], r["label"] or "")
        worst[key] = max(worst.get(key, 0.0), r["err"])
    terminalreporter.write_sep("-", "recorded errors (max|err| / RMS(ref))")
    for (test, label), e in sorted(worst.items()):
        terminalreporter.write_line(f"{e:10.3e}  {test}  {label or ''}")
