import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    """GPU tests are skipped, not failed, on a machine without a GPU."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _gpu_guards_and_margins(request):
    """GPU tests: the test id under which tolerance checks record their
    errors, and afterwards the check that no kernel wrote outside a buffer
    allocated by the test helpers."""
    if "gpu" not in request.keywords:
        yield
        return
    from tests import gpu_util
    gpu_util.CURRENT_TEST["id"] = request.node.nodeid
    yield
    gpu_util.check_guards()


def pytest_sessionfinish(session, exitstatus):
    out = os.environ.get("MOE_MARGINS_OUT")
    mod = sys.modules.get("tests.gpu_util")
    if not out or mod is None or not mod.MARGINS:
        return
    import json
    with open(out, "w") as fh:
        json.dump(mod.MARGINS, fh, indent=0)
