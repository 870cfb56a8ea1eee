import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, minutes on the GPU box")


def pytest_collection_modifyitems(config, items):
    # GPU tests are only meaningful with a device; on a CPU machine they are skipped
    # (the driver selects them explicitly with -m gpu on the GPU machine).
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _debug_library_status_clean(request):
    """With the binding on the debug library (DIT_ATTN_DEBUG=1), every GPU
    test must leave the device status word clean: no bounds check failed and
    no bounded wait ran out."""
    yield
    if os.environ.get("DIT_ATTN_DEBUG") == "1" and "gpu" in request.keywords:
        from dit_long_sequence_gb300 import binding
        assert binding.is_debug_library
        rc, info = binding.check_watchdog()
        assert rc == 0, f"debug library status {rc} {info} after {request.node.nodeid}"
