import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "plants_bad_descriptor: expects failed index checks")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


@pytest.fixture(autouse=True)
def _index_checks(request):
    """Under DPSYNC_VARIANT=checked (the library built with device index checks),
    every GPU test must end with no failed check."""
    yield
    if os.environ.get("DPSYNC_VARIANT") == "checked" and request.node.get_closest_marker("gpu") \
            and not request.node.get_closest_marker("plants_bad_descriptor"):
        import gradient_sync_zero_gb300 as dps
        n = dps.dp_bounds_violations(reset=True)
        assert n == 0, f"{n} device index check(s) failed during {request.node.name}"
