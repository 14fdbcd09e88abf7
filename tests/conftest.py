import ctypes
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name):
    """Rows of a whitespace-separated golden file, comments stripped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def golden():
    return read_golden


@pytest.fixture(autouse=True)
def _bounds_record_stays_clean(request):
    """When the bounds-checked build of the library is the one loaded (its
    path in BMMC_GB300_LIBRARY), every GPU test must leave the device-side
    failure record empty: no kernel access outside its buffers or shared
    arrays."""
    if not os.environ.get("BMMC_GB300_LIBRARY") or request.node.get_closest_marker("gpu") is None:
        yield
        return
    from bmmc_index_transforms_gb300 import _capi

    L = _capi.lib()
    r = _capi.BoundsReport()
    assert L.bmmc_bounds_report(ctypes.byref(r), 1) == _capi.OK
    assert r.enabled == 1, "BMMC_GB300_LIBRARY does not name a bounds-checked build"
    yield
    assert L.bmmc_bounds_report(ctypes.byref(r), 1) == _capi.OK
    assert r.failures == 0, (f"{r.failures} kernel accesses outside their buffers; first at site {r.site} "
                             f"(file tag * 100000 + line), address {r.address:#x}, {r.bytes} bytes, "
                             f"range [{r.lo:#x}, {r.hi:#x})")
