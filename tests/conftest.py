import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libw4")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_lines(name):
    """Non-comment, non-empty lines of tests/golden/<name>."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


def golden_kv(name):
    out = {}
    for parts in golden_lines(name):
        out[parts[0]] = parts[1:]
    return out


@pytest.fixture(scope="session")
def gpu_lib():
    """The built product library (libw4) with a CUDA device, else skip."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_weight_mixed_gb300 as w4
    w4.load()
    return w4


@pytest.fixture(autouse=True)
def no_device_timeouts(request):
    """After every GPU test: no kernel recorded a device-side wait timeout in
    any workspace the binding handed out (a timed-out wait can still leave
    correct outputs, so results alone would not show it)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import int4_weight_mixed_gb300 as w4
    for ws in list(w4._ws_cache.values()):
        assert w4.check_status(ws) == w4.OK, "a device-side wait timed out"
