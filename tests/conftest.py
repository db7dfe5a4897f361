import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Set in the child process that runs a no_device test.
_NO_DEVICE_CHILD = "Z3_TEST_NO_DEVICE_CHILD"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs through the C-ABI library)")
    config.addinivalue_line("markers", "slow: long CPU test")
    config.addinivalue_line(
        "markers",
        "no_device: passes made-up device addresses to the library to check its host-side "
        "validation; runs in a child process that sees no CUDA device, so a validation "
        "that let a call through would fail to launch instead of touching memory")


@pytest.hookimpl(tryfirst=True)
def pytest_pyfunc_call(pyfuncitem):
    """Run a no_device test in a child process with CUDA_VISIBLE_DEVICES set
    to the empty string.  In that process the CUDA runtime finds no device,
    so a launch with a made-up address can only fail with an error."""
    if pyfuncitem.get_closest_marker("no_device") is None:
        return None
    if os.environ.get(_NO_DEVICE_CHILD) == "1":
        assert os.environ.get("CUDA_VISIBLE_DEVICES") == "", "no_device child sees a device"
        return None
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", **{_NO_DEVICE_CHILD: "1"})
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        pyfuncitem.nodeid], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    if r.returncode != 0:
        pytest.fail(f"{pyfuncitem.nodeid} failed in its no-device child process:\n"
                    f"{r.stdout[-4000:]}\n{r.stderr[-2000:]}", pytrace=False)
    return True


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
