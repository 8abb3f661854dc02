import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU")
    config.addinivalue_line("markers", "slow: full-scale case (minutes)")


def _ensure_built():
    """Build the CPU-side libraries (generator, oracle) and the product library
    if they are missing; nvcc cross-compiles without a GPU."""
    import synth
    import oracle

    if not (os.path.exists(synth.HOST_LIB) and os.path.exists(synth.DEV_LIB)):
        synth.build()
    if not os.path.exists(oracle.BUILT_LIB):
        oracle.build()
    try:
        import persistent_moe_decode_sm_gb300 as mk
    except ImportError:
        return
    if getattr(mk, "LIB_PATH", None) and not os.path.exists(mk.LIB_PATH):
        mk.build()


@pytest.fixture(scope="session", autouse=True)
def built_libraries():
    _ensure_built()
