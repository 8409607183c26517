import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The test session runs the library in checked mode: before every launch each
# buffer's device allocation must hold what the call touches (MOER_EEXTENT
# otherwise), so every GPU test also checks the extents the entry points
# compute.  The library reads this at its first call; set MOER_CHECK_EXTENTS=0
# to run the tests unchecked.  test_gpu_extent.py covers both modes.
os.environ.setdefault("MOER_CHECK_EXTENTS", "1")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size case (minutes)")
