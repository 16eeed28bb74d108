import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")

# the property tests need hypothesis, which not every machine that runs the
# suite has; without it the module is left out rather than reported skipped
try:
    import hypothesis  # noqa: F401
except ImportError:
    collect_ignore = ["test_pack_properties.py"]
