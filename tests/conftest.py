import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_sessionstart(session):
    # Build the CUDA library and the float64 oracle before collection: test
    # modules import the package, which refuses to load without librlcs.so.
    # Both builds skip what is already up to date.
    import __graft_entry__
    __graft_entry__.build()
