import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")


def pytest_sessionstart(session):
    # On a GPU machine make sure the CUDA library exists before GPU tests import it.
    try:
        import torch
    except ImportError:
        return
    if torch.cuda.is_available():
        import __graft_entry__
        __graft_entry__.build()
