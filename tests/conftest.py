import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--oracle-lib", default=None,
                     help="run the oracle from this compiled library instead of oracle/oracle.c "
                          "(the mutation test uses it to run the pins against planted mistakes)")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    lib = config.getoption("--oracle-lib")
    if lib:
        import oracle

        oracle._SRC = oracle._LIB_PATH = os.path.abspath(lib)  # already built: build() keeps it
        oracle._lib = None
