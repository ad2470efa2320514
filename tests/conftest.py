import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled sm_103a library")


@pytest.fixture(scope="session")
def orc():
    import oracle

    return oracle.get()


@pytest.fixture(scope="session")
def golden():
    import json

    with open(os.path.join(HERE, "golden", "page_examples.json"), encoding="utf-8") as f:
        return json.load(f)
