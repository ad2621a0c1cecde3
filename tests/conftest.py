import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: large CPU oracle run")


@pytest.fixture(scope="session")
def golden():
    import json
    with open(os.path.join(ROOT, "tests", "golden", "apa_page_constants.json")) as f:
        return {k: v["value"] for k, v in json.load(f).items() if not k.startswith("_")}
