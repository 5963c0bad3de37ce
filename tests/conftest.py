import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


def load_fixture(name):
    """Parse a tests/golden text fixture: 'key = v1 v2 ...' lines, '#' comments."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, vals = line.partition("=")
            toks = vals.split()
            parsed = []
            for t in toks:
                parsed.append(int(t, 16) if t.lower().startswith("0x") else float(t))
            out[key.strip()] = parsed
    return out


@pytest.fixture
def fixture_loader():
    return load_fixture
