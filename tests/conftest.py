import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_ignore_collect(collection_path, config):
    """The oracle's property tests (CPU only, unmarked) need hypothesis; under `-m gpu` they
    are deselected anyway, so where hypothesis is missing they are not collected there instead
    of showing up as a skipped module."""
    if collection_path.name == "test_oracle_properties.py" and "gpu" in (config.getoption("-m") or "") \
            and "not gpu" not in (config.getoption("-m") or ""):
        try:
            import hypothesis  # noqa: F401
        except ImportError:
            return True
    return None


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads (GPU)")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name: str) -> dict:
    """Parse a 'key: v1 v2 ...' fixture file; '#' starts a comment line."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, vals = line.partition(":")
            out[key.strip()] = vals.split()
    return out


@pytest.fixture(scope="session")
def golden():
    return read_golden
