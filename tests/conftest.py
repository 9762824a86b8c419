import os
import pathlib
import shutil
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


# Scratch files (mutated oracle builds, test shims) stay inside the repository,
# in a git-ignored directory, and are removed when the test is done.
SCRATCH = os.path.join(ROOT, ".scratch")


def _scratch_dir():
    os.makedirs(SCRATCH, exist_ok=True)
    return pathlib.Path(tempfile.mkdtemp(dir=SCRATCH))


@pytest.fixture
def repo_tmp():
    d = _scratch_dir()
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.fixture(scope="module")
def repo_tmp_module():
    d = _scratch_dir()
    yield d
    shutil.rmtree(d, ignore_errors=True)
