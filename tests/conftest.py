"""Shared pytest set-up: the ``gpu`` marker and the repository root on ``sys.path``."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture
def repo_tmp(request):
    """A scratch directory inside the repository's git-ignored build folder (tests that
    compile small programs keep their files there, not in a system temp folder)."""
    import pathlib
    import re
    import shutil
    name = re.sub(r"[^A-Za-z0-9_.-]", "_", request.node.name)
    d = pathlib.Path(ROOT) / "bucketized_guidance_step_gb300" / "_build" / "tests_tmp" / name
    shutil.rmtree(d, ignore_errors=True)
    d.mkdir(parents=True)
    yield d
    shutil.rmtree(d, ignore_errors=True)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
