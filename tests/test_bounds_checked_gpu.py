"""The bounds-checked build (CSSCAN_BOUNDS_CHECK, GPU only): the tiny parity suite of
bounds_checked_suite.py through libcsscan_checked.so, in a process of its own; every call must
leave the device status clean and match the oracle."""
import os
import subprocess
import sys

import pytest
import torch

from selective_state_space_diagonal_b300 import build as libbuild

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounds_checked_suite():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    libbuild.build_checked()
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_checked_suite.py")], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, f"bounds-checked suite failed:\n{r.stdout[-3000:]}\n{r.stderr[-3000:]}"
    assert "clean and within tolerance" in r.stdout
