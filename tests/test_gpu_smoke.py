"""The package's smoke run (one small call of every route against the
oracle, then a three-GEMV decode chain) as a GPU test."""
import os
import sys

import pytest

pytestmark = pytest.mark.gpu

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_smoke_runs_clean(lq, cuda_dev):
    import __graft_entry__ as entry
    entry.smoke()
