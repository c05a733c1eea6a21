"""Shared test set-up: the ``gpu`` marker and small helpers.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on a CPU-only machine.
"""
import numpy as np
import pytest


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU and the compiled sm_103a library")


def rel_l2(x, ref):
    """||x - ref||_2 / ||ref||_2 over the whole array, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    return float(num / den) if den > 0 else float(num)


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle
