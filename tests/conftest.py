import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


@pytest.fixture(scope="session")
def full_oracle():
    """Full oracle result (C_ref, W) of a named workload, computed once per
    test session: the large workloads take seconds to tens of seconds on
    the host cores, and several tests compare against the same one."""
    import gemm_inputs
    import oracle

    cache = {}

    def get(name):
        if name not in cache:
            A, B = gemm_inputs.make_workload(name)
            cache[name] = oracle.sgemm(A.numpy(), B.numpy(), with_w=True)
        return cache[name]

    return get
