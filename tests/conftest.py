import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library through its C ABI)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle

TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree for sm_103a; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_27_gb300 import api, build
    build.build_library()
    return api.load()


@pytest.fixture(params=["persistent", "cluster"])
def kernel_path(request, cuda_lib):
    """Runs the test once with each verify kernel: the persistent kernel
    (cluster threshold 0, one-hot row limit 0) and the one-cluster-per-row
    kernel (threshold above any test's rows; rows that are not 16-byte
    vectors still take the persistent kernel). The thresholds are restored
    afterwards. The one-hot row kernel has its own tests."""
    from speculative_decoding_verification_27_gb300 import api
    persistent = request.param == "persistent"
    prev = api.sv_set_cluster_rows(0 if persistent else 1 << 20)
    prev_oh = api.sv_set_onehot_row_bytes(0 if persistent else -1)
    yield request.param
    api.sv_set_cluster_rows(prev)
    api.sv_set_onehot_row_bytes(prev_oh)
