import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running test")


@pytest.fixture(scope="session")
def mq_lib():
    """The C-ABI library, built in-tree if missing or stale."""
    from quantized_decode_matvec_gb300 import build as mqbuild
    mqbuild.build()
    from quantized_decode_matvec_gb300 import mq
    return mq


@pytest.fixture(scope="session")
def cuda_ready(mq_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()
    mq_lib.init(torch.cuda.current_device())
    return mq_lib


@pytest.fixture(params=["auto", "register"])
def variant(request, cuda_ready):
    """Run a test under each kernel family: bulk-copy ring where it applies (auto), and register streaming."""
    mq = cuda_ready
    pol = mq.MQ_VARIANT_AUTO if request.param == "auto" else mq.MQ_VARIANT_FORCE_REGISTER
    assert mq.mq_debug_set_variant(pol) == mq.MQ_OK
    yield request.param
    assert mq.mq_debug_set_variant(mq.MQ_VARIANT_AUTO) == mq.MQ_OK
