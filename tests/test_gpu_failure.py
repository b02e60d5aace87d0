"""The failure path of the kernels' bounded waits, without a GPU fault.

Every mbarrier wait in the tensor-core kernels gives up after about a second,
records a timeout in the device status word and lets the kernel finish.  The
self-test entry point runs one such wait on a barrier that nothing arrives at;
the status must read SDPA_ERR_TIMEOUT once, then SDPA_OK, and the context must
stay usable: a following forward call matches the oracle.
"""
import pytest
import torch

import oracle
import scaled_dot_product_sm_gb300 as sdpa
from test_gpu_parity import check_forward
from workloads import random_inputs

pytestmark = pytest.mark.gpu

SDPA_ERR_TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdpa.build()
    sdpa.load_library()


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    assert sdpa.last_device_status() == 0
    sdpa.selftest_wait_timeout()
    assert sdpa.last_device_status() == SDPA_ERR_TIMEOUT
    assert sdpa.last_device_status() == 0          # read and cleared
    q, k, v, _, _ = random_inputs(1, 4, 2, 300, 260, 128, 128, torch.bfloat16, seed=240)
    o, lse = sdpa.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), None, None, True, True)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.ref_forward(q, k, v, None, None, True, True)
    check_forward(o, lse, ref_o, ref_lse, True)
    assert sdpa.last_device_status() == 0
