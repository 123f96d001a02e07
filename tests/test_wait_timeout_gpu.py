"""Failure detection on the GPU without a fault: a bounded device wait that is
made to expire (an mbarrier that nothing arrives on) is reported to the host as
LAPNYS_ETIMEOUT by lapnys_device_status, the kernel returns, and the context
stays usable (a forward afterwards still matches the oracle)."""
import numpy as np
import pytest
import torch

from laplacian_nystr_linear_gb300 import _lib, api
from laplacian_nystr_linear_gb300.inputs import WORKLOADS, make_inputs

from tests._parity import compare, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert api.device_status(clear=True) in (_lib.LAPNYS_OK, _lib.LAPNYS_ETIMEOUT)
    assert api.device_status() == _lib.LAPNYS_OK
    api.wait_selftest(1000)
    assert api.device_status(clear=True) == _lib.LAPNYS_ETIMEOUT
    assert api.device_status() == _lib.LAPNYS_OK          # cleared
    # the context is intact: the path still runs and matches the oracle
    w = WORKLOADS["tiny"]
    inp = make_inputs(w)
    compare(w, gpu_run(w, inp), oracle_run(w, inp), backward=False)
    assert api.device_status() == _lib.LAPNYS_OK
    x = torch.arange(8, device="cuda", dtype=torch.float32)
    np.testing.assert_array_equal((x * 2).cpu().numpy(), np.arange(8) * 2.0)
