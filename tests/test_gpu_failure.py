"""Failure detection on the GPU without a fault: a bounded wait that can never
complete gives up, records a timeout in the device status word, and the kernel
exits normally -- the context stays usable and later calls are correct."""
import numpy as np
import pytest

import csa_workloads as w
import oracle
from gpu_util import Dev, run_fwd

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports(csa=None):
    import torch
    import sparse_attention_kv_csa_gb300 as csa
    assert csa.csa_device_status(clear=True) == 0
    csa.csa_selftest_bounded_wait(50_000_000)  # 50 ms
    torch.cuda.synchronize()
    assert csa.csa_device_status() == 7  # CSA_ERR_DEVICE_TIMEOUT
    assert "bounded wait" in csa.csa_last_error_message()
    assert csa.csa_device_status(clear=True) == 7
    assert csa.csa_device_status() == 0
    # the context is still usable: a pipelined call after it is correct
    c = w.make_case("after", 4, 2, 512, [64, 37], extra_rows=2, seed=9)
    assert np.array_equal(run_fwd(Dev(c), csa), oracle.case_fwd_f32(c))
    assert csa.csa_device_status() == 0
