"""Failure detection without a GPU fault: every pipelined kernel waits through a bounded mbarrier
wait that, when it runs out, raises the block's abort flag, records a code in the device error
word and returns.  The self-test drives that wait on a barrier nothing arrives on (a short
limit), then the host reads the code, and the context must still run the layer."""
import ctypes

import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
from moe_expert_layer_gemm_gb300 import _lib as L

from .test_gpu_route import check_route

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_context_survives():
    moe.check_device_error()                      # start from a clear error word
    observed = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    moe.moe_selftest_wait_timeout(observed)
    code = ctypes.c_int32(0)
    rc = L.lib().moe_check_device_error(L._stream(None), ctypes.byref(code))
    assert rc == -6 and code.value == 1, (rc, code.value)   # MOE_ERR_DEVICE_CHECK, wait timeout
    assert observed[0].item() == 2                # the wait failed and raised the abort flag
    moe.check_device_error()                      # the read cleared the word
    # the context is intact: routing still matches the oracle bit for bit
    lg = torch.randn(500, 64, generator=torch.Generator().manual_seed(3)) * 2.0
    check_route(500, 64, 6, 1, 1, lg)
    np.testing.assert_equal(observed[1:].cpu().numpy(), [-1, -1, -1])
