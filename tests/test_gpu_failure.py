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


def test_corrupt_slot_map_in_the_mxfp8_backward_is_reported():
    """A slot outside [0, N) in the saved map reaches the MXFP8 combine backward (which also
    quantises dy_perm) and the permute backward. Both check every slot they read: they record the
    bad-slot code in the device error word and skip the row, and the context stays usable. The
    clean map then gives the same gradients as a run that never saw the bad one."""
    import moe_inputs
    import oracle.moe_oracle as O
    lc = moe_inputs.LayerConfig("mx bad slot", 160, 256, 8, 2, 96, f_shared=64,
                                score_fn=O.SOFTMAX, renorm=1)
    inp = moe_inputs.make_layer_inputs(lc, seed=4, device="cuda")
    cfg = moe.cfg_from(lc)
    m = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"])
    mxd = moe.alloc_mxfp8_dgrad(cfg, inp["W1"], inp["W2"])
    saved = moe.alloc_saved(cfg)
    y = torch.empty_like(inp["x"])
    moe.moe_layer_fwd_mxfp8(cfg, inp["x"], inp["W_r"], inp["b_r"], m, inp["Ws1"], inp["Ws2"], None,
                            y, saved, moe.workspace(cfg, moe.WS_LAYER_FWD))
    f32 = torch.float32
    E, d, f, fs = lc.E, lc.d, lc.f, lc.f_shared
    ws = moe.workspace(cfg, moe.WS_LAYER_BWD)

    def backward():
        g = dict(dx=torch.empty_like(inp["x"]), dW_r=torch.empty(E, d, dtype=f32, device="cuda"),
                 dW1=torch.empty(E, 2 * f, d, dtype=f32, device="cuda"),
                 dW2=torch.empty(E, d, f, dtype=f32, device="cuda"),
                 dWs1=torch.empty(2 * fs, d, dtype=f32, device="cuda"),
                 dWs2=torch.empty(d, fs, dtype=f32, device="cuda"))
        moe.moe_layer_bwd_mxfp8(cfg, inp["dy"], inp["x"], inp["W_r"], mxd, inp["Ws1"], inp["Ws2"],
                                None, saved, g["dx"], g["dW_r"], g["dW1"], g["dW2"], g["dWs1"],
                                g["dWs2"], None, ws)
        torch.cuda.synchronize()
        return g

    moe.check_device_error()
    ref = backward()
    moe.check_device_error()                      # the clean map raises nothing
    good = saved["slot_of_pair"][3, 1].item()
    saved["slot_of_pair"][3, 1] = lc.T * lc.k + 5
    backward()
    code = ctypes.c_int32(0)
    rc = L.lib().moe_check_device_error(L._stream(None), ctypes.byref(code))
    assert rc == -6 and code.value == 3, (rc, code.value)   # MOE_ERR_DEVICE_CHECK, bad slot
    saved["slot_of_pair"][3, 1] = good
    again = backward()
    moe.check_device_error()
    for name in ref:
        assert torch.equal(again[name], ref[name]), name
