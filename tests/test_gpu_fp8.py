"""FP8 (E4M3) path on the GPU against the FP8 oracle, through the C ABI.

  * moe_quantize_e4m3: codes bit-identical to the oracle's tensorwise quantisation of the same
    bf16 values, scales and amax exact (integer decision taken in the same fp32 arithmetic);
  * moe_grouped_swiglu_fwd_fp8: [a | u] and h within the bf16 output tolerance of the oracle's
    fp64 product of the same decoded operands; h's codes bit-identical to the oracle's
    quantisation of the GPU's h; y_perm within tolerance of the oracle's fc2 on those codes;
    and, against the unquantised bf16 layer, within the E4M3 rounding bound.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import oracle.fp8_oracle as F8
import oracle.moe_oracle as O

from .helpers import assert_close, np64, rel_err

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2        # bf16 outputs of an fp32-accumulated product of exact E4M3 values


def quantize_gpu(x, groups):
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    scale = torch.empty(max(groups, 4), device="cuda")
    amax = torch.empty(max(groups, 4), device="cuda")
    moe.moe_quantize_e4m3(x, groups, q, scale, amax)
    torch.cuda.synchronize()
    moe.check_device_error()
    return q, scale[:groups], amax[:groups]


@pytest.mark.parametrize("shape,groups", [((64, 48), 1), ((5, 32, 16), 5), ((3000, 96), 1),
                                          ((8, 272, 128), 8)])
def test_quantize_codes_are_exact(shape, groups):
    g = torch.Generator().manual_seed(sum(shape))
    rows = torch.logspace(-3, 2, shape[0]).view(-1, *([1] * (len(shape) - 1)))
    x = (torch.randn(*shape, generator=g) * rows).bfloat16()
    if groups > 1:
        x[1] = 0                                  # an all-zero tensor: scale 1, codes 0
    q, scale, amax = quantize_gpu(x.cuda(), groups)
    rq, rs = F8.quantize_tensorwise(x.float().numpy(), groups)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(scale.cpu().numpy(), rs)
    ref_amax = np.abs(x.float().numpy().reshape(groups, -1)).max(1)
    assert np.array_equal(amax.cpu().numpy(), ref_amax.astype(np.float32))


def routed(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    return O.route(torch.randn(T, E, generator=g).numpy(), k, E, O.SOFTMAX, 1)


@pytest.mark.parametrize("T,d,E,k,f", [(600, 256, 8, 2, 144), (1024, 2048, 128, 8, 768),
                                       (300, 384, 16, 4, 256)])
def test_fp8_grouped_swiglu_forward(T, d, E, k, f):
    r = routed(T, E, k, d)
    N = T * k
    g = torch.Generator().manual_seed(f)
    xp = torch.randn(N, d, generator=g).bfloat16().cuda()
    W1 = (torch.randn(E, 2 * f, d, generator=g) * 0.05).bfloat16().cuda()
    W2 = (torch.randn(E, d, f, generator=g) * 0.05).bfloat16().cuda()
    off = torch.from_numpy(r["offsets"]).cuda()
    cfg = moe.make_cfg(T, d, E, k, f)
    xq, xs, _ = quantize_gpu(xp, 1)
    W1q, s1, _ = quantize_gpu(W1, E)
    W2q, s2, _ = quantize_gpu(W2, E)
    bf = torch.bfloat16
    h = torch.empty(N, f, dtype=bf, device="cuda")
    act = torch.empty(N, 2 * f, dtype=bf, device="cuda")
    hq = torch.empty(N, f, dtype=torch.uint8, device="cuda")
    hs = torch.empty(4, device="cuda")
    ha = torch.empty(4, device="cuda")
    yp = torch.empty(N, d, dtype=bf, device="cuda")
    moe.moe_grouped_swiglu_fwd_fp8(cfg, xq, xs, off, W1q, s1, W2q, s2, h, act, hq, hs, ha, yp)
    torch.cuda.synchronize()
    moe.check_device_error()
    o = r["offsets"]
    ref_h, ref_act = F8.fc1_swiglu_fp8(xq.cpu().numpy(), xs.cpu().numpy(), W1q.cpu().numpy(),
                                       s1.cpu().numpy(), o)
    e_act = assert_close("act", np64(act), ref_act, TOL_OUT)
    e_h = assert_close("h", np64(h), ref_h, TOL_OUT)
    # h's codes: the oracle's quantisation of the GPU's (bf16) h
    rq, rs = F8.quantize_tensorwise(h.float().cpu().numpy())
    assert np.array_equal(hq.cpu().numpy(), rq) and hs[0].item() == rs[0]
    ref_y = F8.fc2_fp8(rq, rs, W2q.cpu().numpy(), s2.cpu().numpy(), o)
    e_y = assert_close("y_perm", np64(yp), ref_y, TOL_OUT)
    # against the unquantised layer: E4M3 keeps 3 mantissa bits (relative rounding <= 2^-4)
    X = np64(xp)
    y_bf = np.zeros((N, d))
    for e in range(E):
        sl = slice(o[e], o[e + 1])
        if o[e + 1] > o[e]:
            y_bf[sl] = O.swiglu_ffn(np64(W1[e]), np64(W2[e]), X[sl])[0]
    e_q = rel_err(np64(yp), y_bf)
    assert e_q < 0.1, e_q
    print(f"act {e_act:.2e} h {e_h:.2e} y {e_y:.2e}; vs unquantised {e_q:.3f}")


@pytest.mark.parametrize("T,d,E,k", [(1000, 256, 16, 4), (4097, 2048, 128, 8), (7, 64, 4, 1)])
def test_permute_quantize_equals_quantizing_the_permuted_matrix(T, d, E, k):
    r = routed(T, E, k, T)
    g = torch.Generator().manual_seed(d)
    x = (torch.randn(T, d, generator=g) * 3).bfloat16().cuda()
    cfg = moe.make_cfg(T, d, E, k, 64)
    sop = torch.from_numpy(r["slot_of_pair"]).cuda()
    xq = torch.empty(T * k, d, dtype=torch.uint8, device="cuda")
    xs, xa = torch.empty(4, device="cuda"), torch.empty(4, device="cuda")
    moe.moe_permute_quantize_e4m3(cfg, x, sop, xq, xs, xa)
    xp = torch.empty(T * k, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, x, sop, xp)
    q2, s2, a2 = quantize_gpu(xp, 1)
    torch.cuda.synchronize()
    moe.check_device_error()
    assert torch.equal(xq, q2) and xs[0].item() == s2[0].item() and xa[0].item() == a2[0].item()
    rq, rs = F8.quantize_tensorwise(xp.float().cpu().numpy())
    assert np.array_equal(xq.cpu().numpy(), rq) and xs[0].item() == rs[0]
