"""FP8 (E4M3) path on the GPU against the FP8 oracle, through the C ABI.

  * moe_quantize_e4m3: codes bit-identical to the oracle's tensorwise quantisation of the same
    bf16 values, scales and amax exact (integer decision taken in the same fp32 arithmetic);
  * moe_grouped_swiglu_fwd_fp8: [a | u] and h within the bf16 output tolerance of the oracle's
    fp64 product of the same decoded operands; h's codes bit-identical to the oracle's
    quantisation of the GPU's h; y_perm within tolerance of the oracle's fc2 on those codes;
    and, against the unquantised bf16 layer, within the E4M3 rounding bound;
  * moe_grouped_swiglu_bwd_fp8, stage by stage on the GPU's own intermediates: dy_perm's codes
    bit-identical to the oracle's quantisation; [da | du] within the bf16 tolerance of the
    oracle's SwiGLU backward of its fc2 data gradient; [da | du]'s codes bit-identical to the
    oracle's quantisation of the GPU's [da | du] (amax exact); dx_perm within the bf16 tolerance,
    dW1 and dW2 within the fp32 tolerance of the oracle's products of the same codes; and the
    whole backward against the unquantised fp64 one within the E4M3 rounding bound.
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
TOL_F32 = 1e-5        # fp32 outputs (weight gradients): exact products, fp32 accumulation


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


def offsets_of(counts):
    o = np.zeros(len(counts) + 1, np.int32)
    o[1:] = np.cumsum(counts)
    return o


def run_fp8_fwd_bwd(T, d, E, k, f, counts, seed):
    """The FP8 forward, then its backward for a random upstream gradient; returns the GPU
    tensors of both."""
    N = T * k
    o = offsets_of(counts)
    assert o[-1] == N
    g = torch.Generator().manual_seed(seed)
    bf = torch.bfloat16
    xp = torch.randn(N, d, generator=g).to(bf).cuda()
    W1 = (torch.randn(E, 2 * f, d, generator=g) * 0.05).to(bf).cuda()
    W2 = (torch.randn(E, d, f, generator=g) * 0.05).to(bf).cuda()
    dy = (torch.randn(N, d, generator=g) * 0.01).to(bf).cuda()
    off = torch.from_numpy(o).cuda()
    cfg = moe.make_cfg(T, d, E, k, f)
    xq, xs, _ = quantize_gpu(xp, 1)
    W1q, s1, _ = quantize_gpu(W1, E)
    W2q, s2, _ = quantize_gpu(W2, E)
    dev = dict(device="cuda")
    t = dict(xp=xp, W1=W1, W2=W2, dy=dy, off=off, o=o, xq=xq, xs=xs, W1q=W1q, s1=s1, W2q=W2q, s2=s2,
             h=torch.empty(N, f, dtype=bf, **dev), act=torch.empty(N, 2 * f, dtype=bf, **dev),
             hq=torch.empty(N, f, dtype=torch.uint8, **dev), hs=torch.empty(4, **dev),
             ha=torch.empty(4, **dev), yp=torch.empty(N, d, dtype=bf, **dev),
             dyq=torch.empty(N, d, dtype=torch.uint8, **dev), dys=torch.empty(4, **dev),
             dya=torch.empty(4, **dev), dH1=torch.empty(N, 2 * f, dtype=bf, **dev),
             dH1q=torch.empty(N, 2 * f, dtype=torch.uint8, **dev), dhs=torch.empty(4, **dev),
             dha=torch.empty(4, **dev), dxp=torch.empty(N, d, dtype=bf, **dev),
             dW1=torch.full((E, 2 * f, d), float("nan"), **dev),
             dW2=torch.full((E, d, f), float("nan"), **dev))
    moe.moe_grouped_swiglu_fwd_fp8(cfg, xq, xs, off, W1q, s1, W2q, s2, t["h"], t["act"], t["hq"],
                                   t["hs"], t["ha"], t["yp"])
    ws = moe.workspace(cfg, moe.WS_FFN_BWD_FP8)
    moe.moe_grouped_swiglu_bwd_fp8(cfg, xq, xs, off, W1q, s1, W2q, s2, t["act"], t["hq"], t["hs"],
                                   dy, t["dyq"], t["dys"], t["dya"], t["dH1"], t["dH1q"], t["dhs"],
                                   t["dha"], t["dxp"], t["dW1"], t["dW2"], ws)
    torch.cuda.synchronize()
    moe.check_device_error()
    return t


def check_fp8_bwd(t, E, f):
    o = t["o"]
    c = {k: v.cpu().numpy() for k, v in t.items() if isinstance(v, torch.Tensor) and v.dtype == torch.uint8}
    sc = lambda k: t[k][:1].cpu().numpy()                                   # noqa: E731
    s1, s2 = t["s1"].cpu().numpy(), t["s2"].cpu().numpy()
    # dy_perm's codes
    rq, rs = F8.quantize_tensorwise(t["dy"].float().cpu().numpy())
    assert np.array_equal(c["dyq"], rq) and sc("dys")[0] == rs[0]
    # [da | du] from the oracle's fc2 data gradient on the same codes
    dh = F8.fc2_dgrad_fp8(c["dyq"], sc("dys"), c["W2q"], s2, o)
    ref_dH1 = F8.swiglu_backward(dh, np64(t["act"]))
    e_dH1 = assert_close("dH1", np64(t["dH1"]), ref_dH1, TOL_OUT)
    # its codes: the oracle's quantisation of the GPU's [da | du]
    gq, gs = F8.quantize_tensorwise(t["dH1"].float().cpu().numpy())
    assert np.array_equal(c["dH1q"], gq) and sc("dhs")[0] == gs[0]
    assert sc("dha")[0] == np.float32(np.abs(t["dH1"].float().cpu().numpy()).max())
    e_dx = assert_close("dx_perm", np64(t["dxp"]),
                        F8.fc1_dgrad_fp8(gq, gs, c["W1q"], s1, o), TOL_OUT)
    ref_dW1 = F8.wgrad_fp8(gq, gs, c["xq"], sc("xs"), o)
    ref_dW2 = F8.wgrad_fp8(c["dyq"], sc("dys"), c["hq"], sc("hs"), o)
    e_w1 = assert_close("dW1", np64(t["dW1"]), ref_dW1, TOL_F32)
    e_w2 = assert_close("dW2", np64(t["dW2"]), ref_dW2, TOL_F32)
    for e in range(E):
        if o[e + 1] == o[e]:
            assert not t["dW1"][e].any() and not t["dW2"][e].any()
    return e_dH1, e_dx, e_w1, e_w2


FP8_BWD_CASES = [
    # T, d, E, k, f, counts (None: routed at random)
    (600, 256, 8, 2, 144, None),
    (300, 384, 16, 4, 256, None),
    (1024, 2048, 128, 8, 768, None),
    # empty experts, an expert of one row, one of more than a full k-block of rows
    (100, 128, 6, 2, 64, [0, 1, 130, 0, 69, 0]),
]


@pytest.mark.parametrize("T,d,E,k,f,counts", FP8_BWD_CASES)
def test_fp8_grouped_swiglu_backward(T, d, E, k, f, counts):
    if counts is None:
        counts = np.diff(routed(T, E, k, d + 1)["offsets"])
    t = run_fp8_fwd_bwd(T, d, E, k, f, counts, seed=T + f)
    errs = check_fp8_bwd(t, E, f)
    # against the unquantised backward (fp64 on the bf16 inputs, the FP8 forward's [a | u])
    o = t["o"]
    X, dY, act = np64(t["xp"]), np64(t["dy"]), np64(t["act"])
    dx_ref = np.zeros_like(X)
    dW1_ref = np.zeros(t["dW1"].shape)
    dW2_ref = np.zeros(t["dW2"].shape)
    for e in range(E):
        lo, hi = o[e], o[e + 1]
        if hi == lo:
            continue
        a, u = act[lo:hi, :f], act[lo:hi, f:]
        h = O.silu(a) * u
        dx_ref[lo:hi], dW1_ref[e], dW2_ref[e] = O.swiglu_ffn_backward(
            np64(t["W1"][e]), np64(t["W2"][e]), X[lo:hi], a, u, h, dY[lo:hi])
    e_q = [rel_err(np64(t[k]), r) for k, r in (("dxp", dx_ref), ("dW1", dW1_ref), ("dW2", dW2_ref))]
    assert max(e_q) < 0.15, e_q
    print("stagewise dH1 %.2e dx %.2e dW1 %.2e dW2 %.2e; vs unquantised %s"
          % (*errs, ", ".join(f"{v:.3f}" for v in e_q)))
