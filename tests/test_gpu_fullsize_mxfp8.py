"""The MXFP8 forward at the benchmark's full size (the DeepSeek-style workload; the stage calls
`bench.py` times for its MXFP8 comparison, and the layer call), against the MXFP8 oracle on what
it can compute one row at a time from the GPU's own codes:

  * the layer's y_perm bit-identical to the stage calls on its routing;
  * x's codes and block scales on sampled slots bit-identical to the oracle's quantisation of
    their tokens' rows;
  * h on sampled slots (heaviest, median and lightest non-empty experts, and each expert's last
    row) within the bf16 tolerance of the oracle's fp64 fc1 + SwiGLU of the decoded operands; h's
    codes and scales bit-identical to the oracle's quantisation of the GPU's bf16 h;
  * y_perm on those slots within the bf16 tolerance of the oracle's fc2 of h's codes.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import moe_inputs
import oracle.moe_oracle as O
import oracle.mxfp8_oracle as MX

from .helpers import assert_close, mx_unpack_act_scales, np64

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2


@pytest.fixture(scope="module")
def run():
    lc = moe_inputs.CONFIGS["deepseek"]
    inp = moe_inputs.make_layer_inputs(lc, seed=0, device="cuda")
    cfg = moe.cfg_from(lc)
    N, d, f = lc.N, lc.d, lc.f
    bf = torch.bfloat16
    m = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"])
    saved = moe.alloc_saved(cfg)
    saved["x_perm"] = saved["act"] = saved["h"] = None
    y = torch.empty_like(inp["x"])
    moe.moe_layer_fwd_mxfp8(cfg, inp["x"], inp["W_r"], inp["b_r"], m, inp["Ws1"], inp["Ws2"], None,
                            y, saved, moe.workspace(cfg, moe.WS_LAYER_FWD))
    st = dict(xq=torch.empty_like(m["x_perm_q"]), xs=torch.empty_like(m["x_perm_s"]),
              hq=torch.empty_like(m["h_q"]), hs=torch.empty_like(m["h_s"]),
              h=torch.empty(N, f, dtype=bf, device="cuda"),
              act=torch.empty(N, 2 * f, dtype=bf, device="cuda"),
              yp=torch.empty(N, d, dtype=bf, device="cuda"))
    off = saved["offsets"]
    moe.moe_permute_quantize_mxfp8(cfg, inp["x"], saved["slot_of_pair"], off, st["xq"], st["xs"])
    moe.moe_grouped_swiglu_fwd_mxfp8(cfg, st["xq"], st["xs"], off, m["W1_q"], m["W1_sp"], m["W2_q"],
                                     m["W2_sp"], st["h"], st["act"], st["hq"], st["hs"], st["yp"])
    torch.cuda.synchronize()
    moe.check_device_error()
    return lc, inp, m, saved, st


def test_layer_equals_stage_calls(run):
    lc, inp, m, saved, st = run
    assert torch.equal(saved["y_perm"], st["yp"])
    assert torch.equal(m["x_perm_q"], st["xq"]) and torch.equal(m["h_q"], st["hq"])


def sample_slots(off):
    counts = np.diff(off)
    live = np.flatnonzero(counts)
    order = live[np.argsort(counts[live], kind="stable")]
    experts = [order[-1], order[len(order) // 2], order[0]]
    rng = np.random.default_rng(0)
    slots = []
    for e in experts:
        lo, hi = off[e], off[e + 1]
        slots += list(rng.integers(lo, hi, size=min(8, hi - lo))) + [hi - 1]
    return experts, np.array(sorted(set(int(s) for s in slots)))


def test_sampled_rows_against_the_oracle(run):
    lc, inp, m, saved, st = run
    N, d, f = lc.N, lc.d, lc.f
    off = np64(saved["offsets"]).astype(np.int64)
    tos = np64(saved["token_of_slot"]).astype(np.int64)
    experts, slots = sample_slots(off)
    # x: codes and scales of the sampled slots = the oracle's quantisation of their tokens' rows
    xrows = np64(inp["x"][torch.from_numpy(tos[slots]).cuda()])
    rq, rs = MX.mx_quantize(xrows)
    xq = st["xq"][torch.from_numpy(slots).cuda()].cpu().numpy()
    xs_all = mx_unpack_act_scales(st["xs"].cpu().numpy(), off, N, d)
    assert np.array_equal(xq, rq) and np.array_equal(xs_all[slots], rs)
    hs_all = mx_unpack_act_scales(st["hs"].cpu().numpy(), off, N, f)
    idx = torch.from_numpy(slots).cuda()
    h_gpu = np64(st["h"][idx])
    hq_gpu = st["hq"][idx].cpu().numpy()
    y_gpu = np64(st["yp"][idx])
    ref_h = np.zeros_like(h_gpu)
    ref_y = np.zeros_like(y_gpu)
    X = MX.mx_decode(xq, xs_all[slots])
    for e in experts:
        rows = np.flatnonzero((slots >= off[e]) & (slots < off[e + 1]))
        W1 = MX.mx_decode(m["W1_q"][e].cpu().numpy(), m["W1_s"][e].cpu().numpy())
        W2 = MX.mx_decode(m["W2_q"][e].cpu().numpy(), m["W2_s"][e].cpu().numpy())
        au = X[rows] @ W1.T
        ref_h[rows] = O.silu(au[:, :f]) * au[:, f:]
        ref_y[rows] = MX.mx_decode(hq_gpu[rows], hs_all[slots[rows]]) @ W2.T
    assert_close("h", h_gpu, ref_h, TOL_OUT)
    # h's codes and scales: the oracle's block quantisation of the GPU's bf16 h
    q2, s2 = MX.mx_quantize(h_gpu)
    assert np.array_equal(hq_gpu, q2) and np.array_equal(hs_all[slots], s2)
    assert_close("y_perm", y_gpu, ref_y, TOL_OUT)


def test_weight_gradients_on_sampled_experts(run):
    """moe_grouped_swiglu_wgrad_mxfp8 at full size on the layer's routing and bf16 h, x_perm from
    the permute, seeded dy_perm and [da | du]: for the heaviest, median and lightest non-empty
    experts, 64 sampled rows of dW1[e] and dW2[e] within fp32 accumulation of the oracle's fp64
    token-block products.  A row i of dW1[e] needs only column i of [da | du] (column blocks are
    independent) and all of x_perm's rows of e."""
    lc, inp, m, saved, st = run
    cfg = moe.cfg_from(lc)
    N, d, f, E = lc.N, lc.d, lc.f, lc.E
    bf = torch.bfloat16
    off = saved["offsets"]
    o = np64(off).astype(np.int64)
    x_perm = torch.empty(N, d, dtype=bf, device="cuda")
    moe.moe_permute(cfg, inp["x"], saved["slot_of_pair"], x_perm)
    g = torch.Generator(device="cuda").manual_seed(7)
    dy = (torch.randn(N, d, generator=g, device="cuda") * 0.1).to(bf)
    dH = (torch.randn(N, 2 * f, generator=g, device="cuda") * 0.1).to(bf)
    dW1 = torch.empty(E, 2 * f, d, device="cuda")
    dW2 = torch.empty(E, d, f, device="cuda")
    moe.moe_grouped_swiglu_wgrad_mxfp8(cfg, off, x_perm, st["h"], dy, dH, dW1, dW2,
                                       moe.workspace(cfg, moe.WS_WGRAD_MXFP8))
    torch.cuda.synchronize()
    moe.check_device_error()
    counts = np.diff(o)
    order = [e for e in np.argsort(-counts, kind="stable") if counts[e] > 0]
    rng = np.random.default_rng(3)
    for e in (order[0], order[len(order) // 2], order[-1]):
        lo, hi = int(o[e]), int(o[e + 1])
        seg = [0, hi - lo]
        r1 = np.sort(rng.choice(2 * f, 64, replace=False))
        r2 = np.sort(rng.choice(d, 64, replace=False))
        B1 = MX.mx_decode_segments(*MX.mx_quantize_segments(np64(x_perm[lo:hi]), seg), seg)
        B2 = MX.mx_decode_segments(*MX.mx_quantize_segments(np64(st["h"][lo:hi]), seg), seg)
        A1 = MX.mx_decode_segments(*MX.mx_quantize_segments(np64(dH[lo:hi, r1]), seg), seg)
        A2 = MX.mx_decode_segments(*MX.mx_quantize_segments(np64(dy[lo:hi, r2]), seg), seg)
        assert_close(f"dW1[{e}] ({hi - lo} rows)", np64(dW1[e][r1]), A1.T @ B1, 2e-5)
        assert_close(f"dW2[{e}] ({hi - lo} rows)", np64(dW2[e][r2]), A2.T @ B2, 2e-5)
    for e in np.nonzero(counts == 0)[0][:4]:
        assert not dW1[e].any() and not dW2[e].any()
