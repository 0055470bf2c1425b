"""The FP8 layer at the benchmark's full size (the DeepSeek-style workload, the calls and
arguments `bench.py --fp8` times), against the FP8 oracle on what it can compute one piece at a
time from the GPU's own codes:

  * the layer's weight gradients bit-identical to the FP8 stage calls composed on its routing
    (so the sampled checks below, made on the stage calls' intermediates, cover the layer);
  * x's E4M3 codes on sampled slots bit-identical to the oracle's quantisation;
  * h, y_perm, [da | du] and dx_perm on sampled slots within the bf16 tolerance of the oracle's
    fp64 products of the decoded codes;
  * dW1 and dW2 of sampled experts (all of a light expert, sampled rows of the heaviest) within
    the fp32 tolerance.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import moe_inputs
import oracle.fp8_oracle as F8

from .helpers import assert_close, np64

pytestmark = pytest.mark.gpu

TOL_OUT, TOL_F32 = 1e-2, 1e-5


def _dec(codes):
    return F8.e4m3_decode(codes)


@pytest.fixture(scope="module")
def run():
    lc = moe_inputs.CONFIGS["deepseek"]
    inp = moe_inputs.make_layer_inputs(lc, seed=0, device="cuda")
    cfg = moe.cfg_from(lc)
    dev = "cuda"
    T, d, E, k, f, fs, N = lc.T, lc.d, lc.E, lc.k, lc.f, lc.f_shared, lc.N
    bf, u8, f32 = torch.bfloat16, torch.uint8, torch.float32
    saved = moe.alloc_saved(cfg, dev)
    saved["x_perm"] = None
    q = moe.alloc_fp8_experts(cfg, inp["W1"], inp["W2"], dev, Ws1=inp["Ws1"], Ws2=inp["Ws2"])
    y = torch.empty_like(inp["x"])
    g = dict(dx=torch.empty_like(inp["x"]), dW_r=torch.empty(E, d, dtype=f32, device=dev),
             dW1=torch.empty(E, 2 * f, d, dtype=f32, device=dev),
             dW2=torch.empty(E, d, f, dtype=f32, device=dev),
             dWs1=torch.empty(2 * fs, d, dtype=f32, device=dev),
             dWs2=torch.empty(d, fs, dtype=f32, device=dev))
    moe.moe_layer_fwd_fp8(cfg, inp["x"], inp["W_r"], inp["b_r"], q, inp["Ws1"], inp["Ws2"], None,
                          y, saved, moe.workspace(cfg, moe.WS_LAYER_FWD))
    moe.moe_layer_bwd_fp8(cfg, inp["dy"], inp["x"], inp["W_r"], q, inp["Ws1"], inp["Ws2"], None,
                          saved, g["dx"], g["dW_r"], g["dW1"], g["dW2"], g["dWs1"], g["dWs2"], None,
                          moe.workspace(cfg, moe.WS_LAYER_BWD_FP8))
    # the same expert path as stage calls, with every intermediate exposed
    sop, off = saved["slot_of_pair"], saved["offsets"]
    st = {}
    st["xq"] = torch.empty(N, d, dtype=u8, device=dev)
    st["xs"], st["xa"] = torch.empty(4, device=dev), torch.empty(4, device=dev)
    moe.moe_permute_quantize_e4m3(cfg, inp["x"], sop, st["xq"], st["xs"], st["xa"])
    st["h"], st["act"] = torch.empty(N, f, dtype=bf, device=dev), torch.empty(N, 2 * f, dtype=bf, device=dev)
    st["hq"], st["hs"], st["ha"] = torch.empty(N, f, dtype=u8, device=dev), torch.empty(4, device=dev), torch.empty(4, device=dev)
    st["yp"] = torch.empty(N, d, dtype=bf, device=dev)
    moe.moe_grouped_swiglu_fwd_fp8(cfg, st["xq"], st["xs"], off, q["W1_q"], q["W1_scale"], q["W2_q"],
                                   q["W2_scale"], st["h"], st["act"], st["hq"], st["hs"], st["ha"],
                                   st["yp"])
    st["dyp"] = torch.empty(N, d, dtype=bf, device=dev)
    dgate = torch.empty(T, k, device=dev)
    dsh = torch.empty_like(inp["x"])
    moe.moe_unpermute_combine_bwd(cfg, inp["dy"], st["yp"], saved["gate"], sop, saved["s_out"],
                                  None, st["dyp"], dgate, dsh, None)
    st["dyq"], st["dH1q"] = torch.empty(N, d, dtype=u8, device=dev), torch.empty(N, 2 * f, dtype=u8, device=dev)
    st["dH1"], st["dxp"] = torch.empty(N, 2 * f, dtype=bf, device=dev), torch.empty(N, d, dtype=bf, device=dev)
    st["sc"] = [torch.empty(4, device=dev) for _ in range(4)]
    st["dW1"], st["dW2"] = torch.empty_like(g["dW1"]), torch.empty_like(g["dW2"])
    moe.moe_grouped_swiglu_bwd_fp8(cfg, st["xq"], st["xs"], off, q["W1_q"], q["W1_scale"], q["W2_q"],
                                   q["W2_scale"], st["act"], st["hq"], st["hs"], st["dyp"], st["dyq"],
                                   st["sc"][0], st["sc"][1], st["dH1"], st["dH1q"], st["sc"][2],
                                   st["sc"][3], st["dxp"], st["dW1"], st["dW2"],
                                   moe.workspace(cfg, moe.WS_FFN_BWD_FP8))
    torch.cuda.synchronize()
    moe.check_device_error()
    yield lc, inp, saved, q, g, st
    del inp, saved, q, g, st
    torch.cuda.empty_cache()


def test_fullsize_fp8_layer_equals_stage_calls(run):
    lc, inp, saved, q, g, st = run
    assert torch.equal(q["x_perm_q"], st["xq"]) and torch.equal(q["h_q"], st["hq"])
    assert torch.equal(saved["y_perm"], st["yp"]) and torch.equal(saved["act"], st["act"])
    assert torch.equal(g["dW1"], st["dW1"]) and torch.equal(g["dW2"], st["dW2"])


def test_fullsize_fp8_sampled_against_oracle(run):
    lc, inp, saved, q, g, st = run
    d, f, E = lc.d, lc.f, lc.E
    rng = np.random.default_rng(0)
    off = np64(saved["offsets"]).astype(np.int64)
    tos = np64(saved["token_of_slot"]).astype(np.int64)
    counts = np.diff(off)
    slots = np.sort(rng.choice(lc.N, 32, replace=False))
    expert_of = np.searchsorted(off, slots, side="right") - 1
    sc = lambda t: t[:1].cpu().numpy()                                   # noqa: E731
    s1, s2 = q["W1_scale"].cpu().numpy(), q["W2_scale"].cpu().numpy()
    # x's codes on the sampled slots: the oracle's quantisation of the token rows, the scale
    # taken from the whole of x
    x = inp["x"].float().cpu().numpy()
    amax = np.float32(np.abs(x).max())
    assert st["xa"][0].item() == amax
    inv = np.float32(448.0) / amax
    ref_codes = F8.e4m3_encode((x[tos[slots]] * inv).astype(np.float32))
    assert np.array_equal(st["xq"][torch.from_numpy(slots).cuda()].cpu().numpy(), ref_codes)
    xq, hq = st["xq"].cpu().numpy(), st["hq"].cpu().numpy()
    dyq, dH1q = st["dyq"].cpu().numpy(), st["dH1q"].cpu().numpy()
    W1q, W2q = q["W1_q"].cpu().numpy(), q["W2_q"].cpu().numpy()
    act, h, yp = np64(st["act"]), np64(st["h"]), np64(st["yp"])
    dH1, dxp = np64(st["dH1"]), np64(st["dxp"])
    ref = {n: [] for n in ("act", "y", "dH1", "dx")}
    got = {n: [] for n in ref}
    for s, e in zip(slots, expert_of):
        W1 = _dec(W1q[e]) * float(s1[e])
        W2 = _dec(W2q[e]) * float(s2[e])
        au = (_dec(xq[s]) * float(sc(st["xs"])[0])) @ W1.T
        ref["act"].append(au)
        got["act"].append(act[s])
        ref["y"].append((_dec(hq[s]) * float(sc(st["hs"])[0])) @ W2.T)
        got["y"].append(yp[s])
        dh = (_dec(dyq[s]) * float(sc(st["sc"][0])[0])) @ W2
        ref["dH1"].append(F8.swiglu_backward(dh[None, :], act[s][None, :])[0])
        got["dH1"].append(dH1[s])
        ref["dx"].append((_dec(dH1q[s]) * float(sc(st["sc"][2])[0])) @ W1)
        got["dx"].append(dxp[s])
    for n in ref:
        assert_close(n, np.array(got[n]), np.array(ref[n]), TOL_OUT)
    # weight gradients: a light expert in full, sampled rows of the heaviest
    sx, sh = float(sc(st["xs"])[0]), float(sc(st["hs"])[0])
    sdy, sdh = float(sc(st["sc"][0])[0]), float(sc(st["sc"][2])[0])
    light = int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    heavy = int(np.argmax(counts))
    for e, rows_m in ((light, None), (heavy, np.sort(rng.choice(2 * f, 16, replace=False)))):
        lo, hi = off[e], off[e + 1]
        B1 = _dec(xq[lo:hi]) * sx
        B2 = _dec(hq[lo:hi]) * sh
        if rows_m is None:
            A1 = _dec(dH1q[lo:hi]) * sdh
            A2 = _dec(dyq[lo:hi]) * sdy
            assert_close(f"dW1[{e}]", np64(st["dW1"][e]), A1.T @ B1, TOL_F32)
            assert_close(f"dW2[{e}]", np64(st["dW2"][e]), A2.T @ B2, TOL_F32)
        else:
            rm2 = rows_m[rows_m < d]
            A1 = _dec(dH1q[lo:hi][:, rows_m]) * sdh
            A2 = _dec(dyq[lo:hi][:, rm2]) * sdy
            assert_close(f"dW1[{e}] rows", np64(st["dW1"][e])[rows_m], A1.T @ B1, TOL_F32)
            assert_close(f"dW2[{e}] rows", np64(st["dW2"][e])[rm2], A2.T @ B2, TOL_F32)
