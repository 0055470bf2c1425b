"""The layer with FP8 routed experts (moe_layer_fwd_fp8 / moe_layer_bwd_fp8) through the C ABI.

The FP8 expert stages are checked against the oracle in test_gpu_fp8.py; here the layer's wiring:
  * routing identical to the bf16 layer's (same kernels, same logits);
  * every FP8 buffer and output bit-identical to the stage calls composed by hand on the
    layer's own routing (permute + quantise, FP8 experts, combine; combine backward, FP8 expert
    backward);
  * with the shared expert in FP8: its outputs, codes and weight gradients bit-identical to the
    FP8 stage calls on one group of all tokens (x's codes in token order);
  * router gradients (and a bf16 shared expert's) bit-identical to the bf16 layer backward run on
    the same saved forward state (they do not depend on the routed experts' backward);
  * y and dx within the E4M3 rounding bound of the unquantised fp64 oracle layer.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import moe_inputs

from .helpers import clean_inputs, inputs_to, np64, oracle_layer, rel_err

pytestmark = pytest.mark.gpu

CASES = [
    moe_inputs.DEEPSEEK_128E.replace(name="deepseek-style small T512 d256 E16 top4 f128 s128",
                                     T=512, d=256, E=16, k=4, f=128, f_shared=128),
    moe_inputs.MTP_256E.replace(name="mtp-style small T384 d128 E32 top8 f64 s64 gate",
                                T=384, d=128, E=32, k=8, f=64, f_shared=64),
    moe_inputs.QWEN3_30B_A3B.replace(name="qwen3-style small T300 d384 E24 top4 f144",
                                     T=300, d=384, E=24, k=4, f=144, backward=True),
    moe_inputs.MTP_256E.replace(name="mtp-e256 small T400 d128 E256 top8 f64 s64 gate",
                                T=400, d=128, E=256, k=8, f=64, f_shared=64),
]


def run_fp8_layer(lc, inp, cfg, sfp8=False):
    dev = inp["x"].device
    saved = moe.alloc_saved(cfg, dev)
    saved["x_perm"] = None                              # the FP8 layer does not use it
    q = moe.alloc_fp8_experts(cfg, inp["W1"], inp["W2"], dev,
                              Ws1=inp["Ws1"] if sfp8 else None, Ws2=inp["Ws2"] if sfp8 else None)
    y = torch.empty_like(inp["x"])
    moe.moe_layer_fwd_fp8(cfg, inp["x"], inp["W_r"], inp["b_r"], q, inp["Ws1"], inp["Ws2"],
                          inp["w_sg"], y, saved, moe.workspace(cfg, moe.WS_LAYER_FWD, dev))
    E, d, f, fs = cfg.E, cfg.d, cfg.f, cfg.f_shared
    f32 = torch.float32
    g = dict(dx=torch.empty_like(inp["x"]), dW_r=torch.empty(E, d, dtype=f32, device=dev),
             dW1=torch.empty(E, 2 * f, d, dtype=f32, device=dev),
             dW2=torch.empty(E, d, f, dtype=f32, device=dev),
             dWs1=torch.empty(2 * fs, d, dtype=f32, device=dev) if fs else None,
             dWs2=torch.empty(d, fs, dtype=f32, device=dev) if fs else None,
             dw_sg=torch.empty(d, dtype=f32, device=dev) if cfg.shared_gate else None)
    moe.moe_layer_bwd_fp8(cfg, inp["dy"], inp["x"], inp["W_r"], q, inp["Ws1"], inp["Ws2"],
                          inp["w_sg"], saved, g["dx"], g["dW_r"], g["dW1"], g["dW2"], g["dWs1"],
                          g["dWs2"], g["dw_sg"], moe.workspace(cfg, moe.WS_LAYER_BWD_FP8, dev))
    torch.cuda.synchronize()
    moe.check_device_error()
    return y, saved, q, g


PARAMS = [(lc, False) for lc in CASES] + [(lc, True) for lc in CASES if lc.f_shared]


@pytest.mark.parametrize("lc,sfp8", PARAMS,
                         ids=lambda v: v.name.split()[0] if hasattr(v, "name") else
                         ("shared-fp8" if v else "shared-bf16"))
def test_fp8_layer(lc, sfp8):
    cpu_inp, _ = clean_inputs(lc)
    inp = inputs_to(cpu_inp, "cuda")
    cfg = moe.cfg_from(lc)
    y, saved, q, g = run_fp8_layer(lc, inp, cfg, sfp8)
    dev = "cuda"
    N, d, f, E = lc.N, lc.d, lc.f, lc.E
    bf, u8 = torch.bfloat16, torch.uint8

    # routing: the bf16 layer's, bit for bit
    ref_saved = moe.alloc_saved(cfg, dev)
    y16 = torch.empty_like(inp["x"])
    moe.moe_layer_fwd(cfg, inp["x"], inp["W_r"], inp["b_r"], inp["W1"], inp["W2"], inp["Ws1"],
                      inp["Ws2"], inp["w_sg"], y16, ref_saved, moe.workspace(cfg, moe.WS_LAYER_FWD))
    for n in ("logits", "idx", "gate", "counts", "offsets", "slot_of_pair", "token_of_slot"):
        assert torch.equal(saved[n], ref_saved[n]), n

    # forward: the stage calls on the layer's routing
    sop, off = saved["slot_of_pair"], saved["offsets"]
    xq, xs, xa = torch.empty(N, d, dtype=u8, device=dev), torch.empty(4, device=dev), torch.empty(4, device=dev)
    moe.moe_permute_quantize_e4m3(cfg, inp["x"], sop, xq, xs, xa)
    h, act = torch.empty(N, f, dtype=bf, device=dev), torch.empty(N, 2 * f, dtype=bf, device=dev)
    hq, hs, ha = torch.empty(N, f, dtype=u8, device=dev), torch.empty(4, device=dev), torch.empty(4, device=dev)
    yp = torch.empty(N, d, dtype=bf, device=dev)
    moe.moe_grouped_swiglu_fwd_fp8(cfg, xq, xs, off, q["W1_q"], q["W1_scale"], q["W2_q"],
                                   q["W2_scale"], h, act, hq, hs, ha, yp)
    y2 = torch.empty_like(y)
    moe.moe_unpermute_combine(cfg, yp, saved["gate"], sop, saved["s_out"], saved["s_coef"], y2)
    torch.cuda.synchronize()
    assert torch.equal(q["x_perm_q"], xq) and torch.equal(q["h_q"], hq)
    assert torch.equal(q["scales"][:4], torch.stack([xs[0], xa[0], hs[0], ha[0]]))
    for a, b, n in ((saved["act"], act, "act"), (saved["h"], h, "h"), (saved["y_perm"], yp, "y_perm"),
                    (y, y2, "y")):
        assert torch.equal(a, b), n

    # backward: combine backward + the FP8 expert backward on the layer's state
    dyp = torch.empty(N, d, dtype=bf, device=dev)
    dgate = torch.empty(lc.T, lc.k, device=dev)
    dsh = torch.empty_like(inp["x"]) if lc.f_shared else None
    dcoef = torch.empty(lc.T, device=dev) if lc.shared_gate else None
    moe.moe_unpermute_combine_bwd(cfg, inp["dy"], saved["y_perm"], saved["gate"], sop,
                                  saved["s_out"], saved["s_coef"], dyp, dgate, dsh, dcoef)
    dyq, dH1q = torch.empty(N, d, dtype=u8, device=dev), torch.empty(N, 2 * f, dtype=u8, device=dev)
    dH1, dxp = torch.empty(N, 2 * f, dtype=bf, device=dev), torch.empty(N, d, dtype=bf, device=dev)
    sc = [torch.empty(4, device=dev) for _ in range(4)]
    dW1, dW2 = torch.empty_like(g["dW1"]), torch.empty_like(g["dW2"])
    x_scale, h_scale = q["scales"][0:1].clone(), q["scales"][2:3].clone()   # 16-byte aligned
    moe.moe_grouped_swiglu_bwd_fp8(cfg, q["x_perm_q"], x_scale, off, q["W1_q"], q["W1_scale"],
                                   q["W2_q"], q["W2_scale"], saved["act"], q["h_q"], h_scale, dyp,
                                   dyq, sc[0], sc[1], dH1, dH1q, sc[2], sc[3], dxp, dW1, dW2,
                                   moe.workspace(cfg, moe.WS_FFN_BWD_FP8))
    torch.cuda.synchronize()
    moe.check_device_error()
    assert torch.equal(g["dW1"], dW1) and torch.equal(g["dW2"], dW2)
    assert torch.equal(q["scales"][4:8], torch.stack([sc[0][0], sc[1][0], sc[2][0], sc[3][0]]))

    # router and shared-expert gradients: the bf16 backward on the same saved forward state
    saved16 = dict(saved)
    saved16["x_perm"] = torch.empty(N, d, dtype=bf, device=dev)
    moe.moe_permute(cfg, inp["x"], sop, saved16["x_perm"])
    g16 = {k: (None if v is None else torch.empty_like(v)) for k, v in g.items()}
    moe.moe_layer_bwd(cfg, inp["dy"], inp["x"], inp["W_r"], inp["W1"], inp["W2"], inp["Ws1"],
                      inp["Ws2"], inp["w_sg"], saved16, g16["dx"], g16["dW_r"], g16["dW1"],
                      g16["dW2"], g16["dWs1"], g16["dWs2"], g16["dw_sg"],
                      moe.workspace(cfg, moe.WS_LAYER_BWD))
    torch.cuda.synchronize()
    moe.check_device_error()
    for n in ("dW_r", "dw_sg") + (() if sfp8 else ("dWs1", "dWs2")):
        if g[n] is not None:
            assert torch.equal(g[n], g16[n]), n

    if sfp8:
        # the shared expert: FP8 stage calls on one group of all T tokens
        T, fs = lc.T, lc.f_shared
        tos = saved["token_of_slot"][:N].long()
        assert torch.equal(q["x_q"][tos], q["x_perm_q"])         # x's codes in token order
        cfg1 = moe.make_cfg(T, d, 1, 1, fs)
        off1 = torch.tensor([0, T], dtype=torch.int32, device=dev)
        x_scale = q["scales"][0:1].clone()
        sh_, sa_ = torch.empty(T, fs, dtype=bf, device=dev), torch.empty(T, 2 * fs, dtype=bf, device=dev)
        shq = torch.empty(T, fs, dtype=u8, device=dev)
        shs, sha = torch.empty(4, device=dev), torch.empty(4, device=dev)
        so = torch.empty(T, d, dtype=bf, device=dev)
        moe.moe_grouped_swiglu_fwd_fp8(cfg1, q["x_q"], x_scale, off1, q["Ws1_q"], q["Ws1_scale"],
                                       q["Ws2_q"], q["Ws2_scale"], sh_, sa_, shq, shs, sha, so)
        sdyq, sdH1q = torch.empty(T, d, dtype=u8, device=dev), torch.empty(T, 2 * fs, dtype=u8, device=dev)
        sdH1, sdx = torch.empty(T, 2 * fs, dtype=bf, device=dev), torch.empty(T, d, dtype=bf, device=dev)
        ssc = [torch.empty(4, device=dev) for _ in range(4)]
        dWs1, dWs2 = torch.empty_like(g["dWs1"]), torch.empty_like(g["dWs2"])
        moe.moe_grouped_swiglu_bwd_fp8(cfg1, q["x_q"], x_scale, off1, q["Ws1_q"], q["Ws1_scale"],
                                       q["Ws2_q"], q["Ws2_scale"], sa_, shq, shs, dsh, sdyq,
                                       ssc[0], ssc[1], sdH1, sdH1q, ssc[2], ssc[3], sdx, dWs1, dWs2,
                                       moe.workspace(cfg1, moe.WS_FFN_BWD_FP8))
        torch.cuda.synchronize()
        moe.check_device_error()
        for a, b, n in ((saved["s_h"], sh_, "s_h"), (saved["s_act"], sa_, "s_act"),
                        (saved["s_out"], so, "s_out"), (q["s_h_q"], shq, "s_h_q"),
                        (g["dWs1"], dWs1, "dWs1"), (g["dWs2"], dWs2, "dWs2")):
            assert torch.equal(a, b), n
        assert torch.equal(q["scales"][8:14], torch.stack(
            [shs[0], sha[0], ssc[0][0], ssc[1][0], ssc[2][0], ssc[3][0]]))

    # against the unquantised fp64 layer: E4M3 rounding (3 mantissa bits) of x, h, the
    # weights, dy_perm and [da | du]
    ref = oracle_layer(lc, cpu_inp)
    e = {"y": rel_err(np64(y), ref["fwd"]["y"]), "dx": rel_err(np64(g["dx"]), ref["bwd"]["dx"]),
         "dW1": rel_err(np64(g["dW1"]), ref["bwd"]["dW1"]),
         "dW2": rel_err(np64(g["dW2"]), ref["bwd"]["dW2"])}
    if sfp8:
        e.update(dWs1=rel_err(np64(g["dWs1"]), ref["bwd"]["dWs1"]),
                 dWs2=rel_err(np64(g["dWs2"]), ref["bwd"]["dWs2"]))
    assert max(e.values()) < 0.15, e
    print(lc.name, {k: round(v, 4) for k, v in e.items()})


def test_fp8_layer_zero_tokens():
    lc = CASES[1].replace(T=0)
    cfg = moe.cfg_from(lc)
    # buffers of one row, a layer of zero tokens: nothing may be read or written per token
    inp = inputs_to(moe_inputs.make_layer_inputs(lc.replace(T=1), seed=1), "cuda")
    y, saved, q, g = run_fp8_layer(lc, inp, cfg, sfp8=True)
    assert int(saved["offsets"].abs().sum()) == 0
    for n in ("dW_r", "dW1", "dW2", "dWs1", "dWs2", "dw_sg"):
        assert not g[n].any(), n
