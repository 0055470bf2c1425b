"""MXFP8 (block-scaled E4M3) path on the GPU against the MXFP8 oracle, through the C ABI.

  * moe_quantize_mxfp8: codes and E8M0 scale bytes bit-identical to the oracle's block
    quantisation of the same bf16 values (the decisions are exact: a power-of-two division and
    one E4M3 rounding);
  * moe_mxfp8_pack_expert_scales: every scale at its documented place in the packed layout, and
    every other byte 127;
  * moe_permute_quantize_mxfp8: the codes of every permuted row equal the oracle's codes of its
    token's row, and the packed scales read back equal the oracle's;
  * moe_grouped_swiglu_fwd_mxfp8: [a | u] and h within the bf16 output tolerance of the oracle's
    fp64 product of the same decoded operands; h's codes and scales bit-identical to the oracle's
    quantisation of the GPU's bf16 h; y_perm within tolerance of the oracle's fc2 on those codes;
    and against the unquantised bf16 experts within the format's rounding bound;
  * moe_layer_fwd_mxfp8: routing and shared expert identical to the bf16 layer's, y bit-identical
    to the composed stage calls, and within the format's rounding of the unquantised layer;
  * the data gradients: the weights' column-blocked codes and scales bit-identical to the
    oracle's (packed scales at their places), dy's codes bit-identical, [da | du] within the bf16
    tolerance of the oracle's SwiGLU backward of its fc2 data gradient on the same codes, its codes
    bit-identical to the oracle's quantisation of the GPU's bf16 [da | du], dx_perm within the bf16
    tolerance of the oracle's fc1 data gradient of those codes; moe_layer_bwd_mxfp8 against the
    bf16 backward on the same saved state and the unquantised oracle.
Shapes cover several tiles with ragged tails, experts without rows, K not a multiple of 128 (a
partial last scale chunk) and f not a multiple of the 96-column SwiGLU tile.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import moe_inputs
import oracle.moe_oracle as O
import oracle.mxfp8_oracle as MX

import oracle.fp8_oracle as F8

from .helpers import (assert_close, clean_inputs, mx_act_pad_bytes, mx_unpack_act_scales,
                      mx_weight_index, mx_weight_index_cols, np64, oracle_layer, rel_err, run_layer)

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2   # bf16 outputs of an fp32-accumulated product of exact block-scaled E4M3 values


def sync():
    torch.cuda.synchronize()
    moe.check_device_error()


def varied(shape, seed, spread=4.0):
    """bf16 values whose magnitude changes from one 32-block to the next (2^-spread .. 2^spread),
    with some all-zero blocks."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g)
    nb = shape[-1] // 32
    mag = torch.exp2(torch.empty(*shape[:-1], nb).uniform_(-spread, spread, generator=g))
    mag[..., ::7] = 0 if nb > 3 else mag[..., ::7]
    return (x * mag.repeat_interleave(32, dim=-1)).bfloat16()


@pytest.mark.parametrize("rows,cols", [(1, 32), (100, 96), (513, 2688), (64, 1856)])
def test_quantize_codes_and_scales_are_exact(rows, cols):
    x = varied((rows, cols), rows + cols)
    x[0, :4] = torch.tensor([480.0, -448.0, 1e-30, 0.0]).bfloat16()   # saturation, tiny, zero
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, cols // 32, dtype=torch.uint8, device="cuda")
    moe.moe_quantize_mxfp8(x.cuda(), q, s)
    sync()
    rq, rs = MX.mx_quantize(x.double().numpy())
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def mx_experts(cfg, seed, scale=0.05):
    E, d, f = cfg.E, cfg.d, cfg.f
    W1 = (varied((E, 2 * f, d), seed, 2.0).float() * scale).bfloat16().cuda()
    W2 = (varied((E, d, f), seed + 1, 2.0).float() * scale).bfloat16().cuda()
    m = moe.alloc_mxfp8_experts(cfg, W1, W2)
    sync()
    return W1, W2, m


@pytest.mark.parametrize("E,d,f", [(3, 256, 160), (2, 2688, 1856), (4, 384, 96)])
def test_packed_weight_scales_are_at_their_places(E, d, f):
    cfg = moe.make_cfg(64, d, E, 2, f)
    W1, W2, m = mx_experts(cfg, E + d)
    rq1, rs1 = MX.mx_quantize(W1.double().cpu().numpy())
    rq2, rs2 = MX.mx_quantize(W2.double().cpu().numpy())
    assert np.array_equal(m["W1_q"].cpu().numpy(), rq1) and np.array_equal(m["W1_s"].cpu().numpy(), rs1)
    assert np.array_equal(m["W2_q"].cpu().numpy(), rq2) and np.array_equal(m["W2_s"].cpu().numpy(), rs2)
    for packed, rs, R, K, sf in ((m["W1_sp"], rs1, 2 * f, d, f), (m["W2_sp"], rs2, d, f, 0)):
        p = packed.cpu().numpy()
        idx = mx_weight_index(E, R, K, sf)
        assert np.array_equal(p[idx], rs)
        rest = np.ones(p.size, bool)
        rest[idx.ravel()] = False
        assert (p[rest] == 127).all()


def routed(T, E, k, seed, empty=0):
    g = torch.Generator().manual_seed(seed)
    lg = torch.randn(T, E, generator=g)
    if empty:
        lg[:, E - empty:] = -1e4      # the last `empty` experts receive nothing
    return O.route(lg.numpy(), k, E, O.SOFTMAX, 1)


@pytest.mark.parametrize("T,d,E,k,empty", [(1000, 256, 16, 4, 3), (4097, 2048, 128, 8, 0),
                                           (7, 64, 4, 1, 0), (300, 2688, 8, 6, 1), (900, 224, 256, 8, 30)])
def test_permute_quantize_mx(T, d, E, k, empty):
    r = routed(T, E, k, T, empty)
    x = varied((T, d), d).cuda()
    cfg = moe.make_cfg(T, d, E, k, 64)
    N = T * k
    sop = torch.from_numpy(r["slot_of_pair"]).cuda()
    off = torch.from_numpy(r["offsets"]).cuda()
    xq = torch.empty(N, d, dtype=torch.uint8, device="cuda")
    xs = torch.full((moe.mxfp8_scale_bytes(cfg, moe.MX_SCALES_X),), 0xEE, dtype=torch.uint8,
                    device="cuda")
    moe.moe_permute_quantize_mxfp8(cfg, x, sop, off, xq, xs)
    sync()
    rq, rs = MX.mx_quantize(x.double().cpu().numpy())
    tos = r["token_of_slot"]
    assert np.array_equal(xq.cpu().numpy(), rq[tos])
    p = xs.cpu().numpy()
    assert np.array_equal(mx_unpack_act_scales(p, r["offsets"], N, d), rs[tos])
    assert (mx_act_pad_bytes(p, r["offsets"], N, d) == 127).all()


@pytest.mark.parametrize("T,d,E,k,f,empty", [(600, 256, 8, 2, 160, 2), (1024, 2048, 128, 8, 768, 0),
                                             (300, 384, 16, 4, 96, 5), (257, 2688, 8, 6, 1856, 0),
                                             (700, 224, 256, 8, 128, 40), (129, 96, 3, 3, 32, 0)])
def test_mxfp8_grouped_swiglu_forward(T, d, E, k, f, empty):
    r = routed(T, E, k, d + f, empty)
    N = T * k
    o = r["offsets"]
    cfg = moe.make_cfg(T, d, E, k, f)
    x = varied((T, d), T).cuda()
    W1, W2, m = mx_experts(cfg, d)
    sop = torch.from_numpy(r["slot_of_pair"]).cuda()
    off = torch.from_numpy(o).cuda()
    moe.moe_permute_quantize_mxfp8(cfg, x, sop, off, m["x_perm_q"], m["x_perm_s"])
    bf = torch.bfloat16
    h = torch.empty(N, f, dtype=bf, device="cuda")
    act = torch.empty(N, 2 * f, dtype=bf, device="cuda")
    yp = torch.empty(N, d, dtype=bf, device="cuda")
    moe.moe_grouped_swiglu_fwd_mxfp8(cfg, m["x_perm_q"], m["x_perm_s"], off, m["W1_q"], m["W1_sp"],
                                     m["W2_q"], m["W2_sp"], h, act, m["h_q"], m["h_s"], yp)
    sync()
    xq = m["x_perm_q"].cpu().numpy()
    xs = mx_unpack_act_scales(m["x_perm_s"].cpu().numpy(), o, N, d)
    W1q, W1s = m["W1_q"].cpu().numpy(), m["W1_s"].cpu().numpy()
    W2q, W2s = m["W2_q"].cpu().numpy(), m["W2_s"].cpu().numpy()
    ref_h, ref_act = MX.fc1_swiglu_mx(xq, xs, W1q, W1s, o)
    e_act = assert_close("act", np64(act), ref_act, TOL_OUT)
    e_h = assert_close("h", np64(h), ref_h, TOL_OUT)
    # h's codes and scales: the oracle's block quantisation of the GPU's (bf16) h
    rq, rs = MX.mx_quantize(np64(h))
    assert np.array_equal(m["h_q"].cpu().numpy(), rq)
    hs = m["h_s"].cpu().numpy()
    assert np.array_equal(mx_unpack_act_scales(hs, o, N, f), rs)
    assert (mx_act_pad_bytes(hs, o, N, f) == 127).all()
    ref_y = MX.fc2_mx(rq, rs, W2q, W2s, o)
    e_y = assert_close("y_perm", np64(yp), ref_y, TOL_OUT)
    # against the unquantised experts: four E4M3 roundings (x, W1, h, W2), each within 2^-4
    # of its value (3 mantissa bits); on these inputs the result moves by 6-10%
    X = np64(x)[r["token_of_slot"]]
    y_bf = np.zeros((N, d))
    for e in range(E):
        sl = slice(o[e], o[e + 1])
        if o[e + 1] > o[e]:
            y_bf[sl] = O.swiglu_ffn(np64(W1[e]), np64(W2[e]), X[sl])[0]
    e_q = rel_err(np64(yp), y_bf)
    assert e_q < 0.25, e_q
    print(f"act {e_act:.2e} h {e_h:.2e} y {e_y:.2e}; vs unquantised {e_q:.3f}")


def test_mxfp8_forward_without_bf16_side_outputs_and_zero_tokens():
    """h and [a | u] are optional (NULL): the codes and y_perm are the same; T = 0 is a no-op."""
    T, d, E, k, f = 200, 256, 8, 2, 128
    r = routed(T, E, k, 3)
    cfg = moe.make_cfg(T, d, E, k, f)
    x = varied((T, d), 5).cuda()
    W1, W2, m = mx_experts(cfg, 9)
    sop = torch.from_numpy(r["slot_of_pair"]).cuda()
    off = torch.from_numpy(r["offsets"]).cuda()
    moe.moe_permute_quantize_mxfp8(cfg, x, sop, off, m["x_perm_q"], m["x_perm_s"])
    N = T * k
    outs = []
    for with_h in (True, False):
        h = torch.empty(N, f, dtype=torch.bfloat16, device="cuda") if with_h else None
        yp = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
        moe.moe_grouped_swiglu_fwd_mxfp8(cfg, m["x_perm_q"], m["x_perm_s"], off, m["W1_q"],
                                         m["W1_sp"], m["W2_q"], m["W2_sp"], h, None, m["h_q"],
                                         m["h_s"], yp)
        sync()
        outs.append((m["h_q"].clone(), yp))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    cfg0 = moe.make_cfg(0, d, E, k, f)
    moe.moe_grouped_swiglu_fwd_mxfp8(cfg0, m["x_perm_q"], m["x_perm_s"], off, m["W1_q"], m["W1_sp"],
                                     m["W2_q"], m["W2_sp"], None, None, m["h_q"], m["h_s"], outs[0][1])
    sync()


LAYER_CASES = {
    # the DeepSeek-style layer's kind (sigmoid + renorm, Zipf-biased router, ungated shared
    # expert) and the MTP kind (softmax, gated shared expert), at sizes the oracle runs quickly
    "sigmoid-shared": moe_inputs.LayerConfig("mx sigmoid shared", 300, 256, 16, 4, 160, f_shared=128,
                                             score_fn=O.SIGMOID, renorm=1, router_bias="zipf1.2"),
    "softmax-gated": moe_inputs.LayerConfig("mx softmax gated", 257, 384, 32, 8, 96, f_shared=64,
                                            score_fn=O.SOFTMAX, renorm=1, shared_gate=1,
                                            router_init="uniform"),
    "no-shared": moe_inputs.LayerConfig("mx plain", 500, 2688, 8, 2, 1856),
    # d = 224 and 2f = 192: the last 128-wide scale chunk of a row is partly padding
    "ragged-d": moe_inputs.LayerConfig("mx ragged d", 131, 224, 8, 3, 96, f_shared=64,
                                       score_fn=O.SOFTMAX, renorm=1, shared_gate=1),
}


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_mxfp8_layer_forward_is_the_composed_stages(name):
    """moe_layer_fwd_mxfp8 = the bf16 layer's routing and shared expert + the MXFP8 stage calls +
    the combine, bit for bit; and within the format's rounding of the unquantised oracle layer."""
    lc = LAYER_CASES[name]
    inp = {k: (None if v is None else v.cuda())
           for k, v in moe_inputs.make_layer_inputs(lc, seed=1).items()}
    ref16 = run_layer(lc, inp, backward=False)
    cfg = moe.cfg_from(lc)
    m = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"])
    saved = moe.alloc_saved(cfg)
    saved["x_perm"] = saved["act"] = saved["h"] = None
    y = torch.empty_like(inp["x"])
    moe.moe_layer_fwd_mxfp8(cfg, inp["x"], inp["W_r"], inp["b_r"], m, inp["Ws1"], inp["Ws2"],
                            inp["w_sg"], y, saved, moe.workspace(cfg, moe.WS_LAYER_FWD))
    sync()
    s16 = ref16["saved"]
    for key in ("logits", "idx", "gate", "counts", "offsets", "slot_of_pair", "token_of_slot"):
        assert torch.equal(saved[key], s16[key]), key
    if lc.f_shared:
        assert torch.equal(saved["s_out"], s16["s_out"])
    # the same call composed from the stage functions
    N = lc.T * lc.k
    xq = torch.empty_like(m["x_perm_q"])
    xs = torch.empty_like(m["x_perm_s"])
    moe.moe_permute_quantize_mxfp8(cfg, inp["x"], s16["slot_of_pair"], s16["offsets"], xq, xs)
    hq, hs = torch.empty_like(m["h_q"]), torch.empty_like(m["h_s"])
    yp = torch.empty(N, lc.d, dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_swiglu_fwd_mxfp8(cfg, xq, xs, s16["offsets"], m["W1_q"], m["W1_sp"], m["W2_q"],
                                     m["W2_sp"], None, None, hq, hs, yp)
    yc = torch.empty_like(y)
    moe.moe_unpermute_combine(cfg, yp, s16["gate"], s16["slot_of_pair"],
                              s16["s_out"] if lc.f_shared else None,
                              s16["s_coef"] if lc.shared_gate else None, yc)
    sync()
    assert torch.equal(m["x_perm_q"], xq) and torch.equal(m["h_q"], hq)
    assert torch.equal(saved["y_perm"], yp) and torch.equal(y, yc)
    # against the unquantised fp64 layer
    ref = oracle_layer(lc, {k: (None if v is None else v.cpu()) for k, v in inp.items()},
                       backward=False)
    e = rel_err(np64(y), ref["fwd"]["y"])
    assert e < 0.15, e
    print(f"{name}: y vs unquantised {e:.3f}")


def test_mxfp8_forward_saves_the_bf16_state_for_the_bf16_backward():
    """With saved.x_perm / act / h given, moe_layer_fwd_mxfp8 writes the permuted bf16 rows, the bf16
    [a | u] and h of its MXFP8 products (bit-identical to the stage calls), y is unchanged, and
    moe_layer_bwd on that state gives gradients within the forward's rounding of the oracle's."""
    lc = LAYER_CASES["sigmoid-shared"]
    host, _ = clean_inputs(lc)       # routing clear of near-ties: the oracle selects the same sets
    inp = {k: (None if v is None else v.cuda()) for k, v in host.items()}
    cfg = moe.cfg_from(lc)
    m = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"])
    ws_f = moe.workspace(cfg, moe.WS_LAYER_FWD)
    lean = moe.alloc_saved(cfg)
    lean["x_perm"] = lean["act"] = lean["h"] = None
    y0 = torch.empty_like(inp["x"])
    moe.moe_layer_fwd_mxfp8(cfg, inp["x"], inp["W_r"], inp["b_r"], m, inp["Ws1"], inp["Ws2"],
                            inp["w_sg"], y0, lean, ws_f)
    saved = moe.alloc_saved(cfg)
    y = torch.empty_like(inp["x"])
    moe.moe_layer_fwd_mxfp8(cfg, inp["x"], inp["W_r"], inp["b_r"], m, inp["Ws1"], inp["Ws2"],
                            inp["w_sg"], y, saved, ws_f)
    sync()
    assert torch.equal(y, y0)
    xp = torch.empty_like(saved["x_perm"])
    moe.moe_permute(cfg, inp["x"], saved["slot_of_pair"], xp)
    h = torch.empty_like(saved["h"])
    act = torch.empty_like(saved["act"])
    moe.moe_grouped_swiglu_fwd_mxfp8(cfg, m["x_perm_q"], m["x_perm_s"], saved["offsets"], m["W1_q"],
                                     m["W1_sp"], m["W2_q"], m["W2_sp"], h, act,
                                     torch.empty_like(m["h_q"]), torch.empty_like(m["h_s"]),
                                     torch.empty_like(saved["y_perm"]))
    sync()
    assert torch.equal(saved["x_perm"], xp)
    assert torch.equal(saved["h"], h) and torch.equal(saved["act"], act)
    f32 = torch.float32
    E, d, f, fs = lc.E, lc.d, lc.f, lc.f_shared
    g = dict(dx=torch.empty_like(inp["x"]), dW_r=torch.empty(E, d, dtype=f32, device="cuda"),
             dW1=torch.empty(E, 2 * f, d, dtype=f32, device="cuda"),
             dW2=torch.empty(E, d, f, dtype=f32, device="cuda"),
             dWs1=torch.empty(2 * fs, d, dtype=f32, device="cuda"),
             dWs2=torch.empty(d, fs, dtype=f32, device="cuda"))
    moe.moe_layer_bwd(cfg, inp["dy"], inp["x"], inp["W_r"], inp["W1"], inp["W2"], inp["Ws1"],
                      inp["Ws2"], None, saved, g["dx"], g["dW_r"], g["dW1"], g["dW2"], g["dWs1"],
                      g["dWs2"], None, moe.workspace(cfg, moe.WS_LAYER_BWD))
    sync()
    ref = oracle_layer(lc, {k: (None if v is None else v.cpu()) for k, v in inp.items()})
    errs = {}
    for name in ("dx", "dW1", "dW2", "dW_r", "dWs1", "dWs2"):
        gpu = np64(g[name])
        assert np.isfinite(gpu).all(), name
        errs[name] = rel_err(gpu, ref["bwd"][name])
        assert errs[name] < 0.15, (name, errs[name])
    print("mxfp8 forward + bf16 backward vs unquantised:", {k: f"{v:.3f}" for k, v in errs.items()})


@pytest.mark.parametrize("E,d,f", [(3, 256, 160), (2, 2688, 1856), (4, 224, 96)])
def test_dgrad_weight_copies(E, d, f):
    cfg = moe.make_cfg(64, d, E, 2, f)
    W1 = (varied((E, 2 * f, d), d, 2.0).float() * 0.05).bfloat16().cuda()
    W2 = (varied((E, d, f), d + 1, 2.0).float() * 0.05).bfloat16().cuda()
    m = moe.alloc_mxfp8_dgrad(cfg, W1, W2)
    sync()
    for W, pre, K, N, tile in ((W1, "W1c", 2 * f, d, 256), (W2, "W2c", d, f, 128)):
        rq, rs = MX.mx_quantize_cols(W.double().cpu().numpy())
        assert np.array_equal(m[pre + "_q"].cpu().numpy(), rq)
        assert np.array_equal(m[pre + "_s"].cpu().numpy(), rs)
        p = m[pre + "_sp"].cpu().numpy()
        idx = mx_weight_index_cols(E, N, K, tile)
        assert np.array_equal(p[idx], rs)
        rest = np.ones(p.size, bool)
        rest[idx.ravel()] = False
        assert (p[rest] == 127).all()


@pytest.mark.parametrize("T,d,E,k,f,empty", [(600, 256, 8, 2, 160, 2), (1024, 2048, 128, 8, 768, 0),
                                             (257, 2688, 8, 6, 1856, 0), (700, 224, 256, 8, 128, 40)])
def test_mxfp8_data_gradients(T, d, E, k, f, empty):
    r = routed(T, E, k, d + f + 1, empty)
    N = T * k
    o = r["offsets"]
    cfg = moe.make_cfg(T, d, E, k, f)
    W1 = (varied((E, 2 * f, d), d, 2.0).float() * 0.05).bfloat16().cuda()
    W2 = (varied((E, d, f), d + 1, 2.0).float() * 0.05).bfloat16().cuda()
    m = moe.alloc_mxfp8_dgrad(cfg, W1, W2)
    dyp = varied((N, d), N).cuda()
    g = torch.Generator().manual_seed(N)
    act = (torch.randn(N, 2 * f, generator=g) * 2).bfloat16().cuda()
    off = torch.from_numpy(o).cuda()
    dH1 = torch.empty(N, 2 * f, dtype=torch.bfloat16, device="cuda")
    dxp = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_swiglu_dgrad_mxfp8(cfg, dyp, off, act, m, dH1, dxp)
    sync()
    # dy's codes and scales
    rq, rs = MX.mx_quantize(np64(dyp))
    assert np.array_equal(m["dy_q"].cpu().numpy(), rq)
    assert np.array_equal(mx_unpack_act_scales(m["dy_s"].cpu().numpy(), o, N, d), rs)
    # fc2's data gradient and the SwiGLU backward on those codes
    W2cq, W2cs = m["W2c_q"].cpu().numpy(), m["W2c_s"].cpu().numpy()
    dh = MX.fc2_dgrad_mx(rq, rs, W2cq, W2cs, o)
    ref_dH1 = F8.swiglu_backward(dh, np64(act))
    e_dh1 = assert_close("dH1", np64(dH1), ref_dH1, TOL_OUT)
    # [da | du]'s codes and scales: the oracle's quantisation of the GPU's bf16 [da | du]
    hq, hs = MX.mx_quantize(np64(dH1))
    assert np.array_equal(m["dH1_q"].cpu().numpy(), hq)
    dhs = m["dH1_s"].cpu().numpy()
    assert np.array_equal(mx_unpack_act_scales(dhs, o, N, 2 * f), hs)
    assert (mx_act_pad_bytes(dhs, o, N, 2 * f) == 127).all()
    ref_dx = MX.fc1_dgrad_mx(hq, hs, m["W1c_q"].cpu().numpy(), m["W1c_s"].cpu().numpy(), o)
    e_dx = assert_close("dx_perm", np64(dxp), ref_dx, TOL_OUT)
    print(f"dH1 {e_dh1:.2e} dx_perm {e_dx:.2e}")


@pytest.mark.parametrize("name", ["sigmoid-shared", "ragged-d"])
def test_mxfp8_layer_backward(name):
    """moe_layer_bwd_mxfp8 after moe_layer_fwd_mxfp8: the weight gradients and dx against the bf16
    backward on the same saved state (they differ by the data gradients' MXFP8 rounding) and
    against the unquantised oracle."""
    lc = LAYER_CASES[name]
    host, _ = clean_inputs(lc)
    inp = {k: (None if v is None else v.cuda()) for k, v in host.items()}
    cfg = moe.cfg_from(lc)
    m = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"])
    mxd = moe.alloc_mxfp8_dgrad(cfg, inp["W1"], inp["W2"])
    saved = moe.alloc_saved(cfg)
    y = torch.empty_like(inp["x"])
    moe.moe_layer_fwd_mxfp8(cfg, inp["x"], inp["W_r"], inp["b_r"], m, inp["Ws1"], inp["Ws2"],
                            inp["w_sg"], y, saved, moe.workspace(cfg, moe.WS_LAYER_FWD))
    f32 = torch.float32
    E, d, f, fs = lc.E, lc.d, lc.f, lc.f_shared

    def grads():
        return dict(dx=torch.empty_like(inp["x"]), dW_r=torch.empty(E, d, dtype=f32, device="cuda"),
                    dW1=torch.empty(E, 2 * f, d, dtype=f32, device="cuda"),
                    dW2=torch.empty(E, d, f, dtype=f32, device="cuda"),
                    dWs1=torch.empty(2 * fs, d, dtype=f32, device="cuda"),
                    dWs2=torch.empty(d, fs, dtype=f32, device="cuda"),
                    dw_sg=torch.empty(d, dtype=f32, device="cuda") if lc.shared_gate else None)
    ws = moe.workspace(cfg, moe.WS_LAYER_BWD)
    g16, gmx = grads(), grads()
    moe.moe_layer_bwd(cfg, inp["dy"], inp["x"], inp["W_r"], inp["W1"], inp["W2"], inp["Ws1"],
                      inp["Ws2"], inp["w_sg"], saved, g16["dx"], g16["dW_r"], g16["dW1"],
                      g16["dW2"], g16["dWs1"], g16["dWs2"], g16["dw_sg"], ws)
    moe.moe_layer_bwd_mxfp8(cfg, inp["dy"], inp["x"], inp["W_r"], mxd, inp["Ws1"], inp["Ws2"],
                            inp["w_sg"], saved, gmx["dx"], gmx["dW_r"], gmx["dW1"], gmx["dW2"],
                            gmx["dWs1"], gmx["dWs2"], gmx["dw_sg"], ws)
    sync()
    # dy_perm's codes and scales, written by the combine backward: the oracle's quantisation of
    # dy_perm[slot(t, j)] = bf16(gate[t, j] * dy[t]) (an fp32 product rounded once, as stored)
    N = lc.T * lc.k
    sop = np64(saved["slot_of_pair"]).astype(np.int64).reshape(-1)
    prod = (saved["gate"].cpu().float()[..., None] * inp["dy"].cpu().float()[:, None, :])
    dy_perm = np.zeros((N, d))
    dy_perm[sop] = np64(prod.to(torch.bfloat16).reshape(N, d))
    rq, rs = MX.mx_quantize(dy_perm)
    o = np64(saved["offsets"]).astype(np.int64)
    assert np.array_equal(mxd["dy_q"].cpu().numpy(), rq)
    assert np.array_equal(mx_unpack_act_scales(mxd["dy_s"].cpu().numpy(), o, N, d), rs)
    assert (mx_act_pad_bytes(mxd["dy_s"].cpu().numpy(), o, N, d) == 127).all()
    # the router's and shared expert's gradients do not depend on the routed data gradients
    for g in ("dW_r", "dWs1", "dWs2", "dW2") + (("dw_sg",) if lc.shared_gate else ()):
        assert torch.equal(gmx[g], g16[g]), g
    ref = oracle_layer(lc, {k: (None if v is None else v.cpu()) for k, v in inp.items()})
    errs = {}
    for g in ("dx", "dW1"):
        errs[g + " vs bf16"] = rel_err(np64(gmx[g]), np64(g16[g]))
        assert errs[g + " vs bf16"] < 0.1, errs
        errs[g + " vs oracle"] = rel_err(np64(gmx[g]), ref["bwd"][g])
        assert errs[g + " vs oracle"] < 0.15, errs
    print("mxfp8 layer backward:", {k: f"{v:.3f}" for k, v in errs.items()})
