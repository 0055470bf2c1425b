"""Router variants on the GPU against the oracle, through the C ABI: the selection-only expert
bias (routing stage and whole layer), the load-balancing loss (value and gradient), and the
expert-bias update.

Selection is an integer decided in floating point.  Given the same fp32 logits, both sides form
the same fp32 keys (score + bias) up to the last bits of exp/sigmoid, so the chosen experts must
be identical on every row whose k-th/(k+1)-th key gap clears KEY_GAP; on the few rows closer than
that the GPU's choice must be a valid top-k of the oracle's keys within KEY_GAP.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import moe_inputs
import oracle.moe_oracle as O
from moe_inputs import SIGMOID, SOFTMAX, LayerConfig

from .helpers import (MARGIN, TOL, boundary_gap, compare_layer, inputs_to, np64, oracle_layer,
                      run_layer)

pytestmark = pytest.mark.gpu

KEY_GAP = 2e-6


def route_stage(cfg, logits, bias):
    T, E, k = cfg.T, cfg.E, cfg.k
    dev = "cuda"
    i32 = torch.int32
    out = dict(idx=torch.empty(T, k, dtype=i32, device=dev),
               gate=torch.empty(T, k, dtype=torch.float32, device=dev),
               counts=torch.empty(E, dtype=i32, device=dev),
               offsets=torch.empty(E + 1, dtype=i32, device=dev),
               sop=torch.empty(T, k, dtype=i32, device=dev),
               tos=torch.empty(max(T * k, 1), dtype=i32, device=dev))
    ws = moe.workspace(cfg, moe.WS_ROUTE)
    moe.moe_route_topk(cfg, None, None, bias, logits, None, out["idx"], out["gate"],
                       out["counts"], out["offsets"], out["sop"], out["tos"], ws)
    torch.cuda.synchronize()
    moe.check_device_error()
    return {n: np64(v) for n, v in out.items()}


def check_selection(keys, idx, k):
    """Exact on clear rows, a valid top-k within KEY_GAP on the rest; returns #near-tie rows."""
    o_idx = O.select_topk(keys, k).astype(np.int64)
    gap = boundary_gap(keys.astype(np.float64), k)
    clear = gap > KEY_GAP
    assert (np.sort(idx[clear], 1) == np.sort(o_idx[clear], 1)).all()
    for t in np.nonzero(~clear)[0]:
        sel = keys[t, idx[t]].astype(np.float64)
        rest = np.delete(keys[t], idx[t]).astype(np.float64)
        assert len(set(idx[t].tolist())) == k
        if rest.size:
            assert sel.min() >= rest.max() - KEY_GAP, t
    # order inside the set: descending key wherever consecutive keys are clear
    srt = np.take_along_axis(keys.astype(np.float64), idx, 1)
    assert (np.diff(srt, axis=1) <= KEY_GAP).all()
    return int((~clear).sum())


@pytest.mark.parametrize("E,k", [(8, 2), (64, 6), (128, 8), (256, 8), (40, 1)])
@pytest.mark.parametrize("score_fn,renorm", [(SIGMOID, 1), (SIGMOID, 0), (SOFTMAX, 1), (SOFTMAX, 0)])
def test_route_with_selection_bias(E, k, score_fn, renorm):
    T = 4097
    g = torch.Generator().manual_seed(E * 10 + k)
    lg = (torch.randn(T, E, generator=g) * 2.0).float()
    bias = (torch.randn(E, generator=g) * (0.05 if score_fn == SIGMOID else 0.01)).float()
    cfg = moe.make_cfg(T, 128, E, k, 128, score_fn=score_fn, renorm=renorm,
                       bias_mode=moe.BIAS_SELECT)
    r = route_stage(cfg, lg.cuda(), bias.cuda())
    keys = O.selection_keys(lg.numpy(), score_fn, bias.numpy())
    idx = r["idx"].astype(np.int64)
    near = check_selection(keys, idx, k)
    assert near < T // 50
    # the bias must matter: the selection differs from the unbiased one on many rows
    assert (np.sort(idx, 1) != np.sort(O.select_topk(lg.numpy(), k), 1)).any(axis=1).sum() > 10
    # gates: from the logits of the chosen experts, never from the bias
    gate = O.gate_weights(lg.numpy().astype(np.float64), idx, score_fn, renorm)
    assert np.abs(r["gate"] - gate).max() <= 2e-6 * max(1.0, np.abs(gate).max())
    counts, offsets, sop, tos = O.routing_maps(idx, E)
    assert (r["counts"] == counts).all() and (r["offsets"] == offsets).all()
    assert (r["sop"] == sop).all() and (r["tos"][: T * k] == tos).all()


def test_selection_bias_forces_experts_on_gpu():
    T, E, k = 1000, 32, 4
    g = torch.Generator().manual_seed(3)
    lg = (torch.randn(T, E, generator=g) * 3).float()
    bias = torch.zeros(E)
    bias[[5, 17]] = 2.0
    cfg = moe.make_cfg(T, 128, E, k, 128, score_fn=SIGMOID, renorm=1, bias_mode=moe.BIAS_SELECT)
    r = route_stage(cfg, lg.cuda(), bias.cuda())
    assert all({5, 17} <= set(row.tolist()) for row in r["idx"])
    assert (r["counts"][[5, 17]] == T).all()


@pytest.mark.parametrize("score_fn", [SOFTMAX, SIGMOID])
@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (300, 8, 2), (4097, 128, 6), (16384, 256, 8)])
def test_aux_loss_value(score_fn, T, E, k):
    g = torch.Generator().manual_seed(T + E)
    lg = (torch.randn(T, E, generator=g) * 1.5).float()
    cfg = moe.make_cfg(T, 128, E, k, 128, score_fn=score_fn, renorm=1, aux_coeff=1e-2)
    r = route_stage(cfg, lg.cuda(), None)
    out = torch.zeros(4, device="cuda")
    ws = moe.workspace(cfg, moe.WS_ROUTE)
    moe.moe_router_aux_loss(cfg, lg.cuda(), torch.as_tensor(r["counts"]).cuda(), out, ws)
    torch.cuda.synchronize()
    ref = O.aux_loss(lg.numpy().astype(np.float64), r["counts"], k, 1e-2, score_fn)
    assert abs(float(out[0]) - ref) <= 2e-6 * abs(ref), (float(out[0]), ref)
    # rerun: fixed-order sums give the same bits
    out2 = torch.zeros(4, device="cuda")
    moe.moe_router_aux_loss(cfg, lg.cuda(), torch.as_tensor(r["counts"]).cuda(), out2, ws)
    assert torch.equal(out[:1], out2[:1])


def test_aux_loss_uniform_probabilities_is_the_coefficient():
    T, E, k = 5000, 64, 4
    cfg = moe.make_cfg(T, 128, E, k, 128, score_fn=SIGMOID, renorm=1, aux_coeff=1e-4)
    lg = torch.full((T, E), 0.3, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    counts[:k] = T                                   # any counts summing to T*k
    out = torch.zeros(4, device="cuda")
    moe.moe_router_aux_loss(cfg, lg, counts, out, moe.workspace(cfg, moe.WS_ROUTE))
    torch.cuda.synchronize()
    assert abs(float(out[0]) - 1e-4) <= 1e-6 * 1e-4


def test_expert_bias_update_is_exact():
    E, T, k = 256, 4096, 8
    g = torch.Generator().manual_seed(9)
    bias = (torch.randn(E, generator=g) * 0.1).float()
    counts = torch.randint(0, 2 * T * k // E, (E,), generator=g, dtype=torch.int32)
    counts[:3] = T * k // E                          # exactly at the mean: unchanged
    cfg = moe.make_cfg(T, 128, E, k, 128, score_fn=SIGMOID, bias_mode=moe.BIAS_SELECT)
    b = bias.cuda()
    moe.moe_expert_bias_update(cfg, counts.cuda(), b, 1e-3)
    torch.cuda.synchronize()
    ref = O.expert_bias_update(bias.numpy(), counts.numpy(), T, k, 1e-3)
    assert np.array_equal(b.cpu().numpy(), ref)
    assert np.array_equal(b.cpu().numpy()[:3], bias.numpy()[:3])


# ----------------------------------------------------------------------------- whole layer

def clean_select_inputs(lc, tries=80):
    """Inputs whose fp32 selection keys (score + expert bias) keep every row's chosen set clear
    of the next expert by more than the router GEMM's rounding can move them."""
    for s in range(tries):
        inp = moe_inputs.make_layer_inputs(lc, seed=s, device="cpu")
        lg = O.router_logits(np64(inp["x"]), np64(inp["W_r"]))
        keys = O.selection_keys(lg.astype(np.float32), lc.score_fn, np64(inp["b_r"]))
        if boundary_gap(keys.astype(np.float64), lc.k).min() > MARGIN * max(1.0, np.abs(lg).max()):
            return inp, keys
    raise AssertionError("no seed with a clear selection margin")


LAYERS = {
    "fp32_sigmoid_select_aux": LayerConfig("f32 sel aux", 256, 128, 8, 2, 96, score_fn=SIGMOID,
                                           renorm=1, dtype="f32", router_bias="normal0.05",
                                           bias_mode=1, aux_coeff=300.0),
    "fp32_softmax_aux_norenorm": LayerConfig("f32 aux", 200, 64, 6, 3, 64, score_fn=SOFTMAX,
                                             renorm=0, dtype="f32", aux_coeff=300.0),
    "bf16_sigmoid_select_aux_shared": LayerConfig("bf16 sel aux", 700, 256, 32, 6, 128,
                                                  f_shared=128, score_fn=SIGMOID, renorm=1,
                                                  router_bias="normal0.05", bias_mode=1,
                                                  aux_coeff=3000.0),
    "bf16_softmax_select": LayerConfig("bf16 sel", 513, 192, 16, 4, 96, score_fn=SOFTMAX,
                                       renorm=1, router_bias="normal0.05", bias_mode=1),
}


@pytest.mark.parametrize("name", list(LAYERS))
def test_layer_with_router_variants(name):
    lc = LAYERS[name]
    if lc.bias_mode == 1:
        inp, keys = clean_select_inputs(lc)
    else:
        from .helpers import clean_inputs
        inp, _ = clean_inputs(lc)
        keys = None
    gpu = run_layer(lc, inputs_to(inp, "cuda"))
    ref = oracle_layer(lc, inp)
    errs = compare_layer(lc, gpu, ref, TOL[lc.dtype], order_keys=keys)
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})


def test_aux_gradient_alone_reaches_router_only():
    """dy = 0: the only gradient is the balancing loss's, through the router."""
    lc = LAYERS["fp32_sigmoid_select_aux"].replace(aux_coeff=1.0)
    inp, _ = clean_select_inputs(lc)
    inp["dy"] = torch.zeros_like(inp["dy"])
    gpu = run_layer(lc, inputs_to(inp, "cuda"))
    ref = oracle_layer(lc, inp)
    b = ref["bwd"]
    assert np.abs(b["dW_r"]).max() > 0
    for n in ["dx", "dW_r"]:
        e = np.abs(np64(gpu[n]) - b[n]).max() / np.abs(b[n]).max()
        assert e <= 1e-5, (n, e)
    assert float(gpu["dW1"].abs().max()) == 0.0 and float(gpu["dW2"].abs().max()) == 0.0
