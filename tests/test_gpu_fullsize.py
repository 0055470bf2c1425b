"""Parity at the benchmark workloads' full sizes, in the configuration bench.py times (the same
device-generated seeded inputs, the same C-ABI calls), against the oracle on what it can
compute one piece at a time:

  * router logits for every token (fp64 matmul) within the logit tolerance;
  * expert selection equal to the oracle's on every row whose k-th/(k+1)-th logit gap clears
    twice the measured logit error; on the few near-tie rows the GPU's set must be a valid top-k
    (its weakest selected logit is within that error of the strongest unselected one);
  * counts, offsets and both slot maps exactly the stable counting sort of the selection;
  * y and dx on sampled tokens (whole forward and backward of those tokens, their experts,
    the shared expert and the router);
  * dW1, dW2 of sampled experts (all of an expert's rows, when none of them is a near tie);
  * dW_r, dWs1, dWs2 and dw_sg as whole tensors: the router's weight gradient (split over
    tokens, then a fixed-order sum) and the shared expert's (one group of all T rows, a
    reduction of K = T = 16384 or 32768 rows), against the oracle's whole forward + backward
    routed on the GPU's fp32 logits (so that near-tie rows take the same experts);
  * a second run of the same step gives bit-identical outputs (no float atomics, fixed-order
    sums, tiles claimed at run time but each reduced by one CTA).
"""
import numpy as np
import pytest
import torch

import moe_inputs
import oracle.moe_oracle as O

from .helpers import GRAD_NAMES, TOL, assert_close, np64, run_layer

pytestmark = pytest.mark.gpu

WORKLOADS = ["qwen3", "deepseek", "mtp256"]


def _host(t):
    return None if t is None else t.float().cpu().numpy()


@pytest.fixture(scope="module", params=WORKLOADS)
def full_run(request):
    lc = moe_inputs.CONFIGS[request.param]
    inp = moe_inputs.make_layer_inputs(lc, seed=0, device="cuda")
    gpu = run_layer(lc, inp, backward=lc.backward)
    host = {k: _host(v) for k, v in inp.items()}
    yield lc, inp, gpu, host
    del gpu, inp
    torch.cuda.empty_cache()


def test_fullsize_routing(full_run):
    lc, inp, gpu, host = full_run
    s = gpu["saved"]
    lg = O.router_logits(host["x"], host["W_r"], host["b_r"])
    g_lg = np64(s["logits"])
    err = np.abs(g_lg - lg).max()
    assert err <= 1e-5 * np.abs(lg).max(), f"logit error {err}"
    idx = np64(s["idx"]).astype(np.int64)
    o_idx = O.select_topk(lg.astype(np.float32), lc.k).astype(np.int64)
    srt = -np.sort(-lg, axis=1)
    gap = srt[:, lc.k - 1] - srt[:, lc.k]
    clear = gap > 2 * err + 1e-12
    assert (np.sort(idx[clear], 1) == np.sort(o_idx[clear], 1)).all()
    # near ties: the GPU's set is a top-k of logits within `err` of the exact ones
    for t in np.nonzero(~clear)[0]:
        sel = lg[t, idx[t]]
        rest = np.delete(lg[t], idx[t])
        assert sel.min() >= rest.max() - 2 * err - 1e-12, t
    assert len(set(map(tuple, np.sort(idx, 1)))) > 1
    counts, offsets, sop, tos = O.routing_maps(idx, lc.E)
    assert (np64(s["counts"]) == counts).all()
    assert (np64(s["offsets"]) == offsets).all()
    assert (np64(s["slot_of_pair"]) == sop).all()
    assert (np64(s["token_of_slot"])[: lc.N] == tos).all()
    full_run[3]["_clear"] = clear
    full_run[3]["_idx"] = idx


def _subset_layer(lc, host, toks, backward):
    sub = dict(host)
    sub["x"] = host["x"][toks]
    sub["dy"] = host["dy"][toks]
    lc_s = lc.replace(T=len(toks))
    fwd = O.layer_forward(lc_s, sub)
    bwd = O.layer_backward(lc_s, sub, fwd, sub["dy"]) if backward else None
    return fwd, bwd


def test_fullsize_sampled_tokens(full_run):
    lc, inp, gpu, host = full_run
    if "_clear" not in host:
        test_fullsize_routing(full_run)
    clear = host["_clear"]
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(np.nonzero(clear)[0], size=48, replace=False))
    fwd, bwd = _subset_layer(lc, host, toks, lc.backward)
    assert (np.sort(fwd["idx"], 1) == np.sort(host["_idx"][toks], 1)).all()
    tol = TOL[lc.dtype]
    assert_close("y[sampled]", np64(gpu["y"])[toks], fwd["y"], tol)
    if lc.backward:
        assert_close("dx[sampled]", np64(gpu["dx"])[toks], bwd["dx"], tol)


def test_fullsize_sampled_expert_weight_gradients(full_run):
    lc, inp, gpu, host = full_run
    if not lc.backward:
        pytest.skip("forward-only workload")
    if "_clear" not in host:
        test_fullsize_routing(full_run)
    clear, idx = host["_clear"], host["_idx"]
    # experts none of whose tokens is a near tie, one hot (many rows) and one cold
    counts = np.bincount(idx.ravel(), minlength=lc.E)
    dirty = set(idx[~clear].ravel().tolist())
    cand = [e for e in np.argsort(-counts) if e not in dirty and counts[e] > 0]
    picks = [cand[0], cand[len(cand) // 2]]
    lg = O.router_logits(host["x"], host["W_r"], host["b_r"])
    x, dy = host["x"], host["dy"]
    for e in picks:
        t_list, j_list = np.nonzero(idx == e)
        g = O.gate_weights(lg[t_list], idx[t_list], lc.score_fn, lc.renorm)[np.arange(len(t_list)), j_list]
        X = x[t_list].astype(np.float64)
        o, a, u, h = O.swiglu_ffn(host["W1"][e], host["W2"][e], X)
        do = g[:, None] * dy[t_list].astype(np.float64)
        _, dW1e, dW2e = O.swiglu_ffn_backward(host["W1"][e], host["W2"][e], X, a, u, h, do)
        assert_close(f"dW1[{e}] ({len(t_list)} rows)", np64(gpu["dW1"][e]), dW1e, TOL[lc.dtype])
        assert_close(f"dW2[{e}] ({len(t_list)} rows)", np64(gpu["dW2"][e]), dW2e, TOL[lc.dtype])


def test_fullsize_router_and_shared_weight_gradients(full_run):
    lc, inp, gpu, host = full_run
    if not lc.backward:
        pytest.skip("forward-only workload")
    s = gpu["saved"]
    lg32 = np64(s["logits"]).astype(np.float32)
    fwd = O.layer_forward(lc, host, selection_logits32=lg32)
    assert (fwd["idx"] == np64(s["idx"])).all()
    bwd = O.layer_backward(lc, host, fwd, host["dy"])
    checked = []
    for n in ("dW_r", "dWs1", "dWs2", "dw_sg"):
        if gpu.get(n) is None:
            assert bwd.get(n) is None, n
            continue
        checked.append((n, assert_close(n, np64(gpu[n]), bwd[n], TOL[lc.dtype])))
    assert [n for n, _ in checked][:3] == ["dW_r", "dWs1", "dWs2"]
    print(lc.name, {n: f"{e:.2e}" for n, e in checked})


def test_fullsize_rerun_is_bit_identical(full_run):
    lc, inp, gpu, host = full_run
    again = run_layer(lc, inp, backward=lc.backward)
    for n in ["y"] + (GRAD_NAMES if lc.backward else []):
        if gpu.get(n) is not None:
            assert torch.equal(gpu[n], again[n]), n
    for n in ("act", "h", "y_perm"):
        assert torch.equal(gpu["saved"][n], again["saved"][n]), n
