"""Pins for the CPU oracle: checks against facts fixed by the pages and by mathematics, not
against the oracle's own formulas.  CPU only.

  * selection    -- brute force (full sort, key (-logit, expert)) and hand-computable ties
  * routing maps -- brute-force slot assignment, bijection and segment invariants
  * expert math  -- special cases that reduce to library routines (torch fp64 on the CPU):
                    E=1,k=1 is a plain SwiGLU MLP; k=E softmax+renorm is the dense
                    softmax-weighted mixture of all experts
  * gradients    -- central finite differences in fp64 for every input and weight
  * closed forms -- 3*d*f parameters per expert (printed on the pages as about 15M / 1.9B)
  * planted mistakes in the oracle must make at least one pin fail
"""
import json
import os
import types

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cfg_ns(T=5, d=6, E=4, k=2, f=3, f_shared=0, score_fn=O.SOFTMAX, renorm=1, shared_gate=0):
    return types.SimpleNamespace(T=T, d=d, E=E, k=k, f=f, f_shared=f_shared, score_fn=score_fn,
                                 renorm=renorm, shared_gate=shared_gate)


def rand_inputs(cfg, seed=0, bias=False):
    rng = np.random.default_rng(seed)
    inp = dict(
        x=rng.standard_normal((cfg.T, cfg.d)),
        W_r=rng.standard_normal((cfg.E, cfg.d)) * 0.7,
        b_r=rng.standard_normal(cfg.E) if bias else None,
        W1=rng.standard_normal((cfg.E, 2 * cfg.f, cfg.d)) * 0.5,
        W2=rng.standard_normal((cfg.E, cfg.d, cfg.f)) * 0.5,
    )
    if cfg.f_shared:
        inp["Ws1"] = rng.standard_normal((2 * cfg.f_shared, cfg.d)) * 0.5
        inp["Ws2"] = rng.standard_normal((cfg.d, cfg.f_shared)) * 0.5
        inp["w_sg"] = rng.standard_normal(cfg.d) * 0.5 if cfg.shared_gate else None
    return inp


# ----------------------------------------------------------------------------- selection

def brute_topk(row, k):
    return sorted(range(len(row)), key=lambda e: (-float(row[e]), e))[:k]


@pytest.mark.parametrize("kind", ["normal", "int_ties", "all_equal", "signed_zero"])
def test_select_topk_matches_brute_force(kind):
    rng = np.random.default_rng(1)
    T, E, k = 64, 13, 5
    if kind == "normal":
        lg = rng.standard_normal((T, E)).astype(np.float32)
    elif kind == "int_ties":
        lg = rng.integers(0, 4, (T, E)).astype(np.float32)
    elif kind == "all_equal":
        lg = np.full((T, E), 0.25, np.float32)
    else:
        lg = rng.choice(np.array([0.0, -0.0, 1.0], np.float32), size=(T, E))
    idx = O.select_topk(lg, k)
    for t in range(T):
        assert list(idx[t]) == brute_topk(lg[t], k)


def test_select_all_equal_takes_lowest_indices():
    lg = np.zeros((3, 10), np.float32)
    assert (O.select_topk(lg, 4) == np.arange(4)).all()


def test_golden_router_example_tie_order():
    g = json.load(open(os.path.join(GOLDEN, "router_example.json")))
    E, k = g["experts"], g["k"]
    lg = np.zeros((len(g["tokens"]), E), np.float32)
    for t, experts in enumerate(g["tokens"]):
        lg[t, experts] = 1.0
    idx = O.select_topk(lg, k)
    assert idx.tolist() == g["tokens"]


# ----------------------------------------------------------------------------- routing maps

def brute_slots(idx, E):
    pairs = sorted(((int(idx[t, j]), t, j) for t in range(idx.shape[0]) for j in range(idx.shape[1])))
    sop = np.empty(idx.shape, np.int64)
    tos = np.empty(idx.size, np.int64)
    for s, (e, t, j) in enumerate(pairs):
        sop[t, j] = s
        tos[s] = t
    return sop, tos


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_routing_maps_brute_force_and_invariants(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 97, 11, 3
    lg = rng.integers(0, 3, (T, E)).astype(np.float32) if seed == 2 else \
        rng.standard_normal((T, E)).astype(np.float32)
    idx = O.select_topk(lg, k)
    counts, offsets, sop, tos = O.routing_maps(idx, E)
    bsop, btos = brute_slots(idx, E)
    assert (sop == bsop).all() and (tos == btos).all()
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    assert (np.diff(offsets) == counts).all() and (np.diff(offsets) >= 0).all()
    # bijection: every pair lands in exactly one slot, and the inverse map agrees
    assert sorted(sop.ravel().tolist()) == list(range(T * k))
    for t in range(T):
        for j in range(k):
            s = sop[t, j]
            assert tos[s] == t
            e = idx[t, j]
            assert offsets[e] <= s < offsets[e + 1]   # the slot lies in its expert's segment
    for e in range(E):                                # ascending tokens inside a segment
        seg = tos[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()


def test_golden_grouped_gemm_counts():
    g = json.load(open(os.path.join(GOLDEN, "grouped_gemm_counts.json")))
    E = g["experts"]
    want = np.zeros(E, np.int64)
    for e, c in g["counts_printed"].items():
        want[int(e)] = c
    # one token per pair, k = 1: token t picks expert e when it is among that expert's tokens
    idx = np.concatenate([np.full(c, e) for e, c in enumerate(want)]).astype(np.int32)[:, None]
    rng = np.random.default_rng(0)
    idx = idx[rng.permutation(len(idx))]
    counts, offsets, sop, tos = O.routing_maps(idx, E)
    assert counts.tolist() == want.tolist()
    assert offsets.tolist()[:4] == [0, 20, 25, 60] and offsets[-1] == 68 and offsets[15] == 60


# ----------------------------------------------------------------------------- gates

def test_gates_sum_to_one_and_softmax_over_all():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((20, 9))
    idx = O.select_topk(lg.astype(np.float32), 9)
    full = O.gate_weights(lg, idx, O.SOFTMAX, 0)
    ref = torch.softmax(torch.from_numpy(lg), dim=1).numpy()
    np.testing.assert_allclose(full, np.take_along_axis(ref, idx.astype(np.int64), 1), rtol=1e-13)
    idx3 = O.select_topk(lg.astype(np.float32), 3)
    for sf in (O.SOFTMAX, O.SIGMOID):
        g = O.gate_weights(lg, idx3, sf, 1)
        np.testing.assert_allclose(g.sum(1), 1.0, rtol=1e-13)
    sg = O.gate_weights(lg, idx3, O.SIGMOID, 0)
    np.testing.assert_allclose(
        sg, torch.sigmoid(torch.from_numpy(np.take_along_axis(lg, idx3.astype(np.int64), 1))).numpy(),
        rtol=1e-13)


def test_softmax_renorm_equals_softmax_over_selected_and_shift_invariant():
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((10, 7))
    idx = O.select_topk(lg.astype(np.float32), 3)
    g = O.gate_weights(lg, idx, O.SOFTMAX, 1)
    sel = torch.from_numpy(np.take_along_axis(lg, idx.astype(np.int64), 1))
    np.testing.assert_allclose(g, torch.softmax(sel, 1).numpy(), rtol=1e-13)
    np.testing.assert_allclose(O.gate_weights(lg + 5.0, idx, O.SOFTMAX, 1), g, rtol=1e-12)


# ----------------------------------------------------------------------------- expert math

def torch_swiglu(x, W1, W2):
    f = W1.shape[0] // 2
    return F.linear(F.silu(F.linear(x, W1[:f])) * F.linear(x, W1[f:]), W2)


@pytest.mark.parametrize("score_fn", [O.SOFTMAX, O.SIGMOID])
def test_single_expert_top1_is_plain_swiglu_mlp(score_fn):
    cfg = cfg_ns(T=9, d=8, E=1, k=1, f=5, score_fn=score_fn, renorm=1)
    inp = rand_inputs(cfg, 5)
    y = O.layer_forward(cfg, inp)["y"]
    ref = torch_swiglu(torch.from_numpy(inp["x"]), torch.from_numpy(inp["W1"][0]),
                       torch.from_numpy(inp["W2"][0])).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_topk_all_experts_softmax_renorm_is_dense_mixture():
    cfg = cfg_ns(T=7, d=6, E=5, k=5, f=4)
    inp = rand_inputs(cfg, 6)
    y = O.layer_forward(cfg, inp)["y"]
    x = torch.from_numpy(inp["x"])
    p = torch.softmax(x @ torch.from_numpy(inp["W_r"]).T, dim=1)
    outs = torch.stack([torch_swiglu(x, torch.from_numpy(inp["W1"][e]), torch.from_numpy(inp["W2"][e]))
                        for e in range(cfg.E)], dim=1)
    ref = torch.einsum("te,ted->td", p, outs).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_routed_output_matches_per_token_library_evaluation():
    """Sigmoid, no renorm, with a router bias and a gated shared expert: every token's output
    recomputed one token at a time with torch routines."""
    cfg = cfg_ns(T=11, d=6, E=6, k=2, f=3, f_shared=4, score_fn=O.SIGMOID, renorm=0, shared_gate=1)
    inp = rand_inputs(cfg, 7, bias=True)
    fwd = O.layer_forward(cfg, inp)
    T = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v) for k, v in inp.items()}
    for t in range(cfg.T):
        xt = T["x"][t:t + 1]
        lg = (xt @ T["W_r"].T + T["b_r"])[0]
        order = sorted(range(cfg.E), key=lambda e: (-float(lg[e].float()), e))[:cfg.k]
        yt = sum(torch.sigmoid(lg[e]) * torch_swiglu(xt, T["W1"][e], T["W2"][e]) for e in order)
        yt = yt + torch.sigmoid(xt @ T["w_sg"]) * torch_swiglu(xt, T["Ws1"], T["Ws2"])
        np.testing.assert_allclose(fwd["y"][t], yt[0].numpy(), rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- gradients

VARIANTS = [
    dict(score_fn=O.SOFTMAX, renorm=1),
    dict(score_fn=O.SOFTMAX, renorm=0),
    dict(score_fn=O.SIGMOID, renorm=1),
    dict(score_fn=O.SIGMOID, renorm=0),
    dict(score_fn=O.SIGMOID, renorm=1, f_shared=3),
    dict(score_fn=O.SOFTMAX, renorm=1, f_shared=3, shared_gate=1),
]


def fd_check(cfg, inp, seed):
    rng = np.random.default_rng(seed + 100)
    dy = rng.standard_normal((cfg.T, cfg.d))
    fwd = O.layer_forward(cfg, inp)
    grads = O.layer_backward(cfg, inp, fwd, dy)
    base_idx = fwd["idx"]
    names = [("x", "dx"), ("W_r", "dW_r"), ("W1", "dW1"), ("W2", "dW2")]
    if cfg.f_shared:
        names += [("Ws1", "dWs1"), ("Ws2", "dWs2")]
        if cfg.shared_gate:
            names += [("w_sg", "dw_sg")]
    eps = 1e-6
    checked = 0
    for pname, gname in names:
        P = inp[pname]
        for c in np.ndindex(P.shape):
            old = P[c]
            P[c] = old + eps
            fp = O.layer_forward(cfg, inp)
            P[c] = old - eps
            fm = O.layer_forward(cfg, inp)
            P[c] = old
            if not ((fp["idx"] == base_idx).all() and (fm["idx"] == base_idx).all()):
                continue  # the perturbation moved a token to another expert
            fd = ((fp["y"] - fm["y"]) * dy).sum() / (2 * eps)
            an = grads[gname][c]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (pname, c, fd, an)
            checked += 1
    return checked


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: "-".join(f"{k}{v[k]}" for k in v))
def test_finite_difference_gradients(variant):
    cfg = cfg_ns(T=5, d=4, E=4, k=2, f=3, **variant)
    inp = rand_inputs(cfg, 11, bias=True)
    assert fd_check(cfg, inp, 11) > 100


# ----------------------------------------------------------------------------- closed forms

def test_golden_param_count():
    g = json.load(open(os.path.join(GOLDEN, "param_count.json")))
    per = O.expert_param_count(g["d_model"], g["ffn"])
    assert per == 3 * 2688 * 1856 == 14966784
    assert round(per, -6) == g["per_expert_printed"]
    assert round(per * g["experts"], -8) == g["all_experts_printed"]
    # the oracle's weight shapes hold exactly that many numbers
    cfg = cfg_ns(d=g["d_model"] // 64, f=g["ffn"] // 64)
    inp = rand_inputs(cfg)
    assert inp["W1"][0].size + inp["W2"][0].size == O.expert_param_count(cfg.d, cfg.f)


# ----------------------------------------------------------------------------- planted mistakes

def _pins_pass():
    try:
        test_single_expert_top1_is_plain_swiglu_mlp(O.SOFTMAX)
        test_topk_all_experts_softmax_renorm_is_dense_mixture()
        test_routed_output_matches_per_token_library_evaluation()
        for v in VARIANTS:
            test_finite_difference_gradients(v)
        test_gates_sum_to_one_and_softmax_over_all()
        test_softmax_renorm_equals_softmax_over_selected_and_shift_invariant()
    except AssertionError:
        return False
    return True


MUTANTS = {
    # forward mistakes
    "silu_without_gate": ("silu", lambda a: a),
    "sigmoid_sign": ("sigmoid", lambda z, _s=O.sigmoid: _s(-np.asarray(z, float))),
    "gate_up_swapped": ("swiglu_ffn", lambda W1e, W2e, X, _f=O.swiglu_ffn: _f(
        np.concatenate([np.asarray(W1e)[len(W1e) // 2:], np.asarray(W1e)[:len(W1e) // 2]]), W2e, X)),
    "w2_transposed": ("swiglu_ffn", lambda W1e, W2e, X, _f=O.swiglu_ffn: _f(
        W1e, np.asarray(W2e).T.reshape(np.asarray(W2e).shape), X)),
    # backward mistakes
    "silu_grad_dropped_term": ("silu_grad", lambda a: O.sigmoid(a)),
    "gate_backward_wrong_sign": ("gate_backward", lambda *a, _g=O.gate_backward: -_g(*a)),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    assert _pins_pass()
    attr, repl = MUTANTS[name]
    monkeypatch.setattr(O, attr, repl)
    assert not _pins_pass(), f"mutant {name} survived every pin"


# ----------------------------------------------------------------------------- degenerate routing

@pytest.mark.parametrize("case", ["all_to_8", "32_empty", "int_ties"])
def test_degenerate_routing_cases(case):
    import moe_inputs
    T, E, k = 300, 128, 8
    lg = moe_inputs.make_stress_logits(case, T, E, seed=0).numpy()
    idx = O.select_topk(lg, k)
    counts, offsets, sop, tos = O.routing_maps(idx, E)
    if case == "all_to_8":
        assert counts[:8].tolist() == [T] * 8 and counts[8:].sum() == 0
        assert (np.sort(idx, 1) == np.arange(8)).all()
    elif case == "32_empty":
        assert counts[E - 32:].sum() == 0 and counts.sum() == T * k
    else:
        # integer logits: the top value class is taken whole, lowest indices first
        for t in range(T):
            assert list(idx[t]) == brute_topk(lg[t], k)
            assert (np.diff(lg[t][idx[t]]) <= 0).all()
