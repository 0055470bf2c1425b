"""Pins for the oracle's router variants (CPU only): the load-balancing loss, its gradient, the
selection-only expert bias and the expert-bias update.  Each is checked against what the
mathematics fixes -- closed forms, invariants, finite differences, hand-computed cases -- not
against a restatement of the oracle's own formulas; planted mistakes must fail a pin.

  * balancing loss -- equals its coefficient whenever the probabilities are uniform (whatever
    the counts); equals coeff * E / k when every token and all probability sit on the same k
    experts; central finite differences of the loss (counts fixed) match its gradient; the
    softmax gradient of every token sums to zero (shift invariance of the softmax)
  * layer gradients with the loss and with a selection-only bias -- finite differences of
    sum(y * dy) + L_aux through the whole oracle layer
  * expert bias -- a bias larger than any score range forces its experts into every token's
    choice; the gates never change with the bias; zero bias selects as the logits do; two
    hand-worked softmax rows where score + bias, logit + bias and sigmoid + bias choose
    different experts; the update moves each bias by -rate, 0 or +rate by the sign of
    (mean load - load)
"""
import types

import numpy as np
import pytest

import oracle.moe_oracle as O


def cfg_ns(T=6, d=4, E=5, k=2, f=3, score_fn=O.SOFTMAX, renorm=1, bias_mode=O.BIAS_LOGIT,
           aux_coeff=0.0, f_shared=0, shared_gate=0):
    return types.SimpleNamespace(T=T, d=d, E=E, k=k, f=f, f_shared=f_shared, score_fn=score_fn,
                                 renorm=renorm, shared_gate=shared_gate, bias_mode=bias_mode,
                                 aux_coeff=aux_coeff)


def rand_inputs(cfg, seed=0, bias_std=1.0):
    rng = np.random.default_rng(seed)
    return dict(
        x=rng.standard_normal((cfg.T, cfg.d)),
        W_r=rng.standard_normal((cfg.E, cfg.d)) * 0.7,
        b_r=rng.standard_normal(cfg.E) * bias_std,
        W1=rng.standard_normal((cfg.E, 2 * cfg.f, cfg.d)) * 0.5,
        W2=rng.standard_normal((cfg.E, cfg.d, cfg.f)) * 0.5,
    )


def random_counts(rng, T, k, E):
    """Non-negative integer counts summing to T*k (any routing of T tokens to k experts)."""
    c = rng.multinomial(T * k, np.ones(E) / E)
    assert c.sum() == T * k
    return c


SCORES = [O.SOFTMAX, O.SIGMOID]


# ----------------------------------------------------------------------------- balancing loss

@pytest.mark.parametrize("score_fn", SCORES)
def test_aux_loss_is_its_coefficient_for_uniform_probabilities(score_fn):
    rng = np.random.default_rng(1)
    for T, E, k in [(7, 5, 2), (16, 8, 3), (3, 4, 4)]:
        lg = np.full((T, E), 0.37)            # equal logits: p = 1/E for both score functions
        for _ in range(3):
            c = random_counts(rng, T, k, E)
            assert O.aux_loss(lg, c, k, 0.25, score_fn) == pytest.approx(0.25, rel=1e-13)


@pytest.mark.parametrize("score_fn", SCORES)
def test_aux_loss_collapsed_routing_closed_form(score_fn):
    T, E, k = 9, 8, 3
    lg = np.full((T, E), -40.0)
    lg[:, :k] = 40.0                          # probability 1/k on experts 0..k-1, ~0 elsewhere
    c = np.zeros(E, dtype=np.int64)
    c[:k] = T                                 # every token routed to the same k experts
    assert O.aux_loss(lg, c, k, 1e-4, score_fn) == pytest.approx(1e-4 * E / k, rel=1e-12)


@pytest.mark.parametrize("score_fn", SCORES)
def test_aux_loss_gradient_finite_differences(score_fn):
    rng = np.random.default_rng(2)
    T, E, k, coeff = 5, 6, 2, 0.7
    lg = rng.standard_normal((T, E)) * 1.5
    c = random_counts(rng, T, k, E)
    an = O.aux_loss_grad(lg, c, k, coeff, score_fn)
    eps = 1e-6
    for i in np.ndindex(lg.shape):
        lp, lm = lg.copy(), lg.copy()
        lp[i] += eps
        lm[i] -= eps
        fd = (O.aux_loss(lp, c, k, coeff, score_fn) - O.aux_loss(lm, c, k, coeff, score_fn)) / (2 * eps)
        assert abs(fd - an[i]) <= 1e-8 + 1e-6 * abs(an[i]), (i, fd, an[i])


def test_aux_loss_softmax_gradient_rows_sum_to_zero():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((11, 7))
    c = random_counts(rng, 11, 3, 7)
    g = O.aux_loss_grad(lg, c, 3, 0.3, O.SOFTMAX)
    assert np.abs(g.sum(axis=1)).max() <= 1e-15 + 1e-12 * np.abs(g).max()
    assert np.abs(g).max() > 0


# ----------------------------------------------------------------------------- layer gradients

def fd_layer(cfg, inp, seed):
    """Finite differences of sum(y * dy) + L_aux with respect to x and W_r (coordinates whose
    perturbation changes the selection are skipped)."""
    rng = np.random.default_rng(seed)
    dy = rng.standard_normal((cfg.T, cfg.d))
    fwd = O.layer_forward(cfg, inp)
    grads = O.layer_backward(cfg, inp, fwd, dy)

    def objective(f):
        return (f["y"] * dy).sum() + f.get("aux_loss", 0.0)

    eps, checked = 1e-6, 0
    for pname, gname in [("x", "dx"), ("W_r", "dW_r"), ("W1", "dW1")]:
        P = inp[pname]
        for c in np.ndindex(P.shape):
            old = P[c]
            P[c] = old + eps
            fp = O.layer_forward(cfg, inp)
            P[c] = old - eps
            fm = O.layer_forward(cfg, inp)
            P[c] = old
            if not ((fp["idx"] == fwd["idx"]).all() and (fm["idx"] == fwd["idx"]).all()):
                continue
            fd = (objective(fp) - objective(fm)) / (2 * eps)
            an = grads[gname][c]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (pname, c, fd, an)
            checked += 1
    return checked


LAYER_VARIANTS = [
    dict(score_fn=O.SOFTMAX, renorm=1, aux_coeff=0.5),
    dict(score_fn=O.SOFTMAX, renorm=0, aux_coeff=0.5),
    dict(score_fn=O.SIGMOID, renorm=1, aux_coeff=0.5),
    dict(score_fn=O.SIGMOID, renorm=1, bias_mode=O.BIAS_SELECT),
    dict(score_fn=O.SIGMOID, renorm=1, bias_mode=O.BIAS_SELECT, aux_coeff=0.5),
    dict(score_fn=O.SOFTMAX, renorm=1, bias_mode=O.BIAS_SELECT, aux_coeff=0.5),
]


@pytest.mark.parametrize("variant", LAYER_VARIANTS,
                         ids=lambda v: "-".join(f"{k}{v[k]}" for k in v))
def test_layer_gradients_with_aux_loss_and_selection_bias(variant):
    cfg = cfg_ns(**variant)
    inp = rand_inputs(cfg, 21, bias_std=0.1)
    assert fd_layer(cfg, inp, 22) > 60


def test_aux_loss_reaches_the_router_weights():
    cfg0 = cfg_ns(score_fn=O.SIGMOID)
    cfg1 = cfg_ns(score_fn=O.SIGMOID, aux_coeff=0.5)
    inp = rand_inputs(cfg0, 5)
    dy = np.zeros((cfg0.T, cfg0.d))          # no upstream gradient: only the loss drives W_r
    g0 = O.layer_backward(cfg0, inp, O.layer_forward(cfg0, inp), dy)
    g1 = O.layer_backward(cfg1, inp, O.layer_forward(cfg1, inp), dy)
    assert np.abs(g0["dW_r"]).max() == 0.0
    assert np.abs(g1["dW_r"]).max() > 1e-4
    assert np.abs(g1["dW1"]).max() == 0.0    # the loss does not reach the experts


# ----------------------------------------------------------------------------- expert bias

def test_selection_bias_forces_its_experts_and_never_moves_the_gates():
    T, E, k = 40, 6, 3
    rng = np.random.default_rng(4)
    lg = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    bias = np.zeros(E, dtype=np.float32)
    bias[[1, 3]] = 2.0                        # wider than the whole sigmoid range (0, 1)
    idx = O.select_topk(O.selection_keys(lg, O.SIGMOID, bias), k)
    assert all({1, 3} <= set(row.tolist()) for row in idx)
    # the third expert is the best of the rest by sigmoid score, i.e. by logit
    rest = np.array([[e for e in np.argsort(-lg[t], kind="stable") if e not in (1, 3)][0]
                     for t in range(T)])
    assert (np.sort(idx, 1) == np.sort(np.stack([np.ones(T, int), np.full(T, 3), rest], 1), 1)).all()
    # the gates depend on the logits of the chosen experts only, never on the bias
    cfg = cfg_ns(T=T, d=3, E=E, k=k, score_fn=O.SIGMOID, bias_mode=O.BIAS_SELECT)
    inp = rand_inputs(cfg, 6)
    inp["b_r"] = bias.astype(np.float64)
    f1 = O.layer_forward(cfg, inp)
    inp2 = dict(inp, b_r=inp["b_r"] * 1.5)    # still forcing 1 and 3: same choice
    f2 = O.layer_forward(cfg, inp2)
    assert (f1["idx"] == f2["idx"]).all()
    assert np.array_equal(f1["gate"], f2["gate"])
    s = O.sigmoid(np.take_along_axis(f1["logits"], f1["idx"].astype(np.int64), axis=1))
    assert np.allclose(f1["gate"], s / s.sum(1, keepdims=True), rtol=0, atol=1e-15)
    # and the logits the layer reports carry no bias
    assert np.allclose(f1["logits"], inp["x"] @ inp["W_r"].T, rtol=0, atol=1e-13)


def test_softmax_selection_keys_by_hand():
    """Softmax routing with a selection-only bias ("Megatron-Bridge 深度剖析", §Nemotron-3-Nano
    配置, expert-bias correction; the reading that the bias is added to the softmax over all E
    experts).  Two hand-worked rows, chosen so that the three plausible keys disagree:

    row A, logits [2, 0, 0], bias [0, 0.75, 0]:
      softmax over E: e^2 / (e^2 + 2) = 7.389056 / 9.389056 = 0.786986, 1 / 9.389056 = 0.106507
      keys = [0.786986, 0.856507, 0.106507] -> top-1 is expert 1, top-2 is (1, 0);
      logit + bias = [2, 0.75, 0] would pick expert 0.
    row B, logits [1, 0], bias [0, 0.3]:
      softmax: e / (e + 1) = 0.731059, 1 / (e + 1) = 0.268941
      keys = [0.731059, 0.568941] -> top-1 is expert 0;
      sigmoid + bias = [0.731059, 0.5 + 0.3 = 0.8] would pick expert 1.
    """
    kA = O.selection_keys(np.array([[2.0, 0.0, 0.0]], np.float32), O.SOFTMAX,
                          np.array([0.0, 0.75, 0.0], np.float32))
    assert kA.dtype == np.float32
    assert np.allclose(kA[0], [0.786986, 0.856507, 0.106507], rtol=0, atol=2e-6)
    assert O.select_topk(kA, 1).tolist() == [[1]]
    assert O.select_topk(kA, 2).tolist() == [[1, 0]]
    kB = O.selection_keys(np.array([[1.0, 0.0]], np.float32), O.SOFTMAX,
                          np.array([0.0, 0.3], np.float32))
    assert np.allclose(kB[0], [0.731059, 0.568941], rtol=0, atol=2e-6)
    assert O.select_topk(kB, 1).tolist() == [[0]]
    # the same row B under sigmoid routing does pick expert 1 (the two branches differ here)
    kS = O.selection_keys(np.array([[1.0, 0.0]], np.float32), O.SIGMOID,
                          np.array([0.0, 0.3], np.float32))
    assert np.allclose(kS[0], [0.731059, 0.8], rtol=0, atol=2e-6)
    assert O.select_topk(kS, 1).tolist() == [[1]]


@pytest.mark.parametrize("score_fn", SCORES)
def test_zero_selection_bias_selects_as_the_logits(score_fn):
    rng = np.random.default_rng(7)
    lg = (rng.standard_normal((200, 16)) * 3).astype(np.float32)
    keys = O.selection_keys(lg, score_fn, np.zeros(16, np.float32))
    # keys are monotone in the logits; distinct logits this far apart give distinct keys
    assert (O.select_topk(keys, 4) == O.select_topk(lg, 4)).all()


def test_expert_bias_update_by_hand():
    b = np.array([0.5, -0.25, 0.0, 1.0], dtype=np.float32)
    counts = np.array([5, 3, 4, 4])           # T*k = 16 over E = 4: mean load 4
    out = O.expert_bias_update(b, counts, 8, 2, 0.125)
    assert out.dtype == np.float32
    assert out.tolist() == [0.375, -0.125, 0.0, 1.0]


def test_expert_bias_update_pushes_load_toward_balance():
    # fixed skewed logits; repeated corrections must lower the load of the hottest expert
    rng = np.random.default_rng(8)
    T, E, k = 256, 8, 2
    lg = (rng.standard_normal((T, E)) + np.linspace(2, 0, E)).astype(np.float32)
    b = np.zeros(E, np.float32)
    first = None
    for _ in range(60):
        idx = O.select_topk(O.selection_keys(lg, O.SIGMOID, b), k)
        counts = np.bincount(idx.ravel(), minlength=E)
        first = counts if first is None else first
        b = O.expert_bias_update(b, counts, T, k, 0.01)
    assert counts.max() < first.max()
    assert counts.max() - counts.min() < first.max() - first.min()


# ----------------------------------------------------------------------------- planted mistakes

def _variant_pins_pass():
    try:
        for s in SCORES:
            test_aux_loss_is_its_coefficient_for_uniform_probabilities(s)
            test_aux_loss_collapsed_routing_closed_form(s)
            test_aux_loss_gradient_finite_differences(s)
        test_aux_loss_softmax_gradient_rows_sum_to_zero()
        test_selection_bias_forces_its_experts_and_never_moves_the_gates()
        test_softmax_selection_keys_by_hand()
        test_expert_bias_update_by_hand()
    except AssertionError:
        return False
    return True


def _aux_sum_not_mean(logits, counts, k, coeff, score_fn):
    p = O.score_probs(logits, score_fn)
    T, E = p.shape
    return float(coeff * E * np.dot(np.asarray(counts, float) / (T * k), p.sum(axis=0)))


MUTANTS = {
    "aux_probability_summed_not_averaged": ("aux_loss", _aux_sum_not_mean),
    "aux_gradient_sign": ("aux_loss_grad", lambda *a, _g=O.aux_loss_grad: -_g(*a)),
    "aux_gradient_without_centering": (
        "aux_loss_grad",
        lambda l, c, k, coeff, s, _p=O.score_probs: _p(l, s) * (
            coeff * np.asarray(l).shape[1] * np.asarray(c, float) / (k * np.asarray(l).shape[0] ** 2))[None, :]),
    "sigmoid_probabilities_unnormalised": (
        "score_probs", lambda l, s, _f=O.score_probs: O.sigmoid(l) if s == O.SIGMOID else _f(l, s)),
    "selection_ignores_bias": (
        "selection_keys", lambda l, s, b, _f=O.selection_keys: _f(l, s, np.zeros_like(b))),
    # softmax routing that adds the bias to the raw logits, or to the sigmoid, instead of to the
    # softmax over all experts
    "softmax_keys_are_logit_plus_bias": (
        "selection_keys", lambda l, s, b, _f=O.selection_keys: (
            np.asarray(l, np.float32) + np.asarray(b, np.float32)[None, :]).astype(np.float32)
        if s == O.SOFTMAX else _f(l, s, b)),
    "softmax_keys_are_sigmoid_plus_bias": (
        "selection_keys", lambda l, s, b, _f=O.selection_keys: _f(l, O.SIGMOID, b)),
    "bias_update_reversed": (
        "expert_bias_update", lambda b, c, T, k, r, _f=O.expert_bias_update: _f(b, c, T, k, -r)),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_router_variant_mistakes_are_caught(name, monkeypatch):
    assert _variant_pins_pass()
    attr, repl = MUTANTS[name]
    monkeypatch.setattr(O, attr, repl)
    assert not _variant_pins_pass(), f"mutant {name} survived every pin"
