"""Oracle: a plain, slow, fp64 CPU statement of one mixture-of-experts layer and its backward.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
may import this module.  The CUDA library never does, and this module imports nothing of
the library: it shares no code with it.

What the layer computes, and where the pages say so:
  * router, then top-k with a softmax or a sigmoid score function -- "Megatron-Bridge 深度剖析"
    (§Motivation: "128 个 expert，每个 token 激活 top-6，sigmoid routing"; §核心模块架构:
    TransformerConfig fields moe_router_topk / moe_router_score_function; §Expert Parallel
    基础, workflow figure Step 1 "Router(x) -> TopK scores");
  * tokens regrouped by expert, the experts run, the results sent back to token order --
    §Expert Parallel 基础, workflow figure Steps 2-3 (dispatch / combine; on one GPU the
    all-to-all becomes a local permutation) and §Permute Fusion (tokens are permuted so that
    each expert's tokens are contiguous);
  * every expert is a SwiGLU FFN (gate_proj, up_proj, down_proj; 3*d*f parameters) --
    §Motivation; fc1 stores gate rows then up rows, (2*ffn_hidden, hidden) --
    §权重映射策略 (GatedMLPMapping);
  * a shared expert that every token goes through, added to the routed output --
    §Shared Expert Overlap; its sigmoid gate -- "Add Megatron-Core MTP training for Qwen3.5
    MoE" (What's in it: "routed experts, shared expert and shared-expert gate").

Readings where the pages are silent (each also listed in the design notes):
  * selection runs on fp32 logits, descending, equal logits -> lower expert index first;
  * renorm: the k selected gates are divided by their sum (softmax+renorm is the softmax over
    the k selected logits);
  * dropless: every (token, expert) pair is computed; no capacity;
  * the gate multiplies the expert output in the combine; no biases in the experts;
  * shared gate c_t = sigmoid(w_sg . x_t), a scalar per token;
  * inside one expert's contiguous segment the tokens are in ascending token order;
  * the router bias b_r is an input, not a trained parameter: added to the logits (to make
    hot experts) or, with the expert-bias correction, to the scores for the selection only;
  * the load-balancing loss is coeff * E * sum_e f_e P_e (share of routed pairs times mean
    probability), its gradient reaches the logits with the counts held fixed; the expert-bias
    update is b_e += rate * sign(mean load - load_e).

Evaluation order.  Each (token, expert) pair's FFN is independent of every other pair.  The
oracle evaluates all pairs that picked the same expert as one matrix product whose rows are
those pairs; no sum is reordered by this, it only runs the per-pair definition in one call.
"""
from __future__ import annotations

import numpy as np

SOFTMAX = 0
SIGMOID = 1


# ----------------------------------------------------------------------------- elementwise

def sigmoid(z):
    """Logistic function 1 / (1 + e^-z), evaluated without overflow for either sign."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def silu(a):
    """SiLU(a) = a * sigmoid(a), the gate nonlinearity of SwiGLU."""
    return a * sigmoid(a)


def silu_grad(a):
    """d SiLU / da = s + a*s*(1-s) with s = sigmoid(a)."""
    s = sigmoid(a)
    return s + a * s * (1.0 - s)


def f64(a):
    return np.asarray(a, dtype=np.float64)


# ----------------------------------------------------------------------------- routing

def router_logits(x, W_r, b_r=None):
    """l[t, e] = x_t . W_r[e] (+ b_r[e]).  The router is a plain linear map (router.weight
    [E, d]); the optional bias only shapes synthetic workloads."""
    l = f64(x) @ f64(W_r).T
    if b_r is not None:
        l = l + f64(b_r)[None, :]
    return l


def select_topk(logits32, k):
    """idx[t, 0..k-1]: the k experts with the largest fp32 logits, in descending order;
    experts with equal logits are taken lower index first.  A stable sort on the negated
    logits gives exactly that order (negation is exact in fp32)."""
    lg = np.asarray(logits32, dtype=np.float32)
    order = np.argsort(-lg, axis=1, kind="stable")
    return np.ascontiguousarray(order[:, :k]).astype(np.int32)


def gate_weights(logits, idx, score_fn, renorm):
    """Combine weights g[t, j] of the k selected experts.

    softmax, renorm:    softmax over the k selected logits
    softmax, no renorm: softmax over all E logits, read at the selected experts
    sigmoid, renorm:    sigmoid(l) of the selected, divided by their sum
    sigmoid, no renorm: sigmoid(l) of the selected
    """
    l = f64(logits)
    sel = np.take_along_axis(l, idx.astype(np.int64), axis=1)
    if score_fn == SOFTMAX:
        if renorm:
            z = np.exp(sel - sel.max(axis=1, keepdims=True))
            return z / z.sum(axis=1, keepdims=True)
        p = np.exp(l - l.max(axis=1, keepdims=True))
        p = p / p.sum(axis=1, keepdims=True)
        return np.take_along_axis(p, idx.astype(np.int64), axis=1)
    s = sigmoid(sel)
    if renorm:
        return s / s.sum(axis=1, keepdims=True)
    return s


def routing_maps(idx, E):
    """Per-expert histogram, exclusive prefix sum and the token<->slot permutation.

    counts[e]   = number of (t, j) pairs with idx[t, j] == e
    offsets[0]  = 0, offsets[e+1] = offsets[e] + counts[e]   (offsets[E] = T*k)
    slot_of_pair[t, j] = offsets[e] + (number of tokens t' < t that picked e), e = idx[t, j]
    token_of_slot[s]   = the token whose pair was given slot s
    This is a stable counting sort of the pairs by expert: each expert's rows are
    contiguous and, inside, in ascending token order.
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for e in idx.ravel():
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    next_free = offsets[:-1].copy()
    slot_of_pair = np.empty((T, k), dtype=np.int64)
    token_of_slot = np.empty(T * k, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            s = next_free[e]
            next_free[e] += 1
            slot_of_pair[t, j] = s
            token_of_slot[s] = t
    return (counts.astype(np.int32), offsets.astype(np.int32), slot_of_pair.astype(np.int32),
            token_of_slot.astype(np.int32))


def route(logits, k, E, score_fn, renorm):
    """Selection on fp32 logits, gates from the same logits in fp64, and the routing maps."""
    l32 = np.asarray(logits, dtype=np.float32)
    idx = select_topk(l32, k)
    g = gate_weights(logits, idx, score_fn, renorm)
    counts, offsets, sop, tos = routing_maps(idx, E)
    return dict(idx=idx, gate=g, counts=counts, offsets=offsets, slot_of_pair=sop,
                token_of_slot=tos)


# ----------------------------------------------------------------------------- router variants
# "Megatron-Bridge 深度剖析", §Nemotron-3-Nano 配置 and its comparison with DeepSeek V3: the
# sigmoid routing runs with an expert-bias correction (moe_router_enable_expert_bias) and a
# load-balancing loss of coefficient 1e-4 (moe_aux_loss_coeff) that pushes the tokens to spread
# evenly over the experts and keeps them from collapsing onto a few.  The pages name both and
# give no formula; the readings below are the published forms they refer to.

BIAS_LOGIT = 0    # b_r is added to the logits: it moves selection and gates alike
BIAS_SELECT = 1   # b_r is added to the scores for the selection only; gates never see it


def score_probs(logits, score_fn):
    """Per-token distribution over all E experts read by the balancing loss:
    softmax(l_t) for softmax routing, s_t / sum(s_t) with s = sigmoid(l_t) for sigmoid."""
    l = f64(logits)
    if score_fn == SOFTMAX:
        z = np.exp(l - l.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    s = sigmoid(l)
    return s / s.sum(axis=1, keepdims=True)


def selection_keys(logits32, score_fn, e_bias):
    """Selection keys under a selection-only expert bias: score + bias in fp32, the score being
    the softmax over all E (softmax routing) or the sigmoid (sigmoid routing) of the fp32
    logits.  The keys are formed in fp32 because that is the precision the choice is made in."""
    l = np.asarray(logits32, dtype=np.float32)
    b = np.asarray(e_bias, dtype=np.float32)[None, :]
    if score_fn == SOFTMAX:
        z = np.exp(l - l.max(axis=1, keepdims=True), dtype=np.float32)
        sc = z / z.sum(axis=1, keepdims=True, dtype=np.float32)
    else:
        sc = np.float32(1.0) / (np.float32(1.0) + np.exp(-l, dtype=np.float32))
    return (sc.astype(np.float32) + b).astype(np.float32)


def aux_loss(logits, counts, k, coeff, score_fn):
    """Load-balancing loss L = coeff * E * sum_e f_e * P_e over one batch of T tokens, where
    f_e = counts_e / (T*k) is expert e's share of the routed (token, expert) pairs and
    P_e = (1/T) sum_t p[t, e] its mean probability (p from score_probs).  With uniform p it is
    exactly coeff, whatever the counts; it grows as tokens and probability pile on few experts."""
    p = score_probs(logits, score_fn)
    T, E = p.shape
    f = f64(counts) / (T * k)
    P = p.mean(axis=0)
    return float(coeff * E * np.dot(f, P))


def aux_loss_grad(logits, counts, k, coeff, score_fn):
    """dL_aux/dlogits [T, E], the counts held fixed (they are piecewise constant).
    w_e = dL/dp[t, e] = coeff * E * counts_e / (k * T^2);  G_t = sum_e p[t, e] w_e;
      softmax: dl[t, e] = p[t, e] (w_e - G_t)
      sigmoid: p = s / S_t, dl[t, e] = s (1 - s) (w_e - G_t) / S_t."""
    l = f64(logits)
    T, E = l.shape
    w = coeff * E * f64(counts) / (k * T * T)
    if score_fn == SOFTMAX:
        p = score_probs(l, SOFTMAX)
        G = p @ w
        return p * (w[None, :] - G[:, None])
    s = sigmoid(l)
    S = s.sum(axis=1, keepdims=True)
    G = (s / S) @ w
    return s * (1.0 - s) * (w[None, :] - G[:, None]) / S


def expert_bias_update(e_bias, counts, T, k, rate):
    """Expert-bias correction after a step (the auxiliary-loss-free balancing of DeepSeek V3):
    b_e <- b_e + rate * sign(T*k/E - counts_e): experts above the mean load lose selection
    priority, those below gain it, those exactly at it keep their bias.  fp32, as stored."""
    b = np.asarray(e_bias, dtype=np.float32)
    E = b.shape[0]
    mean = np.float32(T * k) / np.float32(E)
    sgn = np.sign(mean - np.asarray(counts, dtype=np.float32)).astype(np.float32)
    return (b + np.float32(rate) * sgn).astype(np.float32)


def permute(x, token_of_slot):
    """x_perm[s] = x[token_of_slot[s]]: tokens regrouped into expert-contiguous rows."""
    return f64(x)[np.asarray(token_of_slot, dtype=np.int64)]


# ----------------------------------------------------------------------------- experts

def swiglu_ffn(W1e, W2e, X):
    """One SwiGLU expert on rows X [n, d]: a = X Wg^T, u = X Wu^T (fc1 = [Wg; Wu], gate rows
    first), h = SiLU(a) * u, o = h W2^T.  Returns o and the intermediates."""
    W1e = f64(W1e)
    f = W1e.shape[0] // 2
    a = X @ W1e[:f].T
    u = X @ W1e[f:].T
    h = silu(a) * u
    o = h @ f64(W2e).T
    return o, a, u, h


def swiglu_ffn_backward(W1e, W2e, X, a, u, h, do):
    """Backward of swiglu_ffn for upstream gradient do [n, d].
    Returns dX [n, d], dW1e [2f, d], dW2e [d, f]."""
    W1e = f64(W1e)
    W2e = f64(W2e)
    f = W1e.shape[0] // 2
    dh = do @ W2e
    dW2e = do.T @ h
    da = dh * u * silu_grad(a)
    du = dh * silu(a)
    dH1 = np.concatenate([da, du], axis=1)
    dW1e = dH1.T @ X
    dX = dH1 @ W1e
    return dX, dW1e, dW2e


# ----------------------------------------------------------------------------- the layer

def layer_forward(cfg, inp, selection_logits32=None):
    """y = sum_j g[t,j] * FFN_{idx[t,j]}(x_t)  (+ c_t * FFN_shared(x_t)).

    cfg: object with T, d, E, k, f, f_shared, score_fn, renorm, shared_gate.
    inp: dict with x, W_r, b_r, W1, W2, Ws1, Ws2, w_sg (any float dtype; read as fp64).
    selection_logits32: optional fp32 logits to select on; by default the fp64 logits
    rounded once to fp32 (router scores are computed in fp32).
    """
    x = f64(inp["x"])
    T = x.shape[0]
    E, k = cfg.E, cfg.k
    select_bias = getattr(cfg, "bias_mode", BIAS_LOGIT) == BIAS_SELECT and inp.get("b_r") is not None
    l = router_logits(x, inp["W_r"], None if select_bias else inp.get("b_r"))
    l32 = l.astype(np.float32) if selection_logits32 is None else np.asarray(
        selection_logits32, dtype=np.float32)
    keys = selection_keys(l32, cfg.score_fn, inp["b_r"]) if select_bias else l32
    idx = select_topk(keys, k)
    g = gate_weights(l, idx, cfg.score_fn, cfg.renorm)
    y = np.zeros_like(x)
    pair_out = np.zeros((T, k, x.shape[1]))
    cache = {}
    for e in range(E):
        t_list, j_list = np.nonzero(idx == e)
        if t_list.size == 0:
            continue
        X = x[t_list]
        o, a, u, h = swiglu_ffn(inp["W1"][e], inp["W2"][e], X)
        pair_out[t_list, j_list] = o
        cache[e] = (t_list, j_list, a, u, h)
    for j in range(k):
        y += g[:, j:j + 1] * pair_out[:, j]
    out = dict(logits=l, idx=idx, gate=g, pair_out=pair_out, expert_cache=cache)
    coeff = getattr(cfg, "aux_coeff", 0.0)
    if coeff:
        counts = np.bincount(idx.ravel(), minlength=E)
        out["counts"] = counts
        out["aux_loss"] = aux_loss(l, counts, k, coeff, cfg.score_fn)
    if cfg.f_shared > 0:
        s_out, s_a, s_u, s_h = swiglu_ffn(inp["Ws1"], inp["Ws2"], x)
        if cfg.shared_gate:
            z = x @ f64(inp["w_sg"])
            c = sigmoid(z)
        else:
            c = np.ones(T)
        y = y + c[:, None] * s_out
        out.update(shared_out=s_out, shared_a=s_a, shared_u=s_u, shared_h=s_h, shared_coef=c)
    out["y"] = y
    return out


def gate_backward(logits, idx, g, dg, score_fn, renorm):
    """dL/dlogits [T, E] from dL/dg [T, k] through the gate functions of gate_weights.
    Selection is piecewise constant in the logits, so no gradient flows through idx.

    softmax, renorm:    dl_j = g_j (dg_j - sum_i g_i dg_i)                 (selected j)
    softmax, no renorm: dl_e = p_e (dG_e - sum_j g_j dg_j), dG_e = dg_j if e = idx_j else 0
    sigmoid, renorm:    dl_j = (dg_j - sum_i g_i dg_i) s_j (1 - s_j) / sum_i s_i
    sigmoid, no renorm: dl_j = dg_j s_j (1 - s_j)
    """
    l = f64(logits)
    T, E = l.shape
    ii = idx.astype(np.int64)
    dl = np.zeros((T, E))
    if score_fn == SOFTMAX:
        if renorm:
            inner = (g * dg).sum(axis=1, keepdims=True)
            np.put_along_axis(dl, ii, g * (dg - inner), axis=1)
        else:
            p = np.exp(l - l.max(axis=1, keepdims=True))
            p = p / p.sum(axis=1, keepdims=True)
            dG = np.zeros((T, E))
            np.put_along_axis(dG, ii, dg, axis=1)
            inner = (g * dg).sum(axis=1, keepdims=True)
            dl = p * (dG - inner)
    else:
        s = sigmoid(np.take_along_axis(l, ii, axis=1))
        if renorm:
            inner = (g * dg).sum(axis=1, keepdims=True)
            np.put_along_axis(dl, ii, (dg - inner) * s * (1 - s) / s.sum(axis=1, keepdims=True),
                              axis=1)
        else:
            np.put_along_axis(dl, ii, dg * s * (1 - s), axis=1)
    return dl


def layer_backward(cfg, inp, fwd, dy):
    """Gradients of L = sum(y * dy) (+ L_aux when the configuration has a balancing-loss
    coefficient) with respect to x and every weight (fp64).

    Returns dict: dx, dW_r, dW1, dW2 (+ dWs1, dWs2, dw_sg with the shared expert), and the
    intermediates dg [T, k], dlogits [T, E].
    """
    x = f64(inp["x"])
    dy = f64(dy)
    T, d = x.shape
    E, k, f = cfg.E, cfg.k, cfg.f
    g = fwd["gate"]
    idx = fwd["idx"]
    dx = np.zeros_like(x)
    dW1 = np.zeros((E, 2 * f, d))
    dW2 = np.zeros((E, d, f))
    # combine: y_t = sum_j g_tj o_tj  ->  do_tj = g_tj dy_t,  dg_tj = <dy_t, o_tj>
    dg = np.einsum("td,tjd->tj", dy, fwd["pair_out"])
    for e, (t_list, j_list, a, u, h) in fwd["expert_cache"].items():
        do = g[t_list, j_list][:, None] * dy[t_list]
        dX, dW1e, dW2e = swiglu_ffn_backward(inp["W1"][e], inp["W2"][e], x[t_list], a, u, h, do)
        dW1[e] = dW1e
        dW2[e] = dW2e
        np.add.at(dx, t_list, dX)
    dl = gate_backward(fwd["logits"], idx, g, dg, cfg.score_fn, cfg.renorm)
    coeff = getattr(cfg, "aux_coeff", 0.0)
    if coeff:
        dl = dl + aux_loss_grad(fwd["logits"], fwd["counts"], k, coeff, cfg.score_fn)
    dW_r = dl.T @ x
    dx += dl @ f64(inp["W_r"])
    out = dict(dx=dx, dW_r=dW_r, dW1=dW1, dW2=dW2, dg=dg, dlogits=dl)
    if cfg.f_shared > 0:
        c = fwd["shared_coef"]
        dS = c[:, None] * dy
        dXs, dWs1, dWs2 = swiglu_ffn_backward(inp["Ws1"], inp["Ws2"], x, fwd["shared_a"],
                                              fwd["shared_u"], fwd["shared_h"], dS)
        dx += dXs
        out.update(dWs1=dWs1, dWs2=dWs2)
        if cfg.shared_gate:
            dc = (dy * fwd["shared_out"]).sum(axis=1)
            dz = dc * c * (1 - c)
            out["dw_sg"] = dz @ x
            dx += dz[:, None] * f64(inp["w_sg"])[None, :]
            out["dz_shared_gate"] = dz
    out["dx"] = dx
    return out


# ----------------------------------------------------------------------------- closed forms

def expert_param_count(d, f):
    """Parameters of one SwiGLU expert without biases: gate_proj and up_proj (f x d each)
    plus down_proj (d x f) = 3*d*f."""
    return 2 * f * d + d * f


def layer_flops(cfg, backward=True):
    """Algorithmic multiply-add FLOPs (2 per MAC) of the layer's matrix products:
    router 2*T*d*E; routed experts 6*T*k*d*f; shared expert 6*T*d*f_s (+2*T*d gate);
    the backward doubles each product (data and weight gradients)."""
    T = cfg.T
    fl = 2.0 * T * cfg.d * cfg.E + 6.0 * T * cfg.k * cfg.d * cfg.f
    if cfg.f_shared:
        fl += 6.0 * T * cfg.d * cfg.f_shared
        if cfg.shared_gate:
            fl += 2.0 * T * cfg.d
    return fl * (3.0 if backward else 1.0)
