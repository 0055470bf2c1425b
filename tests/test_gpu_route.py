"""Routing stage (moe_route_topk with given fp32 logits) against the oracle: expert indices,
counts, offsets and both permutation maps bit-for-bit; gates within fp32 rounding.

Includes the routing/permute stress workload at full size (T=65536, E=128, top-8 sigmoid) with
its degenerate cases: every token on the same 8 experts, 32 experts that receive nothing, and
integer logits with massive exact ties; a histogram past the size every slots block reads whole
(the scan path); and the bf16 router GEMM, whose epilogue routes the tokens from its
accumulator, against the top-k kernel on the logits that GEMM wrote -- bit for bit.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import moe_inputs
import oracle.moe_oracle as O

from .helpers import np64

pytestmark = pytest.mark.gpu


def route_gpu(T, E, k, score_fn, renorm, logits, x=None, W_r=None, b_r=None,
              bias_mode=moe.BIAS_LOGIT, logits_out=None):
    d = 8 if x is None else x.shape[1]
    cfg = moe.make_cfg(T, d, E, k, 8, score_fn=score_fn, renorm=renorm, bias_mode=bias_mode)
    dev = "cuda"
    i32 = torch.int32
    out = dict(idx=torch.full((T, k), -7, dtype=i32, device=dev),
               gate=torch.full((T, k), float("nan"), device=dev),
               counts=torch.full((E,), -7, dtype=i32, device=dev),
               offsets=torch.full((E + 1,), -7, dtype=i32, device=dev),
               slot_of_pair=torch.full((T, k), -7, dtype=i32, device=dev),
               token_of_slot=torch.full((max(T * k, 1),), -7, dtype=i32, device=dev))
    ws = moe.workspace(cfg, moe.WS_ROUTE, dev)
    moe.moe_route_topk(cfg, x, W_r, b_r, logits, logits_out, out["idx"], out["gate"],
                       out["counts"], out["offsets"], out["slot_of_pair"], out["token_of_slot"], ws)
    torch.cuda.synchronize()
    moe.check_device_error()
    return {n: t.cpu().numpy() for n, t in out.items()}


def check_route(T, E, k, score_fn, renorm, logits):
    g = route_gpu(T, E, k, score_fn, renorm, logits.cuda())
    lg = logits.cpu().numpy()
    r = O.route(lg, k, E, score_fn, renorm)
    assert (g["idx"] == r["idx"]).all(), "idx"
    assert (g["counts"] == r["counts"]).all(), "counts"
    assert (g["offsets"] == r["offsets"]).all(), "offsets"
    assert (g["slot_of_pair"] == r["slot_of_pair"]).all(), "slot_of_pair"
    assert (g["token_of_slot"][: T * k] == r["token_of_slot"]).all(), "token_of_slot"
    err = np.abs(g["gate"] - r["gate"]).max() / np.abs(r["gate"]).max()
    assert err < 2e-6, f"gate error {err}"
    return g


@pytest.mark.parametrize("E,k", [(8, 2), (5, 3), (1, 1), (32, 6), (128, 8), (256, 8), (256, 1),
                                 (64, 8)])
@pytest.mark.parametrize("score_fn,renorm", [(0, 1), (0, 0), (1, 1), (1, 0)])
def test_route_random_logits(E, k, score_fn, renorm):
    T = 777
    lg = torch.randn(T, E, generator=torch.Generator().manual_seed(E * 31 + k)) * 2.0
    check_route(T, E, k, score_fn, renorm, lg)


@pytest.mark.parametrize("case", moe_inputs.STRESS_CASES)
def test_route_stress_full_size(case):
    lc = moe_inputs.ROUTE_STRESS
    lg = moe_inputs.make_stress_logits(case, lc.T, lc.E, seed=0)
    g = check_route(lc.T, lc.E, lc.k, lc.score_fn, lc.renorm, lg)
    if case == "all_to_8":
        assert (g["counts"][:8] == lc.T).all() and (g["counts"][8:] == 0).all()
    if case == "32_empty":
        assert (g["counts"][lc.E - 32:] == 0).all()


@pytest.mark.parametrize("T", [1, 7, 255, 256, 257, 4097])
def test_route_token_counts_around_block_edges(T):
    lg = torch.randint(0, 3, (T, 16), generator=torch.Generator().manual_seed(T)).float()
    check_route(T, 16, 4, 1, 1, lg)


@pytest.mark.parametrize("E,k", [(64, 4), (128, 8)])
def test_route_nan_logits_stay_in_range(E, k):
    """NaN logits are outside the inputs' contract, but routing must stay memory-safe: a NaN key
    ranks as -inf, so every selected expert is in [0, E), each row's set is distinct, and the
    maps remain a bijection.  Rows without NaN are routed as the oracle routes them."""
    T = 300
    lg = torch.randn(T, E, generator=torch.Generator().manual_seed(E + k)) * 2.0
    lg[:10] = float("nan")                      # whole rows
    lg[10:20, ::2] = float("nan")               # half rows
    g = route_gpu(T, E, k, 1, 1, lg.cuda())
    idx = g["idx"]
    assert ((idx >= 0) & (idx < E)).all()
    assert all(len(set(r)) == k for r in idx.tolist())
    assert g["counts"].sum() == T * k and g["offsets"][-1] == T * k
    assert np.array_equal(np.sort(g["token_of_slot"][: T * k]), np.repeat(np.arange(T), k))
    r = O.route(lg[20:].numpy(), k, E, 1, 1)
    assert (idx[20:] == r["idx"]).all()
    # whole-NaN rows: every key ranks as -inf, ties go to the lowest experts
    assert (idx[:10] == np.arange(k)).all()


def test_route_large_histogram_takes_the_scan_path():
    """T=140000, E=128: 1094 histogram rows of 128 bytes, past the 128 KB every slots block reads
    whole, so a scan kernel forms the per-row prefixes first."""
    T, E, k = 140000, 128, 8
    lg = torch.randint(-20, 20, (T, E), generator=torch.Generator().manual_seed(3)).float()
    lg[: T // 2, :8] += 100.0                 # half the tokens on the same 8 experts
    check_route(T, E, k, 1, 0, lg)


def _router_inputs(T, d, E, seed, integer=False):
    g = torch.Generator().manual_seed(seed)
    if integer:
        # logits are exact integer sums of +-1 products: many exact ties between experts
        x = torch.randint(-1, 2, (T, d), generator=g).float()
        W = torch.randint(-1, 2, (E, d), generator=g).float()
        b = torch.randint(-2, 3, (E,), generator=g).float()
    else:
        x = torch.randn(T, d, generator=g)
        W = torch.randn(E, d, generator=g) * 0.05
        b = torch.randn(E, generator=g) * 0.3
    return x.bfloat16().cuda(), W.bfloat16().cuda(), b.cuda()


def _gemm_vs_kernel(T, d, E, k, score_fn, renorm, bias_mode, seed, integer=False):
    x, W, b = _router_inputs(T, d, E, seed, integer)
    lg = torch.empty(T, E, device="cuda")
    fused = route_gpu(T, E, k, score_fn, renorm, None, x=x, W_r=W, b_r=b, bias_mode=bias_mode,
                      logits_out=lg)
    # the same logits through the standalone top-k kernel (the selection bias, if any, again)
    alone = route_gpu(T, E, k, score_fn, renorm, lg.clone(), b_r=b, bias_mode=bias_mode)
    for n in ("idx", "counts", "offsets", "slot_of_pair", "token_of_slot"):
        assert np.array_equal(fused[n], alone[n]), n
    assert np.array_equal(fused["gate"].view(np.uint32), alone["gate"].view(np.uint32)), "gate bits"
    # and both against the oracle on those logits (selection exact: the keys are fp32 logits)
    if bias_mode == moe.BIAS_LOGIT:
        r = O.route(lg.cpu().numpy(), k, E, score_fn, renorm)
        assert np.array_equal(fused["idx"], r["idx"])
        assert np.array_equal(fused["slot_of_pair"], r["slot_of_pair"])
        err = np.abs(fused["gate"] - r["gate"]).max() / np.abs(r["gate"]).max()
        assert err < 2e-6, f"gate error {err}"
    return fused


@pytest.mark.parametrize("E,k", [(8, 2), (5, 3), (64, 6), (128, 8), (160, 4), (256, 8), (256, 1)])
@pytest.mark.parametrize("score_fn,renorm", [(0, 1), (0, 0), (1, 1), (1, 0)])
def test_router_gemm_epilogue_routes_as_the_topk_kernel(E, k, score_fn, renorm):
    _gemm_vs_kernel(1000, 256, E, k, score_fn, renorm, moe.BIAS_LOGIT, seed=E * 7 + k)


@pytest.mark.parametrize("E,k", [(64, 6), (256, 8)])
@pytest.mark.parametrize("score_fn,renorm", [(0, 1), (0, 0), (1, 1), (1, 0)])
def test_router_gemm_epilogue_with_selection_bias(E, k, score_fn, renorm):
    _gemm_vs_kernel(777, 192, E, k, score_fn, renorm, moe.BIAS_SELECT, seed=E + k)


@pytest.mark.parametrize("T,E,k", [(4097, 128, 8), (300, 16, 4), (129, 256, 8)])
def test_router_gemm_epilogue_integer_ties(T, E, k):
    f = _gemm_vs_kernel(T, 128, E, k, 1, 1, moe.BIAS_LOGIT, seed=T, integer=True)
    assert len(set(map(tuple, f["idx"].tolist()))) > 1
