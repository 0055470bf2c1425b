"""MXFP8 weight gradients on the GPU against the oracle, through the C ABI.

  * moe_mxfp8_quantize_tokens: codes bit-identical to the oracle's token-direction blocks inside
    every expert segment, every scale byte at its documented place in the token-chunk layout, the
    blocks past a segment's rows in its last chunk 127, and the chunk bases;
  * moe_grouped_swiglu_wgrad_mxfp8: dW1 and dW2 within fp32 accumulation of the oracle's fp64
    products of the decoded operands, zero blocks for experts without rows;
  * moe_layer_bwd_mxfp8 with the weight-gradient scratch: dW2 against the oracle's MXFP8 product of
    the layer's own dy_perm and saved h; dW1 beside the bf16 backward's; every other gradient
    identical to the layer's bf16 weight-gradient run.
Segments cover empty experts, segments of 1, 31, 32, 33, 127, 128, 129 and several hundred rows,
and columns that leave the last 128-column tile partly empty.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import oracle.mxfp8_oracle as MX

from .helpers import assert_close, clean_inputs, np64, oracle_layer, rel_err
from .test_gpu_mxfp8 import LAYER_CASES, sync, varied

pytestmark = pytest.mark.gpu

TOL_ACC = 2e-5   # fp32 accumulation of exact products of block-scaled E4M3 values

SEGMENTS = {
    "ragged": [0, 1, 31, 32, 33, 127, 128, 129, 300, 0, 2],
    "one-expert": [700],
    "empty-ends": [0, 96, 5, 0],
}


def offsets_of(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)


def token_scale_index(c, kc, j, kct):
    """Byte of column c, token chunk kc and block j of the chunk in the token-chunk layout."""
    return ((c // 128) * kct + kc) * 512 + (c % 32) * 16 + (c % 128 // 32) * 4 + j


def check_token_scales(s_packed, ref_scales, offsets, C, N, E, cbase):
    kct = N // 128 + E
    cols = np.arange(C)
    cb = 0
    for e in range(E):
        n = int(offsets[e + 1] - offsets[e])
        assert cbase[e] == cb, ("cbase", e)
        nb = -(-n // 32)
        for b in range(nb):
            got = s_packed[token_scale_index(cols, cb + b // 4, b % 4, kct)]
            assert np.array_equal(got, ref_scales[e][b]), ("scale", e, b)
        if nb % 4:   # the last chunk's blocks past the segment's rows
            for j in range(nb % 4, 4):
                assert (s_packed[token_scale_index(cols, cb + (nb - 1) // 4, j, kct)] == 127).all()
        cb += -(-n // 128)
    assert cbase[E] == cb


def quantize_tokens(cfg, x, offsets_t):
    N, C = x.shape
    q = torch.empty(N, C, dtype=torch.uint8, device="cuda")
    s = torch.full((-(-C // 128) * (N // 128 + cfg.E) * 512,), 0xEE, dtype=torch.uint8,
                   device="cuda")
    cbase = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
    moe.moe_mxfp8_quantize_tokens(cfg, x, offsets_t, q, s, cbase)
    sync()
    return q.cpu().numpy(), s.cpu().numpy(), cbase.cpu().numpy()


@pytest.mark.parametrize("segs", list(SEGMENTS))
@pytest.mark.parametrize("C", [64, 160, 2688])
def test_token_blocks_are_exact(segs, C):
    lengths = SEGMENTS[segs]
    off = offsets_of(lengths)
    N, E = int(off[-1]), len(lengths)
    cfg = moe.make_cfg(N, 64, E, 1, 64)
    # magnitudes that change every few rows, exact zeros and saturating values
    x = varied((C, N + (-N) % 32), seed=C + N, spread=6.0).T[:N].contiguous()
    x[::17, 3] = 0
    q, s, cbase = quantize_tokens(cfg, x.cuda(), torch.from_numpy(off).int().cuda())
    rq, rs = MX.mx_quantize_segments(np64(x), off)
    assert np.array_equal(q, rq)
    check_token_scales(s, rs, off, C, N, E, cbase)


def test_token_blocks_reject_bad_offsets():
    """Offsets past N are reported through the device error word and nothing is written."""
    cfg = moe.make_cfg(64, 64, 2, 1, 64)
    x = torch.ones(64, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(64, 64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(64 * 512, dtype=torch.uint8, device="cuda")
    cbase = torch.zeros(3, dtype=torch.int32, device="cuda")
    bad = torch.tensor([0, 40, 80], dtype=torch.int32, device="cuda")
    moe.moe_mxfp8_quantize_tokens(cfg, x, bad, q, s, cbase)
    torch.cuda.synchronize()
    with pytest.raises(RuntimeError):
        moe.check_device_error()
    assert not q.any() and not s.any()


@pytest.mark.parametrize("segs", list(SEGMENTS))
@pytest.mark.parametrize("d,f", [(160, 96), (256, 192)])
def test_grouped_weight_gradients(segs, d, f):
    lengths = SEGMENTS[segs]
    off = offsets_of(lengths)
    N, E = int(off[-1]), len(lengths)
    cfg = moe.make_cfg(N, d, E, 1, f)
    ops = {n: varied((N, C), seed=i * 101 + N, spread=3.0)
           for i, (n, C) in enumerate((("x", d), ("h", f), ("dy", d), ("dH1", 2 * f)))}
    dev = {n: v.cuda() for n, v in ops.items()}
    dW1 = torch.full((E, 2 * f, d), float("nan"), device="cuda")
    dW2 = torch.full((E, d, f), float("nan"), device="cuda")
    ws = moe.workspace(cfg, moe.WS_WGRAD_MXFP8)
    moe.moe_grouped_swiglu_wgrad_mxfp8(cfg, torch.from_numpy(off).int().cuda(), dev["x"], dev["h"],
                                       dev["dy"], dev["dH1"], dW1, dW2, ws)
    sync()
    q = {n: MX.mx_quantize_segments(np64(v), off) for n, v in ops.items()}
    ref1 = MX.wgrad_mx(*q["dH1"], *q["x"], off)
    ref2 = MX.wgrad_mx(*q["dy"], *q["h"], off)
    e1 = assert_close("dW1", np64(dW1), ref1, TOL_ACC)
    e2 = assert_close("dW2", np64(dW2), ref2, TOL_ACC)
    for e in range(E):
        if lengths[e] == 0:
            assert not dW1[e].any() and not dW2[e].any(), e
    print(f"dW1 {e1:.2e} dW2 {e2:.2e}")


@pytest.mark.parametrize("name", ["sigmoid-shared", "ragged-d"])
def test_layer_backward_with_mxfp8_weight_gradients(name):
    lc = LAYER_CASES[name]
    host, _ = clean_inputs(lc)
    inp = {k: (None if v is None else v.cuda()) for k, v in host.items()}
    cfg = moe.cfg_from(lc)
    m = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"])
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
    mxd = moe.alloc_mxfp8_dgrad(cfg, inp["W1"], inp["W2"])
    args = (inp["Ws1"], inp["Ws2"], inp["w_sg"], saved)
    moe.moe_layer_bwd_mxfp8(cfg, inp["dy"], inp["x"], inp["W_r"], mxd, *args, g16["dx"],
                            g16["dW_r"], g16["dW1"], g16["dW2"], g16["dWs1"], g16["dWs2"],
                            g16["dw_sg"], ws)
    mxd["wgrad_ws"] = moe.workspace(cfg, moe.WS_WGRAD_MXFP8)
    moe.moe_layer_bwd_mxfp8(cfg, inp["dy"], inp["x"], inp["W_r"], mxd, *args, gmx["dx"],
                            gmx["dW_r"], gmx["dW1"], gmx["dW2"], gmx["dWs1"], gmx["dWs2"],
                            gmx["dw_sg"], ws)
    sync()
    # every gradient but the routed experts' weight gradients is the same computation
    for g in ("dx", "dW_r", "dWs1", "dWs2") + (("dw_sg",) if lc.shared_gate else ()):
        assert torch.equal(gmx[g], g16[g]), g
    # dW2 = dy_perm^T h on token blocks: dy_perm[slot(t, j)] = bf16(gate[t, j] * dy[t]) and the
    # saved bf16 h
    N = lc.T * lc.k
    sop = np64(saved["slot_of_pair"]).astype(np.int64).reshape(-1)
    prod = saved["gate"].cpu().float()[..., None] * inp["dy"].cpu().float()[:, None, :]
    dy_perm = np.zeros((N, d))
    dy_perm[sop] = np64(prod.to(torch.bfloat16).reshape(N, d))
    o = np64(saved["offsets"]).astype(np.int64)
    ref2 = MX.wgrad_mx(*MX.mx_quantize_segments(dy_perm, o),
                       *MX.mx_quantize_segments(np64(saved["h"]), o), o)
    e2 = assert_close("dW2", np64(gmx["dW2"]), ref2, TOL_ACC)
    # The MXFP8 weight gradients against the bf16 ones and the unquantised oracle: both operands
    # of every product are rounded to E4M3 (a 3-bit mantissa: relative error <= 2^-4 each), so a
    # product is off by at most 2^-3 + 2^-8 of itself and a sum of them by that much of the sum of
    # their magnitudes; with few rows per expert and mixed signs that reaches ~0.13 of max |ref|.
    ref = oracle_layer(lc, {k: (None if v is None else v.cpu()) for k, v in inp.items()})
    errs = {"dW2 vs token-block oracle": e2}
    for g in ("dW1", "dW2"):
        errs[g + " vs bf16"] = rel_err(np64(gmx[g]), np64(g16[g]))
        assert errs[g + " vs bf16"] < 0.15, errs
        errs[g + " vs oracle"] = rel_err(np64(gmx[g]), ref["bwd"][g])
        assert errs[g + " vs oracle"] < 0.2, errs
    print("mxfp8 weight gradients:", {k: f"{v:.3e}" for k, v in errs.items()})


def test_zero_tokens():
    """T = 0: the grouped weight gradients are zero blocks; the quantiser writes only the chunk
    bases (all zero)."""
    cfg = moe.make_cfg(0, 64, 4, 1, 64)
    dev = "cuda"
    # operand buffers (not read when there are no rows; one row each so that they are not null)
    empty = torch.zeros(1, 64, dtype=torch.bfloat16, device=dev)
    off = torch.zeros(5, dtype=torch.int32, device=dev)
    dW1 = torch.full((4, 128, 64), float("nan"), device=dev)
    dW2 = torch.full((4, 64, 64), float("nan"), device=dev)
    ws = moe.workspace(cfg, moe.WS_WGRAD_MXFP8)
    moe.moe_grouped_swiglu_wgrad_mxfp8(cfg, off, empty, empty, empty,
                                       torch.zeros(1, 128, dtype=torch.bfloat16, device=dev),
                                       dW1, dW2, ws)
    cbase = torch.full((5,), -1, dtype=torch.int32, device=dev)
    q = torch.empty(1, 64, dtype=torch.uint8, device=dev)
    s = torch.empty(4 * 512, dtype=torch.uint8, device=dev)
    moe.moe_mxfp8_quantize_tokens(cfg, empty, off, q, s, cbase)
    sync()
    assert not dW1.any() and not dW2.any()
    assert not cbase.any()
