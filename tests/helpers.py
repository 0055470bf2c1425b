"""Shared test utilities: running the CUDA layer through the C ABI, running the oracle on the
same inputs, and the comparison metric.

Tolerance metric (per tensor): max_i |gpu_i - ref_i| / max_i |ref_i|.  Bounds: 2e-2 for bf16
layers (bf16 operands, fp32 accumulation), 1e-5 for fp32 layers.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_expert_layer_gemm_gb300 as moe
import moe_inputs
import oracle.moe_oracle as O

TOL = {"bf16": 2e-2, "f32": 1e-5}


def np64(t):
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy() if t.is_floating_point() else \
        t.detach().cpu().numpy()


def rel_err(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.abs(ref).max()
    if scale == 0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu - ref).max() / scale)


def assert_close(name, gpu, ref, tol):
    e = rel_err(gpu, ref)
    assert np.isfinite(np.asarray(gpu, np.float64)).all(), f"{name}: non-finite values"
    assert e <= tol, f"{name}: max|gpu-ref|/max|ref| = {e:.3e} > {tol:.1e}"
    return e


def inputs_to(inp, device):
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def oracle_inputs(inp):
    return {k: np64(v) for k, v in inp.items() if k != "dy"}


def boundary_gap(logits, k):
    """Per row: gap between the k-th and (k+1)-th largest logit (how close the row is to
    selecting a different set of experts)."""
    if k >= logits.shape[1]:
        return np.full(logits.shape[0], np.inf)
    s = -np.sort(-logits, axis=1)
    return s[:, k - 1] - s[:, k]


def order_gap(logits, k):
    """Per row: smallest gap between consecutive logits among the top k+1."""
    s = -np.sort(-logits, axis=1)[:, : k + 1]
    if s.shape[1] < 2:
        return np.full(logits.shape[0], np.inf)
    return np.min(s[:, :-1] - s[:, 1:], axis=1)


LOGIT_TOL = 1e-5      # router logits: max|gpu - fp64| / max|fp64| (fp32 accumulation)
MARGIN = 4 * LOGIT_TOL


def clean_inputs(lc, seed=0, tries=80):
    """CPU-generated inputs whose fp64 router logits keep every row's selected set clear of the
    next expert by more than twice the logit tolerance, so that rounding in the router GEMM
    cannot change which experts are selected.  Only the oracle is consulted."""
    for s in range(seed, seed + tries):
        inp = moe_inputs.make_layer_inputs(lc, seed=s, device="cpu")
        lg = O.router_logits(np64(inp["x"]), np64(inp["W_r"]), np64(inp["b_r"]))
        if boundary_gap(lg, lc.k).min() > MARGIN * max(1.0, np.abs(lg).max()):
            return inp, s
    raise AssertionError("no seed with a clear routing margin")


def run_layer(lc, inp, backward=True, T=None, side=True, stream=None, sync=True):
    """Forward (and backward) through the C ABI; returns dict of torch tensors on the device.
    side=True: the shared expert and the router backward run on a caller-owned side stream
    (moe_side_stream), as bench.py runs them; False: one stream; or a moe.SideStream.
    stream: the calls' stream (default: the current one); sync=False returns without waiting
    for the GPU (the caller synchronises and checks the device error word)."""
    cfg = moe.cfg_from(lc, T=T)
    dev = inp["x"].device
    if side is True:
        side = moe.SideStream(dev)
    elif side is False:
        side = None
    saved = moe.alloc_saved(cfg, dev)
    y = torch.empty_like(inp["x"])
    ws_f = moe.workspace(cfg, moe.WS_LAYER_FWD, dev)
    moe.moe_layer_fwd(cfg, inp["x"], inp["W_r"], inp["b_r"], inp["W1"], inp["W2"], inp["Ws1"],
                      inp["Ws2"], inp["w_sg"], y, saved, ws_f, stream=stream, side=side)
    out = dict(y=y, saved=saved, cfg=cfg, _keep=[ws_f, side])   # alive until the GPU is done
    if backward:
        E, d, f, fs = cfg.E, cfg.d, cfg.f, cfg.f_shared
        f32 = torch.float32
        g = dict(
            dx=torch.empty_like(inp["x"]),
            dW_r=torch.empty(E, d, dtype=f32, device=dev),
            dW1=torch.empty(E, 2 * f, d, dtype=f32, device=dev),
            dW2=torch.empty(E, d, f, dtype=f32, device=dev),
            dWs1=torch.empty(2 * fs, d, dtype=f32, device=dev) if fs else None,
            dWs2=torch.empty(d, fs, dtype=f32, device=dev) if fs else None,
            dw_sg=torch.empty(d, dtype=f32, device=dev) if cfg.shared_gate else None,
        )
        ws_b = moe.workspace(cfg, moe.WS_LAYER_BWD, dev)
        moe.moe_layer_bwd(cfg, inp["dy"], inp["x"], inp["W_r"], inp["W1"], inp["W2"], inp["Ws1"],
                          inp["Ws2"], inp["w_sg"], saved, g["dx"], g["dW_r"], g["dW1"], g["dW2"],
                          g["dWs1"], g["dWs2"], g["dw_sg"], ws_b, stream=stream, side=side)
        out.update(g)
        out["_keep"].append(ws_b)
    if sync:
        torch.cuda.synchronize()
        moe.check_device_error()
    return out


def oracle_layer(lc, inp, backward=True):
    oi = oracle_inputs(inp)
    fwd = O.layer_forward(lc, oi)
    out = dict(fwd=fwd)
    if backward:
        out["bwd"] = O.layer_backward(lc, oi, fwd, np64(inp["dy"]))
    return out


GRAD_NAMES = ["dx", "dW_r", "dW1", "dW2", "dWs1", "dWs2", "dw_sg"]


def compare_layer(lc, gpu, ref, tol, backward=True, order_keys=None):
    """Routing exact, float outputs within tol.  Returns the per-tensor errors.

    The selected SET of every row must equal the oracle's (inputs come from clean_inputs); the
    order inside the set must match wherever the oracle's top-(k+1) selection keys (the logits,
    or `order_keys` when the selection runs on other keys) are farther apart than the router
    GEMM's rounding can move them."""
    fwd = ref["fwd"]
    s = gpu["saved"]
    errs = {}
    lg = fwd["logits"]
    scale = max(1.0, np.abs(lg).max())
    errs["logits"] = assert_close("logits", np64(s["logits"]), lg, LOGIT_TOL if tol > 1e-4 else 1e-6)
    idx = np64(s["idx"]).astype(np.int64)
    oidx = fwd["idx"].astype(np.int64)
    assert (np.sort(idx, 1) == np.sort(oidx, 1)).all(), "selected experts differ from the oracle"
    keys = lg if order_keys is None else np.asarray(order_keys, np.float64)
    clear = order_gap(keys, lc.k) > MARGIN * scale
    assert (idx[clear] == oidx[clear]).all(), "selection order differs on rows with clear margins"
    counts, offsets, sop, tos = O.routing_maps(oidx, lc.E)
    assert (np64(s["counts"]) == counts).all()
    assert (np64(s["offsets"]) == offsets).all()
    # slots depend on the selected sets only: compare per (token, expert)
    gs = np.take_along_axis(np64(s["slot_of_pair"]), np.argsort(idx, 1), 1)
    os_ = np.take_along_axis(sop, np.argsort(oidx, 1), 1)
    assert (gs == os_).all()
    assert (np64(s["token_of_slot"])[: lc.N] == tos).all()
    gg = np.take_along_axis(np64(s["gate"]), np.argsort(idx, 1), 1)
    og = np.take_along_axis(fwd["gate"], np.argsort(oidx, 1), 1)
    errs["gate"] = assert_close("gate", gg, og, 1e-4 if tol > 1e-4 else 1e-5)
    errs["y"] = assert_close("y", np64(gpu["y"]), fwd["y"], tol)
    if "aux_loss" in fwd:
        errs["aux_loss"] = assert_close("aux_loss", np64(s["aux_loss"])[:1],
                                        np.array([fwd["aux_loss"]]), 1e-4 if tol > 1e-4 else 1e-5)
    if backward:
        b = ref["bwd"]
        for n in GRAD_NAMES:
            if gpu.get(n) is None:
                continue
            errs[n] = assert_close(n, np64(gpu[n]), b[n], tol)
    return errs


# ----------------------------------------------------------------------------- MXFP8 layouts
# The packed block-scale layouts of the C ABI (include/moe_gb300.h, MOE_MX_SCALES_*), restated
# here from that documentation to read the GPU's buffers back into row-major [rows, K/32] scales.

def mx_unpack_act_scales(packed, offsets, N, K):
    """Row-major scales [N, K/32] of the permuted rows from the MOE_MX_SCALES_X/_H layout."""
    packed = np.asarray(packed)
    off = np.asarray(offsets, np.int64)
    kch, nb = (K + 127) // 128, K // 32
    pre = np.concatenate([[0], np.cumsum((np.diff(off) + 127) // 128)])
    s = np.arange(N)
    e = np.searchsorted(off, s, side="right") - 1          # the expert that holds row s
    rr = s - off[e]
    mt = pre[e] + rr // 128
    b = np.arange(nb)
    r = rr % 128
    idx = (mt[:, None] * kch + b[None, :] // 4) * 512 + (r % 32)[:, None] * 16 + \
        (r // 32)[:, None] * 4 + (b % 4)[None, :]
    return packed[idx]


def mx_act_pad_bytes(packed, offsets, N, K):
    """The bytes of blocks past K in every row's last chunk (must all be 127)."""
    off = np.asarray(offsets, np.int64)
    kch, nb = (K + 127) // 128, K // 32
    if nb % 4 == 0:
        return np.array([127], np.uint8)
    pre = np.concatenate([[0], np.cumsum((np.diff(off) + 127) // 128)])
    s = np.arange(N)
    e = np.searchsorted(off, s, side="right") - 1
    rr = s - off[e]
    mt = pre[e] + rr // 128
    b = np.arange(nb % 4, 4)
    idx = (mt[:, None] * kch + kch - 1) * 512 + ((rr % 128) % 32)[:, None] * 16 + \
        ((rr % 128) // 32)[:, None] * 4 + b[None, :]
    return np.asarray(packed)[idx]


def mx_weight_index(E, R, K, swiglu_f):
    """Index [E, R, K/32] into the packed weight layout (MOE_MX_SCALES_W1 with swiglu_f = f, R = 2f;
    MOE_MX_SCALES_W2 with swiglu_f = 0)."""
    kch, nb = (K + 127) // 128, K // 32
    q = np.arange(R)
    if swiglu_f:
        hc = np.where(q < swiglu_f, q, q - swiglu_f)
        t = hc // 96
        rt = np.where(q < swiglu_f, hc % 96, 96 + hc % 96)
        NT = (swiglu_f + 95) // 96
    else:
        t, rt = q // 192, q % 192
        NT = (R + 191) // 192
    e = np.arange(E)[:, None, None]
    b = np.arange(nb)[None, None, :]
    t, rt = t[None, :, None], rt[None, :, None]
    return ((e * NT + t) * kch + b // 4) * 1024 + (rt // 128) * 512 + (rt % 32) * 16 + \
        ((rt % 128) // 32) * 4 + b % 4


def mx_weight_index_cols(E, N, K, tile=256):
    """Index [E, K/32, N] into a packed weight layout whose B-rows are the weight's N columns in
    tiles of `tile` (MOE_MX_SCALES_W1C / _W2C: scales of 32-row blocks down each column)."""
    kch, nb = (K + 127) // 128, K // 32
    NT = (N + tile - 1) // tile
    n = np.arange(N)[None, None, :]
    t, rt = n // tile, n % tile
    e = np.arange(E)[:, None, None]
    b = np.arange(nb)[None, :, None]
    return ((e * NT + t) * kch + b // 4) * ((tile + 127) // 128 * 512) + (rt // 128) * 512 + \
        (rt % 32) * 16 + ((rt % 128) // 32) * 4 + b % 4
