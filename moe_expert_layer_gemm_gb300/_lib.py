"""ctypes binding of libmoe_gb300.so (declared in include/moe_gb300.h).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.  The
functions take torch CUDA tensors (PyTorch provides device memory and streams) and raise
RuntimeError with the library's message when a call fails.  There is no fallback: without the
built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "_build", "libmoe_gb300.so")
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")

MOE_OK = 0
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_WORKSPACE",
          -4: "MOE_ERR_ALIGNMENT", -5: "MOE_ERR_CUDA", -6: "MOE_ERR_DEVICE_CHECK"}
SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1
DTYPE_BF16, DTYPE_F32 = 0, 1
BIAS_LOGIT, BIAS_SELECT = 0, 1
WS_ROUTE, WS_FFN_FWD, WS_FFN_BWD, WS_LAYER_FWD, WS_LAYER_BWD, WS_FFN_BWD_FP8, WS_LAYER_BWD_FP8, \
    WS_WGRAD_MXFP8 = range(8)
MX_SCALES_X, MX_SCALES_H, MX_SCALES_W1, MX_SCALES_W2, MX_SCALES_DH1, MX_SCALES_W1C, MX_SCALES_W2C, \
    MX_SCALES_TOK_D, MX_SCALES_TOK_F, MX_SCALES_TOK_2F = range(10)


class MoeCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d", "E", "k", "f", "f_shared", "score_fn", "renorm", "shared_gate", "dtype",
                 "bias_mode")] + [("aux_coeff", ctypes.c_float)]


class MoeSaved(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("logits", "idx", "gate", "counts", "offsets", "slot_of_pair", "token_of_slot",
                 "x_perm", "act", "h", "y_perm", "s_act", "s_h", "s_out", "s_coef", "aux_loss")]


class MoeFp8Experts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W1_q", "W1_scale", "W2_q", "W2_scale", "x_perm_q", "h_q", "scales",
                 "Ws1_q", "Ws1_scale", "Ws2_q", "Ws2_scale", "x_q", "s_h_q")]


class MoeMxfp8Experts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W1_q", "W1_sp", "W2_q", "W2_sp", "x_perm_q", "x_perm_s", "h_q", "h_s")]


class MoeMxfp8Dgrad(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("W1c_q", "W1c_sp", "W2c_q", "W2c_sp", "dy_q", "dy_s", "dH1_q", "dH1_s",
                 "wgrad_ws")] + [("wgrad_ws_bytes", ctypes.c_size_t)]


class MoeSideStream(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("stream", "fork", "join")]


class SideStream:
    """A caller-owned second stream for the layer calls (moe_side_stream): a torch CUDA stream and
    two events, on `device`.  Pass it as `side=` to moe_layer_fwd* / moe_layer_bwd* so that the
    shared expert (and, in the backward, the router's backward) runs beside the routed experts.
    One SideStream serves one sequence of calls; concurrent callers each need their own."""

    def __init__(self, device="cuda"):
        import torch
        self.stream = torch.cuda.Stream(device=device)
        self.fork = torch.cuda.Event()
        self.join = torch.cuda.Event()
        # torch creates an event's CUDA handle on its first record
        with torch.cuda.device(self.stream.device):
            self.fork.record(self.stream)
            self.join.record(self.stream)
        self.struct = MoeSideStream(self.stream.cuda_stream, self.fork.cuda_event,
                                    self.join.cuda_event)


def _side(side):
    return None if side is None else ctypes.byref(side.struct)


_VP = ctypes.c_void_p
_SZ = ctypes.c_size_t
_CFG = ctypes.POINTER(MoeCfg)
_SIDE = ctypes.POINTER(MoeSideStream)
_SIGS = {
    "moe_workspace_bytes": (_SZ, [_CFG, ctypes.c_int]),
    "moe_route_topk": (ctypes.c_int, [_CFG] + [_VP] * 12 + [_SZ, _VP]),
    "moe_route_topk_noalloc": (ctypes.c_int, [_CFG] + [_VP] * 12),
    "moe_permute": (ctypes.c_int, [_CFG, _VP, _VP, _VP, _VP]),
    "moe_grouped_swiglu_fwd": (ctypes.c_int, [_CFG] + [_VP] * 8 + [_SZ, _VP]),
    "moe_grouped_swiglu_bwd": (ctypes.c_int, [_CFG] + [_VP] * 11 + [_SZ, _VP]),
    "moe_grouped_swiglu_fwd_gathered": (ctypes.c_int, [_CFG] + [_VP] * 9 + [_SZ, _VP]),
    "moe_grouped_swiglu_bwd_gathered": (ctypes.c_int, [_CFG] + [_VP] * 12 + [_SZ, _VP]),
    "moe_quantize_e4m3": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_int32, _VP, _VP, _VP, _VP]),
    "moe_grouped_swiglu_fwd_fp8": (ctypes.c_int, [_CFG] + [_VP] * 14),
    "moe_grouped_swiglu_bwd_fp8": (ctypes.c_int, [_CFG] + [_VP] * 22 + [_SZ, _VP]),
    "moe_permute_quantize_e4m3": (ctypes.c_int, [_CFG] + [_VP] * 6),
    "moe_mxfp8_scale_bytes": (_SZ, [_CFG, ctypes.c_int]),
    "moe_quantize_mxfp8": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.c_int32, _VP, _VP, _VP]),
    "moe_mxfp8_pack_expert_scales": (ctypes.c_int, [_CFG] + [_VP] * 5),
    "moe_permute_quantize_mxfp8": (ctypes.c_int, [_CFG] + [_VP] * 6),
    "moe_grouped_swiglu_fwd_mxfp8": (ctypes.c_int, [_CFG] + [_VP] * 13),
    "moe_layer_fwd_mxfp8": (ctypes.c_int, [_CFG] + [_VP] * 3 + [ctypes.POINTER(MoeMxfp8Experts)]
                            + [_VP] * 4 + [ctypes.POINTER(MoeSaved), _VP, _SZ, _VP, _SIDE]),
    "moe_mxfp8_prepare_dgrad_weights": (ctypes.c_int, [_CFG] + [_VP] * 9),
    "moe_grouped_swiglu_dgrad_mxfp8": (ctypes.c_int, [_CFG] + [_VP] * 14),
    "moe_mxfp8_quantize_tokens": (ctypes.c_int, [_CFG, _VP, ctypes.c_int32] + [_VP] * 5),
    "moe_grouped_swiglu_wgrad_mxfp8": (ctypes.c_int, [_CFG] + [_VP] * 8 + [_SZ, _VP]),
    "moe_layer_bwd_mxfp8": (ctypes.c_int, [_CFG] + [_VP] * 3 + [ctypes.POINTER(MoeMxfp8Dgrad)]
                            + [_VP] * 3 + [ctypes.POINTER(MoeSaved)] + [_VP] * 8 + [_SZ, _VP, _SIDE]),
    "moe_unpermute_combine": (ctypes.c_int, [_CFG] + [_VP] * 7),
    "moe_unpermute_combine_bwd": (ctypes.c_int, [_CFG] + [_VP] * 11),
    "moe_layer_fwd": (ctypes.c_int, [_CFG] + [_VP] * 9 + [ctypes.POINTER(MoeSaved), _VP, _SZ, _VP,
                                                       _SIDE]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [_VP, _VP]),
    "moe_layer_fwd_fp8": (ctypes.c_int, [_CFG] + [_VP] * 3 + [ctypes.POINTER(MoeFp8Experts)]
                          + [_VP] * 4 + [ctypes.POINTER(MoeSaved), _VP, _SZ, _VP, _SIDE]),
    "moe_layer_bwd_fp8": (ctypes.c_int, [_CFG] + [_VP] * 3 + [ctypes.POINTER(MoeFp8Experts)]
                          + [_VP] * 3 + [ctypes.POINTER(MoeSaved)] + [_VP] * 8 + [_SZ, _VP, _SIDE]),
    "moe_layer_bwd": (ctypes.c_int, [_CFG] + [_VP] * 8 + [ctypes.POINTER(MoeSaved)] + [_VP] * 8
                      + [_SZ, _VP, _SIDE]),
    "moe_router_aux_loss": (ctypes.c_int, [_CFG, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_expert_bias_update": (ctypes.c_int, [_CFG, _VP, _VP, ctypes.c_float, _VP]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_check_device_error": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_int32)]),
    "moe_launch_count": (ctypes.c_uint64, []),
    "moe_gemm_wait_stats": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint64), ctypes.c_int]),
    "moe_trace_enable": (ctypes.c_int, [ctypes.c_int]),
    "moe_trace_read": (ctypes.c_int, [ctypes.c_char_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(ctypes.c_double), ctypes.c_int]),
    "moe_version": (ctypes.c_int, []),
}

_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"MoE CUDA library not built ({LIB_PATH} missing): run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_functions():
    """Names of the functions include/moe_gb300.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(",
                                 text, re.M)))


def _check(rc, what):
    if rc != MOE_OK:
        msg = lib().moe_last_error().decode(errors="replace")
        raise RuntimeError(f"{what}: {STATUS.get(rc, rc)}: {msg}")


def make_cfg(T, d, E, k, f, f_shared=0, score_fn=0, renorm=1, shared_gate=0, dtype=DTYPE_BF16,
             bias_mode=BIAS_LOGIT, aux_coeff=0.0):
    return MoeCfg(T, d, E, k, f, f_shared, score_fn, renorm, shared_gate, dtype, bias_mode,
                  aux_coeff)


def cfg_from(lc, T=None):
    """MoeCfg from a moe_inputs.LayerConfig-like object."""
    return make_cfg(lc.T if T is None else T, lc.d, lc.E, lc.k, lc.f, lc.f_shared, lc.score_fn,
                    lc.renorm, lc.shared_gate, DTYPE_BF16 if lc.dtype == "bf16" else DTYPE_F32,
                    getattr(lc, "bias_mode", BIAS_LOGIT), getattr(lc, "aux_coeff", 0.0))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def workspace_bytes(cfg, which):
    return int(lib().moe_workspace_bytes(ctypes.byref(cfg), which))


def workspace(cfg, which, device="cuda"):
    import torch
    n = workspace_bytes(cfg, which)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------- stage calls

def moe_route_topk(cfg, x, W_r, b_r, logits_in, logits_out, idx, gate, counts, offsets,
                   slot_of_pair, token_of_slot, ws, stream=None):
    _check(lib().moe_route_topk(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), _p(logits_in),
                                _p(logits_out), _p(idx), _p(gate), _p(counts), _p(offsets),
                                _p(slot_of_pair), _p(token_of_slot), _p(ws),
                                0 if ws is None else ws.numel(), _stream(stream)),
           "moe_route_topk")


def moe_route_topk_noalloc(cfg, x, W_r, b_r, logits_in, logits_out, idx, gate, counts, offsets,
                           slot_of_pair, token_of_slot, stream=None):
    """moe_route_topk without a workspace (scratch inside the library; see the header)."""
    _check(lib().moe_route_topk_noalloc(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), _p(logits_in),
                                        _p(logits_out), _p(idx), _p(gate), _p(counts), _p(offsets),
                                        _p(slot_of_pair), _p(token_of_slot), _stream(stream)),
           "moe_route_topk_noalloc")


def moe_permute(cfg, x, slot_of_pair, x_perm, stream=None):
    _check(lib().moe_permute(ctypes.byref(cfg), _p(x), _p(slot_of_pair), _p(x_perm),
                             _stream(stream)), "moe_permute")


def moe_grouped_swiglu_fwd(cfg, x_perm, offsets, W1, W2, h, act, y_perm, ws=None, stream=None):
    _check(lib().moe_grouped_swiglu_fwd(ctypes.byref(cfg), _p(x_perm), _p(offsets), _p(W1), _p(W2),
                                        _p(h), _p(act), _p(y_perm), _p(ws),
                                        0 if ws is None else ws.numel(), _stream(stream)),
           "moe_grouped_swiglu_fwd")


def moe_grouped_swiglu_bwd(cfg, x_perm, offsets, W1, W2, act, h, dy_perm, dx_perm, dW1, dW2, ws,
                           stream=None):
    _check(lib().moe_grouped_swiglu_bwd(ctypes.byref(cfg), _p(x_perm), _p(offsets), _p(W1), _p(W2),
                                        _p(act), _p(h), _p(dy_perm), _p(dx_perm), _p(dW1), _p(dW2),
                                        _p(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "moe_grouped_swiglu_bwd")


def moe_grouped_swiglu_fwd_gathered(cfg, x, token_of_slot, offsets, W1, W2, h, act, y_perm,
                                    ws=None, stream=None):
    _check(lib().moe_grouped_swiglu_fwd_gathered(
        ctypes.byref(cfg), _p(x), _p(token_of_slot), _p(offsets), _p(W1), _p(W2), _p(h), _p(act),
        _p(y_perm), _p(ws), 0 if ws is None else ws.numel(), _stream(stream)),
        "moe_grouped_swiglu_fwd_gathered")


def moe_grouped_swiglu_bwd_gathered(cfg, x, token_of_slot, offsets, W1, W2, act, h, dy_perm,
                                    dx_perm, dW1, dW2, ws, stream=None):
    _check(lib().moe_grouped_swiglu_bwd_gathered(
        ctypes.byref(cfg), _p(x), _p(token_of_slot), _p(offsets), _p(W1), _p(W2), _p(act), _p(h),
        _p(dy_perm), _p(dx_perm), _p(dW1), _p(dW2), _p(ws), 0 if ws is None else ws.numel(),
        _stream(stream)), "moe_grouped_swiglu_bwd_gathered")


def moe_quantize_e4m3(x, groups, q, scale, amax, stream=None):
    """E4M3 codes (uint8 tensor shaped like x) and per-group scales of the bf16 tensor x."""
    _check(lib().moe_quantize_e4m3(_p(x), x.numel() // groups, groups, _p(q), _p(scale), _p(amax),
                                   _stream(stream)), "moe_quantize_e4m3")


def moe_permute_quantize_e4m3(cfg, x, slot_of_pair, x_perm_q, x_scale, x_amax, stream=None):
    _check(lib().moe_permute_quantize_e4m3(ctypes.byref(cfg), _p(x), _p(slot_of_pair), _p(x_perm_q),
                                           _p(x_scale), _p(x_amax), _stream(stream)),
           "moe_permute_quantize_e4m3")


def moe_grouped_swiglu_fwd_fp8(cfg, x_perm_q, x_scale, offsets, W1_q, W1_scale, W2_q, W2_scale, h,
                               act, h_q, h_scale, h_amax, y_perm, stream=None):
    _check(lib().moe_grouped_swiglu_fwd_fp8(
        ctypes.byref(cfg), _p(x_perm_q), _p(x_scale), _p(offsets), _p(W1_q), _p(W1_scale),
        _p(W2_q), _p(W2_scale), _p(h), _p(act), _p(h_q), _p(h_scale), _p(h_amax), _p(y_perm),
        _stream(stream)), "moe_grouped_swiglu_fwd_fp8")


def moe_grouped_swiglu_bwd_fp8(cfg, x_perm_q, x_scale, offsets, W1_q, W1_scale, W2_q, W2_scale, act,
                               h_q, h_scale, dy_perm, dy_q, dy_scale, dy_amax, dH1, dH1_q,
                               dH1_scale, dH1_amax, dx_perm, dW1, dW2, ws, stream=None):
    _check(lib().moe_grouped_swiglu_bwd_fp8(
        ctypes.byref(cfg), _p(x_perm_q), _p(x_scale), _p(offsets), _p(W1_q), _p(W1_scale),
        _p(W2_q), _p(W2_scale), _p(act), _p(h_q), _p(h_scale), _p(dy_perm), _p(dy_q), _p(dy_scale),
        _p(dy_amax), _p(dH1), _p(dH1_q), _p(dH1_scale), _p(dH1_amax), _p(dx_perm), _p(dW1),
        _p(dW2), _p(ws), 0 if ws is None else ws.numel(), _stream(stream)),
        "moe_grouped_swiglu_bwd_fp8")


def mxfp8_scale_bytes(cfg, which):
    return lib().moe_mxfp8_scale_bytes(ctypes.byref(cfg), which)


def moe_quantize_mxfp8(x, q, scales, stream=None):
    """MXFP8 codes (uint8, x's shape) and row-major block scales (uint8 [..., cols/32]) of the bf16
    tensor x along its last dimension."""
    cols = x.shape[-1]
    _check(lib().moe_quantize_mxfp8(_p(x), x.numel() // max(cols, 1), cols, _p(q), _p(scales),
                                    _stream(stream)), "moe_quantize_mxfp8")


def moe_mxfp8_pack_expert_scales(cfg, W1_s, W2_s, W1_sp, W2_sp, stream=None):
    _check(lib().moe_mxfp8_pack_expert_scales(ctypes.byref(cfg), _p(W1_s), _p(W2_s), _p(W1_sp),
                                              _p(W2_sp), _stream(stream)),
           "moe_mxfp8_pack_expert_scales")


def moe_permute_quantize_mxfp8(cfg, x, slot_of_pair, offsets, x_perm_q, x_perm_s, stream=None):
    _check(lib().moe_permute_quantize_mxfp8(ctypes.byref(cfg), _p(x), _p(slot_of_pair), _p(offsets),
                                            _p(x_perm_q), _p(x_perm_s), _stream(stream)),
           "moe_permute_quantize_mxfp8")


def moe_grouped_swiglu_fwd_mxfp8(cfg, x_perm_q, x_perm_s, offsets, W1_q, W1_sp, W2_q, W2_sp, h, act,
                                 h_q, h_s, y_perm, stream=None):
    _check(lib().moe_grouped_swiglu_fwd_mxfp8(
        ctypes.byref(cfg), _p(x_perm_q), _p(x_perm_s), _p(offsets), _p(W1_q), _p(W1_sp), _p(W2_q),
        _p(W2_sp), _p(h), _p(act), _p(h_q), _p(h_s), _p(y_perm), _stream(stream)),
        "moe_grouped_swiglu_fwd_mxfp8")


def alloc_mxfp8_experts(cfg, W1, W2, device="cuda", stream=None):
    """MXFP8 state of the routed experts (torch tensors): W1 and W2 quantised once along their
    reduction dimensions (codes, row-major scales and the packed scales the GEMMs read), and the
    buffers the MXFP8 stage calls write."""
    import torch
    E, d, f = cfg.E, cfg.d, cfg.f
    N = max(cfg.T, 1) * cfg.k
    u8 = torch.uint8
    m = dict(W1_q=torch.empty(E, 2 * f, d, dtype=u8, device=device),
             W1_s=torch.empty(E, 2 * f, d // 32, dtype=u8, device=device),
             W2_q=torch.empty(E, d, f, dtype=u8, device=device),
             W2_s=torch.empty(E, d, f // 32, dtype=u8, device=device),
             W1_sp=torch.empty(mxfp8_scale_bytes(cfg, MX_SCALES_W1), dtype=u8, device=device),
             W2_sp=torch.empty(mxfp8_scale_bytes(cfg, MX_SCALES_W2), dtype=u8, device=device),
             x_perm_q=torch.empty(N, d, dtype=u8, device=device),
             x_perm_s=torch.empty(mxfp8_scale_bytes(cfg, MX_SCALES_X), dtype=u8, device=device),
             h_q=torch.empty(N, f, dtype=u8, device=device),
             h_s=torch.empty(mxfp8_scale_bytes(cfg, MX_SCALES_H), dtype=u8, device=device))
    moe_quantize_mxfp8(W1, m["W1_q"], m["W1_s"], stream)
    moe_quantize_mxfp8(W2, m["W2_q"], m["W2_s"], stream)
    moe_mxfp8_pack_expert_scales(cfg, m["W1_s"], m["W2_s"], m["W1_sp"], m["W2_sp"], stream)
    return m


def mx_struct(m):
    return MoeMxfp8Experts(*[m[n].data_ptr() for n, _ in MoeMxfp8Experts._fields_])


def moe_layer_fwd_mxfp8(cfg, x, W_r, b_r, mx, Ws1, Ws2, w_sg, y, saved, ws, stream=None, side=None):
    st, ms = saved_struct(saved), mx_struct(mx)
    _check(lib().moe_layer_fwd_mxfp8(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), ctypes.byref(ms),
                                     _p(Ws1), _p(Ws2), _p(w_sg), _p(y), ctypes.byref(st), _p(ws),
                                     ws.numel(), _stream(stream), _side(side)), "moe_layer_fwd_mxfp8")


def alloc_mxfp8_dgrad(cfg, W1, W2, device="cuda", stream=None):
    """The data gradients' MXFP8 state (torch tensors): W1 and W2 quantised once in blocks down
    their rows (codes, plain and packed scales), and the buffers the MXFP8 backward writes."""
    import torch
    E, d, f = cfg.E, cfg.d, cfg.f
    N = max(cfg.T, 1) * cfg.k
    u8 = torch.uint8
    m = dict(W1c_q=torch.empty(E, 2 * f, d, dtype=u8, device=device),
             W1c_s=torch.empty(E, 2 * f // 32, d, dtype=u8, device=device),
             W1c_sp=torch.empty(mxfp8_scale_bytes(cfg, MX_SCALES_W1C), dtype=u8, device=device),
             W2c_q=torch.empty(E, d, f, dtype=u8, device=device),
             W2c_s=torch.empty(E, d // 32, f, dtype=u8, device=device),
             W2c_sp=torch.empty(mxfp8_scale_bytes(cfg, MX_SCALES_W2C), dtype=u8, device=device),
             dy_q=torch.empty(N, d, dtype=u8, device=device),
             dy_s=torch.empty(mxfp8_scale_bytes(cfg, MX_SCALES_X), dtype=u8, device=device),
             dH1_q=torch.empty(N, 2 * f, dtype=u8, device=device),
             dH1_s=torch.empty(mxfp8_scale_bytes(cfg, MX_SCALES_DH1), dtype=u8, device=device))
    _check(lib().moe_mxfp8_prepare_dgrad_weights(
        ctypes.byref(cfg), _p(W1), _p(W2), _p(m["W1c_q"]), _p(m["W1c_s"]), _p(m["W1c_sp"]),
        _p(m["W2c_q"]), _p(m["W2c_s"]), _p(m["W2c_sp"]), _stream(stream)),
        "moe_mxfp8_prepare_dgrad_weights")
    return m


def moe_grouped_swiglu_dgrad_mxfp8(cfg, dy_perm, offsets, act, mxd, dH1, dx_perm, stream=None):
    _check(lib().moe_grouped_swiglu_dgrad_mxfp8(
        ctypes.byref(cfg), _p(dy_perm), _p(offsets), _p(act), _p(mxd["W1c_q"]), _p(mxd["W1c_sp"]),
        _p(mxd["W2c_q"]), _p(mxd["W2c_sp"]), _p(mxd["dy_q"]), _p(mxd["dy_s"]), _p(dH1),
        _p(mxd["dH1_q"]), _p(mxd["dH1_s"]), _p(dx_perm), _stream(stream)),
        "moe_grouped_swiglu_dgrad_mxfp8")


def moe_mxfp8_quantize_tokens(cfg, x, offsets, q, s, cbase, stream=None):
    """Token-direction MXFP8 of x [N, C] inside the expert segments (see the header)."""
    _check(lib().moe_mxfp8_quantize_tokens(ctypes.byref(cfg), _p(x), int(x.shape[1]), _p(offsets),
                                           _p(q), _p(s), _p(cbase), _stream(stream)),
           "moe_mxfp8_quantize_tokens")


def moe_grouped_swiglu_wgrad_mxfp8(cfg, offsets, x_perm, h, dy_perm, dH1, dW1, dW2, ws,
                                   stream=None):
    _check(lib().moe_grouped_swiglu_wgrad_mxfp8(
        ctypes.byref(cfg), _p(offsets), _p(x_perm), _p(h), _p(dy_perm), _p(dH1), _p(dW1), _p(dW2),
        _p(ws), 0 if ws is None else ws.numel(), _stream(stream)), "moe_grouped_swiglu_wgrad_mxfp8")


def mxd_struct(m):
    """The struct of an mxfp8_dgrad_state dict; with m["wgrad_ws"] (a uint8 tensor of
    workspace_bytes(cfg, WS_WGRAD_MXFP8)) the weight gradients run in MXFP8 too."""
    ws = m.get("wgrad_ws")
    ptrs = [m[n].data_ptr() for n, _ in MoeMxfp8Dgrad._fields_[:8]]
    return MoeMxfp8Dgrad(*ptrs, None if ws is None else ws.data_ptr(),
                         0 if ws is None else ws.numel())


def moe_layer_bwd_mxfp8(cfg, dy, x, W_r, mxd, Ws1, Ws2, w_sg, saved, dx, dW_r, dW1, dW2, dWs1, dWs2,
                        dw_sg, ws, stream=None, side=None):
    st, ms = saved_struct(saved), mxd_struct(mxd)
    _check(lib().moe_layer_bwd_mxfp8(ctypes.byref(cfg), _p(dy), _p(x), _p(W_r), ctypes.byref(ms),
                                     _p(Ws1), _p(Ws2), _p(w_sg), ctypes.byref(st), _p(dx), _p(dW_r),
                                     _p(dW1), _p(dW2), _p(dWs1), _p(dWs2), _p(dw_sg), _p(ws),
                                     ws.numel(), _stream(stream), _side(side)), "moe_layer_bwd_mxfp8")


def moe_unpermute_combine(cfg, y_perm, gate, slot_of_pair, shared_out, shared_coef, y, stream=None):
    _check(lib().moe_unpermute_combine(ctypes.byref(cfg), _p(y_perm), _p(gate), _p(slot_of_pair),
                                       _p(shared_out), _p(shared_coef), _p(y), _stream(stream)),
           "moe_unpermute_combine")


def moe_unpermute_combine_bwd(cfg, dy, y_perm, gate, slot_of_pair, shared_out, shared_coef,
                              dy_perm, dgate, dshared, dcoef, stream=None):
    _check(lib().moe_unpermute_combine_bwd(ctypes.byref(cfg), _p(dy), _p(y_perm), _p(gate),
                                           _p(slot_of_pair), _p(shared_out), _p(shared_coef),
                                           _p(dy_perm), _p(dgate), _p(dshared), _p(dcoef),
                                           _stream(stream)), "moe_unpermute_combine_bwd")


def moe_router_aux_loss(cfg, logits, counts, aux_loss, ws, stream=None):
    _check(lib().moe_router_aux_loss(ctypes.byref(cfg), _p(logits), _p(counts), _p(aux_loss),
                                     _p(ws), 0 if ws is None else ws.numel(), _stream(stream)),
           "moe_router_aux_loss")


def moe_expert_bias_update(cfg, counts, e_bias, rate, stream=None):
    _check(lib().moe_expert_bias_update(ctypes.byref(cfg), _p(counts), _p(e_bias), float(rate),
                                        _stream(stream)), "moe_expert_bias_update")


# ----------------------------------------------------------------------------- whole layer

SAVED_FIELDS = [f for f, _ in MoeSaved._fields_]


def alloc_saved(cfg, device="cuda"):
    """Caller-owned buffers a forward pass leaves for the backward (torch tensors)."""
    import torch
    dt = torch.bfloat16 if cfg.dtype == DTYPE_BF16 else torch.float32
    T, d, E, k, f, fs = max(cfg.T, 1), cfg.d, cfg.E, cfg.k, cfg.f, cfg.f_shared
    N = T * k
    i32, f32 = torch.int32, torch.float32
    s = dict(
        logits=torch.empty(T, E, dtype=f32, device=device),
        idx=torch.empty(T, k, dtype=i32, device=device),
        gate=torch.empty(T, k, dtype=f32, device=device),
        counts=torch.empty(E, dtype=i32, device=device),
        offsets=torch.empty(E + 1, dtype=i32, device=device),
        slot_of_pair=torch.empty(T, k, dtype=i32, device=device),
        token_of_slot=torch.empty(max(N, 1), dtype=i32, device=device),
        x_perm=torch.empty(max(N, 1), d, dtype=dt, device=device),
        act=torch.empty(max(N, 1), 2 * f, dtype=dt, device=device),
        h=torch.empty(max(N, 1), f, dtype=dt, device=device),
        y_perm=torch.empty(max(N, 1), d, dtype=dt, device=device),
        s_act=torch.empty(T, 2 * fs, dtype=dt, device=device) if fs else None,
        s_h=torch.empty(T, fs, dtype=dt, device=device) if fs else None,
        s_out=torch.empty(T, d, dtype=dt, device=device) if fs else None,
        s_coef=torch.empty(T, dtype=f32, device=device) if cfg.shared_gate else None,
        aux_loss=torch.empty(4, dtype=f32, device=device) if cfg.aux_coeff > 0 else None,
    )
    return s


def saved_struct(saved):
    return MoeSaved(*[None if saved[n] is None else saved[n].data_ptr() for n in SAVED_FIELDS])


def moe_layer_fwd(cfg, x, W_r, b_r, W1, W2, Ws1, Ws2, w_sg, y, saved, ws, stream=None, side=None):
    st = saved_struct(saved)
    _check(lib().moe_layer_fwd(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), _p(W1), _p(W2), _p(Ws1),
                               _p(Ws2), _p(w_sg), _p(y), ctypes.byref(st), _p(ws), ws.numel(),
                               _stream(stream), _side(side)), "moe_layer_fwd")


def moe_layer_bwd(cfg, dy, x, W_r, W1, W2, Ws1, Ws2, w_sg, saved, dx, dW_r, dW1, dW2, dWs1, dWs2,
                  dw_sg, ws, stream=None, side=None):
    st = saved_struct(saved)
    _check(lib().moe_layer_bwd(ctypes.byref(cfg), _p(dy), _p(x), _p(W_r), _p(W1), _p(W2), _p(Ws1),
                               _p(Ws2), _p(w_sg), ctypes.byref(st), _p(dx), _p(dW_r), _p(dW1),
                               _p(dW2), _p(dWs1), _p(dWs2), _p(dw_sg), _p(ws), ws.numel(),
                               _stream(stream), _side(side)), "moe_layer_bwd")


def alloc_fp8_experts(cfg, W1, W2, device="cuda", stream=None, Ws1=None, Ws2=None):
    """FP8 state of the experts (torch tensors): W1 and W2 (and the shared expert's Ws1, Ws2 when
    given) quantised once to E4M3 with one scale per expert (FP8 parameters), and the buffers
    the FP8 layer calls write."""
    import torch
    E, d, f, fs = cfg.E, cfg.d, cfg.f, cfg.f_shared
    T = max(cfg.T, 1)
    N = T * cfg.k
    u8, f32 = torch.uint8, torch.float32
    q = dict(W1_q=torch.empty(E, 2 * f, d, dtype=u8, device=device),
             W1_scale=torch.empty(E, dtype=f32, device=device),
             W2_q=torch.empty(E, d, f, dtype=u8, device=device),
             W2_scale=torch.empty(E, dtype=f32, device=device),
             x_perm_q=torch.empty(N, d, dtype=u8, device=device),
             h_q=torch.empty(N, f, dtype=u8, device=device),
             scales=torch.zeros(16, dtype=f32, device=device))
    amax = torch.empty(max(E, 4), dtype=f32, device=device)
    moe_quantize_e4m3(W1, E, q["W1_q"], q["W1_scale"], amax, stream)
    moe_quantize_e4m3(W2, E, q["W2_q"], q["W2_scale"], amax, stream)
    if fs and Ws1 is not None:
        q.update(Ws1_q=torch.empty(2 * fs, d, dtype=u8, device=device),
                 Ws1_scale=torch.empty(4, dtype=f32, device=device),
                 Ws2_q=torch.empty(d, fs, dtype=u8, device=device),
                 Ws2_scale=torch.empty(4, dtype=f32, device=device),
                 x_q=torch.empty(T, d, dtype=u8, device=device),
                 s_h_q=torch.empty(T, fs, dtype=u8, device=device))
        moe_quantize_e4m3(Ws1, 1, q["Ws1_q"], q["Ws1_scale"], amax, stream)
        moe_quantize_e4m3(Ws2, 1, q["Ws2_q"], q["Ws2_scale"], amax, stream)
    return q


def fp8_struct(q):
    return MoeFp8Experts(*[None if q.get(n) is None else q[n].data_ptr()
                           for n, _ in MoeFp8Experts._fields_])


def moe_layer_fwd_fp8(cfg, x, W_r, b_r, fp8, Ws1, Ws2, w_sg, y, saved, ws, stream=None, side=None):
    st, qs = saved_struct(saved), fp8_struct(fp8)
    _check(lib().moe_layer_fwd_fp8(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), ctypes.byref(qs),
                                   _p(Ws1), _p(Ws2), _p(w_sg), _p(y), ctypes.byref(st), _p(ws),
                                   ws.numel(), _stream(stream), _side(side)), "moe_layer_fwd_fp8")


def moe_layer_bwd_fp8(cfg, dy, x, W_r, fp8, Ws1, Ws2, w_sg, saved, dx, dW_r, dW1, dW2, dWs1, dWs2,
                      dw_sg, ws, stream=None, side=None):
    st, qs = saved_struct(saved), fp8_struct(fp8)
    _check(lib().moe_layer_bwd_fp8(ctypes.byref(cfg), _p(dy), _p(x), _p(W_r), ctypes.byref(qs),
                                   _p(Ws1), _p(Ws2), _p(w_sg), ctypes.byref(st), _p(dx), _p(dW_r),
                                   _p(dW1), _p(dW2), _p(dWs1), _p(dWs2), _p(dw_sg), _p(ws),
                                   ws.numel(), _stream(stream), _side(side)), "moe_layer_bwd_fp8")


def moe_selftest_wait_timeout(observed, stream=None):
    """Run the bounded-wait self-test (see include/moe_gb300.h); observed: int32 device tensor."""
    _check(lib().moe_selftest_wait_timeout(_p(observed), _stream(stream)), "moe_selftest_wait_timeout")


def check_device_error(stream=None):
    code = ctypes.c_int32(0)
    _check(lib().moe_check_device_error(_stream(stream), ctypes.byref(code)), "device check")


def launch_count():
    return int(lib().moe_launch_count())


WAIT_FIELDS = ("producer_stage_wait", "mma_stage_wait", "mma_accumulator_wait",
               "epilogue_accumulator_wait", "cta_cycles", "kblocks", "ctas")


def gemm_wait_stats():
    """{kernel kind: {field: value}} of the GEMM pipeline wait counters since the last read
    (synchronises the device and clears them), or None when the library was built without
    MOE_WAIT_STATS=1."""
    buf = (ctypes.c_uint64 * (64 * 7))()
    n = lib().moe_gemm_wait_stats(buf, 64 * 7)
    if n == -2:   # MOE_ERR_UNSUPPORTED: built without the counters
        return None
    if n < 0:
        _check(n, "moe_gemm_wait_stats")
    out = {}
    for kind in range(n):
        v = [int(buf[7 * kind + i]) for i in range(7)]
        if v[6]:
            out[kind] = dict(zip(WAIT_FIELDS, v))
    return out


def trace_enable(on=True):
    lib().moe_trace_enable(1 if on else 0)


def trace_read(cap=64):
    """{kernel kind: (launches, total ms)} since the last read (synchronises the device)."""
    stride = 64
    names = ctypes.create_string_buffer(cap * stride)
    launches = (ctypes.c_int * cap)()
    ms = (ctypes.c_double * cap)()
    n = lib().moe_trace_read(names, stride, launches, ms, cap)
    if n < 0:
        _check(n, "moe_trace_read")
    out = {}
    for i in range(min(n, cap)):
        nm = names.raw[i * stride:(i + 1) * stride].split(b"\0", 1)[0].decode()
        out[nm] = (launches[i], ms[i])
    return out
