"""The C-ABI library without a GPU: it loads, exports every function include/moe_gb300.h
declares, and rejects bad arguments on the host with the documented status codes before any
CUDA work is enqueued."""
import ctypes
import os

import pytest

import moe_expert_layer_gemm_gb300 as moe

L = None


def setup_module():
    global L
    if not os.path.exists(moe._lib.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    L = moe.lib()


def test_exports_every_declared_function():
    names = moe.header_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), n
    assert L.moe_version() >= 100


def cfg(**kw):
    base = dict(T=256, d=128, E=8, k=2, f=256, f_shared=0, score_fn=0, renorm=1, shared_gate=0,
                dtype=0, bias_mode=0, aux_coeff=0.0)
    base.update(kw)
    return moe.MoeCfg(*[base[n] for n, _ in moe.MoeCfg._fields_])


P = ctypes.c_void_p(1 << 20)     # a fake, aligned, never-dereferenced address
MIS = ctypes.c_void_p((1 << 20) + 8)


@pytest.mark.parametrize("bad,code", [
    (dict(k=9), -2),                               # k above the maximum
    (dict(k=3, E=2), -1),                          # k > E
    (dict(E=300), -2),                             # too many experts
    (dict(d=100), -2),                             # d not a multiple of 8 (bf16 rows)
    (dict(T=-1), -1),
    (dict(score_fn=3), -1),
    (dict(shared_gate=1), -1),                     # gate without a shared expert
    (dict(dtype=7), -1),
    (dict(bias_mode=2), -1),
    (dict(aux_coeff=-1e-4), -1),
    (dict(aux_coeff=float("nan")), -1),
    (dict(aux_coeff=float("inf")), -1),
])
def test_bad_config_is_rejected(bad, code):
    c = cfg(**bad)
    assert L.moe_permute(ctypes.byref(c), P, P, P, None) == code
    assert L.moe_workspace_bytes(ctypes.byref(c), 4) == 0
    assert L.moe_last_error()


def test_null_and_misaligned_pointers():
    c = cfg()
    assert L.moe_permute(ctypes.byref(c), None, P, P, None) == -1
    assert b"x" in L.moe_last_error()
    assert L.moe_permute(ctypes.byref(c), MIS, P, P, None) == -4
    assert L.moe_unpermute_combine(ctypes.byref(c), P, P, P, None, None, None, None) == -1


def test_workspace_too_small():
    c = cfg()
    need = L.moe_workspace_bytes(ctypes.byref(c), moe.WS_ROUTE)
    assert need > 0
    rc = L.moe_route_topk(ctypes.byref(c), P, P, None, None, None, P, P, P, P, P, P, P, need - 256,
                          None)
    assert rc == -3


def test_workspace_sizes_grow_with_the_layer():
    small = cfg(T=256)
    big = cfg(T=4096)
    for w in (moe.WS_ROUTE, moe.WS_LAYER_BWD, moe.WS_FFN_BWD):
        assert L.moe_workspace_bytes(ctypes.byref(big), w) > L.moe_workspace_bytes(ctypes.byref(small), w)


def test_side_stream_arguments_are_checked_on_the_host():
    """moe_side_stream (the caller's second stream for the layer calls): every field required,
    fork and join distinct, the side stream not the call's own stream.  Rejected before any
    launch; NULL (no side stream) passes this check and fails later on the missing buffers."""
    c = cfg(f_shared=128)
    ws = 1 << 30
    a, b, e1, e2 = (ctypes.c_void_p((1 << 20) * i) for i in (3, 4, 5, 6))
    bad = [moe.MoeSideStream(None, e1, e2), moe.MoeSideStream(b, None, e2),
           moe.MoeSideStream(b, e1, None), moe.MoeSideStream(b, e1, e1),
           moe.MoeSideStream(a, e1, e2)]                 # a is also the call's stream below
    args_f = [P] * 9
    for sd in bad:
        assert L.moe_layer_fwd(ctypes.byref(c), *args_f, None, P, ws, a, ctypes.byref(sd)) == -1
        assert b"side" in L.moe_last_error()
        assert L.moe_layer_bwd(ctypes.byref(c), *([P] * 8), None, *([P] * 7), P, ws, a,
                               ctypes.byref(sd)) == -1
        assert b"side" in L.moe_last_error()
    good = moe.MoeSideStream(b, e1, e2)
    # a good side stream gets past its check: the NULL saved struct is what fails
    assert L.moe_layer_fwd(ctypes.byref(c), *args_f, None, P, ws, a, ctypes.byref(good)) == -1
    assert b"saved" in L.moe_last_error()
    assert L.moe_layer_fwd(ctypes.byref(c), *args_f, None, P, ws, a, None) == -1
    assert b"saved" in L.moe_last_error()


def test_router_variant_entry_points_check_arguments():
    c = cfg(aux_coeff=1e-4)
    ws_n = L.moe_workspace_bytes(ctypes.byref(c), 0)
    assert ws_n > 0
    # balancing loss: needs a coefficient, logits, counts, an output and the routing workspace
    c0 = cfg()
    assert L.moe_router_aux_loss(ctypes.byref(c0), P, P, P, P, ws_n, None) == -1
    assert L.moe_router_aux_loss(ctypes.byref(c), None, P, P, P, ws_n, None) == -1
    assert L.moe_router_aux_loss(ctypes.byref(c), P, P, MIS, P, ws_n, None) == -4
    assert L.moe_router_aux_loss(ctypes.byref(c), P, P, P, P, ws_n - 1, None) == -3
    # bias update: counts and bias required, finite rate
    assert L.moe_expert_bias_update(ctypes.byref(c), None, P, ctypes.c_float(1e-3), None) == -1
    assert L.moe_expert_bias_update(ctypes.byref(c), P, None, ctypes.c_float(1e-3), None) == -1
    assert L.moe_expert_bias_update(ctypes.byref(c), P, P, ctypes.c_float(float("nan")), None) == -1
    assert L.moe_last_error()


def test_mxfp8_entry_points_check_arguments():
    """MXFP8 calls reject, on the host and before any launch: d or f not a multiple of 32 (the
    block), an fp32 layer, a row length not a multiple of 32, missing or misaligned buffers."""
    c = cfg(d=256, f=160)
    for which in range(4):
        assert L.moe_mxfp8_scale_bytes(ctypes.byref(c), which) > 0
    assert L.moe_mxfp8_scale_bytes(ctypes.byref(c), 10) == 0
    assert L.moe_mxfp8_scale_bytes(ctypes.byref(cfg(k=9)), moe.MX_SCALES_X) == 0
    # packed sizes: activations per 128-row tile and 128-element chunk, weights per 192-row tile
    N, E = 256 * 2, 8
    assert L.moe_mxfp8_scale_bytes(ctypes.byref(c), moe.MX_SCALES_X) == ((N + 127 * E) // 128 + 1) * 2 * 512
    assert L.moe_mxfp8_scale_bytes(ctypes.byref(c), moe.MX_SCALES_W1) == E * 2 * 2 * 1024
    assert L.moe_mxfp8_scale_bytes(ctypes.byref(c), moe.MX_SCALES_W2) == E * 2 * 2 * 1024
    assert L.moe_quantize_mxfp8(P, 4, 48, P, P, None) == -2          # 48 is not a multiple of 32
    assert L.moe_quantize_mxfp8(P, -1, 64, P, P, None) == -1
    assert L.moe_quantize_mxfp8(P, 4, 64, MIS, P, None) == -4
    bad_f = cfg(d=256, f=144)
    assert L.moe_permute_quantize_mxfp8(ctypes.byref(bad_f), P, P, P, P, P, None) == -2
    assert L.moe_permute_quantize_mxfp8(ctypes.byref(cfg(dtype=1)), P, P, P, P, P, None) == -2
    assert L.moe_permute_quantize_mxfp8(ctypes.byref(c), P, P, None, P, P, None) == -1
    assert L.moe_mxfp8_pack_expert_scales(ctypes.byref(c), P, P, P, MIS, None) == -4
    args = [P] * 13
    assert L.moe_grouped_swiglu_fwd_mxfp8(ctypes.byref(bad_f), *args) == -2
    args[3] = None                                                     # W1_q
    assert L.moe_grouped_swiglu_fwd_mxfp8(ctypes.byref(c), *args) == -1
    assert b"W1_q" in L.moe_last_error()
    assert L.moe_layer_fwd_mxfp8(ctypes.byref(c), P, P, None, None, None, None, None, P, None, P,
                                 1 << 30, None, None) == -1
    # the weight gradients' token-chunk layouts: ceil(C/128) column tiles x (N/128 + E) chunks
    for which, C in ((moe.MX_SCALES_TOK_D, 256), (moe.MX_SCALES_TOK_F, 160),
                     (moe.MX_SCALES_TOK_2F, 320)):
        assert L.moe_mxfp8_scale_bytes(ctypes.byref(c), which) == -(-C // 128) * (N // 128 + E) * 512
    assert L.moe_mxfp8_quantize_tokens(ctypes.byref(c), P, 48, P, P, P, P, None) == -2
    assert L.moe_mxfp8_quantize_tokens(ctypes.byref(c), P, 64, None, P, P, P, None) == -1
    assert L.moe_mxfp8_quantize_tokens(ctypes.byref(bad_f), P, 64, P, P, P, P, None) == -2
    ws_need = L.moe_workspace_bytes(ctypes.byref(c), moe.WS_WGRAD_MXFP8)
    assert ws_need >= N * (2 * 256 + 3 * 160)
    assert L.moe_grouped_swiglu_wgrad_mxfp8(ctypes.byref(c), P, P, P, P, P, P, P, P, ws_need - 1,
                                            None) == -3
    assert L.moe_grouped_swiglu_wgrad_mxfp8(ctypes.byref(c), P, P, None, P, P, P, P, P, ws_need,
                                            None) == -1
    assert b"h" in L.moe_last_error()


def test_wait_stats_need_their_build_option():
    """The default library has no pipeline wait counters: the entry point says so on the host
    (no device call) and the binding reads that as None."""
    import ctypes
    buf = (ctypes.c_uint64 * 448)()
    assert moe.lib().moe_gemm_wait_stats(buf, 448) == -2
    assert b"MOE_WAIT_STATS" in moe.lib().moe_last_error()
    assert moe.gemm_wait_stats() is None


def test_binding_argument_counts_match_the_header():
    """Every ctypes signature of the binding takes as many arguments as the header declares."""
    import re
    hdr = open(moe._lib.HEADER).read()
    decls = {m.group(1): m.group(2) for m in re.finditer(
        r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(([^;]*?)\);", hdr, re.M | re.S)}
    for name, (_, args) in moe._lib._SIGS.items():
        assert name in decls, name
        params = [p for p in (q.strip() for q in decls[name].split(",")) if p and p != "void"]
        assert len(params) == len(args), (name, len(params), len(args))


C_CLIENT = r"""
#include <stdio.h>
#include "moe_gb300.h"
int main(void) {
  moe_cfg c = {256, 128, 8, 2, 256, 0, MOE_SCORE_SOFTMAX, 1, 0, MOE_DTYPE_BF16, MOE_BIAS_LOGIT,
               0.0f};
  size_t ws = moe_workspace_bytes(&c, MOE_WS_LAYER_BWD);
  int rc = moe_route_topk(NULL, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0);
  printf("%d %zu %d %s\n", moe_version(), ws, rc, moe_last_error());
  return (ws > 0 && rc == MOE_ERR_INVALID_ARG) ? 0 : 1;
}
"""


def test_plain_c_client_builds_against_the_header_and_links(tmp_path):
    """The header is strict C11 and the library links into a plain C program (no C++, no Python),
    which sizes a workspace and gets a host-side argument error back."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(moe._lib.LIB_PATH)
    exe = tmp_path / "client"
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I" + os.path.join(root, "include"), str(src), "-L" + libdir,
                        "-lmoe_gb300", "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, LD_LIBRARY_PATH=libdir)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, (r.stdout, r.stderr)
    assert "cfg is NULL" in r.stdout
