"""Stage entry points (moe_permute, moe_grouped_swiglu_fwd/bwd, moe_unpermute_combine(_bwd))
against the oracle's definitions on the same inputs."""
import numpy as np
import pytest
import torch

import moe_expert_layer_gemm_gb300 as moe
import oracle.moe_oracle as O

from .helpers import assert_close, np64

pytestmark = pytest.mark.gpu


def routed(T, E, k, seed=0):
    g = torch.Generator().manual_seed(seed)
    lg = torch.randn(T, E, generator=g)
    r = O.route(lg.numpy(), k, E, O.SOFTMAX, 1)
    return r


@pytest.mark.parametrize("dtype", [moe.DTYPE_BF16, moe.DTYPE_F32])
def test_permute_is_exact_copy(dtype):
    T, d, E, k = 1000, 264, 16, 4
    r = routed(T, E, k)
    cfg = moe.make_cfg(T, d, E, k, 64, dtype=dtype)
    tdt = torch.bfloat16 if dtype == moe.DTYPE_BF16 else torch.float32
    x = torch.randn(T, d).to(tdt).cuda()
    xp = torch.full((T * k, d), float("nan"), dtype=tdt, device="cuda")
    moe.moe_permute(cfg, x, torch.from_numpy(r["slot_of_pair"]).cuda(), xp)
    torch.cuda.synchronize()
    ref = x.cpu()[torch.from_numpy(r["token_of_slot"]).long()]
    assert torch.equal(xp.cpu(), ref)


def test_grouped_swiglu_fwd_bwd_stage():
    T, d, E, k, f = 600, 256, 8, 2, 136
    r = routed(T, E, k, 3)
    N = T * k
    cfg = moe.make_cfg(T, d, E, k, f)
    g = torch.Generator().manual_seed(5)
    xp = torch.randn(N, d, generator=g).bfloat16()
    W1 = (torch.randn(E, 2 * f, d, generator=g) * 0.05).bfloat16()
    W2 = (torch.randn(E, d, f, generator=g) * 0.05).bfloat16()
    dyp = torch.randn(N, d, generator=g).bfloat16()
    off = torch.from_numpy(r["offsets"])
    c = {n: t.cuda() for n, t in dict(xp=xp, W1=W1, W2=W2, dyp=dyp, off=off).items()}
    h = torch.empty(N, f, dtype=torch.bfloat16, device="cuda")
    act = torch.empty(N, 2 * f, dtype=torch.bfloat16, device="cuda")
    yp = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_swiglu_fwd(cfg, c["xp"], c["off"], c["W1"], c["W2"], h, act, yp)
    dxp = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    dW1 = torch.empty(E, 2 * f, d, device="cuda")
    dW2 = torch.empty(E, d, f, device="cuda")
    ws = moe.workspace(cfg, moe.WS_FFN_BWD)
    moe.moe_grouped_swiglu_bwd(cfg, c["xp"], c["off"], c["W1"], c["W2"], act, h, c["dyp"], dxp, dW1,
                               dW2, ws)
    torch.cuda.synchronize()
    moe.check_device_error()
    X, dY = np64(xp), np64(dyp)
    ref_y = np.zeros((N, d))
    ref_dx = np.zeros((N, d))
    o = r["offsets"]
    for e in range(E):
        sl = slice(o[e], o[e + 1])
        y_e, a, u, hh = O.swiglu_ffn(np64(W1[e]), np64(W2[e]), X[sl])
        ref_y[sl] = y_e
        dX, dW1e, dW2e = O.swiglu_ffn_backward(np64(W1[e]), np64(W2[e]), X[sl], a, u, hh, dY[sl])
        ref_dx[sl] = dX
        assert_close(f"dW1[{e}]", np64(dW1[e]), dW1e, 2e-2)
        assert_close(f"dW2[{e}]", np64(dW2[e]), dW2e, 2e-2)
    assert_close("y_perm", np64(yp), ref_y, 2e-2)
    assert_close("dx_perm", np64(dxp), ref_dx, 2e-2)


def test_tall_tiles_on_ragged_groups():
    """fc2 and fc1's data gradient on 256-row tiles: with 8192 rows and d = 2048 the library takes
    them (two waves of 256 x 256 tiles against four of 128 x 256 on a GPU of about 150 SMs).  The
    groups' sizes cover the tall tile's cases: empty groups, a single row, tails of at most 128
    rows (only the first half's MMAs), tails of 129 and 200 rows (a partial second half), whole
    tiles of 256 and 512 rows, a 255-row group and one large group.  Every output row is written
    (the buffers start as NaN) and matches the oracle's per-expert products."""
    E, d, f = 16, 2048, 128
    sizes = [0, 1, 100, 128, 129, 200, 256, 300, 385, 512, 640, 0, 1000, 1, 255]
    sizes.append(8192 - sum(sizes))
    N = sum(sizes)
    off_np = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    cfg = moe.make_cfg(N, d, E, 1, f)
    g = torch.Generator().manual_seed(21)
    xp = torch.randn(N, d, generator=g).bfloat16()
    W1 = (torch.randn(E, 2 * f, d, generator=g) * 0.03).bfloat16()
    W2 = (torch.randn(E, d, f, generator=g) * 0.05).bfloat16()
    dyp = torch.randn(N, d, generator=g).bfloat16()
    c = {n: t.cuda() for n, t in dict(xp=xp, W1=W1, W2=W2, dyp=dyp,
                                       off=torch.from_numpy(off_np)).items()}
    nan = float("nan")
    h = torch.full((N, f), nan, dtype=torch.bfloat16, device="cuda")
    act = torch.full((N, 2 * f), nan, dtype=torch.bfloat16, device="cuda")
    yp = torch.full((N, d), nan, dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_swiglu_fwd(cfg, c["xp"], c["off"], c["W1"], c["W2"], h, act, yp)
    dxp = torch.full((N, d), nan, dtype=torch.bfloat16, device="cuda")
    dW1 = torch.empty(E, 2 * f, d, device="cuda")
    dW2 = torch.empty(E, d, f, device="cuda")
    ws = moe.workspace(cfg, moe.WS_FFN_BWD)
    moe.moe_grouped_swiglu_bwd(cfg, c["xp"], c["off"], c["W1"], c["W2"], act, h, c["dyp"], dxp, dW1,
                               dW2, ws)
    torch.cuda.synchronize()
    moe.check_device_error()
    assert not torch.isnan(yp).any() and not torch.isnan(dxp).any()
    X, dY = np64(xp), np64(dyp)
    ref_y = np.zeros((N, d))
    ref_dx = np.zeros((N, d))
    for e in range(E):
        sl = slice(off_np[e], off_np[e + 1])
        if sizes[e] == 0:
            continue
        y_e, a, u, hh = O.swiglu_ffn(np64(W1[e]), np64(W2[e]), X[sl])
        ref_y[sl] = y_e
        ref_dx[sl] = O.swiglu_ffn_backward(np64(W1[e]), np64(W2[e]), X[sl], a, u, hh, dY[sl])[0]
    assert_close("y_perm", np64(yp), ref_y, 2e-2)
    assert_close("dx_perm", np64(dxp), ref_dx, 2e-2)


@pytest.mark.parametrize("shared", [0, 1, 2])
def test_combine_and_backward(shared):
    T, d, E, k = 500, 136, 12, 3
    r = routed(T, E, k, 7)
    N = T * k
    cfg = moe.make_cfg(T, d, E, k, 64)
    g = torch.Generator().manual_seed(9)
    yp = torch.randn(N, d, generator=g).bfloat16()
    gate = torch.from_numpy(r["gate"]).float()
    so = torch.randn(T, d, generator=g).bfloat16() if shared else None
    coef = torch.rand(T, generator=g) if shared == 2 else None
    dy = torch.randn(T, d, generator=g).bfloat16()
    sop = torch.from_numpy(r["slot_of_pair"])
    cu = lambda t: None if t is None else t.cuda()
    y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.moe_unpermute_combine(cfg, cu(yp), cu(gate), cu(sop), cu(so), cu(coef), y)
    dyp = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    dg = torch.empty(T, k, device="cuda")
    dso = torch.empty(T, d, dtype=torch.bfloat16, device="cuda") if shared else None
    dc = torch.empty(T, device="cuda") if shared == 2 else None
    moe.moe_unpermute_combine_bwd(cfg, cu(dy), cu(yp), cu(gate), cu(sop), cu(so), cu(coef), dyp, dg,
                                  dso, dc)
    torch.cuda.synchronize()
    Y, G, SOP, DY = np64(yp), r["gate"], r["slot_of_pair"], np64(dy)
    c = np64(coef) if shared == 2 else np.ones(T)
    ref = np.einsum("tj,tjd->td", G, Y[SOP])
    if shared:
        ref = ref + c[:, None] * np64(so)
    assert_close("y", np64(y), ref, 1e-2)
    ref_dyp = np.zeros((N, d))
    ref_dyp[SOP] = G[:, :, None] * DY[:, None, :]
    assert_close("dy_perm", np64(dyp), ref_dyp, 1e-2)
    assert_close("dgate", np64(dg), np.einsum("td,tjd->tj", DY, Y[SOP]), 1e-3)
    if shared:
        assert_close("dshared", np64(dso), c[:, None] * DY, 1e-2)
    if shared == 2:
        assert_close("dcoef", np64(dc), (DY * np64(so)).sum(1), 1e-3)


@pytest.mark.parametrize("T,d,E,k,f", [(600, 256, 8, 2, 136), (1000, 384, 32, 6, 200),
                                       (77, 128, 4, 3, 64)])
def test_gathered_stages_equal_permute_then_stage(T, d, E, k, f):
    """The permutation folded into the operand loads (rows of x gathered by token_of_slot):
    bit-identical to moe_permute followed by the x_perm stage calls, and within the bf16
    tolerance of the oracle."""
    r = routed(T, E, k, 11)
    N = T * k
    cfg = moe.make_cfg(T, d, E, k, f)
    g = torch.Generator().manual_seed(13)
    x = torch.randn(T, d, generator=g).bfloat16().cuda()
    W1 = (torch.randn(E, 2 * f, d, generator=g) * 0.05).bfloat16().cuda()
    W2 = (torch.randn(E, d, f, generator=g) * 0.05).bfloat16().cuda()
    dyp = torch.randn(N, d, generator=g).bfloat16().cuda()
    off = torch.from_numpy(r["offsets"]).cuda()
    sop = torch.from_numpy(r["slot_of_pair"]).cuda()
    tos = torch.from_numpy(r["token_of_slot"]).cuda()
    bf = torch.bfloat16

    def run(gathered):
        h = torch.empty(N, f, dtype=bf, device="cuda")
        act = torch.empty(N, 2 * f, dtype=bf, device="cuda")
        yp = torch.empty(N, d, dtype=bf, device="cuda")
        dxp = torch.empty(N, d, dtype=bf, device="cuda")
        dW1 = torch.empty(E, 2 * f, d, device="cuda")
        dW2 = torch.empty(E, d, f, device="cuda")
        ws = moe.workspace(cfg, moe.WS_FFN_BWD)
        if gathered:
            moe.moe_grouped_swiglu_fwd_gathered(cfg, x, tos, off, W1, W2, h, act, yp)
            moe.moe_grouped_swiglu_bwd_gathered(cfg, x, tos, off, W1, W2, act, h, dyp, dxp, dW1,
                                                dW2, ws)
        else:
            xp = torch.empty(N, d, dtype=bf, device="cuda")
            moe.moe_permute(cfg, x, sop, xp)
            moe.moe_grouped_swiglu_fwd(cfg, xp, off, W1, W2, h, act, yp)
            moe.moe_grouped_swiglu_bwd(cfg, xp, off, W1, W2, act, h, dyp, dxp, dW1, dW2, ws)
        torch.cuda.synchronize()
        moe.check_device_error()
        return dict(h=h, act=act, yp=yp, dxp=dxp, dW1=dW1, dW2=dW2)

    a, b = run(True), run(False)
    for n in a:
        assert torch.equal(a[n], b[n]), n
    X = np64(x)[r["token_of_slot"]]
    o = r["offsets"]
    ref_y = np.zeros((N, d))
    for e in range(E):
        sl = slice(o[e], o[e + 1])
        ref_y[sl] = O.swiglu_ffn(np64(W1[e]), np64(W2[e]), X[sl])[0]
    assert_close("y_perm", np64(a["yp"]), ref_y, 2e-2)
