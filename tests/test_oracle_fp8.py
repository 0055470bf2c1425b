"""Pins for the FP8 oracle (CPU only): the E4M3 codec against PyTorch's float8_e4m3fn (a
library implementation of the same format), exact round trips, the tensorwise scale's closed
forms, and the quantised GEMM against a library fp64 evaluation on operands that are exactly
representable (so quantisation is the identity up to an exact power-of-two scale).  Planted
mistakes must fail a pin."""
import numpy as np
import pytest
import torch

import oracle.fp8_oracle as F8


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def torch_encode(x32):
    t = torch.from_numpy(np.clip(np.asarray(x32, np.float32), -448, 448))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_codes_matches_library():
    codes = np.arange(256)
    a, b = F8.e4m3_decode(codes), torch_decode(codes)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    ok = ~np.isnan(a)
    assert np.array_equal(a[ok], b[ok])
    assert np.nanmax(a) == 448.0 and F8.e4m3_decode(0x01) == 2.0 ** -9


def test_encode_matches_library_on_values_ties_and_extremes():
    vals = F8.e4m3_decode(np.arange(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2                      # exact ties between neighbours
    rng = np.random.default_rng(0)
    xs = [vals, -vals, mids, -mids, np.array([0.0, -0.0, 448.0, 449.0, 464.0, 1e9, -1e9, 2.0 ** -10,
                                              -(2.0 ** -10), 2.0 ** -11])]
    for sc in [1e-3, 0.1, 1.0, 30.0, 500.0]:
        xs.append(rng.standard_normal(4000) * sc)
    x = np.concatenate(xs).astype(np.float32)
    assert np.array_equal(F8.e4m3_encode(x), torch_encode(x))


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(F8.e4m3_encode(F8.e4m3_decode(codes).astype(np.float32)), codes)


def test_tensorwise_scale_closed_forms():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 48)).astype(np.float32)
    q, s = F8.quantize_tensorwise(x)
    i = np.unravel_index(np.abs(x).argmax(), x.shape)
    assert q[i] in (0x7E, 0xFE)                              # amax maps onto +-448
    assert s[0] == np.float32(np.abs(x).max()) / np.float32(448)
    q2, s2 = F8.quantize_tensorwise(x * 4)                   # powers of two scale exactly
    assert np.array_equal(q2, q) and s2[0] == 4 * s[0]
    qz, sz = F8.quantize_tensorwise(np.zeros((3, 5)))
    assert (qz == 0).all() and sz[0] == 1.0
    # per-group blocks are independent tensors
    W = np.stack([x, 8 * x])
    qg, sg = F8.quantize_tensorwise(W, groups=2)
    assert np.array_equal(qg[0], q) and np.array_equal(qg[1], q) and sg[1] == 8 * sg[0]


def representable(rng, shape, amax_code=0x7E):
    """Random E4M3-representable values whose largest magnitude is decode(amax_code)."""
    c = rng.integers(0, 0x7E, size=shape)
    c = c | (rng.integers(0, 2, size=shape) << 7)
    v = F8.e4m3_decode(c)
    v.flat[0] = F8.e4m3_decode(amax_code)
    return v


@pytest.mark.parametrize("shift", [0, 3])
def test_quantised_swiglu_equals_library_on_representable_operands(shift):
    """With operands already on the E4M3 grid and amax = 448 * 2^-shift, the scale is exactly
    2^-shift and quantisation is exact: fc1 + SwiGLU and fc2 must equal torch's fp64 result."""
    rng = np.random.default_rng(2 + shift)
    E, f, d, N = 3, 8, 16, 20
    offsets = np.array([0, 7, 7, 20])
    k = 2.0 ** -shift
    x = representable(rng, (N, d)) * k
    W1 = np.stack([representable(rng, (2 * f, d)) * k for _ in range(E)])
    W2 = np.stack([representable(rng, (d, f)) * k for _ in range(E)])
    xq, sx = F8.quantize_tensorwise(x)
    W1q, s1 = F8.quantize_tensorwise(W1, E)
    W2q, s2 = F8.quantize_tensorwise(W2, E)
    assert sx[0] == k and (s1 == k).all()
    h, act = F8.fc1_swiglu_fp8(xq, sx, W1q, s1, offsets)
    hq, sh = F8.quantize_tensorwise(h.astype(np.float32))
    y = F8.fc2_fp8(hq, sh, W2q, s2, offsets)
    X = torch.from_numpy(x)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        au = X[lo:hi] @ torch.from_numpy(W1[e]).T
        ref_h = torch.nn.functional.silu(au[:, :f]) * au[:, f:]
        ref = ref_h.numpy()
        assert np.abs(h[lo:hi] - ref).max() <= 1e-12 * np.abs(ref).max()
        Hd = torch.from_numpy(F8.dequantize(hq, sh)[lo:hi])
        assert np.allclose(y[lo:hi], (Hd @ torch.from_numpy(W2[e]).T).numpy(), rtol=1e-12, atol=0)


def _pins_pass():
    try:
        test_decode_all_codes_matches_library()
        test_encode_matches_library_on_values_ties_and_extremes()
        test_round_trip_of_every_finite_code()
        test_tensorwise_scale_closed_forms()
        for s in (0, 3):
            test_quantised_swiglu_equals_library_on_representable_operands(s)
    except AssertionError:
        return False
    return True


def _encode_ties_away(x32):
    x = np.asarray(x32, np.float32).astype(np.float64)
    codes = np.arange(0x7F)
    vals = F8.e4m3_decode(codes)
    a = np.minimum(np.abs(x), 448.0)
    idx = np.abs(a[:, None] - vals[None, :])
    best = np.argmin(idx[:, ::-1], axis=1)
    mag = codes[::-1][best]
    return (mag | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


MUTANTS = {
    "ties_away_from_even": ("e4m3_encode", _encode_ties_away),
    "exponent_bias_8": ("e4m3_decode", lambda c, _d=F8.e4m3_decode: _d(c) / 2),
    "scale_not_applied": ("dequantize", lambda c, s, g=1: F8.e4m3_decode(np.asarray(c))),
    "scale_inverted": ("quantize_tensorwise", lambda x, g=1, _q=F8.quantize_tensorwise: (
        _q(x, g)[0], (1.0 / _q(x, g)[1]).astype(np.float32))),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_fp8_mistakes_are_caught(name, monkeypatch):
    assert _pins_pass()
    attr, repl = MUTANTS[name]
    monkeypatch.setattr(F8, attr, repl)
    assert not _pins_pass(), f"mutant {name} survived every pin"


# ----------------------------------------------------------------------------- backward pins

import oracle.moe_oracle as MO  # noqa: E402

# E4M3 rounding of a normal value is within 2^-4 of it (3 mantissa bits, half a step); a value in
# the subnormal range is within half the subnormal step, 2^-10, times the tensor's scale.  bf16
# rounding adds 2^-9 relative.
REL_Q = 2.0 ** -4 + 2.0 ** -9
ABS_SUB = 2.0 ** -10


def _bwd_case(seed, E=3, f=8, d=16, N=20, offsets=(0, 7, 7, 20)):
    """Operands on the E4M3 grid with a distinct power-of-two scale per tensor (and per expert
    for the weights), so that every quantisation is exact and a mixed-up scale shows."""
    rng = np.random.default_rng(seed)
    offsets = np.array(offsets)
    x = representable(rng, (N, d)) * 2.0 ** -2
    h = representable(rng, (N, f)) * 2.0 ** -5
    dy = representable(rng, (N, d)) * 2.0 ** -9
    W1 = np.stack([representable(rng, (2 * f, d)) * 2.0 ** -(3 + e) for e in range(E)])
    W2 = np.stack([representable(rng, (d, f)) * 2.0 ** -(6 + e) for e in range(E)])
    act = F8.bf16_round(rng.standard_normal((N, 2 * f)) * 2)
    xq, sx = F8.quantize_tensorwise(x)
    hq, sh = F8.quantize_tensorwise(h)
    W1q, s1 = F8.quantize_tensorwise(W1, E)
    W2q, s2 = F8.quantize_tensorwise(W2, E)
    assert sx[0] == 2.0 ** -2 and sh[0] == 2.0 ** -5
    assert list(s1) == [2.0 ** -(3 + e) for e in range(E)]
    return dict(offsets=offsets, x=x, h=h, dy=dy, W1=W1, W2=W2, act=act, xq=xq, sx=sx, hq=hq,
                sh=sh, W1q=W1q, s1=s1, W2q=W2q, s2=s2)


def _bwd_pins(seed):
    c = _bwd_case(seed)
    r = F8.grouped_swiglu_bwd_fp8(c["xq"], c["sx"], c["W1q"], c["s1"], c["W2q"], c["s2"], c["act"],
                                  c["hq"], c["sh"], c["dy"], c["offsets"])
    assert r["dy_scale"][0] == 2.0 ** -9
    f = c["h"].shape[1]
    off = c["offsets"]
    for e in range(len(off) - 1):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            assert not r["dW1"][e].any() and not r["dW2"][e].any()
            continue
        a, u = c["act"][lo:hi, :f], c["act"][lo:hi, f:]
        dX, dW1e, dW2e = MO.swiglu_ffn_backward(c["W1"][e], c["W2"][e], c["x"][lo:hi], a, u,
                                                c["h"][lo:hi], c["dy"][lo:hi])
        # exact operands: dW2 and dh carry no quantisation error
        assert np.allclose(r["dW2"][e], dW2e, rtol=1e-12, atol=0)
        dh_ref = c["dy"][lo:hi] @ c["W2"][e]
        assert np.allclose(r["dh"][lo:hi], dh_ref, rtol=1e-12, atol=0)
        dH1_ref = np.concatenate([dh_ref * u * MO.silu_grad(a), dh_ref * MO.silu(a)], axis=1)
        # dx, dW1 see dH1's bf16 and E4M3 rounding only: elementwise bounds from the error of each
        # dH1 value, propagated through |.| of the exact other operand
        sub = ABS_SUB * float(r["dH1_scale"][0])
        W1a, Xa = np.abs(c["W1"][e]), np.abs(c["x"][lo:hi])
        bound_dx = REL_Q * (np.abs(dH1_ref) @ W1a) + sub * W1a.sum(axis=0) + 1e-12
        assert (np.abs(r["dx"][lo:hi] - dX) <= bound_dx).all()
        bound_dw1 = REL_Q * (np.abs(dH1_ref).T @ Xa) + sub * Xa.sum(axis=0)[None, :] + 1e-12
        assert (np.abs(r["dW1"][e] - dW1e) <= bound_dw1).all()
        # and the error is not trivially zero-bounded: the result moved by less than 10% overall
        assert np.abs(r["dx"][lo:hi] - dX).max() <= 0.1 * np.abs(dX).max()


@pytest.mark.parametrize("seed", [5, 6])
def test_fp8_backward_against_exact_fp64_backward(seed):
    _bwd_pins(seed)


def _brute_wgrad(Aq, sa, Bq, sb, offsets):
    """dW[e][i][j] = sum over rows r of expert e of dec(A[r][i])*sa * dec(B[r][j])*sb, by loops."""
    table = {c: float(F8.e4m3_decode(c)) for c in range(256)}
    E = len(offsets) - 1
    m, n = Aq.shape[1], Bq.shape[1]
    out = [[[0.0] * n for _ in range(m)] for _ in range(E)]
    for e in range(E):
        for r in range(int(offsets[e]), int(offsets[e + 1])):
            for i in range(m):
                av = table[int(Aq[r][i])] * float(sa[0])
                for j in range(n):
                    out[e][i][j] += av * table[int(Bq[r][j])] * float(sb[0])
    return np.array(out)


def _brute_dgrad(Gq, sg, Wq, sw, offsets):
    """out[r][j] = sum_i dec(G[r][i])*sg * dec(W[e][i][j])*sw[e] for rows r of expert e, by loops."""
    table = {c: float(F8.e4m3_decode(c)) for c in range(256)}
    n = Wq.shape[2]
    out = [[0.0] * n for _ in range(Gq.shape[0])]
    for e in range(len(offsets) - 1):
        for r in range(int(offsets[e]), int(offsets[e + 1])):
            for j in range(n):
                acc = 0.0
                for i in range(Gq.shape[1]):
                    acc += table[int(Gq[r][i])] * float(sg[0]) * table[int(Wq[e][i][j])] * float(sw[e])
                out[r][j] = acc
    return np.array(out)


def test_fp8_backward_products_against_brute_force():
    rng = np.random.default_rng(9)
    E, N, m, n = 3, 9, 5, 6
    offsets = np.array([0, 4, 4, 9])
    Aq = rng.integers(0, 256, size=(N, m)).astype(np.uint8)
    Bq = rng.integers(0, 256, size=(N, n)).astype(np.uint8)
    Aq[(Aq & 0x7F) == 0x7F] = 0x11                      # no NaN codes
    Bq[(Bq & 0x7F) == 0x7F] = 0x22
    sa, sb = np.array([0.37], np.float32), np.array([1.9], np.float32)
    assert np.allclose(F8.wgrad_fp8(Aq, sa, Bq, sb, offsets), _brute_wgrad(Aq, sa, Bq, sb, offsets),
                       rtol=1e-12, atol=1e-300)
    Wq = rng.integers(0, 256, size=(E, m, n)).astype(np.uint8)
    Wq[(Wq & 0x7F) == 0x7F] = 0x33
    sw = np.array([0.5, 3.0, 0.01], np.float32)
    # fc2's data gradient ([d] . [d, f]) and fc1's ([2f] . [2f, d]) are the same row product
    ref = _brute_dgrad(Aq, sa, Wq, sw, offsets)
    assert np.allclose(F8.fc2_dgrad_fp8(Aq, sa, Wq, sw, offsets), ref, rtol=1e-12, atol=1e-300)
    assert np.allclose(F8.fc1_dgrad_fp8(Aq, sa, Wq, sw, offsets), ref, rtol=1e-12, atol=1e-300)


def _bwd_pins_pass():
    try:
        for s in (5, 6):
            _bwd_pins(s)
        test_fp8_backward_products_against_brute_force()
    except AssertionError:
        return False
    return True


BWD_MUTANTS = {
    "swiglu_bwd_no_u": ("swiglu_backward", lambda dh, act: np.concatenate(
        [dh * MO.silu_grad(np.asarray(act)[:, :dh.shape[1]]),
         dh * MO.silu(np.asarray(act)[:, :dh.shape[1]])], axis=1)),
    "swiglu_bwd_silu_for_grad": ("swiglu_backward", lambda dh, act: np.concatenate(
        [dh * np.asarray(act)[:, dh.shape[1]:] * MO.silu(np.asarray(act)[:, :dh.shape[1]]),
         dh * MO.silu(np.asarray(act)[:, :dh.shape[1]])], axis=1)),
    "wgrad_scale_squared": ("wgrad_fp8", lambda Aq, sa, Bq, sb, off, _w=F8.wgrad_fp8: _w(Aq, sa, Bq, sa, off)),
    "dgrad_first_expert_scale": ("fc1_dgrad_fp8", lambda G, sg, Wq, sw, off, _d=F8.fc1_dgrad_fp8: _d(
        G, sg, Wq, np.full_like(sw, sw[0]), off)),
    "fc2_dgrad_wrong_weight_row": ("fc2_dgrad_fp8", lambda D, sd, Wq, sw, off, _d=F8.fc2_dgrad_fp8: _d(
        D, sd, np.ascontiguousarray(Wq[:, ::-1, :]), sw, off)),
    "wgrad_rows_of_next_expert": ("wgrad_fp8", lambda Aq, sa, Bq, sb, off, _w=F8.wgrad_fp8: _w(
        Aq, sa, Bq, sb, np.concatenate([off[:1], off[1:] + 1]).clip(max=off[-1]))),
}


@pytest.mark.parametrize("name", list(BWD_MUTANTS))
def test_fp8_backward_mistakes_are_caught(name, monkeypatch):
    assert _bwd_pins_pass()
    attr, repl = BWD_MUTANTS[name]
    monkeypatch.setattr(F8, attr, repl)
    assert not _bwd_pins_pass(), f"mutant {name} survived every pin"
