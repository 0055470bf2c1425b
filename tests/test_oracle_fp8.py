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
