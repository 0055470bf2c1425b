"""Pins for the MXFP8 oracle (CPU only): the shared block exponent's closed forms, exact round
trips of blocks already on the E4M3 grid with their own power-of-two scales, the element codes
against PyTorch's float8_e4m3fn (a library implementation of E4M3) after the block's exact
power-of-two division, the elementwise error bound of the format, saturation, and the block-scaled
GEMMs against a library fp64 evaluation on exactly representable operands.  Planted mistakes
must fail a pin."""
import numpy as np
import pytest
import torch

import oracle.fp8_oracle as F8
import oracle.mxfp8_oracle as MX


def torch_encode(x32):
    t = torch.from_numpy(np.clip(np.asarray(x32, np.float32), -448, 448))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_shared_exponent_closed_forms():
    # floor(log2(amax)) - 8, by hand
    table = [(1.0, -8), (448.0, 0), (447.5, 0), (256.0, 0), (255.9, -1), (512.0, 1), (0.75, -9),
             (3.0e38, 119), (2.0 ** -130, -127), (0.0, -127), (2.0 ** -119, -127),
             (2.0 ** -118, -126), (1e-3, -18)]
    got = MX.shared_exponent(np.array([a for a, _ in table]))
    assert list(got) == [e for _, e in table]


def grid_blocks(rng, rows, K, shifts):
    """Rows of K values on the E4M3 grid times 2^shift per 32-block (shifts [rows, K/32]); every
    block's largest magnitude is an E4M3 value in [256, 448], so its shared exponent is exactly
    `shift` and quantisation is the identity."""
    c = rng.integers(0, 0x7E, size=(rows, K)) | (rng.integers(0, 2, size=(rows, K)) << 7)
    v = F8.e4m3_decode(c).reshape(rows, K // 32, 32)
    top = F8.e4m3_decode(rng.integers(0x78, 0x7F, size=(rows, K // 32)))   # 256 .. 448
    pos = rng.integers(0, 32, size=(rows, K // 32))
    np.put_along_axis(v, pos[..., None], top[..., None], axis=2)
    return np.ldexp(v, shifts[..., None]).reshape(rows, K)


def test_grid_blocks_round_trip_exactly():
    rng = np.random.default_rng(0)
    rows, K = 24, 128
    shifts = rng.integers(-20, 12, size=(rows, K // 32))
    x = grid_blocks(rng, rows, K, shifts)
    q, s = MX.mx_quantize(x)
    assert np.array_equal(s.astype(np.int64) - 127, shifts)
    assert np.array_equal(MX.mx_decode(q, s), x)


def test_codes_match_library_after_block_division():
    rng = np.random.default_rng(1)
    rows, K = 40, 256
    # bf16 values with a different magnitude per block, exact ties included
    x = rng.standard_normal((rows, K)) * np.repeat(10.0 ** rng.uniform(-6, 6, (rows, K // 32)), 32, 1)
    x = F8.bf16_round(x)
    q, s = MX.mx_quantize(x)
    e = s.astype(np.int64) - 127
    scaled = np.ldexp(x.reshape(rows, K // 32, 32), -e[..., None]).reshape(rows, K)
    assert np.array_equal(q, torch_encode(scaled.astype(np.float32)))
    amax = np.abs(x.reshape(rows, K // 32, 32)).max(-1)
    assert ((amax >= 2.0 ** (e + 8)) & (amax < 2.0 ** (e + 9))).all()


def test_error_bound_and_saturation():
    rng = np.random.default_rng(2)
    rows, K = 64, 96
    x = rng.standard_normal((rows, K)) * np.repeat(2.0 ** rng.integers(-30, 30, (rows, K // 32)), 32, 1)
    q, s = MX.mx_quantize(x)
    dec = MX.mx_decode(q, s)
    e = np.repeat(s.astype(np.int64) - 127, 32, 1)
    a = np.abs(x) * 2.0 ** -e                       # magnitude inside the block's E4M3 range
    normal = (a >= 2.0 ** -6) & (a <= 448)
    err = np.abs(dec - x)
    # half a step of a 3-bit mantissa; half the subnormal step 2^-9 below the normal range
    assert (err[normal] <= np.ldexp(1.0, np.floor(np.log2(np.abs(x[normal]))).astype(int) - 4)).all()
    assert (err[~normal & (a < 448)] <= np.ldexp(1.0, e[~normal & (a < 448)] - 10)).all()
    over = a > 448
    assert (np.abs(dec[over]) == 448 * 2.0 ** e[over]).all()
    # a block whose largest magnitude is 480 keeps exponent 0 and clamps it to 448
    blk = np.zeros((1, 32))
    blk[0, 3], blk[0, 7] = 480.0, -1.0
    qb, sb = MX.mx_quantize(blk)
    assert sb[0, 0] == 127 and qb[0, 3] == 0x7E and qb[0, 7] == 0xB8
    # all-zero block: exponent -127, zero codes
    qz, sz = MX.mx_quantize(np.zeros((2, 64)))
    assert (sz == 0).all() and (qz == 0).all()


def test_block_scaled_swiglu_equals_library_on_representable_operands():
    """Operands on the grid with a distinct power-of-two scale per block: quantisation is exact,
    so fc1 + SwiGLU and fc2 must equal torch's fp64 products of the unquantised operands."""
    rng = np.random.default_rng(3)
    E, f, d, N = 3, 64, 96, 20
    offsets = np.array([0, 7, 7, 20])
    x = grid_blocks(rng, N, d, rng.integers(-6, 2, size=(N, d // 32)))
    W1 = np.stack([grid_blocks(rng, 2 * f, d, rng.integers(-12, -6, size=(2 * f, d // 32)))
                   for _ in range(E)])
    W2 = np.stack([grid_blocks(rng, d, f, rng.integers(-12, -6, size=(d, f // 32)))
                   for _ in range(E)])
    xq, xs = MX.mx_quantize(x)
    W1q, W1s = MX.mx_quantize(W1)
    W2q, W2s = MX.mx_quantize(W2)
    h, act = MX.fc1_swiglu_mx(xq, xs, W1q, W1s, offsets)
    hq, hs = MX.mx_quantize(F8.bf16_round(h))
    y = MX.fc2_mx(hq, hs, W2q, W2s, offsets)
    X = torch.from_numpy(x)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            assert not h[lo:hi].any()
            continue
        au = X[lo:hi] @ torch.from_numpy(W1[e]).T
        ref_h = (torch.nn.functional.silu(au[:, :f]) * au[:, f:]).numpy()
        assert np.abs(h[lo:hi] - ref_h).max() <= 1e-12 * np.abs(ref_h).max()
        assert np.abs(act[lo:hi] - au.numpy()).max() <= 1e-12 * np.abs(au.numpy()).max()
        Hd = torch.from_numpy(MX.mx_decode(hq, hs)[lo:hi])
        assert np.allclose(y[lo:hi], (Hd @ torch.from_numpy(W2[e]).T).numpy(), rtol=1e-12, atol=0)


def grid_cols(rng, R, C, shifts):
    """An R x C matrix on the E4M3 grid with a power-of-two scale per 32-row block and column
    (shifts [R/32, C]): its column blocks quantise exactly, with exponents `shifts`."""
    return np.swapaxes(grid_blocks(rng, C, R, shifts.T), 0, 1)


def test_column_blocks_round_trip_and_their_scales():
    rng = np.random.default_rng(4)
    R, C = 96, 40
    shifts = rng.integers(-9, 9, size=(R // 32, C))
    x = grid_cols(rng, R, C, shifts)
    q, s = MX.mx_quantize_cols(x)
    assert s.shape == (R // 32, C)
    assert np.array_equal(s.astype(np.int64) - 127, shifts)
    assert np.array_equal(MX.mx_decode_cols(q, s), x)
    # one block by hand: rows 32..63 of column 5 scaled by 2^3 carry exponent 3
    y = np.zeros((64, 8))
    y[40, 5], y[33, 5] = 448.0 * 8, -3.0
    qy, sy = MX.mx_quantize_cols(y)
    # -3 / 2^3 = -0.375 = -1.5 * 2^-2: sign, exponent field 5, mantissa 4 -> 0xAC
    assert sy[1, 5] == 130 and sy[0, 5] == 0 and qy[40, 5] == 0x7E and qy[33, 5] == 0xAC


def test_block_scaled_data_gradients_equal_library_on_representable_operands():
    """dy and [da | du] on the grid in row blocks, W2 and W1 on the grid in column blocks, each
    block with its own power of two: quantisation is exact, so fc2's and fc1's data gradients
    must equal torch's fp64 products of the unquantised operands."""
    rng = np.random.default_rng(5)
    E, f, d, N = 3, 64, 96, 20
    offsets = np.array([0, 9, 9, 20])
    dy = grid_blocks(rng, N, d, rng.integers(-8, 0, size=(N, d // 32)))
    dH = grid_blocks(rng, N, 2 * f, rng.integers(-8, 0, size=(N, 2 * f // 32)))
    W2 = np.stack([grid_cols(rng, d, f, rng.integers(-12, -4, size=(d // 32, f))) for _ in range(E)])
    W1 = np.stack([grid_cols(rng, 2 * f, d, rng.integers(-12, -4, size=(2 * f // 32, d)))
                   for _ in range(E)])
    dyq, dys = MX.mx_quantize(dy)
    dHq, dHs = MX.mx_quantize(dH)
    W2q, W2s = MX.mx_quantize_cols(W2)
    W1q, W1s = MX.mx_quantize_cols(W1)
    dh = MX.fc2_dgrad_mx(dyq, dys, W2q, W2s, offsets)
    dx = MX.fc1_dgrad_mx(dHq, dHs, W1q, W1s, offsets)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        ref_dh = (torch.from_numpy(dy[lo:hi]) @ torch.from_numpy(W2[e])).numpy()
        ref_dx = (torch.from_numpy(dH[lo:hi]) @ torch.from_numpy(W1[e])).numpy()
        assert np.allclose(dh[lo:hi], ref_dh, rtol=1e-12, atol=0)
        assert np.allclose(dx[lo:hi], ref_dx, rtol=1e-12, atol=0)
    assert not dh[9:9].any()


def _pins_pass():
    try:
        test_shared_exponent_closed_forms()
        test_grid_blocks_round_trip_exactly()
        test_codes_match_library_after_block_division()
        test_error_bound_and_saturation()
        test_block_scaled_swiglu_equals_library_on_representable_operands()
        test_column_blocks_round_trip_and_their_scales()
        test_block_scaled_data_gradients_equal_library_on_representable_operands()
    except AssertionError:
        return False
    return True


def _quantize_first_half_amax(x, block=32):
    """A block's exponent from its first 16 elements only (a half-block mistake)."""
    x64 = np.asarray(x, np.float64)
    K = x64.shape[-1]
    b = x64.reshape(x64.shape[:-1] + (K // block, block))
    e = MX.shared_exponent(np.abs(b[..., :16]).max(-1))
    q = F8.e4m3_encode(np.ldexp(b, -e[..., None]).astype(np.float32)).reshape(x64.shape)
    return q, (e + 127).astype(np.uint8)


def _decode_blocks_reversed(codes, scales, block=32):
    """Scales applied to the blocks in reverse order (an index mistake)."""
    return _mx_decode(codes, np.asarray(scales)[..., ::-1], block)


_mx_decode = MX.mx_decode
_shared_exponent = MX.shared_exponent


def _exponent_ceil(amax):
    """ceil(log2(amax)) - 8 (rounding the exponent up: differs from floor except at powers of 2)."""
    a = np.asarray(amax, np.float64)
    m, p = np.frexp(a)
    ce = np.where(m == 0.5, p - 1, p)
    return np.clip(np.where(a > 0, ce - 8, -127), -127, 127).astype(np.int64)


_mx_quantize_cols = MX.mx_quantize_cols
_mx_decode_cols = MX.mx_decode_cols

MUTANTS = {
    "exponent_ceil": ("shared_exponent", lambda a: _exponent_ceil(a)),
    "emax_7": ("shared_exponent", lambda a: np.maximum(_shared_exponent(a) + 1, -127)),
    "exponent_off_low": ("shared_exponent", lambda a: np.maximum(_shared_exponent(a) - 1, -127)),
    "half_block_amax": ("mx_quantize", _quantize_first_half_amax),
    "scales_reversed": ("mx_decode", _decode_blocks_reversed),
    "scale_not_applied": ("mx_decode", lambda c, s, block=32: F8.e4m3_decode(np.asarray(c))),
    # column blocks: each block decoded with its neighbour's scales; exponents one too large
    "column_scales_rolled": ("mx_decode_cols", lambda c, s, block=32: _mx_decode_cols(
        c, np.roll(np.asarray(s), 1, axis=-2), block)),
    "column_exponent_plus_one": ("mx_quantize_cols", lambda x, block=32: (
        _mx_quantize_cols(x, block)[0], (_mx_quantize_cols(x, block)[1] + 1).astype(np.uint8))),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mxfp8_mistakes_are_caught(name, monkeypatch):
    assert _pins_pass()
    attr, repl = MUTANTS[name]
    monkeypatch.setattr(MX, attr, repl)
    assert not _pins_pass(), f"mutant {name} survived every pin"
