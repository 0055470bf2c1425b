"""Pins for the MXFP8 weight-gradient oracle (CPU only): token-direction blocks inside each expert
segment.  A hand-worked three-row segment; a segment boundary whose blocks differ from blocks
counted from row 0; agreement with the column-block quantiser on segments of whole blocks; exact
round trips of segments already on the grid; and the weight-gradient products against a library
fp64 evaluation on exactly representable operands.  Planted mistakes must fail a pin."""
import numpy as np
import pytest
import torch

import oracle.fp8_oracle as F8
import oracle.mxfp8_oracle as MX

from .test_oracle_mxfp8 import grid_cols


def test_three_row_segment_by_hand():
    """Column 0 = [1, 2, 3]: amax 3, exponent floor(log2 3) - 8 = -7 (byte 120); the scaled
    values 128, 256, 384 are E4M3 1.0 * 2^7, 1.0 * 2^8 and 1.5 * 2^8: codes 0x70, 0x78, 0x7C.
    Column 1 = [0.5, -0.25, 0]: exponent -1 - 8 = -9 (byte 118); 256, -128, 0: 0x78, 0xF0, 0x00.
    The block's missing 29 rows are zeros and store nothing."""
    x = np.array([[1.0, 0.5], [2.0, -0.25], [3.0, 0.0]])
    q, s = MX.mx_quantize_segments(x, [0, 3])
    assert q.tolist() == [[0x70, 0x78], [0x78, 0xF0], [0x7C, 0x00]]
    assert len(s) == 1 and s[0].tolist() == [[120, 118]]
    assert np.array_equal(MX.mx_decode_segments(q, s, [0, 3]), x)


def test_blocks_restart_at_every_segment():
    """Experts of 20 and 40 rows in one column: expert 0 holds 0.01s, expert 1 starts with twelve
    100s.  Counted from each segment's first row, expert 0's only block has amax 0.01 (exponent
    floor(log2 0.01) - 8 = -15, byte 112) and expert 1's blocks cover its rows 0-31 (amax 100:
    6 - 8 = -2, byte 125) and 32-39 (amax 1: -8, byte 119).  Blocks counted from row 0 would put
    expert 0's rows beside expert 1's 100s."""
    x = np.zeros((60, 1))
    x[:20] = 0.01
    x[20:32] = 100.0
    x[32:] = 1.0
    q, s = MX.mx_quantize_segments(x, [0, 20, 60])
    assert [b.ravel().tolist() for b in s] == [[112], [125, 119]]
    # 0.01 / 2^-15 = 327.68 rounds to the E4M3 value 320 (step 32 between 256 and 512)
    assert np.allclose(MX.mx_decode_segments(q, s, [0, 20, 60])[:20], 320 * 2.0 ** -15, rtol=0)
    # an empty segment has no blocks
    q2, s2 = MX.mx_quantize_segments(x, [0, 20, 20, 60])
    assert s2[1].shape == (0, 1) and np.array_equal(q2, q)


def test_whole_block_segments_equal_the_column_quantiser():
    rng = np.random.default_rng(11)
    x = F8.bf16_round(rng.standard_normal((160, 24)) * 3.0)
    offsets = [0, 64, 64, 160]
    q, s = MX.mx_quantize_segments(x, offsets)
    for e in range(3):
        lo, hi = offsets[e], offsets[e + 1]
        qc, sc = MX.mx_quantize_cols(x[lo:hi])
        assert np.array_equal(q[lo:hi], qc) and np.array_equal(s[e], sc)


def grid_segments(rng, offsets, C, lo_shift, hi_shift):
    """Rows on the E4M3 grid, each segment's 32-row blocks (counted from its first row) with their
    own power-of-two scale per column; a short last block is drawn whole and cut, and keeps its
    amax row inside the segment.  Quantisation is then exact."""
    N = int(offsets[-1])
    x = np.zeros((N, C))
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        n = hi - lo
        if n == 0:
            continue
        nb = -(-n // 32)
        blk = grid_cols(rng, nb * 32, C, rng.integers(lo_shift, hi_shift, size=(nb, C)))
        # move each block's largest magnitude into the segment (row 0 of the block)
        b = blk.reshape(nb, 32, C)
        top = np.abs(b).argmax(axis=1)
        for i in range(nb):
            for c in range(C):
                r = top[i, c]
                b[i, 0, c], b[i, r, c] = b[i, r, c], b[i, 0, c]
        x[lo:hi] = b.reshape(nb * 32, C)[:n]
    return x


def test_grid_segments_round_trip_exactly():
    rng = np.random.default_rng(12)
    offsets = np.array([0, 5, 5, 70, 133])
    x = grid_segments(rng, offsets, 40, -10, 6)
    q, s = MX.mx_quantize_segments(x, offsets)
    assert np.array_equal(MX.mx_decode_segments(q, s, offsets), x)
    assert [b.shape[0] for b in s] == [1, 0, 3, 2]


def test_weight_gradients_equal_library_on_representable_operands():
    """dW1[e] = dH1_e^T x_e and dW2[e] = dy_e^T h_e with every operand on the grid: the block-scaled
    products must equal torch's fp64 products of the unquantised operands."""
    rng = np.random.default_rng(13)
    d, f = 64, 32
    offsets = np.array([0, 33, 33, 40, 101])
    E = len(offsets) - 1
    x = grid_segments(rng, offsets, d, -4, 2)
    h = grid_segments(rng, offsets, f, -6, 0)
    dy = grid_segments(rng, offsets, d, -8, -2)
    dH = grid_segments(rng, offsets, 2 * f, -8, -2)
    xq, xs = MX.mx_quantize_segments(x, offsets)
    hq, hs = MX.mx_quantize_segments(h, offsets)
    dyq, dys = MX.mx_quantize_segments(dy, offsets)
    dHq, dHs = MX.mx_quantize_segments(dH, offsets)
    dW1 = MX.wgrad_mx(dHq, dHs, xq, xs, offsets)
    dW2 = MX.wgrad_mx(dyq, dys, hq, hs, offsets)
    assert dW1.shape == (E, 2 * f, d) and dW2.shape == (E, d, f)
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        r1 = (torch.from_numpy(dH[lo:hi]).T @ torch.from_numpy(x[lo:hi])).numpy()
        r2 = (torch.from_numpy(dy[lo:hi]).T @ torch.from_numpy(h[lo:hi])).numpy()
        assert np.allclose(dW1[e], r1, rtol=1e-12, atol=0)
        assert np.allclose(dW2[e], r2, rtol=1e-12, atol=0)
    assert not dW1[1].any() and not dW2[1].any()


def _pins_pass():
    try:
        test_three_row_segment_by_hand()
        test_blocks_restart_at_every_segment()
        test_whole_block_segments_equal_the_column_quantiser()
        test_grid_segments_round_trip_exactly()
        test_weight_gradients_equal_library_on_representable_operands()
    except (AssertionError, ValueError, IndexError):
        return False
    return True


_quantize_segments = MX.mx_quantize_segments
_decode_segments = MX.mx_decode_segments
_wgrad = MX.wgrad_mx


def _blocks_from_row_zero(x, offsets, block=32):
    """Blocks counted from row 0 of the whole tensor (across segment boundaries), cut per segment."""
    x64 = np.asarray(x, np.float64)
    N, C = x64.shape
    nb = -(-N // block)
    padded = np.zeros((nb * block, C))
    padded[:N] = x64
    q, s = MX.mx_quantize_cols(padded, block)
    scales = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        n = hi - lo
        scales.append(np.stack([s[min((lo + 32 * i) // 32, nb - 1)] for i in range(-(-n // 32))])
                      if n else np.zeros((0, C), np.uint8))
    return q[:N], scales


def _short_block_padded_with_neighbours(x, offsets, block=32):
    """A segment's short last block filled with the next rows of the tensor, not zeros."""
    x64 = np.asarray(x, np.float64)
    codes = np.zeros(x64.shape, np.uint8)
    scales = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        n = hi - lo
        nb = -(-n // block)
        padded = np.zeros((nb * block, x64.shape[1]))
        take = x64[lo:lo + nb * block]
        padded[:len(take)] = take
        q, s = MX.mx_quantize_cols(padded, block)
        codes[lo:hi] = q[:n]
        scales.append(s)
    return codes, scales


MUTANTS = {
    "blocks_from_row_zero": ("mx_quantize_segments", _blocks_from_row_zero),
    "short_block_takes_next_rows": ("mx_quantize_segments", _short_block_padded_with_neighbours),
    # each block of a segment decoded with the previous block's scales (an index mistake)
    "scales_rolled_within_segment": ("mx_decode_segments", lambda c, s, o, block=32: _decode_segments(
        c, [np.roll(b, 1, axis=0) for b in s], o, block)),
    "exponent_plus_one": ("mx_quantize_segments", lambda x, o, block=32: (
        _quantize_segments(x, o, block)[0],
        [(b.astype(np.int64) + 1).astype(np.uint8) for b in _quantize_segments(x, o, block)[1]])),
    "wgrad_operands_swapped": ("wgrad_mx", lambda aq, a_s, bq, b_s, o: _wgrad(bq, b_s, aq, a_s, o)),
    # the last expert's gradient dropped
    "wgrad_last_expert_dropped": ("wgrad_mx", lambda aq, a_s, bq, b_s, o: _wgrad(
        aq, a_s, bq, b_s, o) * np.array([1.0] * (len(o) - 2) + [0.0])[:, None, None]),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mxfp8_wgrad_mistakes_are_caught(name, monkeypatch):
    assert _pins_pass()
    attr, repl = MUTANTS[name]
    monkeypatch.setattr(MX, attr, repl)
    assert not _pins_pass(), f"mutant {name} survived every pin"
