"""Oracle for the MXFP8 (microscaling FP8) expert GEMMs: block quantisation and the grouped
SwiGLU forward on block-scaled operands (fp64 CPU).

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU leg may import this
module; it imports nothing of the CUDA library and shares no code with it.

What the pages fix ("Megatron-Bridge 深度剖析", §新硬件适配): Blackwell brings a microscaling
FP8 whose scale factors are finer grained than FP8's per-tensor ones (and an FP4 beside it).
The pages stop there; the format is the Open Compute Project's Microscaling (MX) one, whose
MXFP8 variant pairs E4M3 elements with one shared E8M0 (power-of-two) scale per block.
Readings where the pages are silent:
  * a block is 32 consecutive elements along the product's reduction dimension K (d for fc1,
    f for fc2), so every row of an operand has K/32 scales;
  * the shared exponent of a block is floor(log2(amax)) - 8, where 8 is the exponent of E4M3's
    largest normal (448 = 1.75 * 2^8) and amax the block's largest magnitude; it is clamped to
    [-127, 127] and amax = 0 gives -127; the stored E8M0 byte is exponent + 127;
  * an element's code is E4M3(x / 2^e), round to nearest even; magnitudes in [448, 512) * 2^e
    saturate to 448 (the MX rule of clamping to the element format's largest normal);
  * the GEMM multiplies decoded values (code value times its block's scale) and accumulates;
    h is quantised again, in blocks of 32 along f, before fc2, from its bf16 value;
  * each expert's weights are quantised along their own K: W1 [2f, d] in blocks along d, W2
    [d, f] in blocks along f.
"""
from __future__ import annotations

import numpy as np

from .fp8_oracle import bf16_round, e4m3_decode, e4m3_encode  # noqa: F401 (bf16_round: re-export)
from .moe_oracle import silu

BLOCK = 32
E4M3_EMAX = 8          # exponent of the largest normal E4M3 value, 448 = 1.75 * 2^8
SCALE_BIAS = 127       # E8M0: the byte is the exponent plus 127


def shared_exponent(amax):
    """Shared block exponent floor(log2(amax)) - 8, clamped to [-127, 127]; -127 for amax = 0.
    floor(log2(.)) is read off frexp (exact): amax = m * 2^p with m in [0.5, 1) -> p - 1."""
    a = np.asarray(amax, dtype=np.float64)
    _, p = np.frexp(a)
    e = np.where(a > 0, (p.astype(np.int64) - 1) - E4M3_EMAX, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def mx_quantize(x, block=BLOCK):
    """MXFP8 codes of x along its last axis (whose length must be a multiple of `block`).
    Returns (codes uint8 with x's shape, scale bytes uint8 [..., K / block])."""
    x64 = np.asarray(x, dtype=np.float64)
    K = x64.shape[-1]
    if K % block:
        raise ValueError("the blocked axis must be a multiple of the block size")
    blocks = x64.reshape(x64.shape[:-1] + (K // block, block))
    amax = np.abs(blocks).max(axis=-1)
    e = shared_exponent(amax)
    # x / 2^e is exact in fp64; as fp32 it is exact too for the magnitudes that can round to a
    # nonzero E4M3 value (2^e * 2^-10 and up), which is all e4m3_encode looks at
    scaled = np.ldexp(blocks, -e[..., None]).astype(np.float32)
    codes = e4m3_encode(scaled).reshape(x64.shape)
    return codes, (e + SCALE_BIAS).astype(np.uint8)


def mx_decode(codes, scales, block=BLOCK):
    """Decoded values: each code's E4M3 value times 2^(its block's byte - 127) (fp64)."""
    c = np.asarray(codes)
    s = np.asarray(scales, dtype=np.int64)
    K = c.shape[-1]
    v = e4m3_decode(c).reshape(c.shape[:-1] + (K // block, block))
    v = np.ldexp(v, (s - SCALE_BIAS)[..., None])
    return v.reshape(c.shape)


def fc1_swiglu_mx(xq, xs, W1q, W1s, offsets):
    """fc1 + SwiGLU of every expert on MXFP8 operands: for the rows s of expert e,
    [a | u] = dec(xq[s], xs[s]) . dec(W1q[e], W1s[e])^T and h = SiLU(a) * u.  fp64.
    Returns (h [N, f], act = [a | u] [N, 2f])."""
    E = W1q.shape[0]
    f = W1q.shape[1] // 2
    X = mx_decode(xq, xs)
    N = X.shape[0]
    h = np.zeros((N, f))
    act = np.zeros((N, 2 * f))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        au = X[lo:hi] @ mx_decode(W1q[e], W1s[e]).T
        act[lo:hi] = au
        h[lo:hi] = silu(au[:, :f]) * au[:, f:]
    return h, act


def fc2_mx(hq, hs, W2q, W2s, offsets):
    """fc2 of every expert on MXFP8 operands: y[s] = dec(hq[s], hs[s]) . dec(W2q[e], W2s[e])^T
    for the rows s of expert e.  fp64."""
    E = W2q.shape[0]
    H = mx_decode(hq, hs)
    y = np.zeros((H.shape[0], W2q.shape[1]))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            y[lo:hi] = H[lo:hi] @ mx_decode(W2q[e], W2s[e]).T
    return y



# ----------------------------------------------------------------------------- data gradients
# Readings (the pages fix none of it): the data gradients run on MXFP8 operands with blocks along
# each product's own reduction dimension -- dy_perm [N, d] in row blocks along d for fc2's data
# gradient, [da | du] [N, 2f] in row blocks along 2f for fc1's; the weights in blocks along their
# first (K) dimension: W2 [d, f] in 32-row blocks along d, W1 [2f, d] in 32-row blocks along 2f
# (the "columnwise" copies; the forward's copies block the other dimension).  [da | du] is
# quantised from its bf16 value.  The weight gradients stay out of this (they reduce over tokens).

def mx_quantize_cols(x, block=BLOCK):
    """MXFP8 codes of x in blocks of 32 consecutive rows (along axis -2), one scale per block and
    column.  Returns (codes with x's shape, scale bytes [..., R / block, C])."""
    x64 = np.asarray(x, dtype=np.float64)
    q, s = mx_quantize(np.swapaxes(x64, -1, -2), block)
    return np.ascontiguousarray(np.swapaxes(q, -1, -2)), np.ascontiguousarray(np.swapaxes(s, -1, -2))


def mx_decode_cols(codes, scales, block=BLOCK):
    """Decoded values of row-blocked codes: code value times 2^(its block's byte - 127)."""
    v = mx_decode(np.swapaxes(np.asarray(codes), -1, -2), np.swapaxes(np.asarray(scales), -1, -2),
                  block)
    return np.swapaxes(v, -1, -2)


def fc2_dgrad_mx(dyq, dys, W2cq, W2cs, offsets):
    """dh[s] = dec(dyq[s], dys[s]) . decc(W2cq[e], W2cs[e]) for the rows s of expert e: [N, f]."""
    E, d, f = W2cq.shape
    DY = mx_decode(dyq, dys)
    dh = np.zeros((DY.shape[0], f))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            dh[lo:hi] = DY[lo:hi] @ mx_decode_cols(W2cq[e], W2cs[e])
    return dh


def fc1_dgrad_mx(dHq, dHs, W1cq, W1cs, offsets):
    """dx_perm[s] = dec(dHq[s], dHs[s]) . decc(W1cq[e], W1cs[e]) for the rows s of expert e: [N, d]."""
    E, two_f, d = W1cq.shape
    DH = mx_decode(dHq, dHs)
    dx = np.zeros((DH.shape[0], d))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            dx[lo:hi] = DH[lo:hi] @ mx_decode_cols(W1cq[e], W1cs[e])
    return dx


# ----------------------------------------------------------------------------- weight gradients
# The weight gradients reduce over each expert's tokens (dW1[e] = dH1_e^T . x_e, [2f, d];
# dW2[e] = dy_e^T . h_e, [d, f]), so the reduction dimension of their MXFP8 operands is the token
# one.  Readings (the pages fix none of it, §FP8 训练 names fp8_wgrad and §新硬件适配 MXFP8):
#   * inside expert e's rows [offsets[e], offsets[e+1]) every column is cut into blocks of 32
#     consecutive rows counted from the segment's first row; a block never holds rows of two
#     experts, and a segment's last block may be short;
#   * a short block's missing rows count as zeros (they leave its amax unchanged and no code is
#     stored for them);
#   * each block's exponent and codes follow the rules above (the same as the forward's blocks);
#     all four operands are quantised from their bf16 values.

def mx_quantize_segments(x, offsets, block=BLOCK):
    """Token-direction MXFP8 of x [N, C] inside each expert segment.  Returns (codes [N, C]
    uint8, [scales of expert e: uint8 [ceil(n_e / 32), C] for each e])."""
    x64 = np.asarray(x, dtype=np.float64)
    N, C = x64.shape
    codes = np.zeros((N, C), dtype=np.uint8)
    scales = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        n = hi - lo
        nb = -(-n // block)
        padded = np.zeros((nb * block, C))
        padded[:n] = x64[lo:hi]
        q, s = mx_quantize_cols(padded, block)
        codes[lo:hi] = q[:n]
        scales.append(s)
    return codes, scales


def mx_decode_segments(codes, scales, offsets, block=BLOCK):
    """Decoded values [N, C] of segment-blocked codes (fp64)."""
    c = np.asarray(codes)
    out = np.zeros(c.shape)
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        n = hi - lo
        if n == 0:
            continue
        nb = -(-n // block)
        padded = np.zeros((nb * block, c.shape[1]), dtype=np.uint8)
        padded[:n] = c[lo:hi]
        out[lo:hi] = mx_decode_cols(padded, scales[e], block)[:n]
    return out


def wgrad_mx(aq, a_s, bq, b_s, offsets):
    """dW[e] = dec(A_e)^T . dec(B_e) for every expert e (fp64), A_e and B_e the expert's rows of
    the segment-blocked operands A [N, M] and B [N, C]: [E, M, C]."""
    A = mx_decode_segments(aq, a_s, offsets)
    B = mx_decode_segments(bq, b_s, offsets)
    E = len(offsets) - 1
    dW = np.zeros((E, A.shape[1], B.shape[1]))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            dW[e] = A[lo:hi].T @ B[lo:hi]
    return dW
