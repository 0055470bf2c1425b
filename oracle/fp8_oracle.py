"""Oracle for the FP8 expert GEMMs: E4M3 encoding, tensorwise quantisation and the grouped
SwiGLU forward on quantised operands (fp64 CPU).

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU leg may import this
module; it imports nothing of the CUDA library and shares no code with it.

What the pages fix ("Megatron-Bridge 深度剖析", §FP8 训练): FP8 in the E4M3 format (largest
finite magnitude about 480 -- exactly 448 for the finite-only E4M3 variant), a "tensorwise"
scaling recipe (one scale per tensor), and that FP8 halves the bytes the 128-expert grouped
GEMM moves.  Readings where they are silent:
  * the scale maps a tensor's largest magnitude onto 448: q = E4M3(x * (448 / amax)), the stored
    dequantisation scale is amax / 448, both quotients formed in fp32 (amax = 0 -> scales 1);
  * E4M3 rounding is round-to-nearest-even with saturation to +-448 (no infinities);
  * activations are one tensor (one scale); each expert's fc1 and fc2 weight is its own tensor
    (one scale per expert), as the pages' per-parameter "tensorwise" recipe implies;
  * the GEMM multiplies the decoded values and applies both scales to the fp32 result; the
    SwiGLU input h is quantised again (its own tensorwise scale) before fc2;
  * backward ("fp8_wgrad": weight gradients in FP8 too; "e4m3" for every tensor): the upstream
    gradient dy_perm is one tensor, quantised like the activations; fc2's data gradient and the
    SwiGLU backward give [da | du] in bf16, which is quantised as one tensor before fc1's data
    gradient and fc1's weight gradient; the weight gradients multiply the quantised tensors the
    forward made (x_perm_q, h_q) with the quantised gradients, the weights' codes are reused as
    stored.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import silu, silu_grad

E4M3_MAX = 448.0


def e4m3_decode(codes):
    """Value of E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is
    subnormal with value m/8 * 2^-6; code S.1111.111 is NaN, there is no infinity)."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def _finite_table():
    codes = np.arange(0x7F, dtype=np.int64)          # non-negative finite codes 0x00..0x7E
    return codes, e4m3_decode(codes)


def e4m3_encode(x32):
    """E4M3 code of each fp32 value: round to the nearest representable value, ties to the code
    with an even mantissa (the even last bit), magnitudes above 448 saturate to 448."""
    x = np.asarray(x32, dtype=np.float32).astype(np.float64)
    codes, vals = _finite_table()
    a = np.minimum(np.abs(x), E4M3_MAX)
    # nearest value by bracketing: vals is increasing in the code
    hi = np.searchsorted(vals, a, side="left")
    hi = np.clip(hi, 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo = a - vals[lo]
    d_hi = vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    mag = np.where(pick_hi, codes[hi], codes[lo])
    mag = np.where(a == vals[hi], codes[hi], mag)
    # the sign is kept, also on values that round to zero (-0 has its own code, 0x80)
    return (mag | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def quantize_tensorwise(x, groups=1):
    """Tensorwise quantisation of x split into `groups` equal leading blocks (one tensor each):
    per block amax (fp32), inv = fp32(448 / amax), codes = E4M3(fp32(x * inv)),
    scale = fp32(amax / 448).  Returns (codes with x's shape, scale [groups] fp32)."""
    x32 = np.asarray(x, dtype=np.float32)
    blocks = x32.reshape(groups, -1)
    amax = np.abs(blocks).max(axis=1).astype(np.float32)
    inv = np.where(amax > 0, np.float32(E4M3_MAX) / np.where(amax > 0, amax, 1), 1).astype(np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), 1).astype(np.float32)
    scaled = (blocks * inv[:, None]).astype(np.float32)
    return e4m3_encode(scaled).reshape(x32.shape), scale


def dequantize(codes, scale, groups=1):
    """Decoded values times their block's scale (fp64)."""
    c = np.asarray(codes)
    v = e4m3_decode(c.reshape(groups, -1)) * np.asarray(scale, np.float64)[:, None]
    return v.reshape(c.shape)


def fc1_swiglu_fp8(xq, sx, W1q, sw1, offsets):
    """fc1 + SwiGLU of every expert on quantised operands: for rows s of expert e,
    [a | u] = (dec(xq[s]) * sx) . (dec(W1q[e]) * sw1[e])^T, h = SiLU(a) * u.  fp64."""
    E = W1q.shape[0]
    f = W1q.shape[1] // 2
    X = dequantize(xq, sx)
    N = X.shape[0]
    h = np.zeros((N, f))
    act = np.zeros((N, 2 * f))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        W = e4m3_decode(W1q[e]) * float(sw1[e])
        au = X[lo:hi] @ W.T
        a, u = au[:, :f], au[:, f:]
        act[lo:hi] = au
        h[lo:hi] = silu(a) * u
    return h, act


def fc2_fp8(hq, sh, W2q, sw2, offsets):
    """fc2 of every expert on quantised operands: y[s] = (dec(hq[s]) * sh) . (dec(W2q[e]) *
    sw2[e])^T for rows s of expert e.  fp64."""
    E = W2q.shape[0]
    H = dequantize(hq, sh)
    y = np.zeros((H.shape[0], W2q.shape[1]))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            y[lo:hi] = H[lo:hi] @ (e4m3_decode(W2q[e]) * float(sw2[e])).T
    return y


# ----------------------------------------------------------------------------- backward

def _rows(offsets, e):
    return int(offsets[e]), int(offsets[e + 1])


def fc2_dgrad_fp8(dyq, sdy, W2q, sw2, offsets):
    """dh[s] = (dec(dyq[s]) * sdy) . (dec(W2q[e]) * sw2[e]) for rows s of expert e ([d] . [d, f]).
    fp64."""
    E, _, f = W2q.shape
    D = dequantize(dyq, sdy)
    dh = np.zeros((D.shape[0], f))
    for e in range(E):
        lo, hi = _rows(offsets, e)
        if hi > lo:
            dh[lo:hi] = D[lo:hi] @ (e4m3_decode(W2q[e]) * float(sw2[e]))
    return dh


def swiglu_backward(dh, act):
    """[da | du] of h = SiLU(a) * u at the saved pre-activations act = [a | u]:
    da = dh * u * SiLU'(a), du = dh * SiLU(a).  fp64."""
    f = dh.shape[1]
    a, u = np.asarray(act, np.float64)[:, :f], np.asarray(act, np.float64)[:, f:]
    return np.concatenate([dh * u * silu_grad(a), dh * silu(a)], axis=1)


def fc1_dgrad_fp8(dH1q, sdh, W1q, sw1, offsets):
    """dx[s] = (dec(dH1q[s]) * sdh) . (dec(W1q[e]) * sw1[e]) for rows s of expert e
    ([2f] . [2f, d]).  fp64."""
    E, _, d = W1q.shape
    G = dequantize(dH1q, sdh)
    dx = np.zeros((G.shape[0], d))
    for e in range(E):
        lo, hi = _rows(offsets, e)
        if hi > lo:
            dx[lo:hi] = G[lo:hi] @ (e4m3_decode(W1q[e]) * float(sw1[e]))
    return dx


def wgrad_fp8(Aq, sa, Bq, sb, offsets):
    """dW[e] = (dec(Aq[rows of e]) * sa)^T . (dec(Bq[rows of e]) * sb): [m, n] per expert, zero for
    an expert without rows.  fp64."""
    E = len(offsets) - 1
    A = dequantize(Aq, sa)
    B = dequantize(Bq, sb)
    dW = np.zeros((E, A.shape[1], B.shape[1]))
    for e in range(E):
        lo, hi = _rows(offsets, e)
        if hi > lo:
            dW[e] = A[lo:hi].T @ B[lo:hi]
    return dW


def bf16_round(x):
    """x rounded to bfloat16 (round to nearest even) and returned as fp64 (via torch, a library
    implementation of the format)."""
    import torch
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


def grouped_swiglu_bwd_fp8(xq, sx, W1q, sw1, W2q, sw2, act, hq, sh, dy_perm, offsets):
    """The backward of the FP8 grouped SwiGLU, stage by stage:
      dy_perm -> (dyq, sdy) one tensor;  dh = fc2_dgrad_fp8;  dH1 = SwiGLU backward, stored in
      bf16 and quantised as one tensor -> (dH1q, sdh);  dx = fc1_dgrad_fp8;
      dW1 = wgrad_fp8(dH1q, x);  dW2 = wgrad_fp8(dyq, h).
    Returns a dict with every intermediate."""
    dyq, sdy = quantize_tensorwise(np.asarray(dy_perm, np.float32))
    dh = fc2_dgrad_fp8(dyq, sdy, W2q, sw2, offsets)
    dH1 = bf16_round(swiglu_backward(dh, act))
    dH1q, sdh = quantize_tensorwise(dH1.astype(np.float32))
    return {
        "dy_q": dyq, "dy_scale": sdy, "dh": dh, "dH1": dH1, "dH1_q": dH1q, "dH1_scale": sdh,
        "dx": fc1_dgrad_fp8(dH1q, sdh, W1q, sw1, offsets),
        "dW1": wgrad_fp8(dH1q, sdh, xq, sx, offsets),
        "dW2": wgrad_fp8(dyq, sdy, hq, sh, offsets),
    }
