"""Whole-layer parity: moe_layer_fwd / moe_layer_bwd (C ABI) against the fp64 oracle.

Shapes span several 128-row tiles with ragged tails (rows per expert, ffn widths that are not
multiples of 64/128), every score function / renorm combination, the shared expert with and
without its gate, single-expert and 256-expert layers, and the fp32 path.
"""
import numpy as np
import pytest
import torch

import moe_inputs
from moe_inputs import SIGMOID, SOFTMAX, LayerConfig

from .helpers import TOL, clean_inputs, compare_layer, inputs_to, np64, oracle_layer, run_layer

pytestmark = pytest.mark.gpu

CASES = {
    # name: LayerConfig
    "tiny_fp32": moe_inputs.TINY_F32,
    "fp32_sigmoid_shared_gate": LayerConfig("f32 sig", 100, 64, 6, 3, 32, f_shared=24,
                                            score_fn=SIGMOID, renorm=0, shared_gate=1, dtype="f32"),
    "bf16_softmax_shared_gate": LayerConfig("bf16 a", 700, 384, 8, 2, 200, f_shared=136,
                                            score_fn=SOFTMAX, renorm=1, shared_gate=1),
    "bf16_sigmoid_zipf_shared": LayerConfig("bf16 b", 513, 256, 32, 6, 128, f_shared=128,
                                            score_fn=SIGMOID, renorm=1, router_bias="zipf1.2"),
    "bf16_softmax_norenorm": LayerConfig("bf16 c", 300, 192, 16, 4, 96, score_fn=SOFTMAX, renorm=0),
    "bf16_sigmoid_norenorm_top1": LayerConfig("bf16 d", 257, 128, 4, 1, 64, score_fn=SIGMOID,
                                              renorm=0),
    "bf16_single_expert": LayerConfig("bf16 e", 130, 128, 1, 1, 136),
    "bf16_256_experts": LayerConfig("bf16 f", 400, 128, 256, 8, 64, f_shared=64, shared_gate=1),
    "bf16_wide_rows": LayerConfig("bf16 g", 1100, 1024, 8, 2, 320, score_fn=SIGMOID, renorm=1),
    # a handful of tokens: one partial row tile per live expert, most experts without rows
    "bf16_one_token": LayerConfig("bf16 h", 1, 128, 8, 2, 64, f_shared=64, shared_gate=1),
    "bf16_seven_tokens_128e": LayerConfig("bf16 i", 7, 256, 128, 8, 128, score_fn=SIGMOID,
                                          renorm=1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_layer_matches_oracle(name):
    lc = CASES[name]
    inp, seed = clean_inputs(lc)
    gpu = run_layer(lc, inputs_to(inp, "cuda"))
    ref = oracle_layer(lc, inp)
    errs = compare_layer(lc, gpu, ref, TOL[lc.dtype])
    print(name, "seed", seed, {k: f"{v:.2e}" for k, v in errs.items()})


def test_layer_is_deterministic():
    lc = CASES["bf16_sigmoid_zipf_shared"]
    inp, _ = clean_inputs(lc)
    d = inputs_to(inp, "cuda")
    a = run_layer(lc, d)
    b = run_layer(lc, d)
    for n in ["y", "dx", "dW_r", "dW1", "dW2", "dWs1", "dWs2"]:
        assert torch.equal(a[n], b[n]), n
    for n in ["idx", "gate", "offsets", "slot_of_pair", "x_perm", "act", "h", "y_perm"]:
        if a["saved"][n] is not None:
            assert torch.equal(a["saved"][n], b["saved"][n]), n


def test_empty_experts_get_zero_weight_gradients():
    """A router bias that no token can overcome leaves experts without rows: their dW1/dW2 must
    be exactly zero and the rest must still match the oracle."""
    lc = LayerConfig("bf16 empty", 300, 128, 16, 2, 64, score_fn=SOFTMAX, renorm=1)
    inp, _ = clean_inputs(lc)
    inp = dict(inp)
    b = torch.zeros(16)
    b[10:] = -1.0e4
    inp["b_r"] = b
    gpu = run_layer(lc, inputs_to(inp, "cuda"))
    ref = oracle_layer(lc, inp)
    assert (np64(gpu["saved"]["counts"])[10:] == 0).all()
    assert (np64(gpu["dW1"])[10:] == 0).all() and (np64(gpu["dW2"])[10:] == 0).all()
    compare_layer(lc, gpu, ref, TOL["bf16"])


def test_zero_tokens():
    lc = LayerConfig("bf16 T0", 0, 128, 8, 2, 64, f_shared=64, shared_gate=1)
    # buffers of one row, a layer of zero tokens: nothing may be read or written per token
    inp = inputs_to(moe_inputs.make_layer_inputs(lc.replace(T=1), seed=0), "cuda")
    gpu = run_layer(lc, inp)
    for n in ["dW_r", "dW1", "dW2", "dWs1", "dWs2", "dw_sg"]:
        assert (np64(gpu[n]) == 0).all(), n
    assert (np64(gpu["saved"]["offsets"]) == 0).all()


def test_layer_step_replays_from_a_cuda_graph():
    """The layer calls are capturable (no allocation, stream-ordered memsets, the caller's side
    stream forked and joined by its events): a captured forward + backward replayed from a CUDA
    graph gives bit-identical results to the eager calls, and those equal the calls without a
    side stream."""
    import moe_expert_layer_gemm_gb300 as moe
    lc = CASES["bf16_sigmoid_zipf_shared"]
    inp, _ = clean_inputs(lc)
    d = inputs_to(inp, "cuda")
    eager = run_layer(lc, d)                      # also performs the one-time setup uncaptured
    serial = run_layer(lc, d, side=False)
    for n in ["y", "dx", "dW_r", "dW1", "dW2", "dWs1", "dWs2"]:
        assert torch.equal(eager[n], serial[n]), n
    cfg = moe.cfg_from(lc)
    saved = moe.alloc_saved(cfg, "cuda")
    y = torch.empty_like(d["x"])
    g = {n: torch.empty_like(eager[n]) for n in ["dx", "dW_r", "dW1", "dW2", "dWs1", "dWs2"]}
    ws_f = moe.workspace(cfg, moe.WS_LAYER_FWD)
    ws_b = moe.workspace(cfg, moe.WS_LAYER_BWD)
    side = moe.SideStream("cuda")

    def step():
        moe.moe_layer_fwd(cfg, d["x"], d["W_r"], d["b_r"], d["W1"], d["W2"], d["Ws1"], d["Ws2"],
                          d["w_sg"], y, saved, ws_f, side=side)
        moe.moe_layer_bwd(cfg, d["dy"], d["x"], d["W_r"], d["W1"], d["W2"], d["Ws1"], d["Ws2"],
                          d["w_sg"], saved, g["dx"], g["dW_r"], g["dW1"], g["dW2"], g["dWs1"],
                          g["dWs2"], None, ws_b, side=side)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                    # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in [y, *g.values()]:
        t.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    moe.check_device_error()
    assert torch.equal(y, eager["y"])
    for n, t in g.items():
        assert torch.equal(t, eager[n]), n


def test_two_layer_steps_run_concurrently_on_their_own_streams():
    """The library owns no stream or switch: two forward + backward steps issued back to back on
    two streams, each with its own buffers, workspaces and side stream, may run at the same
    time, and each gives the results of the same step run alone."""
    import moe_expert_layer_gemm_gb300 as moe
    lc = CASES["bf16_sigmoid_zipf_shared"]
    runs = []
    for seed in (0, 1):
        inp, _ = clean_inputs(lc, seed=seed)
        runs.append(inputs_to(inp, "cuda"))
    alone = [run_layer(lc, d) for d in runs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    # the second step is enqueued while the first may still run
    together = [run_layer(lc, runs[i], stream=streams[i], sync=False) for i in (0, 1)]
    torch.cuda.synchronize()
    moe.check_device_error()
    for i in (0, 1):
        for n in ["y", "dx", "dW_r", "dW1", "dW2", "dWs1", "dWs2"]:
            assert torch.equal(together[i][n], alone[i][n]), (i, n)
