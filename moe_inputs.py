"""Seeded synthetic inputs for one mixture-of-experts layer.

This module holds only shapes and random draws: no step of the layer's arithmetic.
Both the CUDA path (tests, bench) and the CPU oracle take their inputs from here.

Workload shapes come from the pages:
  * "Megatron-Bridge 深度剖析" (§Motivation): a DeepSeek-style layer with 128 experts,
    top-6 sigmoid routing, expert ffn 1856, hidden 2688, plus a shared expert.
  * "Tevatron Meets Megatron" (§3): Qwen3-30B-A3B, 128 experts, top-8.
  * "Add Megatron-Core MTP training for Qwen3.5 MoE" (Notes): an MTP MoE layer with 256
    experts, shared expert and shared-expert gate, 16 sequences of up to 2k tokens.
The datasets those pages train on are not used: the layer only sees activations, so seeded
Gaussian activations of the same shapes stand in for them.
"""
from __future__ import annotations

import dataclasses
import math

import torch

SOFTMAX = 0
SIGMOID = 1


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int            # tokens
    d: int            # d_model
    E: int            # routed experts
    k: int            # experts per token
    f: int            # routed expert ffn width
    f_shared: int = 0  # shared expert ffn width (0: no shared expert)
    score_fn: int = SOFTMAX
    renorm: int = 1
    shared_gate: int = 0
    dtype: str = "bf16"        # "bf16" or "f32"
    router_init: str = "normal"  # "normal" (N(0, 0.02)) or "uniform" (U(+-1/sqrt(d)))
    router_bias: str = "none"    # "none", "zipf1.2" or "normal0.05"
    backward: bool = True
    bias_mode: int = 0           # 0: b_r added to the logits; 1: to the scores, selection only
    aux_coeff: float = 0.0       # load-balancing loss coefficient (0: no auxiliary loss)

    @property
    def N(self) -> int:
        return self.T * self.k

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def replace(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


# The five workloads.  Names say what each is; sizes are the pages' layer shapes.
TINY_F32 = LayerConfig("tiny-fp32 T256 d128 E8 top2 softmax-renorm f256", 256, 128, 8, 2, 256,
                       dtype="f32")
QWEN3_30B_A3B = LayerConfig("qwen3-30b-a3b-shaped T8192 d2048 E128 top8 softmax-renorm f768",
                            8192, 2048, 128, 8, 768, backward=False)
DEEPSEEK_128E = LayerConfig(
    "deepseek-style T16384 d2688 E128 top6 sigmoid-renorm f1856 shared1856 zipf1.2",
    16384, 2688, 128, 6, 1856, f_shared=1856, score_fn=SIGMOID, renorm=1,
    router_bias="zipf1.2")
MTP_256E = LayerConfig(
    "mtp-256e T32768 d2048 E256 top8 softmax-renorm f512 shared512 sigmoid-gate",
    32768, 2048, 256, 8, 512, f_shared=512, score_fn=SOFTMAX, renorm=1, shared_gate=1,
    router_init="uniform")
ROUTE_STRESS = LayerConfig("routing-stress T65536 d4096 E128 top8 sigmoid", 65536, 4096, 128, 8,
                           512, score_fn=SIGMOID, renorm=0, backward=False)

# A 32-expert slice of the DeepSeek-style layer: same d_model, ffn, top-k and about the same
# rows per expert (T*k/E = 768), a quarter of the tokens -- small enough (about 4 GB on the
# device) for multi-pass profiler captures of the per-expert kernels.
DEEPSEEK_E32 = DEEPSEEK_128E.replace(
    name="deepseek-style slice T4096 d2688 E32 top6 sigmoid-renorm f1856 shared1856 zipf1.2",
    T=4096, E=32)

CONFIGS = {
    "tiny": TINY_F32,
    "qwen3": QWEN3_30B_A3B,
    "deepseek": DEEPSEEK_128E,
    "mtp256": MTP_256E,
    "stress": ROUTE_STRESS,
    "deepseek_e32": DEEPSEEK_E32,
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def zipf_router_bias(E: int, s: float = 1.2, seed: int = 0, device="cpu") -> torch.Tensor:
    """Per-expert logit bias that makes a few experts hot: b[e] = -s * ln(r_e), with r a
    seeded random permutation of 1..E (expert with rank 1 gets bias 0, rank r gets
    -s*ln r), so that exp(b) follows a Zipf(s) law over experts."""
    g = _gen(seed + 7, "cpu")
    r = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (-s * torch.log(r)).to(torch.float32).to(device)


def normal_router_bias(E: int, std: float = 0.05, seed: int = 0, device="cpu") -> torch.Tensor:
    """Per-expert bias ~ N(0, std^2) from its own seeded generator (an expert-bias state of the
    size a balancing correction reaches next to sigmoid scores in (0, 1))."""
    g = _gen(seed + 11, "cpu")
    return (torch.randn(E, generator=g, dtype=torch.float32) * std).to(device)


def make_layer_inputs(cfg: LayerConfig, seed: int = 0, device="cpu", T: int | None = None):
    """All tensors of one layer call, drawn from one seeded generator.

    x ~ N(0,1); expert and shared weights ~ N(0, 0.02); router ~ N(0, 0.02) or
    U(-1/sqrt(d), 1/sqrt(d)); upstream gradient dy ~ N(0,1).  Values are drawn in fp32 and
    rounded once to the layer dtype, so the oracle reads exactly what the GPU reads.
    """
    T = cfg.T if T is None else T
    g = _gen(seed, device)
    dt = cfg.torch_dtype

    def randn(*shape, std=1.0):
        return (torch.randn(*shape, generator=g, device=device) * std).to(dt)

    out = {}
    out["x"] = randn(T, cfg.d)
    if cfg.router_init == "uniform":
        a = 1.0 / math.sqrt(cfg.d)
        out["W_r"] = ((torch.rand(cfg.E, cfg.d, generator=g, device=device) * 2 - 1) * a).to(dt)
    else:
        out["W_r"] = randn(cfg.E, cfg.d, std=0.02)
    if cfg.router_bias == "zipf1.2":
        out["b_r"] = zipf_router_bias(cfg.E, 1.2, seed, device)
    elif cfg.router_bias == "normal0.05":
        out["b_r"] = normal_router_bias(cfg.E, 0.05, seed, device)
    else:
        out["b_r"] = None
    out["W1"] = randn(cfg.E, 2 * cfg.f, cfg.d, std=0.02)
    out["W2"] = randn(cfg.E, cfg.d, cfg.f, std=0.02)
    if cfg.f_shared > 0:
        out["Ws1"] = randn(2 * cfg.f_shared, cfg.d, std=0.02)
        out["Ws2"] = randn(cfg.d, cfg.f_shared, std=0.02)
        out["w_sg"] = randn(cfg.d, std=0.02) if cfg.shared_gate else None
    else:
        out["Ws1"] = out["Ws2"] = out["w_sg"] = None
    out["dy"] = randn(T, cfg.d)
    return out


# Degenerate routing cases of the routing/permute stress workload.
STRESS_CASES = ("normal", "all_to_8", "32_empty", "int_ties")


def make_stress_logits(case: str, T: int, E: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """fp32 router logits [T, E] for the routing stress cases:
      normal   -- N(0,1)
      all_to_8 -- N(0,1) with +100 on experts 0..7, so every token picks exactly those
      32_empty -- N(0,1) with -1e4 on the last 32 experts, so they receive no token
      int_ties -- integers drawn from {0,1,2,3}: massive exact ties
    """
    g = _gen(seed + 11, device)
    if case == "int_ties":
        return torch.randint(0, 4, (T, E), generator=g, device=device).to(torch.float32)
    lg = torch.randn(T, E, generator=g, device=device)
    if case == "all_to_8":
        lg[:, :8] += 100.0
    elif case == "32_empty":
        lg[:, E - 32:] -= 1.0e4
    elif case != "normal":
        raise ValueError(case)
    return lg.contiguous()
