"""Benchmark of the MoE layer forward + backward on GB300.

One step = moe_layer_fwd + moe_layer_bwd (router GEMM, top-k, routing maps, permute, grouped
SwiGLU fc1/fc2, shared expert, combine, and every backward stage) on one batch of seeded
synthetic tokens resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload deepseek]
  python bench.py --impl reference ...   # the fp64 CPU oracle timed on the host cores

Default workload: the DeepSeek-style layer (T=16384 tokens, d_model 2688, 128 experts, top-6
sigmoid routing normalised over the selected experts, expert ffn 1856, one shared expert of
ffn 1856, Zipf(1.2) router bias), forward + backward.  Its inputs (3.8 GB of expert weights,
0.5 GB+ per activation array) are far larger than the 129 MB L2, so no L2 flush is needed
between steps.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_inputs  # noqa: E402

METRIC = "MoE layer fwd+bwd tokens/s; grouped-GEMM TFLOPS and % of bf16 peak, 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ----------------------------------------------------------------------------- work per kernel

def kernel_work(lc, trace=None, steps=1):
    """Algorithmic work of one launch of each kernel kind: ('tensor', FLOPs) or ('hbm', bytes).
    FLOPs count 2 per multiply-add of the products the method needs (no padding, no dense
    all-expert work); bytes count each operand the kernel must read or write once.  The FP8
    layer's E4M3 products (names ending in _fp8) do the same FLOPs as their bf16 twins; its
    quantisation kernels serve several tensors a step, so their bytes per launch are the step's
    total times `steps` over the launches `trace` saw in that many steps."""
    T, d, E, k, f, fs = lc.T, lc.d, lc.E, lc.k, lc.f, lc.f_shared
    N = T * k
    b = 2 if lc.dtype == "bf16" else 4
    g = 1 if lc.shared_gate else 0
    w = {
        "gemm_router": ("tensor", 2.0 * T * d * E),
        "gemm_fc1_swiglu": ("tensor", 4.0 * N * d * f),
        "gemm_fc2": ("tensor", 2.0 * N * d * f),
        "gemm_fc2_dgrad": ("tensor", 2.0 * N * d * f),
        "gemm_fc2_wgrad": ("tensor", 2.0 * N * d * f),
        "gemm_fc1_dgrad": ("tensor", 4.0 * N * d * f),
        "gemm_fc1_wgrad": ("tensor", 4.0 * N * d * f),
        "gemm_router_dgrad": ("tensor", 2.0 * T * d * E),
        "gemm_router_wgrad": ("tensor", 2.0 * T * d * (E + g)),
        "route_topk": ("hbm", T * E * 4 + N * 8),
        "route_scan": ("hbm", 0.0),
        "route_slots": ("hbm", N * 4 + N * 8),
        "permute": ("hbm", T * d * b * (1 + k) + N * 4),
        "combine": ("hbm", T * d * b * (k + 1) + N * 8 + (T * d * b if fs else 0)),
        "combine_bwd": ("hbm", T * d * b * (1 + 2 * k) + N * 12 + (2 * T * d * b if fs else 0)),
        "permute_bwd": ("hbm", T * d * b * (k + 1) + N * 4 + T * d * b * (2 if fs else 1)),
        "router_bwd": ("hbm", T * E * 4 + N * 12 + T * (E + g) * b),
        "split_reduce": ("hbm", 0.0),
        "shared_gate": ("hbm", T * d * b),
    }
    if fs:
        w.update({
            "gemm_shared_fc1_swiglu": ("tensor", 4.0 * T * d * fs),
            "gemm_shared_fc2": ("tensor", 2.0 * T * d * fs),
            "gemm_shared_fc2_dgrad": ("tensor", 2.0 * T * d * fs),
            "gemm_shared_fc2_wgrad": ("tensor", 2.0 * T * d * fs),
            "gemm_shared_fc1_dgrad": ("tensor", 4.0 * T * d * fs),
            "gemm_shared_fc1_wgrad": ("tensor", 4.0 * T * d * fs),
        })
    for n in [n for n in w if n.startswith("gemm_") and "router" not in n]:
        w[n + "_fp8"] = w[n]
    # E4M3 quantisation (bf16 in, one byte out): amax passes read (only x's in the layer: the
    # gradients' amaxes come out of the combine backward), quantise passes read + write
    amax_bytes = T * d * 2
    quant_bytes = N * f * 3 + (T * fs * 3 if fs else 0)
    if lc.backward:
        quant_bytes += N * d * 3 + N * 2 * f * 3 + ((T * d * 3 + T * 2 * fs * 3) if fs else 0)
    per = lambda name, total: total * steps / max(1, (trace or {}).get(name, (steps, 0))[0])  # noqa: E731
    w["fp8_amax"] = ("hbm", per("fp8_amax", amax_bytes))
    w["fp8_quantize"] = ("hbm", per("fp8_quantize", quant_bytes))
    w["fp8_permute_quantize"] = ("hbm", T * d * 2 + N * d + (T * d if fs else 0) + N * 4)
    # MXFP8 (routed experts): the same products; permute + quantise reads x once and writes every
    # pair's codes and its block scales (one byte per 32)
    w["gemm_fc1_swiglu_mxfp8"] = w["gemm_fc1_swiglu"]
    w["gemm_fc2_mxfp8"] = w["gemm_fc2"]
    w["gemm_fc2_dgrad_mxfp8"] = w["gemm_fc2_dgrad"]
    w["gemm_fc1_dgrad_mxfp8"] = w["gemm_fc1_dgrad"]
    # (with a backward, the MXFP8 forward also writes the bf16 x_perm the weight gradient reads)
    w["mxfp8_permute_quantize"] = ("hbm", T * d * 2 + N * d * 33 / 32 + N * 4 +
                                   (N * d * 2 if lc.backward else 0))
    w["mxfp8_quantize_rows"] = ("hbm", N * d * 2 + N * d * 33 / 32)   # dy_perm in expert order
    # the weight gradients' token-direction quantisation: x_perm, dy_perm, h and [da | du] read in
    # bf16, written as codes plus one scale byte per 32 (four launches a step)
    w["mxfp8_quantize_tokens"] = ("hbm", per("mxfp8_quantize_tokens",
                                             N * (2 * d + 3 * f) * (2 + 33 / 32)))
    w["gemm_fc2_wgrad_mxfp8"] = w["gemm_fc2_wgrad"]
    w["gemm_fc1_wgrad_mxfp8"] = w["gemm_fc1_wgrad"]
    # the combine backward that also writes dy_perm's codes and scales
    w["combine_bwd_mxfp8"] = ("hbm", w["combine_bwd"][1] + N * d * 33 / 32)
    return w


def gemm_bytes(lc):
    """Algorithmic DRAM bytes of one launch of each expert GEMM: every operand read once, every
    result written once (bf16 activations out, fp32 weight gradients; E4M3 operands of the _fp8
    kinds one byte each).  A GEMM whose bytes at the measured copy bandwidth take longer than its
    FLOPs at the tensor peak is HBM-bound, and its roofline is the bandwidth."""
    T, d, E, k, f, fs = lc.T, lc.d, lc.E, lc.k, lc.f, lc.f_shared
    out = {}
    for pre, rows, G, ff in (("gemm_", T * k, E, f), ("gemm_shared_", T, 1, fs)):
        if ff == 0:
            continue
        for sfx, b in (("", 2), ("_fp8", 1)):
            out[pre + "fc1_swiglu" + sfx] = rows * d * b + G * 2 * ff * d * b + rows * 3 * ff * 2
            out[pre + "fc2" + sfx] = rows * ff * b + G * d * ff * b + rows * d * 2
            out[pre + "fc2_dgrad" + sfx] = rows * d * b + G * d * ff * b + rows * 4 * ff * 2
            out[pre + "fc2_wgrad" + sfx] = rows * d * b + rows * ff * b + G * d * ff * 4
            out[pre + "fc1_dgrad" + sfx] = rows * 2 * ff * b + G * 2 * ff * d * b + rows * d * 2
            out[pre + "fc1_wgrad" + sfx] = rows * 2 * ff * b + rows * d * b + G * 2 * ff * d * 4
    # MXFP8 forward (layer call): codes plus one scale byte per 32 in, h's codes and scales out
    # of fc1 (no bf16 h or [a | u]), bf16 y_perm out of fc2
    q = 33 / 32
    out["gemm_fc1_swiglu_mxfp8"] = T * k * d * q + E * 2 * f * d * q + T * k * f * q
    out["gemm_fc2_mxfp8"] = T * k * f * q + E * d * f * q + T * k * d * 2
    # data gradients: dy's and the weights' codes in; [da | du] in bf16 and as codes, dx out
    out["gemm_fc2_dgrad_mxfp8"] = T * k * d * q + E * d * f * q + T * k * 2 * f * 2 + \
        T * k * 2 * f * (2 + q)
    out["gemm_fc1_dgrad_mxfp8"] = T * k * 2 * f * q + E * 2 * f * d * q + T * k * d * 2
    # weight gradients: both token-blocked operands' codes and scales in, fp32 blocks out
    out["gemm_fc2_wgrad_mxfp8"] = T * k * (d + f) * q + E * d * f * 4
    out["gemm_fc1_wgrad_mxfp8"] = T * k * (2 * f + d) * q + E * 2 * f * d * 4
    return out


def kernel_source_hash():
    """sha256 over the library's kernel sources and public header (names and bytes)."""
    import glob
    import hashlib
    files = sorted(glob.glob(os.path.join(ROOT, "moe_expert_layer_gemm_gb300", "csrc", "*")))
    files.append(os.path.join(ROOT, "include", "moe_gb300.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()


def captured_traffic(workload, kernel):
    """DRAM bytes (read + write) of one launch of `kernel`, from the ncu capture summarised in
    profiles/traffic.json; None when there is none or the kernel sources changed since."""
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tpath):
        return None
    d = json.load(open(tpath))
    if d.get("source_sha256") != kernel_source_hash():
        return None
    rec = d.get("workloads", {}).get(workload, {}).get(kernel)
    return None if rec is None else rec["total"]


def layer_flops(lc, backward=True):
    fl = 2.0 * lc.T * lc.d * lc.E + 6.0 * lc.T * lc.k * lc.d * lc.f
    if lc.f_shared:
        fl += 6.0 * lc.T * lc.d * lc.f_shared + (2.0 * lc.T * lc.d if lc.shared_gate else 0.0)
    return fl * (3.0 if backward else 1.0)


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(value, device=None):
    """The largest value over all ranks (a job of replicas is as slow as its slowest one);
    the value itself on a single rank.  device: where the collective's tensor lives (the
    rank's GPU under NCCL, the CPU under gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_rank_step, steps, world, ms_max):
    """Whole-job tokens/s of `world` independent replicas, each running `steps` steps of
    tokens_per_rank_step tokens, timed by the slowest rank (ms_max)."""
    return tokens_per_rank_step * steps * world / (ms_max / 1e3)


# ----------------------------------------------------------------------------- clocks

class NvmlClockSampler:
    """SM clock, its maximum, power and the clock-event (throttle) reasons of one GPU, read through
    NVML (read-only queries) every `period` seconds on a host thread during the timed region, so
    that even a short region gets several samples.  The GPU is found by its PCI bus id."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, device, period=0.01):
        import ctypes
        import threading
        import torch
        self.ok = False
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        nv = self.nv
        if nv.nvmlInit_v2() != 0:
            return
        pr = torch.cuda.get_device_properties(device)
        bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0".encode()
        self.h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(self.h)) != 0:
            return
        self.reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.samples = []
        self.period = period
        self.stop_ev = threading.Event()
        self.ok = True
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _read(self):
        import ctypes
        sm, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(sm)) != 0:   # NVML_CLOCK_SM
            return None
        self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(pw))
        self.reason_fn(self.h, ctypes.byref(rs))
        return sm.value, mx.value, pw.value / 1000.0, rs.value

    def _run(self):
        while not self.stop_ev.is_set():
            r = self._read()
            if r is not None:
                self.samples.append(r)
            self.stop_ev.wait(self.period)

    def stop(self):
        if not self.ok:
            return None
        self.stop_ev.set()
        self.thread.join(timeout=5)
        self.nv.nvmlShutdown()
        if not self.samples:
            return None
        reasons = sorted({n for *_, rs in self.samples for b, n in self.REASONS.items() if rs & b})
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "reasons": reasons,
                "samples": len(self.samples), "power_w_max": round(max(s[2] for s in self.samples), 1),
                "source": f"NVML every {int(self.period * 1e3)} ms"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region (used
    when NVML cannot be loaded)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi every 200 ms"}


def start_clock_sampler(device, gpu_index):
    s = NvmlClockSampler(device)
    return s if s.ok else ClockSampler(gpu_index)


# ----------------------------------------------------------------------------- CPU oracle leg

def oracle_sample_inputs(lc, inp, n_tok, seed=1234):
    """A seeded subset of n_tok tokens with every expert's weights, as numpy (fp32 values of the
    bf16 inputs; the oracle reads them as fp64)."""
    import numpy as np
    import torch
    gen = torch.Generator().manual_seed(seed)
    sel = torch.randperm(lc.T, generator=gen)[:n_tok].sort().values
    host = {}
    for name, t in inp.items():
        if t is None:
            host[name] = None
        elif name in ("x", "dy"):
            host[name] = t[sel.to(t.device)].float().cpu().numpy()
        else:
            host[name] = t.float().cpu().numpy()
    return host, lc.replace(T=n_tok)


def time_oracle(lc_s, host, reps=1):
    import oracle.moe_oracle as O
    t0 = time.perf_counter()
    for _ in range(reps):
        fwd = O.layer_forward(lc_s, host)
        if lc_s.backward:
            O.layer_backward(lc_s, host, fwd, host["dy"])
    return (time.perf_counter() - t0) / reps


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- main arm

def run_gpu(args, lc):
    import torch
    import torch.distributed as dist

    import moe_expert_layer_gemm_gb300 as moe
    from moe_expert_layer_gemm_gb300 import build as _build

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    if not os.path.exists(moe._lib.LIB_PATH):
        if rank == 0:
            _build.build()
        if world > 1:
            dist.barrier()
    moe.lib()
    dev = torch.device("cuda", local)
    # each rank is an independent replica on its own tokens (weak scaling; no exchange)
    inp = moe_inputs.make_layer_inputs(lc, seed=args.seed + rank, device=dev)
    cfg = moe.cfg_from(lc)
    saved = moe.alloc_saved(cfg, dev)
    f32 = torch.float32
    y = torch.empty_like(inp["x"])
    grads = dict(
        dx=torch.empty_like(inp["x"]),
        dW_r=torch.empty(lc.E, lc.d, dtype=f32, device=dev),
        dW1=torch.empty(lc.E, 2 * lc.f, lc.d, dtype=f32, device=dev),
        dW2=torch.empty(lc.E, lc.d, lc.f, dtype=f32, device=dev),
        dWs1=torch.empty(2 * lc.f_shared, lc.d, dtype=f32, device=dev) if lc.f_shared else None,
        dWs2=torch.empty(lc.d, lc.f_shared, dtype=f32, device=dev) if lc.f_shared else None,
        dw_sg=torch.empty(lc.d, dtype=f32, device=dev) if lc.shared_gate else None,
    )
    ws_f = moe.workspace(cfg, moe.WS_LAYER_FWD, dev)
    ws_b = moe.workspace(cfg, moe.WS_LAYER_BWD_FP8 if args.fp8 else moe.WS_LAYER_BWD, dev)
    stream = torch.cuda.current_stream()
    # the caller-owned second stream of the layer calls (shared expert and router backward beside
    # the routed experts)
    side = moe.SideStream(dev)
    mxq = None
    if args.mxfp8:
        # MXFP8 routed experts (weights quantised once, outside the timed steps, both copies).
        # Forward-only configurations keep routing and y_perm alone; with a backward, the forward
        # also saves the bf16 x_perm, [a | u] and h, and the backward runs the routed data
        # gradients on MXFP8 operands and the weight gradients on token-blocked MXFP8 operands
        # (bf16 with --mxfp8-bf16-wgrad)
        mxq = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"], dev)
        mxd = moe.alloc_mxfp8_dgrad(cfg, inp["W1"], inp["W2"], dev) if lc.backward else None
        if mxd is not None and not args.mxfp8_bf16_wgrad:
            mxd["wgrad_ws"] = moe.workspace(cfg, moe.WS_WGRAD_MXFP8, dev)
        if not lc.backward:
            saved["x_perm"] = saved["act"] = saved["h"] = None
    fp8q = None
    if args.fp8:
        # E4M3 weights quantised once (FP8 parameters); saved.x_perm is not used
        fp8q = moe.alloc_fp8_experts(cfg, inp["W1"], inp["W2"], dev, Ws1=inp["Ws1"], Ws2=inp["Ws2"])
        saved["x_perm"] = None

    def step(x, dy, yout, dxout, side=side):
        if mxq is not None:
            moe.moe_layer_fwd_mxfp8(cfg, x, inp["W_r"], inp["b_r"], mxq, inp["Ws1"], inp["Ws2"],
                                    inp["w_sg"], yout, saved, ws_f, side=side)
            if lc.backward:
                moe.moe_layer_bwd_mxfp8(cfg, dy, x, inp["W_r"], mxd, inp["Ws1"], inp["Ws2"],
                                        inp["w_sg"], saved, dxout, grads["dW_r"], grads["dW1"],
                                        grads["dW2"], grads["dWs1"], grads["dWs2"],
                                        grads["dw_sg"], ws_b, side=side)
            return
        if fp8q is not None:
            moe.moe_layer_fwd_fp8(cfg, x, inp["W_r"], inp["b_r"], fp8q, inp["Ws1"], inp["Ws2"],
                                  inp["w_sg"], yout, saved, ws_f, side=side)
            if lc.backward:
                moe.moe_layer_bwd_fp8(cfg, dy, x, inp["W_r"], fp8q, inp["Ws1"], inp["Ws2"],
                                      inp["w_sg"], saved, dxout, grads["dW_r"], grads["dW1"],
                                      grads["dW2"], grads["dWs1"], grads["dWs2"], grads["dw_sg"], ws_b,
                                      side=side)
            return
        moe.moe_layer_fwd(cfg, x, inp["W_r"], inp["b_r"], inp["W1"], inp["W2"], inp["Ws1"],
                          inp["Ws2"], inp["w_sg"], yout, saved, ws_f, side=side)
        if lc.backward:
            moe.moe_layer_bwd(cfg, dy, x, inp["W_r"], inp["W1"], inp["W2"], inp["Ws1"], inp["Ws2"],
                              inp["w_sg"], saved, dxout, grads["dW_r"], grads["dW1"], grads["dW2"],
                              grads["dWs1"], grads["dWs2"], grads["dw_sg"], ws_b, side=side)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step(inp["x"], inp["dy"], y, grads["dx"])
    torch.cuda.synchronize()
    moe.check_device_error()

    # One step captured in a CUDA graph (the library allocates nothing and orders its memsets
    # and side-stream fork/join on the stream, so the whole step is capturable); the timed
    # region replays it.  --no-graph times the eager calls instead.
    graph = None
    if not args.no_graph:
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            step(inp["x"], inp["dy"], y, grads["dx"])
        stream.wait_stream(cs)
        graph = torch.cuda.CUDAGraph()
        before = moe.launch_count()
        with torch.cuda.graph(graph):
            step(inp["x"], inp["dy"], y, grads["dx"])
        graph_launches = moe.launch_count() - before
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        moe.check_device_error()

    def timed_step():
        if graph is not None:
            graph.replay()
        else:
            step(inp["x"], inp["dy"], y, grads["dx"])

    # ---- device-timed region: inputs resident in HBM
    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except (ValueError, IndexError):
            pass
    clocks = start_clock_sampler(dev, gpu_index)
    launches0 = moe.launch_count()
    barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        timed_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    # graph replays launch no host calls: count the captured step's launches per replay
    launches = (moe.launch_count() - launches0) if graph is None else graph_launches * args.steps
    clk = clocks.stop()
    ms_total = ev0.elapsed_time(ev1)
    moe.check_device_error()

    # ---- per-kernel attribution: a second timed region with every launch bracketed by CUDA
    # events on its stream, without the side stream (concurrent kernels would share the SMs and
    # their event times would overlap); identical results, serial order.
    n_trace = max(3, min(args.steps, 20))
    moe.trace_read()   # drop anything recorded before
    moe.trace_enable(True)
    torch.cuda.synchronize()
    tr0 = torch.cuda.Event(enable_timing=True)
    tr1 = torch.cuda.Event(enable_timing=True)
    tr0.record(stream)
    for _ in range(n_trace):
        step(inp["x"], inp["dy"], y, grads["dx"], side=None)
    tr1.record(stream)
    torch.cuda.synchronize()
    moe.trace_enable(False)
    trace = moe.trace_read()
    trace_ms_step = tr0.elapsed_time(tr1) / n_trace
    moe.check_device_error()
    ms_max = max_over_ranks(ms_total, dev)
    ms_step = ms_max / args.steps
    value = replica_throughput(lc.T, args.steps, world, ms_max)

    # ---- end-to-end: every step copies its inputs (x, dy) in from pinned host memory and its
    # results (y, dx) out to pinned host memory.  Uploads and downloads run on two copy streams
    # (two copy engines), double-buffered, so that step i+1's upload and step i's download
    # overlap step i's compute; events order every buffer's reuse.
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    x_h = [inp["x"].cpu().pin_memory() for _ in range(2)]
    dy_h = [inp["dy"].cpu().pin_memory() for _ in range(2)]
    y_h = [torch.empty_like(x_h[0]).pin_memory() for _ in range(2)]
    dx_h = [torch.empty_like(x_h[0]).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(inp["x"]) for _ in range(2)]
    dy_d = [torch.empty_like(inp["dy"]) for _ in range(2)]
    y_d = [torch.empty_like(inp["x"]) for _ in range(2)]
    dx_d = [torch.empty_like(inp["x"]) for _ in range(2)]
    up_s = torch.cuda.Stream(device=dev)
    down_s = torch.cuda.Stream(device=dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]
    # the step on each device buffer pair replays a CUDA graph, as in the device-timed region
    e2e_graphs = [None, None]
    if graph is not None:
        for b in range(2):
            x_d[b].copy_(inp["x"])
            dy_d[b].copy_(inp["dy"])
            cs = torch.cuda.Stream(device=dev)
            cs.wait_stream(stream)
            with torch.cuda.stream(cs):
                step(x_d[b], dy_d[b], y_d[b], dx_d[b])
            stream.wait_stream(cs)
            e2e_graphs[b] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graphs[b]):
                step(x_d[b], dy_d[b], y_d[b], dx_d[b])
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up_s.wait_stream(stream)
    down_s.wait_stream(stream)
    with torch.cuda.stream(up_s):
        x_d[0].copy_(x_h[0], non_blocking=True)
        if lc.backward:                    # a forward-only step reads no dy
            dy_d[0].copy_(dy_h[0], non_blocking=True)
        uploaded[0].record(up_s)
    for i in range(e2e_steps):
        b = i & 1
        stream.wait_event(uploaded[b])
        if i >= 2:
            stream.wait_event(downloaded[b])      # step i-2's results are out of y_d[b], dx_d[b]
        if e2e_graphs[b] is not None:
            e2e_graphs[b].replay()
        else:
            step(x_d[b], dy_d[b], y_d[b], dx_d[b])
        computed[b].record(stream)
        if i + 1 < e2e_steps:
            nb = b ^ 1
            with torch.cuda.stream(up_s):
                if i >= 1:
                    up_s.wait_event(computed[nb])  # step i-1 no longer reads x_d[nb], dy_d[nb]
                x_d[nb].copy_(x_h[nb], non_blocking=True)
                if lc.backward:
                    dy_d[nb].copy_(dy_h[nb], non_blocking=True)
                uploaded[nb].record(up_s)
        with torch.cuda.stream(down_s):
            down_s.wait_event(computed[b])
            y_h[b].copy_(y_d[b], non_blocking=True)
            if lc.backward:
                dx_h[b].copy_(dx_d[b], non_blocking=True)
            downloaded[b].record(down_s)
    stream.wait_stream(up_s)
    stream.wait_stream(down_s)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    e2e_value = replica_throughput(lc.T, e2e_steps, world, e2e_ms)
    esz = inp["x"].element_size()
    h2d = (2 if lc.backward else 1) * lc.T * lc.d * esz
    d2h = 2 * lc.T * lc.d * esz if lc.backward else lc.T * lc.d * esz
    assert torch.equal(y_h[(e2e_steps - 1) & 1].to(dev), y), "e2e output differs from the device run"

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    fp8 = None if args.no_fp8 or args.fp8 or args.mxfp8 or lc.dtype != "bf16" else \
        fp8_experts(args, lc, cfg, inp, saved, dev)
    if fp8 is not None:
        fp8["layer"] = fp8_layer(args, lc, cfg, inp, dev, ms_step)
        fp8["mxfp8_layer_fwd"] = mxfp8_layer_fwd(args, lc, cfg, inp, dev)

    # ---- roofline of the dominant kernel (largest share of device time in the timed region)
    peaks, peak_src = load_peaks()
    work = kernel_work(lc, trace, n_trace)
    flops_of = dict(work)      # FLOPs of the GEMMs, whatever bound their roofline takes
    # Peaks: the burst figure (a short timed region: the kernels are timed inside a
    # sub-second region, as a kernel timed alone) and the sustained one beside it.
    bf16_burst = peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained"))
    bf16_sus = peaks.get("bf16_tflops_sustained", bf16_burst)

    def tensor_peak(name, sustained=False):
        # E4M3 products (tensorwise or block-scaled): twice the measured bf16 rate (the nominal
        # dense fp8 : bf16 ratio)
        p = bf16_sus if sustained else bf16_burst
        return 2.0 * p if name.endswith(("_fp8", "_mxfp8")) else p

    gbytes = gemm_bytes(lc) if lc.dtype == "bf16" else {}
    kern = {}
    for name, (n_launch, ms) in trace.items():
        kind, amount = work.get(name, ("hbm", 0.0))
        if kind == "tensor" and name in gbytes and \
                gbytes[name] / (peaks["hbm_gbs"] * 1e9) > amount / (tensor_peak(name) * 1e12):
            kind, amount = "hbm", gbytes[name]      # bound by its bytes, not its FLOPs
        work[name] = (kind, amount)
        avg_ms = ms / max(1, n_launch)
        if kind == "tensor":
            ach = amount / (avg_ms / 1e3) / 1e12
            unit, peak, peak_s = "TFLOP/s", tensor_peak(name), tensor_peak(name, True)
        else:
            ach = amount / (avg_ms / 1e3) / 1e9
            unit, peak = "GB/s", peaks["hbm_gbs"]
            peak_s = peak
        kern[name] = {"launches": n_launch, "ms_per_launch": round(avg_ms, 4),
                      "share": None, "achieved": round(ach, 1), "unit": unit,
                      "frac": round(ach / peak, 4) if amount else None,
                      "frac_sustained": round(ach / peak_s, 4) if amount else None}
    tot = sum(ms for _, ms in trace.values()) or 1.0
    for name, (n_launch, ms) in trace.items():
        kern[name]["share"] = round(ms / tot, 4)
    dom = max(trace.items(), key=lambda kv: kv[1][1])[0] if trace else None
    roof = None
    if dom:
        kd = kern[dom]
        kind = work.get(dom, ("hbm", 0))[0]
        traffic = captured_traffic(lc.name, dom)
        fp8_dom = kind == "tensor" and dom.endswith(("_fp8", "_mxfp8"))
        roof = {"bound": kind, "kernel": dom, "achieved": kd["achieved"],
                "peak": tensor_peak(dom) if kind == "tensor" else peaks["hbm_gbs"],
                "unit": kd["unit"], "frac": kd["frac"], "traffic": traffic,
                "peak_source": f"{peak_src} (" + ("2 x bf16_tflops (burst), nominal fp8:bf16 ratio"
                                                  if fp8_dom else "bf16_tflops (burst)"
                                                  if kind == "tensor" else "hbm_gbs") + ")",
                "peak_sustained": tensor_peak(dom, True) if kind == "tensor" else peaks["hbm_gbs"],
                "frac_sustained": kd["frac_sustained"]}
    # The routing chain of the forward: router GEMM (whose epilogue also selects, with bf16
    # operands), top-k (given or fp32 logits), the scan (large histograms only) and the slot maps.
    # Its algorithmic bytes: x and W_r read, fp32 logits written, idx, gate and both slot maps
    # written (4 x N x 4 bytes).
    chain = [n for n in ("gemm_router", "route_topk", "route_scan", "route_slots") if n in trace]
    routing = None
    if chain:
        r_ms = sum(trace[n][1] for n in chain) / n_trace
        r_bytes = (lc.T * lc.d * (2 if lc.dtype == "bf16" else 4) * 1.0 +
                   lc.E * lc.d * (2 if lc.dtype == "bf16" else 4) + lc.T * lc.E * 4 +
                   16.0 * lc.T * lc.k)
        r_ach = r_bytes / (r_ms / 1e3) / 1e9
        rest = [n for n in chain if n != "gemm_router"]
        routing = {"launches": chain, "ms_per_step": round(r_ms, 4),
                   "bytes": int(r_bytes), "achieved": round(r_ach, 1), "unit": "GB/s",
                   "frac": round(r_ach / peaks["hbm_gbs"], 4),
                   "after_gemm_ms": round(sum(trace[n][1] for n in rest) / n_trace, 4)}
    gemm_ms = sum(ms for n, (_, ms) in trace.items() if n.startswith("gemm_"))
    gemm_flops = sum(flops_of[n][1] * trace[n][0] for n in trace
                     if n.startswith("gemm_") and n in flops_of)
    gemm_tflops = gemm_flops / (gemm_ms / 1e3) / 1e12 if gemm_ms else None

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        n_tok = args.cpu_tokens
        host, lc_s = oracle_sample_inputs(lc, inp, n_tok)
        dt = time_oracle(lc_s, host)
        cpu = {"value": round(n_tok / dt, 2), "unit": "tokens/s", "cores": cpu_cores(),
               "kind": "oracle",
               "sample": f"{n_tok} seeded tokens of the workload, all {lc.E} experts, "
                         f"{'fwd+bwd' if lc.backward else 'fwd'} in fp64 numpy ({dt:.1f} s)"}

    flops_step = layer_flops(lc, lc.backward)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 experts, bf16 router/combine" if args.fp8 else
                  (("mxfp8 expert products (e4m3, e8m0 scale per 32) in the forward and the data "
                    "gradients, bf16 weight gradients, bf16 router/shared/combine"
                    if args.mxfp8_bf16_wgrad else
                    "mxfp8 expert products (e4m3, e8m0 scale per 32) in the forward, the data "
                    "gradients and the weight gradients (token blocks), bf16 router/shared/combine")
                   if lc.backward else
                   "mxfp8 experts (e4m3, e8m0 scale per 32), bf16 router/shared/combine")
                  if args.mxfp8 else lc.dtype),
        "data": "synthetic (seeded N(0,1) tokens, N(0,0.02) weights, random init)",
        "config": {"workload": lc.name, "T": lc.T, "d_model": lc.d, "experts": lc.E, "top_k": lc.k,
                   "ffn": lc.f, "shared_ffn": lc.f_shared,
                   "score_fn": "sigmoid" if lc.score_fn else "softmax", "renorm": bool(lc.renorm),
                   "shared_gate": bool(lc.shared_gate), "router_bias": lc.router_bias,
                   "pass": "fwd+bwd" if lc.backward else "fwd",
                   "global_batch": lc.T * world, "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (expert weights alone exceed 129 MB), no flush"},
        "tflops": round(flops_step / (ms_step / 1e3) / 1e12, 1),
        "pct_bf16_peak": round(flops_step / (ms_step / 1e3) / 1e12 / bf16_burst, 4),
        "pct_bf16_peak_sustained": round(flops_step / (ms_step / 1e3) / 1e12 / bf16_sus, 4),
        "grouped_gemm_tflops": round(gemm_tflops, 1) if gemm_tflops else None,
        "roofline": roof,
        "routing_chain": routing,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "cuda_graph": graph is not None,
        "kernel_trace": {"steps": n_trace, "ms_per_step": round(trace_ms_step, 4),
                         "shared_overlap": False,
                         "note": "per-kernel CUDA-event times (roofline, kernels) from this "
                                 "second timed region, run in serial order"},
        "clocks": clk,
        "cpu_baseline": cpu,
        "fp8": fp8,
        "kernels": kern,
    }
    if world > 1:
        dist.destroy_process_group()
    return out


# ----------------------------------------------------------------------------- FP8 experts

def fp8_experts(args, lc, cfg, inp, saved, dev):
    """The routed experts in bf16 and in FP8 E4M3 on the same routed rows, forward and backward.
    Forward: permute + fc1 + SwiGLU + fc2; backward: the expert backward (both data gradients, both
    weight gradients).  FP8 weights are quantised once (FP8 parameters); activations and gradients
    are quantised every step (x with the permute, h and [da | du] from their GEMMs' epilogues, dy
    inside the backward call).  Device time per step with CUDA events."""
    import torch
    import moe_expert_layer_gemm_gb300 as moe
    E, d, f, N = lc.E, lc.d, lc.f, lc.N
    if d % 16 or f % 16:
        return None
    u8, bf = torch.uint8, torch.bfloat16
    x_perm, off = saved["x_perm"], saved["offsets"]
    W1q = torch.empty(E, 2 * f, d, dtype=u8, device=dev)
    W2q = torch.empty(E, d, f, dtype=u8, device=dev)
    s1, s2, a1, a2 = (torch.empty(max(E, 4), device=dev) for _ in range(4))
    moe.moe_quantize_e4m3(inp["W1"], E, W1q, s1, a1)
    moe.moe_quantize_e4m3(inp["W2"], E, W2q, s2, a2)
    xq = torch.empty(N, d, dtype=u8, device=dev)
    xs, xa, hs, ha, dys, dya, gs, ga = (torch.empty(4, device=dev) for _ in range(8))
    h = torch.empty(N, f, dtype=bf, device=dev)
    act = torch.empty(N, 2 * f, dtype=bf, device=dev)
    hq = torch.empty(N, f, dtype=u8, device=dev)
    yp = torch.empty(N, d, dtype=bf, device=dev)
    g = torch.Generator(device=dev).manual_seed(11)
    dyp = (torch.randn(N, d, device=dev, generator=g) * 0.01).to(bf)
    dyq = torch.empty(N, d, dtype=u8, device=dev)
    dH1 = torch.empty(N, 2 * f, dtype=bf, device=dev)
    dH1q = torch.empty(N, 2 * f, dtype=u8, device=dev)
    dxp = torch.empty(N, d, dtype=bf, device=dev)
    dW1 = torch.empty(E, 2 * f, d, device=dev)
    dW2 = torch.empty(E, d, f, device=dev)
    ws16 = moe.workspace(cfg, moe.WS_FFN_BWD, dev)
    ws8 = moe.workspace(cfg, moe.WS_FFN_BWD_FP8, dev)
    sop = saved["slot_of_pair"]
    # MXFP8 (one E8M0 scale per 32 elements along K): weights quantised once, x with the
    # permute, h in fc1's epilogue; [a | u] saved as for training, bf16 h not written
    mx = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"], dev) if d % 32 == 0 and f % 32 == 0 \
        else None

    def fwd16():
        moe.moe_permute(cfg, inp["x"], sop, x_perm)
        moe.moe_grouped_swiglu_fwd(cfg, x_perm, off, inp["W1"], inp["W2"], h, act, yp)

    def fwd8():
        moe.moe_permute_quantize_e4m3(cfg, inp["x"], sop, xq, xs, xa)
        moe.moe_grouped_swiglu_fwd_fp8(cfg, xq, xs, off, W1q, s1, W2q, s2, h, act, hq, hs, ha, yp)

    def fwdmx():
        moe.moe_permute_quantize_mxfp8(cfg, inp["x"], sop, off, mx["x_perm_q"], mx["x_perm_s"])
        moe.moe_grouped_swiglu_fwd_mxfp8(cfg, mx["x_perm_q"], mx["x_perm_s"], off, mx["W1_q"],
                                         mx["W1_sp"], mx["W2_q"], mx["W2_sp"], None, act, mx["h_q"],
                                         mx["h_s"], yp)

    def bwd16():
        moe.moe_grouped_swiglu_bwd(cfg, x_perm, off, inp["W1"], inp["W2"], act, h, dyp, dxp, dW1,
                                   dW2, ws16)

    def bwd8():
        moe.moe_grouped_swiglu_bwd_fp8(cfg, xq, xs, off, W1q, s1, W2q, s2, act, hq, hs, dyp, dyq,
                                       dys, dya, dH1, dH1q, gs, ga, dxp, dW1, dW2, ws8)

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    n = max(5, min(args.steps, 50))
    peaks, src = load_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops_sustained"]
    out = {"fp8_peak": f"{fp8_peak:.1f} TFLOP/s = 2 x {src} bf16_tflops_sustained (nominal ratio)"}
    for part, f16, f8, flops, gemms, scope in (
            ("forward", fwd16, fwd8, 6.0 * N * d * f, ("gemm_fc1_swiglu_fp8", "gemm_fc2_fp8"),
             "permute + routed fc1+SwiGLU and fc2; x quantised with the permute, h from fc1's "
             "epilogue amax (included)"),
            ("backward", bwd16, bwd8, 12.0 * N * d * f,
             ("gemm_fc2_dgrad_fp8", "gemm_fc2_wgrad_fp8", "gemm_fc1_dgrad_fp8", "gemm_fc1_wgrad_fp8"),
             "routed expert backward: dy quantised, fc2 dgrad + SwiGLU backward, [da | du] "
             "quantised, fc1 dgrad, fc1 and fc2 weight gradients (fp32)")):
        if part == "backward":
            fwd8()          # the backward reads the FP8 forward's h codes and [a | u]
        ms16 = timed(f16, n)
        if part == "backward":
            fwd8()
        moe.trace_read()
        moe.trace_enable(True)
        ms8 = timed(f8, n)
        moe.trace_enable(False)
        tr = moe.trace_read()
        moe.check_device_error()
        per = {k: round(ms / c, 4) for k, (c, ms) in tr.items() if c}
        gemm_ms = sum(per.get(k, 0) for k in gemms)
        out[part] = {"bf16_ms": round(ms16, 4), "fp8_ms": round(ms8, 4),
                     "speedup": round(ms16 / ms8, 3),
                     "fp8_gemm_tflops": round(flops / (gemm_ms / 1e3) / 1e12, 1) if gemm_ms else None,
                     "fp8_gemm_frac": round(flops / (gemm_ms / 1e3) / 1e12 / fp8_peak, 4)
                     if gemm_ms else None,
                     "kernels_ms": per, "scope": scope}
    if mx is not None:
        moe.trace_read()
        moe.trace_enable(True)
        msmx = timed(fwdmx, n)
        moe.trace_enable(False)
        tr = moe.trace_read()
        moe.check_device_error()
        per = {k: round(ms / c, 4) for k, (c, ms) in tr.items() if c}
        gemm_ms = sum(per.get(k, 0) for k in ("gemm_fc1_swiglu_mxfp8", "gemm_fc2_mxfp8"))
        flops = 6.0 * N * d * f
        fw = out["forward"]
        fw.update(mxfp8_ms=round(msmx, 4), mxfp8_speedup=round(fw["bf16_ms"] / msmx, 3),
                  mxfp8_gemm_tflops=round(flops / (gemm_ms / 1e3) / 1e12, 1) if gemm_ms else None,
                  mxfp8_gemm_frac=round(flops / (gemm_ms / 1e3) / 1e12 / fp8_peak, 4)
                  if gemm_ms else None,
                  mxfp8_kernels_ms=per,
                  mxfp8_scope="MXFP8 (E8M0 scale per 32 along K): permute + quantise x, fc1 + "
                              "SwiGLU with h quantised in its epilogue, fc2; [a | u] saved")
    return out


def graph_timed(args, step, dev, n):
    """Device ms per call of step(): 3 eager warm-up calls, then n replays of a CUDA graph of one
    call (eager calls with --no-graph), timed with CUDA events on the current stream."""
    import torch
    import moe_expert_layer_gemm_gb300 as moe
    stream = torch.cuda.current_stream()
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    moe.check_device_error()
    graph = None
    if not args.no_graph:
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            step()
        stream.wait_stream(cs)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        graph.replay() if graph is not None else step()
    e1.record(stream)
    torch.cuda.synchronize()
    moe.check_device_error()
    return e0.elapsed_time(e1) / n, graph is not None


def mxfp8_layer_fwd(args, lc, cfg, inp, dev):
    """The layer forward with MXFP8 routed experts (moe_layer_fwd_mxfp8: x permuted and
    block-quantised in one pass, h quantised in fc1's epilogue; router, bf16 shared expert and
    combine as in bf16) against the bf16 layer forward (moe_layer_fwd), both replayed from CUDA
    graphs.  MXFP8 weights are quantised once, outside the timed calls."""
    import torch
    import moe_expert_layer_gemm_gb300 as moe
    if lc.d % 32 or lc.f % 32:
        return None
    s16 = moe.alloc_saved(cfg, dev)
    smx = moe.alloc_saved(cfg, dev)
    smx["x_perm"] = smx["act"] = smx["h"] = None
    mx = moe.alloc_mxfp8_experts(cfg, inp["W1"], inp["W2"], dev)
    y = torch.empty_like(inp["x"])
    ws_f = moe.workspace(cfg, moe.WS_LAYER_FWD, dev)
    side = moe.SideStream(dev)

    def f16():
        moe.moe_layer_fwd(cfg, inp["x"], inp["W_r"], inp["b_r"], inp["W1"], inp["W2"], inp["Ws1"],
                          inp["Ws2"], inp["w_sg"], y, s16, ws_f, side=side)

    def fmx():
        moe.moe_layer_fwd_mxfp8(cfg, inp["x"], inp["W_r"], inp["b_r"], mx, inp["Ws1"], inp["Ws2"],
                                inp["w_sg"], y, smx, ws_f, side=side)

    n = max(5, min(args.steps, 50))
    ms16, graphed = graph_timed(args, f16, dev, n)
    msmx, _ = graph_timed(args, fmx, dev, n)
    return {"bf16_fwd_ms": round(ms16, 4), "mxfp8_fwd_ms": round(msmx, 4),
            "speedup": round(ms16 / msmx, 3), "tokens_per_s": round(lc.T / (msmx / 1e3), 1),
            "steps": n, "cuda_graph": graphed,
            "scope": "layer forward: routing, permute + quantise, routed experts in MXFP8, "
                     "shared expert in bf16, combine (bf16 forward: the same with bf16 experts)"}


def fp8_layer(args, lc, cfg, inp, dev, ms_bf16):
    """The whole layer step with FP8 experts (moe_layer_fwd_fp8 / moe_layer_bwd_fp8: routed and
    shared experts on E4M3 operands, router, gate and combine as in bf16; E4M3 weights quantised
    once as FP8 parameters, activations and gradients quantised inside the step), replayed from a
    CUDA graph like the bf16 step it is compared with."""
    import torch
    import moe_expert_layer_gemm_gb300 as moe
    saved = moe.alloc_saved(cfg, dev)
    saved["x_perm"] = None
    q = moe.alloc_fp8_experts(cfg, inp["W1"], inp["W2"], dev, Ws1=inp["Ws1"], Ws2=inp["Ws2"])
    f32 = torch.float32
    y = torch.empty_like(inp["x"])
    g = dict(dx=torch.empty_like(inp["x"]), dW_r=torch.empty(lc.E, lc.d, dtype=f32, device=dev),
             dW1=torch.empty(lc.E, 2 * lc.f, lc.d, dtype=f32, device=dev),
             dW2=torch.empty(lc.E, lc.d, lc.f, dtype=f32, device=dev),
             dWs1=torch.empty(2 * lc.f_shared, lc.d, dtype=f32, device=dev) if lc.f_shared else None,
             dWs2=torch.empty(lc.d, lc.f_shared, dtype=f32, device=dev) if lc.f_shared else None,
             dw_sg=torch.empty(lc.d, dtype=f32, device=dev) if lc.shared_gate else None)
    ws_f = moe.workspace(cfg, moe.WS_LAYER_FWD, dev)
    ws_b = moe.workspace(cfg, moe.WS_LAYER_BWD_FP8, dev)
    side = moe.SideStream(dev)

    def step():
        moe.moe_layer_fwd_fp8(cfg, inp["x"], inp["W_r"], inp["b_r"], q, inp["Ws1"], inp["Ws2"],
                              inp["w_sg"], y, saved, ws_f, side=side)
        if lc.backward:
            moe.moe_layer_bwd_fp8(cfg, inp["dy"], inp["x"], inp["W_r"], q, inp["Ws1"], inp["Ws2"],
                                  inp["w_sg"], saved, g["dx"], g["dW_r"], g["dW1"], g["dW2"],
                                  g["dWs1"], g["dWs2"], g["dw_sg"], ws_b, side=side)

    n = max(5, min(args.steps, 50))
    ms, graphed = graph_timed(args, step, dev, n)
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(lc.T / (ms / 1e3), 1),
            "bf16_ms_per_step": round(ms_bf16, 4), "speedup": round(ms_bf16 / ms, 3),
            "steps": n, "cuda_graph": graphed,
            "scope": "whole layer " + ("fwd+bwd" if lc.backward else "fwd") + " with the routed "
                     "and shared experts in E4M3 (router, shared gate and combine in bf16)"}


# ----------------------------------------------------------------------------- reference arm

def run_route_only(args, lc):
    """Routing alone on the workload's tokens: moe_route_topk from x (router GEMM whose epilogue
    selects, then the slot maps) and from given fp32 logits (top-k kernel, then the slot maps),
    each timed as a CUDA graph of `steps` calls after `warmup` eager ones, with a per-kernel
    CUDA-event trace beside it.  The chain's algorithmic bytes: x and W_r read, fp32 logits
    written (the GEMM path) or read (the given-logits path), idx, gate and both slot maps written."""
    import torch

    import moe_expert_layer_gemm_gb300 as moe
    from moe_expert_layer_gemm_gb300 import build as _build

    if not os.path.exists(moe._lib.LIB_PATH):
        _build.build()
    moe.lib()
    dev = torch.device("cuda", 0)
    inp = moe_inputs.make_layer_inputs(lc, seed=args.seed, device=dev)
    x, W_r, b_r = inp["x"], inp["W_r"], inp["b_r"]
    del inp
    torch.cuda.empty_cache()
    cfg = moe.cfg_from(lc)
    T, E, k = lc.T, lc.E, lc.k
    i32 = torch.int32
    o = dict(idx=torch.empty(T, k, dtype=i32, device=dev), gate=torch.empty(T, k, device=dev),
             counts=torch.empty(E, dtype=i32, device=dev),
             offsets=torch.empty(E + 1, dtype=i32, device=dev),
             sop=torch.empty(T, k, dtype=i32, device=dev),
             tos=torch.empty(max(T * k, 1), dtype=i32, device=dev))
    lg = torch.empty(T, E, device=dev)
    lg_in = torch.empty(T, E, device=dev)
    ws = moe.workspace(cfg, moe.WS_ROUTE, dev)
    stream = torch.cuda.Stream(dev)
    peaks, _ = load_peaks()
    b = 2 if lc.dtype == "bf16" else 4
    maps = 16.0 * T * k
    paths = {
        "from_x": (lambda: moe.moe_route_topk(cfg, x, W_r, b_r, None, lg, o["idx"], o["gate"],
                                              o["counts"], o["offsets"], o["sop"], o["tos"], ws,
                                              stream=stream),
                   T * lc.d * b + E * lc.d * b + T * E * 4.0 + maps),
        "from_logits": (lambda: moe.moe_route_topk(cfg, None, None, b_r, lg_in, None, o["idx"],
                                                   o["gate"], o["counts"], o["offsets"], o["sop"],
                                                   o["tos"], ws, stream=stream),
                        T * E * 4.0 + maps),
    }
    out = {}
    with torch.cuda.stream(stream):
        paths["from_x"][0]()
        lg_in.copy_(lg)   # the logits the router GEMM wrote
        for name, (fn, nbytes) in paths.items():
            for _ in range(args.warmup):
                fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(args.steps):
                    fn()
            g.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            stream.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / args.steps
            moe.trace_read()
            moe.trace_enable(True)
            n_tr = max(3, min(args.steps, 20))
            for _ in range(n_tr):
                fn()
            stream.synchronize()
            moe.trace_enable(False)
            tr = moe.trace_read()
            moe.check_device_error()
            out[name] = {"us_per_call": round(us, 2),
                         "achieved": round(nbytes / (us * 1e-6) / 1e9, 1), "unit": "GB/s",
                         "frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                         "bytes": int(nbytes),
                         "kernels_us": {n: round(ms * 1e3 / max(1, c), 2) for n, (c, ms) in tr.items()},
                         "launches_per_call": int(sum(c for c, _ in tr.values()) / n_tr)}
    return {"metric": "routing time per call (moe_route_topk)", "value": out["from_x"]["us_per_call"],
            "unit": "us", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "data": "synthetic (the workload's seeded x, W_r, b_r)",
            "config": {"workload": lc.name, "T": T, "d_model": lc.d, "experts": E, "top_k": k,
                       "score_fn": "sigmoid" if lc.score_fn else "softmax",
                       "renorm": bool(lc.renorm), "timing": "CUDA graph of `steps` calls"},
            "paths": out}


def run_wgrad_routings(args, lc):
    """The routed experts' backward (moe_grouped_swiglu_bwd) on the workload's expert shapes under
    several per-expert row distributions with the same total rows N = T*k where the distribution
    allows: the workload's own routing (moe_route_topk on its seeded tokens), uniform, N/8 rows on
    8 experts (the others empty), 64 rows on every expert and one row on every expert.  Operands
    are seeded Gaussians; each distribution is timed per kernel with the CUDA-event trace over
    `steps` calls after `warmup` eager ones.  For each weight gradient the line gives its
    reduction FLOPs (2 per multiply-add, padded k-blocks not counted) and its fp32 block bytes."""
    import numpy as np
    import torch

    import moe_expert_layer_gemm_gb300 as moe
    from moe_expert_layer_gemm_gb300 import build as _build

    if not os.path.exists(moe._lib.LIB_PATH):
        _build.build()
    moe.lib()
    dev = torch.device("cuda", 0)
    E, d, f, N = lc.E, lc.d, lc.f, lc.T * lc.k
    # the workload's routing: counts from the library's own routing of the seeded tokens
    inp = moe_inputs.make_layer_inputs(lc, seed=args.seed, device=dev)
    cfg_r = moe.cfg_from(lc)
    i32 = torch.int32
    counts = torch.empty(E, dtype=i32, device=dev)
    offsets = torch.empty(E + 1, dtype=i32, device=dev)
    moe.moe_route_topk(cfg_r, inp["x"], inp["W_r"], inp["b_r"], None,
                       torch.empty(lc.T, E, device=dev),
                       torch.empty(lc.T, lc.k, dtype=i32, device=dev),
                       torch.empty(lc.T, lc.k, device=dev), counts, offsets,
                       torch.empty(lc.T, lc.k, dtype=i32, device=dev),
                       torch.empty(N, dtype=i32, device=dev), moe.workspace(cfg_r, moe.WS_ROUTE, dev))
    own = counts.cpu().numpy().astype(np.int64)
    del inp
    torch.cuda.empty_cache()
    uni = np.full(E, N // E, np.int64)
    uni[: N - uni.sum()] += 1
    hot = np.zeros(E, np.int64)
    hot[:8] = N // 8
    hot[: N - hot.sum()] += 1
    dists = {"workload": own, "uniform": uni, "8_experts": hot,
             "64_rows_each": np.full(E, 64, np.int64), "1_row_each": np.ones(E, np.int64)}
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed)
    bf = torch.bfloat16
    rows = max(int(c.sum()) for c in dists.values())
    xp = torch.randn(rows, d, device=dev, generator=g).to(bf)
    act = torch.randn(rows, 2 * f, device=dev, generator=g).to(bf)
    h = torch.randn(rows, f, device=dev, generator=g).to(bf)
    dyp = torch.randn(rows, d, device=dev, generator=g).to(bf)
    dxp = torch.empty(rows, d, device=dev, dtype=bf)
    W1 = (torch.randn(E, 2 * f, d, device=dev, generator=g) * 0.02).to(bf)
    W2 = (torch.randn(E, d, f, device=dev, generator=g) * 0.02).to(bf)
    dW1 = torch.empty(E, 2 * f, d, device=dev)
    dW2 = torch.empty(E, d, f, device=dev)
    out = {}
    for name, c in dists.items():
        n = int(c.sum())
        cfg = moe.make_cfg(n, d, E, 1, f)
        ws = moe.workspace(cfg, moe.WS_FFN_BWD, dev)
        off = torch.tensor(np.concatenate([[0], np.cumsum(c)]), dtype=i32, device=dev)
        call = lambda: moe.moe_grouped_swiglu_bwd(cfg, xp, off, W1, W2, act, h, dyp, dxp, dW1, dW2, ws)
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        moe.trace_read()
        moe.trace_enable(True)
        for _ in range(args.steps):
            call()
        torch.cuda.synchronize()
        moe.trace_enable(False)
        tr = moe.trace_read()
        moe.check_device_error()
        ms = {k_: round(t / max(1, cnt), 4) for k_, (cnt, t) in tr.items()}
        out[name] = {"rows": n, "max_rows": int(c.max()), "experts_with_rows": int((c > 0).sum()),
                     "kernels_ms": ms,
                     "fc1_wgrad": {"tflop": round(4.0 * n * d * f / 1e12, 4),
                                   "fp32_gb": round(E * 2 * f * d * 4 / 1e9, 3)},
                     "fc2_wgrad": {"tflop": round(2.0 * n * d * f / 1e12, 4),
                                   "fp32_gb": round(E * d * f * 4 / 1e9, 3)}}
        del ws
    return {"metric": "routed-expert backward kernel times under per-expert row distributions",
            "value": out["workload"]["kernels_ms"].get("gemm_fc1_wgrad"), "unit": "ms",
            "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "data": "synthetic (seeded Gaussian operands; the workload's own routing counts)",
            "config": {"workload": lc.name, "d_model": d, "experts": E, "ffn": f, "N": N,
                       "timing": "per-kernel CUDA events, eager calls"},
            "distributions": out}


def wait_kind_name(kind):
    """The product a GEMM pipeline wait-statistics kind (moe_gemm_wait_stats) stands for here."""
    if kind >= 48:
        return "tall row tiles, B " + ("MN-major (data gradients)" if kind & 1 else "K-major (fc2)")
    epi = ["bf16 store", "fp32", "SwiGLU forward", "SwiGLU backward"][(kind >> 3) & 3]
    sched = "ragged reduction (weight gradients)" if kind & 4 else "ragged rows"
    return f"one-CTA 128x256, {sched}, {epi}" + (", 8-bit" if kind & 32 else "")


def run_wait_stats(args, lc):
    """Where the tensor-core GEMMs' pipelines wait: the routed experts' forward
    (moe_grouped_swiglu_fwd) and backward (moe_grouped_swiglu_bwd) on the workload's shapes and its
    own routing counts, `steps` calls of each after `warmup`, with the library built with
    MOE_WAIT_STATS=1.  Per kernel kind: the fraction of the CTAs' cycles the producer waited for a
    free stage, the MMA warp for a loaded stage and for a free accumulator, the first epilogue
    warp for a finished accumulator, and the CTA cycles per k-block."""
    import numpy as np
    import torch

    import moe_expert_layer_gemm_gb300 as moe
    from moe_expert_layer_gemm_gb300 import build as _build

    if not os.path.exists(moe._lib.LIB_PATH):
        _build.build()
    moe.lib()
    if moe.gemm_wait_stats() is None:
        return {"metric": "GEMM pipeline wait fractions", "unavailable":
                "the library was built without the counters: rebuild with "
                "MOE_NVCC_EXTRA=-DMOE_WAIT_STATS=1"}
    dev = torch.device("cuda", 0)
    E, d, f, N = lc.E, lc.d, lc.f, lc.T * lc.k
    inp = moe_inputs.make_layer_inputs(lc, seed=args.seed, device=dev)
    cfg_r = moe.cfg_from(lc)
    i32 = torch.int32
    counts = torch.empty(E, dtype=i32, device=dev)
    offsets = torch.empty(E + 1, dtype=i32, device=dev)
    moe.moe_route_topk(cfg_r, inp["x"], inp["W_r"], inp["b_r"], None,
                       torch.empty(lc.T, E, device=dev),
                       torch.empty(lc.T, lc.k, dtype=i32, device=dev),
                       torch.empty(lc.T, lc.k, device=dev), counts, offsets,
                       torch.empty(lc.T, lc.k, dtype=i32, device=dev),
                       torch.empty(N, dtype=i32, device=dev), moe.workspace(cfg_r, moe.WS_ROUTE, dev))
    del inp
    torch.cuda.empty_cache()
    g = torch.Generator(device=dev)
    g.manual_seed(args.seed)
    bf = torch.bfloat16
    xp = torch.randn(N, d, device=dev, generator=g).to(bf)
    W1 = (torch.randn(E, 2 * f, d, device=dev, generator=g) * 0.02).to(bf)
    W2 = (torch.randn(E, d, f, device=dev, generator=g) * 0.02).to(bf)
    h = torch.empty(N, f, device=dev, dtype=bf)
    act = torch.empty(N, 2 * f, device=dev, dtype=bf)
    yp = torch.empty(N, d, device=dev, dtype=bf)
    dyp = torch.randn(N, d, device=dev, generator=g).to(bf)
    dxp = torch.empty(N, d, device=dev, dtype=bf)
    dW1 = torch.empty(E, 2 * f, d, device=dev)
    dW2 = torch.empty(E, d, f, device=dev)
    cfg = moe.make_cfg(N, d, E, 1, f)
    wsf = moe.workspace(cfg, moe.WS_FFN_FWD, dev)
    wsb = moe.workspace(cfg, moe.WS_FFN_BWD, dev)
    calls = {"forward": lambda: moe.moe_grouped_swiglu_fwd(cfg, xp, offsets, W1, W2, h, act, yp, wsf),
             "backward": lambda: moe.moe_grouped_swiglu_bwd(cfg, xp, offsets, W1, W2, act, h, dyp, dxp,
                                                            dW1, dW2, wsb)}
    out = {}
    for name, fn in calls.items():
        for _ in range(args.warmup):
            fn()
        moe.gemm_wait_stats()
        for _ in range(args.steps):
            fn()
        st = moe.gemm_wait_stats()
        moe.check_device_error()
        rows = {}
        for kind, v in sorted(st.items()):
            cyc = max(1, v["cta_cycles"])
            rows[str(kind)] = {
                "kernel": wait_kind_name(kind), "ctas": v["ctas"], "kblocks": v["kblocks"],
                "mma_stage_wait": round(v["mma_stage_wait"] / cyc, 3),
                "mma_accumulator_wait": round(v["mma_accumulator_wait"] / cyc, 3),
                "producer_stage_wait": round(v["producer_stage_wait"] / cyc, 3),
                "epilogue_accumulator_wait": round(v["epilogue_accumulator_wait"] / cyc, 3),
                "cta_cycles_per_kblock": round(cyc / max(1, v["kblocks"]), 1)}
        out[name] = rows
    return {"metric": "GEMM pipeline wait fractions (of each kind's CTA cycles)", "unit": "fraction",
            "steps": args.steps, "warmup": args.warmup,
            "data": "synthetic (seeded Gaussian operands; the workload's own routing counts)",
            "config": {"workload": lc.name, "d_model": d, "experts": E, "ffn": f, "N": N},
            "calls": out}


def run_reference(args, lc):
    """The fp64 CPU oracle as the reference arm: each step is the oracle's forward + backward on
    a bounded, seeded sample of the same workload's tokens (all experts)."""
    import torch
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = moe_inputs.make_layer_inputs(lc, seed=args.seed, device=dev)
    host, lc_s = oracle_sample_inputs(lc, inp, args.ref_tokens)
    del inp
    for _ in range(args.warmup):
        time_oracle(lc_s, host)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(lc_s, host)
    dt = time.perf_counter() - t0
    value = args.ref_tokens * args.steps / dt
    sample = (f"{args.ref_tokens} seeded tokens of the workload per step, all {lc.E} experts, "
              f"fp64 numpy {'forward+backward' if lc.backward else 'forward'}")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": lc.name, "T": lc.T, "pass": "fwd+bwd" if lc.backward else "fwd"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=250)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="deepseek", choices=list(moe_inputs.CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    # the oracle's token sample: the same seeded tokens in cpu_baseline and in --impl reference
    ap.add_argument("--cpu-tokens", type=int, default=256)
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 expert comparison")
    ap.add_argument("--no-graph", action="store_true", help="time eager calls, not a CUDA graph")
    ap.add_argument("--fp8", action="store_true",
                    help="time the layer with its experts in FP8 E4M3 (moe_layer_fwd_fp8 / "
                         "moe_layer_bwd_fp8) instead of bf16")
    ap.add_argument("--mxfp8", action="store_true",
                    help="time the layer with MXFP8 routed experts: moe_layer_fwd_mxfp8, and "
                         "moe_layer_bwd_mxfp8 (MXFP8 data gradients, bf16 weight gradients) where "
                         "the configuration has a backward; --mxfp8-forward-only: the forward alone")
    ap.add_argument("--mxfp8-bf16-wgrad", action="store_true",
                    help="with --mxfp8: the routed weight gradients in bf16 instead of MXFP8")
    ap.add_argument("--mxfp8-forward-only", action="store_true",
                    help="with --mxfp8: the step is the forward, also on workloads with a backward")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--route-only", action="store_true",
                    help="time moe_route_topk alone on the workload's tokens (from x through the "
                         "router GEMM, and from given logits); prints its own JSON line")
    ap.add_argument("--wgrad-routings", action="store_true",
                    help="time the routed experts' backward kernels under several per-expert row "
                         "distributions of the workload's shapes; prints its own JSON line")
    ap.add_argument("--wait-stats", action="store_true",
                    help="where the GEMM pipelines wait (a library built with MOE_WAIT_STATS=1); "
                         "prints its own JSON line")
    args = ap.parse_args()
    if args.fp8 and args.mxfp8:
        ap.error("--fp8 and --mxfp8 are exclusive")
    args.warmup = max(args.warmup, 3) if args.impl == "native" else args.warmup
    lc = moe_inputs.CONFIGS[args.workload]
    if args.mxfp8 and args.mxfp8_forward_only:
        lc = lc.replace(backward=False)
    if args.route_only:
        out = run_route_only(args, lc)
    elif args.wgrad_routings:
        out = run_wgrad_routings(args, lc)
    elif args.wait_stats:
        out = run_wait_stats(args, lc)
    else:
        out = run_reference(args, lc) if args.impl == "reference" else run_gpu(args, lc)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
