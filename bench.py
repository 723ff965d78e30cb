#!/usr/bin/env python
"""Benchmark of the B300 MoE expert layer (forward + backward) through the C ABI.

One step = one pass of the whole layer over one batch: router, top-k (or the
balanced gate), expert sort, grouped gate/up GEMM + SwiGLU, grouped down GEMM,
weighted combine, and the full backward (data and weight gradients).  The
default workload is the Qwen3-30B-A3B-shaped layer with the balanced gate:
4096 tokens, hidden 2048, 128 experts, top-8, SwiGLU intermediate 768.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (a bounded token sample of the same workload).

Multi-GPU: the layer runs as independent replicas, one per rank (no
collective on the data path); value = all ranks' tokens / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s fwd & fwd+bwd, 4096-tok Qwen3-30B-A3B shape; % roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ----------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def blas_threads():
    try:
        import threadpoolctl
        n = [i.get("num_threads", 0) for i in threadpoolctl.threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def layer_model(w, counts=None):
    """Algorithmic FLOPs and minimum HBM bytes of one layer call.

    Forward: router GEMM, gate/up and down GEMMs over the S = T*k slots.
    Bytes: x, W_r, every expert weight that received at least one slot, out,
    routing ids/weights and the sorted order.  Forward+backward adds the
    backward GEMMs (2x the forward FLOPs), the saved gate/up pre-activations
    (write + read), a second read of the active expert weights, the weight
    gradients (all experts), grad_out, grad_x, a second read of x and grad W_r.
    """
    T, H, E, k, I, Is = w.T, w.H, w.E, w.k, w.I, w.I_shared
    S = T * k
    e_act = E if counts is None else int(sum(1 for c in counts if c > 0))
    f_fwd = 2.0 * T * H * E + 2.0 * S * H * 2 * I + 2.0 * S * I * H + 2.0 * T * H * 3 * Is
    w_act = e_act * 3.0 * I * H * 2 + 3.0 * Is * H * 2
    b_fwd = T * H * 2 * 2 + E * H * 2 + w_act + T * k * 8 + S * 8 + (E + 1) * 4
    f_fb = 3.0 * f_fwd
    b_fb = (b_fwd + 2 * (S * 2 * I * 2 + T * 2 * Is * 2) + w_act + (E * 3.0 * I * H * 2 + 3.0 * Is * H * 2)
            + T * H * 2 * 3 + E * H * 2)
    return f_fwd, b_fwd, f_fb, b_fb


def kernel_model(name, w, counts, P):
    """Algorithmic (FLOPs, bytes) of one launch of a library kernel."""
    T, H, E, k, I = w.T, w.H, w.E, w.k, w.I
    S = T * k
    e_act = sum(1 for c in counts if c > 0)
    Wgu, Wd = e_act * 2.0 * I * H * 2, e_act * 1.0 * H * I * 2
    nNB = (I + 255) // 256
    table = {
        # router GEMM + softmax + top-k: x and W_r in, ids and weights out
        "router": (2.0 * T * H * E, T * H * 2 + E * H * 2 + S * 8),
        # sort pass: ids in, both maps out
        "route_sort": (0.0, S * 4 * 3),
        "sort_histogram": (0.0, S * 4),
        "sort_scatter": (0.0, S * 4 * 3),
        "gate_up": (2.0 * S * H * 2 * I, Wgu + T * H * 2 + S * 4 + S * I * 2 + S * 2 * I * 2),
        "down": (2.0 * S * I * H, Wd + S * I * 2 + S * H * 2),
        "combine": (2.0 * S * H, S * H * 2 + T * H * 2 + S * 8),
        "dgrad_down": (2.0 * S * H * I, Wd + T * H * 2 + S * 2 * I * 2 + P * 2 * I * 2 + P * I * 2 + P * nNB * 4),
        "dgrad_gate_up": (2.0 * S * 2 * I * H, Wgu + P * 2 * I * 2 + P * H * 2),
        "wgrad_down": (2.0 * S * H * I, T * H * 2 + P * I * 2 + E * H * I * 2.0),
        "wgrad_gate_up": (2.0 * S * 2 * I * H, P * 2 * I * 2 + T * H * 2 + E * 2.0 * I * H * 2),
        "dx_gather": (2.0 * S * H, S * H * 2 + T * H * 2 + E * H * 2),
        "router_wgrad": (2.0 * S * H, T * H * 2 + E * H * 2 + S * 8),
        "gather_rows": (0.0, S * H * 2 + T * H * 2 + S * 4),
        "gather_rows_bwd": (0.0, 2.0 * P * H * 2 + 2 * T * H * 2 + S * 4),
    }
    return table.get(name, (0.0, 0.0))


def measured_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu capture, or None when the
    kernel sources changed since the capture (or no capture covers it)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        h = hashlib.md5()
        for name in ("gemm.cuh", "gemm_res.cuh", "ptx.cuh", "kernels_misc.cuh"):
            with open(os.path.join(ROOT, "grouped_expert_gemm_top_b300", "csrc", name), "rb") as f:
                h.update(f.read())
        k = rec["kernels"].get(kernel)
        if h.hexdigest() != rec["kernel_source_md5"] or not k or k["workload"] != workload:
            return None
        return k["dram_bytes_per_launch"]
    except Exception:
        return None


class _CtypesNvml:
    """Minimal read-only NVML access through libnvidia-ml (when pynvml is absent)."""

    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")

    def nvmlDeviceGetHandleByIndex(self, i):
        h = self.ct.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(self.ct.c_uint(i), self.ct.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByIndex_v2 failed")
        return h

    def nvmlDeviceGetHandleByPciBusId(self, bus):
        h = self.ct.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), self.ct.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByPciBusId_v2 failed")
        return h

    def _clock(self, fn, h, kind):
        v = self.ct.c_uint()
        if fn(h, self.ct.c_int(kind), self.ct.byref(v)) != 0:
            raise RuntimeError("clock query failed")
        return v.value

    def nvmlDeviceGetClockInfo(self, h, kind):
        return self._clock(self.lib.nvmlDeviceGetClockInfo, h, kind)

    def nvmlDeviceGetMaxClockInfo(self, h, kind):
        return self._clock(self.lib.nvmlDeviceGetMaxClockInfo, h, kind)

    def nvmlDeviceGetCurrentClocksThrottleReasons(self, h):
        v = self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, self.ct.byref(v)) != 0:
            raise RuntimeError("reason query failed")
        return v.value


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while running, and
    for `tail_s` after: NVML's clock and reason readings trail the GPU by about
    0.1 s (they change in steps every ~0.1 s), so samples taken only inside a
    region of tens of milliseconds would show the state before it."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index=0, period_s=0.002, tail_s=0.15):
        self.samples, self.reasons, self.ok = [], set(), False
        self.period = period_s
        self.tail = tail_s
        try:
            try:
                import pynvml
                pynvml.nvmlInit()
            except ImportError:
                pynvml = _CtypesNvml()
            self.nv = pynvml
            self.h = None
            try:
                import torch
                p = torch.cuda.get_device_properties(device_index)
                bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
                self.h = pynvml.nvmlDeviceGetHandleByPciBusId(bus)
            except Exception:
                pass
            if self.h is None:
                self.h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.ok = True
        except Exception as e:  # report, then run without clock samples
            sys.stderr.write(f"clock sampler unavailable: {e!r}\n")
            self.max_mhz = None

    def _run(self):
        nv = self.nv
        get_r = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM))
                r = get_r(self.h)
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            time.sleep(self.tail)
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


# ----------------------------------------------------------------- oracle (CPU)
def oracle_step_fn(w, n_tok, seed=0):
    """Returns f() that runs the oracle forward+backward on the first n_tok tokens."""
    import numpy as np
    from grouped_expert_gemm_top_b300 import inputs as G
    from oracle import moe_oracle as O
    inp = G.make_inputs(w, seed, with_grad=True)
    x = O.widen_bf16(inp["x"][:n_tok])
    go = O.widen_bf16(inp["grad_out"][:n_tok])
    wr, wgu, wd = (O.widen_bf16(inp[k]) for k in ("w_router", "w_gate_up", "w_down"))
    bias = None if inp["router_bias"] is None else inp["router_bias"].astype(np.float64)
    sh = {}
    if w.I_shared:
        sh = dict(w_sh_gu=O.widen_bf16(inp["w_sh_gate_up"]), w_sh_down=O.widen_bf16(inp["w_sh_down"]))
    balanced = w.gate == G.GATE_BALANCED

    def step():
        f = O.layer_forward(x, wr, wgu, wd, w.k, balanced=balanced, bias=bias, **sh)
        O.layer_backward(f, go, x, wr, wgu, wd, w.k, **sh)
    return step


def run_reference(args, w, rank):
    if rank != 0:
        return 0
    n_tok = args.ref_tokens
    step = oracle_step_fn(w, n_tok)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        step()
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    mean = sum(times) / len(times)
    value = n_tok / mean
    cores = blas_threads()
    sample = f"first {n_tok} of {w.T} tokens, forward+backward, float64 numpy oracle"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks_ms(v, world):
    """The slowest rank's time (replicas: the job ends when the last one does)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(v)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return float(v)


def job_tokens_per_s(tokens_per_rank_step, world, steps, max_ms):
    """Whole-job throughput: every rank's tokens over the max-over-ranks time."""
    return tokens_per_rank_step * world * steps / (max_ms / 1e3)


def config_of(w, args):
    return {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "I": w.I,
            "I_shared": w.I_shared, "gate": "balanced" if w.gate == 1 else "softmax_topk",
            "router_bias_std": w.bias_std, "step": "forward+backward", "seed": args.seed,
            "l2": "inputs larger than L2: each step streams 1.21 GB of expert weights and "
                  "writes 1.21 GB of weight gradients (L2 126 MB)",
            "parallelism": f"replicas x{args.gpus}",
            "rest_s": args.rest_s}


# ----------------------------------------------------------------- GPU arm
def time_other_shape(name, args, dev, peaks, timed):
    """Forward (inference, no saved pre-activations) and, for a training
    workload, forward+backward of another large workload, each a captured
    CUDA graph replayed args.steps times, with the layer roofline from the
    routing's actual per-expert histogram.  These shapes are not the headline
    (which is the balanced Qwen3 step); they show ragged routing and the
    shared expert."""
    import numpy as np
    import torch
    from grouped_expert_gemm_top_b300 import inputs as G
    from grouped_expert_gemm_top_b300 import moe as M
    from grouped_expert_gemm_top_b300.pipeline import StepGraph

    w = G.WORKLOADS[name]
    inp = G.make_inputs(w, args.seed, with_grad=w.backward)

    def up(b):
        return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)

    x, wr, wgu, wd = (up(inp[k]) for k in ("x", "w_router", "w_gate_up", "w_down"))
    bias = None if inp["router_bias"] is None else torch.from_numpy(inp["router_bias"]).to(dev)
    wsg = up(inp["w_sh_gate_up"]) if w.I_shared else None
    wsd = up(inp["w_sh_down"]) if w.I_shared else None
    weights = dict(w_router=wr, w_gate_up=wgu, w_down=wd, router_bias=bias, w_sh_gate_up=wsg,
                   w_sh_down=wsd)
    dims = (w.T, w.H, w.E, w.k, w.I, w.I_shared)
    res = {"workload": name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "I": w.I,
           "I_shared": w.I_shared, "gate": "balanced" if w.gate == 1 else "softmax_topk",
           "router_bias_std": w.bias_std}
    layer_inf = M.MoeLayer(dims, gate_mode=w.gate, device=dev, with_backward=False)
    fg = StepGraph(layer_inf, None, weights, x)
    torch.cuda.synchronize(dev)
    time.sleep(args.rest_s)   # a burst from a rested GPU, as the headline
    for _ in range(args.warmup):
        fg.replay()
    ms_f = timed(fg.replay, args.steps)
    assert M.moe_read_device_status(layer_inf.workspace) == 0, "device reported an error"
    counts = np.diff(layer_inf.expert_offsets.cpu().numpy())
    del fg, layer_inf
    f_fwd, b_fwd, f_fb, b_fb = layer_model(w, counts)

    def roof(f, b, ms):
        t = ms / 1e3 / args.steps
        t_roof = max(f / (peaks["bf16_tflops"] * 1e12), b / (peaks["hbm_gbs"] * 1e9))
        return {"ms_per_step": ms / args.steps, "tokens_per_s": w.T / t, "t_roof_us": t_roof * 1e6,
                "t_us": t * 1e6, "frac": t_roof / t, "flops": f, "bytes": b,
                "bound": "tensor" if f / (peaks["bf16_tflops"] * 1e12) >= b / (peaks["hbm_gbs"] * 1e9)
                else "hbm"}

    res["active_experts"] = int((counts > 0).sum())
    res["max_load_over_mean"] = float(counts.max() / counts.mean())
    res["fwd"] = roof(f_fwd, b_fwd, ms_f)
    if w.backward:
        go = up(inp["grad_out"])
        layer = M.MoeLayer(dims, gate_mode=w.gate, device=dev, with_backward=True)
        grads = layer.alloc_grads(with_bias=bias is not None)
        sg = StepGraph(layer, grads, weights, x, go)
        torch.cuda.synchronize(dev)
        time.sleep(args.rest_s)
        for _ in range(args.warmup):
            sg.replay()
        ms_fb = timed(sg.replay, args.steps)
        assert M.moe_read_device_status(layer.workspace) == 0, "device reported an error"
        res["fwd_bwd"] = roof(f_fb, b_fb, ms_fb)
        del sg, layer, grads
    del x, wr, wgu, wd, bias, wsg, wsd, weights
    torch.cuda.empty_cache()
    return res


def run_ours(args, w, rank, world):
    import numpy as np
    import torch
    from grouped_expert_gemm_top_b300 import inputs as G
    from grouped_expert_gemm_top_b300 import moe as M

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    M.load_library()   # raises if the CUDA library is missing: no fallback
    inp = G.make_inputs(w, args.seed, with_grad=True)

    def up(b):
        return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)

    x, wr, wgu, wd, go = (up(inp[k]) for k in ("x", "w_router", "w_gate_up", "w_down", "grad_out"))
    bias = None if inp["router_bias"] is None else torch.from_numpy(inp["router_bias"]).to(dev)
    wsg = up(inp["w_sh_gate_up"]) if w.I_shared else None
    wsd = up(inp["w_sh_down"]) if w.I_shared else None
    dims = (w.T, w.H, w.E, w.k, w.I, w.I_shared)
    layer = M.MoeLayer(dims, gate_mode=w.gate, device=dev, with_backward=True)
    grads = layer.alloc_grads(with_bias=bias is not None)
    # forward-only (inference) layer: same calls, no saved pre-activations
    layer_inf = M.MoeLayer(dims, gate_mode=w.gate, device=dev, with_backward=False)
    # activation recompute: the forward keeps no pre-activations, the backward recomputes them
    layer_rc = M.MoeLayer(dims, gate_mode=w.gate, device=dev, with_backward=True, recompute=True)
    grads_rc = layer_rc.alloc_grads(with_bias=bias is not None)
    # with the auxiliary load-balancing loss (alpha = 0.01)
    layer_aux = M.MoeLayer(dims, gate_mode=w.gate, device=dev, with_backward=True, aux_alpha=0.01)
    grads_aux = layer_aux.alloc_grads(with_bias=bias is not None)
    # with an expert capacity of 0.75 x the even share (slots past it are dropped)
    cap_factor = 0.75
    cap = M.expert_capacity(w.T, w.k, w.E, cap_factor)
    layer_cap = M.MoeLayer(dims, gate_mode=w.gate, device=dev, with_backward=True, capacity=cap)
    grads_cap = layer_cap.alloc_grads(with_bias=bias is not None)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        layer.forward(x, wr, wgu, wd, bias, wsg, wsd)

    def fwd_inf():
        layer_inf.forward(x, wr, wgu, wd, bias, wsg, wsd)

    def step():
        fwd()
        layer.backward(go, x, wr, wgu, wd, grads, wsg, wsd)

    def step_rc():
        layer_rc.forward(x, wr, wgu, wd, bias, wsg, wsd)
        layer_rc.backward(go, x, wr, wgu, wd, grads_rc, wsg, wsd)

    def step_aux():
        layer_aux.forward(x, wr, wgu, wd, bias, wsg, wsd)
        layer_aux.backward(go, x, wr, wgu, wd, grads_aux, wsg, wsd)

    def step_cap():
        layer_cap.forward(x, wr, wgu, wd, bias, wsg, wsd)
        layer_cap.backward(go, x, wr, wgu, wd, grads_cap, wsg, wsd)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(v):
        return max_over_ranks_ms(v, world)

    def timed(fn, k):
        barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert M.moe_read_device_status(layer.workspace) == 0, "device reported an error"
    counts = np.diff(layer.expert_offsets.cpu().numpy())
    P_pad = int(sum((int(c) + 127) // 128 * 128 for c in counts))

    # ---- forward + backward (the headline): the step captured once as a CUDA
    # graph and replayed (every kernel of the step runs each time; the graph
    # only takes the host's launch calls out of the loop), no instrumentation
    from grouped_expert_gemm_top_b300.pipeline import StepGraph
    sg = StepGraph(layer, grads, dict(w_router=wr, w_gate_up=wgu, w_down=wd, router_bias=bias,
                                      w_sh_gate_up=wsg, w_sh_down=wsd), x, go)
    # Each headline number is a short burst from a rested GPU: under a
    # continuous load the board reaches its power limit within ~0.1 s and the
    # SM clock drops (the sustained pass below measures that state).
    torch.cuda.synchronize(dev)
    time.sleep(args.rest_s)
    for _ in range(args.warmup):
        sg.replay()
    with ClockSampler(local) as clocks:
        ms_fb = timed(sg.replay, args.steps)
    # ---- forward only (inference: no saved pre-activations), right after the
    # headline and in the same state of the GPU: a captured graph, clocks sampled
    fg = StepGraph(layer_inf, None, dict(w_router=wr, w_gate_up=wgu, w_down=wd, router_bias=bias,
                                         w_sh_gate_up=wsg, w_sh_down=wsd), x)
    torch.cuda.synchronize(dev)
    time.sleep(args.rest_s)
    for _ in range(max(1, args.warmup // 2)):
        fg.replay()
    with ClockSampler(local) as clocks_f:
        ms_f = timed(fg.replay, args.steps)
    assert M.moe_read_device_status(layer_inf.workspace) == 0, "device reported an error"
    # ---- the same step launched call by call (eager)
    ms_fb_eager = timed(step, args.steps)
    # ---- the same steps again with every kernel bracketed by CUDA events on
    # its stream: per-kernel times and the dominant kernel's roofline
    # (a burst from a rested GPU too, after a few untimed steps)
    torch.cuda.synchronize(dev)
    time.sleep(args.rest_s)
    for _ in range(3):
        step()
    M.moe_timing_enable(True)
    M.moe_kernel_stats(reset=True)
    ms_fb_inst = timed(step, args.steps)
    kstats = M.moe_kernel_stats(reset=True)
    M.moe_timing_enable(False)
    # ---- the forward launched call by call
    ms_f_eager = timed(fwd_inf, args.steps)
    assert M.moe_read_device_status(layer_inf.workspace) == 0, "device reported an error"
    # ---- the variants (activation recompute, auxiliary loss, expert
    # capacity), each timed in alternating blocks with the plain step so that
    # the GPU's drift over a run (it slows as it warms) cancels in the
    # comparison: medians of 3 blocks of each
    def paired(fn, lay):
        for _ in range(max(1, args.warmup // 2)):
            fn()
        a, b = [], []
        for _ in range(3):
            a.append(timed(step, args.steps))
            b.append(timed(fn, args.steps))
        assert M.moe_read_device_status(lay.workspace) == 0, "device reported an error"
        return statistics.median(b), statistics.median(a)

    ms_rc, ms_rc_plain = paired(step_rc, layer_rc)
    ms_aux, ms_aux_plain = paired(step_aux, layer_aux)
    ms_cap, ms_cap_plain = paired(step_cap, layer_cap)
    kept = int(np.minimum(np.diff(layer_cap.expert_offsets.cpu().numpy()), cap).sum())
    # ---- graph replay against the eager step, in alternating blocks
    ms_graph, ms_graph_plain = paired(sg.replay, layer)
    # ---- sustained: the plain step for ~3 s (the GPU's steady state under
    # its power limit), clocks sampled meanwhile
    n_sus = max(args.steps, int(args.sustain_s * 1e3 / (ms_fb / args.steps)))
    ms_sus, clocks_sus = None, None
    if args.sustain_s > 0:
        with ClockSampler(local) as clocks_sus:
            ms_sus = timed(sg.replay, n_sus)   # the headline's step, replayed for seconds

    # ---- end to end: pinned host inputs in, result out, every step
    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    goh = torch.empty(go.shape, dtype=go.dtype, pin_memory=True)
    xh.copy_(x)
    goh.copy_(go)
    outh = torch.empty(layer.out.shape, dtype=layer.out.dtype, pin_memory=True)
    gxh = torch.empty(grads["grad_x"].shape, dtype=torch.bfloat16, pin_memory=True)

    # serial: copy in, compute, copy out, one after the other on one stream
    def e2e_serial_step():
        x.copy_(xh, non_blocking=True)
        go.copy_(goh, non_blocking=True)
        step()
        outh.copy_(layer.out, non_blocking=True)
        gxh.copy_(grads["grad_x"], non_blocking=True)

    for _ in range(2):
        e2e_serial_step()
    ms_e2e_serial = timed(e2e_serial_step, args.steps)
    # pipelined: step i+1's inputs go up and step i-1's results come back on
    # their own streams while step i computes (every copy still made per step)
    from grouped_expert_gemm_top_b300.pipeline import HostStepPipeline
    pipe = HostStepPipeline(layer, grads, dict(w_router=wr, w_gate_up=wgu, w_down=wd,
                                               router_bias=bias, w_sh_gate_up=wsg, w_sh_down=wsd))

    def e2e_pipelined(k):
        for _ in range(k):
            pipe.step(xh, goh, outh, gxh)
        pipe.drain()

    e2e_pipelined(3)
    torch.cuda.synchronize(dev)
    time.sleep(args.rest_s)
    e2e_pipelined(3)
    ms_e2e = timed(lambda: e2e_pipelined(args.steps), 1)   # all K steps and the last read-back
    assert M.moe_read_device_status(layer.workspace) == 0, "device reported an error"
    h2d = pipe.h2d_bytes_per_step
    d2h = pipe.d2h_bytes_per_step

    # ---- the other large workloads: the skewed router (ragged expert tiles,
    # forward) and the shared-expert shape (forward and forward+backward)
    peaks, peak_src = load_peaks()
    other = {}
    if not args.no_other_shapes:
        for name in ("qwen3_30b_a3b_skewed", "shared_expert_skewed"):
            if name != w.name:
                other[name] = time_other_shape(name, args, dev, peaks, timed)

    value = job_tokens_per_s(w.T, world, args.steps, ms_fb)
    fwd_value = job_tokens_per_s(w.T, world, args.steps, ms_f)
    e2e_value = job_tokens_per_s(w.T, world, args.steps, ms_e2e)

    f_fwd, b_fwd, f_fb, b_fb = layer_model(w, counts)
    t_roof_f = max(f_fwd / (peaks["bf16_tflops"] * 1e12), b_fwd / (peaks["hbm_gbs"] * 1e9))
    t_roof_fb = max(f_fb / (peaks["bf16_tflops"] * 1e12), b_fb / (peaks["hbm_gbs"] * 1e9))
    t_f = ms_f / 1e3 / args.steps
    t_fb = ms_fb / 1e3 / args.steps

    kernels = {}
    for name, (n, ms) in kstats.items():
        if n:
            kernels[name] = {"launches": n, "avg_us": ms * 1e3 / n, "share": None}
    tot = sum(v["avg_us"] * v["launches"] for v in kernels.values())
    for v in kernels.values():
        v["share"] = v["avg_us"] * v["launches"] / tot if tot else None
    top = max(kernels, key=lambda n: kernels[n]["avg_us"] * kernels[n]["launches"])
    F, B = kernel_model(top, w, counts, P_pad)
    t_k = kernels[top]["avg_us"] / 1e6
    bound = "tensor" if F / (peaks["bf16_tflops"] * 1e12) >= B / (peaks["hbm_gbs"] * 1e9) else "hbm"
    if bound == "tensor":
        achieved, peak, unit = F / t_k / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = B / t_k / 1e9, peaks["hbm_gbs"], "GB/s"
    roofline = {"kernel": top, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": measured_traffic(top, w.name),
                "peak_source": peak_src,
                "algorithmic_flops": F, "algorithmic_bytes": B, "avg_us": kernels[top]["avg_us"]}
    per_kernel_roof = {}
    for name, v in kernels.items():
        F_, B_ = kernel_model(name, w, counts, P_pad)
        if F_ == 0 and B_ == 0:
            continue
        t_roof_k = max(F_ / (peaks["bf16_tflops"] * 1e12), B_ / (peaks["hbm_gbs"] * 1e9))
        per_kernel_roof[name] = round(t_roof_k / (v["avg_us"] / 1e6), 4)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_tok = args.cpu_tokens
        stepc = oracle_step_fn(w, n_tok, args.seed)
        t0 = time.perf_counter()
        stepc()
        dt = time.perf_counter() - t0
        cpu = {"value": n_tok / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"first {n_tok} of {w.T} tokens of the same workload, forward+backward "
                         f"once, float64 numpy oracle ({dt:.1f} s)"}

    gpu_launches = sum(n for n, _ in kstats.values())
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_fb / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_of(w, args),
        "fwd_tokens_per_s": fwd_value, "fwd_ms_per_step": ms_f / args.steps,
        "fwd_clocks": clocks_f.summary(),
        # the headline steps again with per-kernel CUDA events (source of `kernels`)
        "ms_per_step_instrumented": ms_fb_inst / args.steps,
        # forward+backward with activation recompute: the forward keeps no gate/up
        # pre-activations (S*2I bf16), the backward reruns the gate/up GEMM
        "recompute": {"tokens_per_s": job_tokens_per_s(w.T, world, args.steps, ms_rc),
                      "ms_per_step": ms_rc / args.steps,
                      "plain_ms_per_step_adjacent": ms_rc_plain / args.steps,
                      "saved_bytes_not_held": w.T * w.k * 2 * w.I * 2 + w.T * 2 * w.I_shared * 2,
                      "extra_flops": 2.0 * w.T * w.k * w.H * 2 * w.I + 2.0 * w.T * w.H * 2 * w.I_shared},
        # forward+backward with the auxiliary load-balancing loss (alpha 0.01): its value
        # on the device, and the step time with its dense router gradient
        "aux_loss": {"tokens_per_s": job_tokens_per_s(w.T, world, args.steps, ms_aux),
                     "ms_per_step": ms_aux / args.steps,
                     "plain_ms_per_step_adjacent": ms_aux_plain / args.steps,
                     "value": float(layer_aux.aux_loss.item()), "alpha": 0.01},
        # forward+backward with an expert capacity (token dropping)
        "capacity": {"factor": cap_factor, "capacity": cap,
                     "dropped_fraction": 1.0 - kept / (w.T * w.k),
                     "tokens_per_s": job_tokens_per_s(w.T, world, args.steps, ms_cap),
                     "ms_per_step": ms_cap / args.steps,
                     "plain_ms_per_step_adjacent": ms_cap_plain / args.steps},
        # the headline step is a CUDA-graph replay; the same step launched call
        # by call right after it, and the two in alternating blocks
        "eager": {"tokens_per_s": job_tokens_per_s(w.T, world, args.steps, ms_fb_eager),
                  "ms_per_step": ms_fb_eager / args.steps,
                  "fwd_ms_per_step": ms_f_eager / args.steps,
                  "graph_vs_eager_adjacent_ms": [ms_graph / args.steps, ms_graph_plain / args.steps]},
        # the plain step repeated for ~3 s: steady-state rate and clocks
        "sustained": None if ms_sus is None else {
            "steps": n_sus, "seconds": ms_sus / 1e3,
            "tokens_per_s": job_tokens_per_s(w.T, world, n_sus, ms_sus),
            "ms_per_step": ms_sus / n_sus, "clocks": clocks_sus.summary()},
        "layer_roofline": {
            "fwd": {"t_roof_us": t_roof_f * 1e6, "t_us": t_f * 1e6, "frac": t_roof_f / t_f,
                    "flops": f_fwd, "bytes": b_fwd},
            "fwd_bwd": {"t_roof_us": t_roof_fb * 1e6, "t_us": t_fb * 1e6, "frac": t_roof_fb / t_fb,
                        "flops": f_fb, "bytes": b_fb},
            "peaks": peaks, "peak_source": peak_src},
        "roofline": roofline,
        "kernel_roofline_frac": per_kernel_roof,
        # other workloads, each with its own layer roofline from its histogram
        "other_shapes": other,
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                # copies overlapped with compute on their own streams; the same
                # steps with copy-in, compute and copy-out strictly in sequence:
                "serial_value": job_tokens_per_s(w.T, world, args.steps, ms_e2e_serial)},
        "gpu_launches": gpu_launches,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_30b_a3b_balanced_fwd_bwd")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-tokens", type=int, default=2048)
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-shapes", action="store_true",
                    help="skip timing the skewed-router and shared-expert workloads")
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of the extra steady-state pass (0: no such pass)")
    ap.add_argument("--rest-s", type=float, default=1.0,
                    help="idle seconds before each headline measurement (forward+backward, "
                         "forward, per-kernel times, end to end), so that each is a burst "
                         "from a rested GPU")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from grouped_expert_gemm_top_b300 import inputs as G
    w = G.WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    if args.impl == "reference":
        rc = run_reference(args, w, rank)
    else:
        rc = run_ours(args, w, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
