"""Seeded synthetic inputs for the MoE expert layer.

This module holds no arithmetic of the layer itself: it only draws random
numbers, rounds them to bfloat16 bit patterns and names the workload shapes.
Both the CPU oracle (through the tests) and the CUDA path are fed from here.

Every bf16 tensor is returned as a ``numpy.uint16`` array of raw bfloat16 bits
(round-to-nearest-even from an fp32 normal draw).  Router biases are fp32.

Workloads
---------
The pages measure fine-tuning on "random dummy tokens" at sequence length 4096
and local batch 1 (NeMo AutoModel blog, "单节点30B MoE基准测试 / single-node
30B MoE benchmark" method table).  No dataset is involved; the shapes below
stand in for it:

* ``tiny``: 256 tokens, hidden 256, 8 experts, top-2 softmax router with
  renormalised weights, SwiGLU intermediate 512, x / W ~ N(0, 0.02).
* ``qwen3_30b_a3b_balanced``: Qwen3-30B-A3B-shaped layer (4096 tokens,
  hidden 2048, 128 experts, top-8, intermediate 768) with the balanced gate,
  i.e. exactly 256 token-slots per expert.
* ``qwen3_30b_a3b_skewed``: same shape, softmax top-8 over
  ``x W_r^T + b`` with ``b ~ N(0, 1.5)`` per expert (skewed, some experts empty).
* ``shared_expert_skewed``: 8192 tokens (seq 4096 x batch 2), hidden 2688,
  128 experts, top-6, intermediate 1856, plus one always-on shared expert of
  intermediate 3712, skewed router.

x is drawn N(0, 1) for the large shapes and N(0, 0.02) for ``tiny``; expert
and router weights are N(0, 0.02); grad_out is N(0, 1).
"""

from __future__ import annotations

import dataclasses
import os

import numpy as np

GATE_SOFTMAX_TOPK = 0
GATE_BALANCED = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    I_shared: int = 0
    gate: int = GATE_SOFTMAX_TOPK
    x_std: float = 1.0
    w_std: float = 0.02
    bias_std: float = 0.0  # 0 -> no router bias
    backward: bool = False

    @property
    def S(self) -> int:
        return self.T * self.k

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=256, E=8, k=2, I=512, x_std=0.02),
    "qwen3_30b_a3b_balanced": Workload(
        "qwen3_30b_a3b_balanced", T=4096, H=2048, E=128, k=8, I=768,
        gate=GATE_BALANCED),
    "qwen3_30b_a3b_skewed": Workload(
        "qwen3_30b_a3b_skewed", T=4096, H=2048, E=128, k=8, I=768,
        bias_std=1.5),
    "qwen3_30b_a3b_balanced_fwd_bwd": Workload(
        "qwen3_30b_a3b_balanced_fwd_bwd", T=4096, H=2048, E=128, k=8, I=768,
        gate=GATE_BALANCED, backward=True),
    # same per-expert shape with 32 experts and 1024 tokens (256 slots per expert):
    # a smaller case for counter captures whose expert weights still exceed L2
    "qwen3_30b_a3b_balanced_32experts_1024tok": Workload(
        "qwen3_30b_a3b_balanced_32experts_1024tok", T=1024, H=2048, E=32, k=8, I=768,
        gate=GATE_BALANCED, backward=True),
    "shared_expert_skewed": Workload(
        "shared_expert_skewed", T=8192, H=2688, E=128, k=6, I=1856,
        I_shared=3712, bias_std=1.5, backward=True),
}

# Stream ids keep every tensor's draw independent of the others.
_STREAM = {"x": 1, "w_router": 2, "router_bias": 3, "w_gate_up": 4,
           "w_down": 5, "w_sh_gate_up": 6, "w_sh_down": 7, "grad_out": 8}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); return raw bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of raw bfloat16 bits to fp32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


_CHUNK = 1 << 22  # elements per independently seeded chunk


def _rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), _STREAM[stream]])


def normal_bf16(shape, std: float, seed: int, stream: str) -> np.ndarray:
    """N(0, std^2) draws rounded to bf16 bits.

    The flat tensor is cut into fixed chunks of 2^22 values; chunk c is drawn
    from its own generator seeded with (seed, stream, c), so the result does
    not depend on how many threads draw it.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def one(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.default_rng([int(seed), _STREAM[stream], c])
        out[lo:hi] = f32_to_bf16_bits(g.standard_normal(size=hi - lo, dtype=np.float32) * np.float32(std))

    if nchunks <= 1:
        for c in range(nchunks):
            one(c)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1)) as ex:
            list(ex.map(one, range(nchunks)))
    return out.reshape(shape)


def make_inputs(w: Workload, seed: int = 0, with_grad: bool | None = None) -> dict:
    """All inputs of one layer call as numpy arrays (bf16 as uint16 bits).

    Keys: x [T,H], w_router [E,H], router_bias [E] fp32 or None,
    w_gate_up [E,2I,H] (gate rows first, then up rows), w_down [E,H,I],
    w_sh_gate_up [2I_sh,H] / w_sh_down [H,I_sh] or None, grad_out [T,H] or None.
    """
    if with_grad is None:
        with_grad = w.backward
    d = {
        "x": normal_bf16((w.T, w.H), w.x_std, seed, "x"),
        "w_router": normal_bf16((w.E, w.H), w.w_std, seed, "w_router"),
        "w_gate_up": normal_bf16((w.E, 2 * w.I, w.H), w.w_std, seed, "w_gate_up"),
        "w_down": normal_bf16((w.E, w.H, w.I), w.w_std, seed, "w_down"),
        "router_bias": None,
        "w_sh_gate_up": None,
        "w_sh_down": None,
        "grad_out": None,
    }
    if w.bias_std > 0:
        d["router_bias"] = (_rng(seed, "router_bias").standard_normal(
            size=(w.E,), dtype=np.float32) * np.float32(w.bias_std))
    if w.I_shared > 0:
        d["w_sh_gate_up"] = normal_bf16((2 * w.I_shared, w.H), w.w_std, seed, "w_sh_gate_up")
        d["w_sh_down"] = normal_bf16((w.H, w.I_shared), w.w_std, seed, "w_sh_down")
    if with_grad:
        d["grad_out"] = normal_bf16((w.T, w.H), 1.0, seed, "grad_out")
    return d
