"""Cross-kernel overlap (the down GEMM starting on the SMs the gate/up GEMM
frees, the gate/up data gradient on those the down data gradient frees): a
consumer unit must read its rows only after the producer kernel has written
them.

Each unit of the consumer waits for a count of finished producer units on its
256-row block; units are handed out in the order the CTAs ask for them, so the
timing differs from run to run.  A unit that read its rows too early would
read stale or partial rows and change the result, so every step here must
reproduce the first one bit for bit (outputs, saved pre-activations, every
gradient), over many steps, replayed from a captured graph and launched call
by call, at the full Qwen3 shape and at a ragged one.  The values themselves
are checked against the oracle by the parity tests.
"""

import numpy as np
import pytest
import torch

import gpu_util as U
from grouped_expert_gemm_top_b300 import inputs as G
from grouped_expert_gemm_top_b300 import moe as M
from grouped_expert_gemm_top_b300.pipeline import StepGraph

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _snapshot(layer, grads):
    ts = [layer.out, layer.y_perm, layer.gu_saved, layer.topk_w, layer.slot_perm]
    ts += [grads[k] for k in sorted(grads) if grads[k] is not None]
    return [_bits(t).clone() for t in ts if t is not None]


@pytest.mark.parametrize("name,steps", [("qwen3_30b_a3b_balanced_fwd_bwd", 24),
                                        ("qwen3_30b_a3b_skewed", 12)])
def test_overlapped_steps_are_bit_identical(name, steps):
    w = G.WORKLOADS[name]
    di = U.DeviceInputs(w, seed=0, with_grad=True)
    layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True)
    grads = layer.alloc_grads(with_bias=di.router_bias is not None)
    weights = dict(w_router=di.w_router, w_gate_up=di.w_gate_up, w_down=di.w_down,
                   router_bias=di.router_bias)

    def eager():
        layer.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias)
        layer.backward(di.grad_out, di.x, di.w_router, di.w_gate_up, di.w_down, grads)

    eager()
    torch.cuda.synchronize()
    assert M.moe_read_device_status(layer.workspace) == 0
    ref = _snapshot(layer, grads)
    g = StepGraph(layer, grads, weights, di.x, di.grad_out)
    for i in range(steps):
        if i % 3 == 2:
            eager()
        else:
            g.replay()
        torch.cuda.synchronize()
        got = _snapshot(layer, grads)
        for j, (a, b) in enumerate(zip(ref, got)):
            assert torch.equal(a, b), (i, j)
    assert M.moe_read_device_status(layer.workspace) == 0


@pytest.mark.parametrize("name", ["qwen3_30b_a3b_balanced", "qwen3_30b_a3b_skewed"])
def test_overlapped_forward_only_is_bit_identical(name):
    """The inference forward (no saved pre-activations) repeated, against its
    first run and against the training forward's output; the skewed routing
    also runs the gate/up GEMM's narrow units."""
    w = G.WORKLOADS[name]
    di = U.DeviceInputs(w, seed=2, with_grad=False)
    inf = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=False)
    tr = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True)
    tr.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias)
    outs = []
    for _ in range(16):
        inf.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias)
        torch.cuda.synchronize()
        outs.append((_bits(inf.out).clone(), _bits(inf.y_perm).clone()))
    for o, y in outs:
        assert torch.equal(o, _bits(tr.out))
        assert torch.equal(y, _bits(tr.y_perm))
    assert M.moe_read_device_status(inf.workspace) == 0
