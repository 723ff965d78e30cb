"""The host-fed step pipeline against plain steps.

Copies overlapped with compute must not change a bit of any step's results:
five steps with different host inputs through the pipeline give the same
out and grad_x per step, and the same weight gradients after the last step,
as the same steps run one after the other on one stream.
"""

import numpy as np
import pytest
import torch

import gpu_util as U
from grouped_expert_gemm_top_b300 import inputs as G
from grouped_expert_gemm_top_b300 import moe as M
from grouped_expert_gemm_top_b300.pipeline import HostStepPipeline

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shared,use_graph", [(False, False), (False, True), (True, True)])
def test_pipelined_steps_match_plain_steps(shared, use_graph):
    w = G.Workload("pipe", T=320, H=256, E=8, k=2, I=192, I_shared=128 if shared else 0, bias_std=0.5)
    di = U.DeviceInputs(w, seed=5, with_grad=True)
    weights = dict(w_router=di.w_router, w_gate_up=di.w_gate_up, w_down=di.w_down,
                   router_bias=di.router_bias, w_sh_gate_up=di.w_sh_gate_up, w_sh_down=di.w_sh_down)
    r = np.random.default_rng(9)
    steps = []
    for _ in range(5):   # every slot reused twice
        x = torch.from_numpy(r.normal(size=(w.T, w.H)).astype(np.float32)).to(torch.bfloat16)
        go = torch.from_numpy(r.normal(size=(w.T, w.H)).astype(np.float32)).to(torch.bfloat16)
        steps.append((x.pin_memory(), go.pin_memory()))

    # plain: copy in, compute, copy out, one stream
    plain = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True)
    pg = plain.alloc_grads(with_bias=True)
    ref = []
    for xh, goh in steps:
        x, go = xh.cuda(), goh.cuda()
        plain.forward(x, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                      di.w_sh_down)
        plain.backward(go, x, di.w_router, di.w_gate_up, di.w_down, pg, di.w_sh_gate_up, di.w_sh_down)
        ref.append((plain.out.cpu(), pg["grad_x"].cpu()))
    torch.cuda.synchronize()

    layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True)
    grads = layer.alloc_grads(with_bias=True)
    pipe = HostStepPipeline(layer, grads, weights, use_graph=use_graph)
    outs = [(torch.empty(w.T, w.H, dtype=torch.bfloat16).pin_memory(),
             torch.empty(w.T, w.H, dtype=torch.bfloat16).pin_memory()) for _ in steps]
    for (xh, goh), (oh, gh) in zip(steps, outs):
        pipe.step(xh, goh, oh, gh)
    pipe.drain()
    torch.cuda.synchronize()
    assert M.moe_read_device_status(layer.workspace) == 0
    for (o_ref, g_ref), (oh, gh) in zip(ref, outs):
        assert torch.equal(oh, o_ref)
        assert torch.equal(gh, g_ref)
    for key, v in pg.items():
        if v is not None and key != "grad_x":
            assert torch.equal(grads[key], v), key
    assert pipe.h2d_bytes_per_step == 2 * w.T * w.H * 2


@pytest.mark.parametrize("shared", [False, True])
def test_graph_replay_matches_eager_steps(shared):
    """A captured step replayed on new inputs gives the eager step's bits."""
    from grouped_expert_gemm_top_b300.pipeline import StepGraph
    w = G.Workload("graph", T=300, H=256, E=8, k=2, I=192, I_shared=128 if shared else 0, bias_std=0.5)
    di = U.DeviceInputs(w, seed=6, with_grad=True)
    weights = dict(w_router=di.w_router, w_gate_up=di.w_gate_up, w_down=di.w_down,
                   router_bias=di.router_bias, w_sh_gate_up=di.w_sh_gate_up, w_sh_down=di.w_sh_down)
    layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True)
    grads = layer.alloc_grads(with_bias=True)
    x = torch.empty_like(di.x)
    go = torch.empty_like(di.grad_out)
    x.copy_(di.x)
    go.copy_(di.grad_out)
    g = StepGraph(layer, grads, weights, x, go)
    eager = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True)
    eg = eager.alloc_grads(with_bias=True)
    r = np.random.default_rng(2)
    for _ in range(2):
        xn = torch.from_numpy(r.normal(size=(w.T, w.H)).astype(np.float32)).to(torch.bfloat16).cuda()
        gn = torch.from_numpy(r.normal(size=(w.T, w.H)).astype(np.float32)).to(torch.bfloat16).cuda()
        x.copy_(xn)
        go.copy_(gn)
        g.replay()
        eager.forward(xn, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                      di.w_sh_down)
        eager.backward(gn, xn, di.w_router, di.w_gate_up, di.w_down, eg, di.w_sh_gate_up, di.w_sh_down)
        torch.cuda.synchronize()
        assert M.moe_read_device_status(layer.workspace) == 0
        assert torch.equal(layer.out, eager.out)
        for key, v in eg.items():
            if v is not None:
                assert torch.equal(grads[key], v), key


def test_forward_only_graph_matches_eager_forward():
    from grouped_expert_gemm_top_b300.pipeline import StepGraph
    w = G.Workload("graph_fwd", T=300, H=256, E=8, k=2, I=192, bias_std=0.5)
    di = U.DeviceInputs(w, seed=8, with_grad=False)
    weights = dict(w_router=di.w_router, w_gate_up=di.w_gate_up, w_down=di.w_down,
                   router_bias=di.router_bias)
    layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=False)
    x = di.x.clone()
    g = StepGraph(layer, None, weights, x)
    eager = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=False)
    xn = (di.x.float() * -1.5).to(torch.bfloat16)
    x.copy_(xn)
    g.replay()
    eager.forward(xn, di.w_router, di.w_gate_up, di.w_down, di.router_bias)
    torch.cuda.synchronize()
    assert torch.equal(layer.out, eager.out)
    assert torch.equal(layer.topk_idx, eager.topk_idx)
