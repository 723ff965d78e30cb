"""Degenerate shapes and feature combinations, whole layer against the oracle.

Each case runs forward+backward on the device and compares every output and
gradient with the float64 oracle on the device's routing: one token; one
expert (the layer is a dense SwiGLU MLP); every token to every expert (k = E);
the smallest hidden and intermediate sizes; one expert receiving almost every
token; 160000 token-slots; 128, 200 and 256 experts; and the optional features together (capacity with the auxiliary loss;
activation recompute with capacity and a shared expert).
"""

import numpy as np
import pytest
import torch

import gpu_util as U
from grouped_expert_gemm_top_b300 import inputs as G
from grouped_expert_gemm_top_b300 import moe as M
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

W = G.Workload
EDGE = {
    "one_token": W("one_token", T=1, H=128, E=4, k=2, I=128, bias_std=0.5),
    "one_expert": W("one_expert", T=200, H=128, E=1, k=1, I=192),
    "k_equals_E": W("k_equals_E", T=150, H=128, E=4, k=4, I=128, bias_std=0.5),
    "smallest_dims": W("smallest_dims", T=130, H=64, E=3, k=2, I=64, bias_std=0.5),
    "one_hot_expert": W("one_hot_expert", T=600, H=128, E=8, k=2, I=128, bias_std=6.0),
    # 160000 slots: the multi-block sort and row indices past 2^17 through the whole layer
    "many_tokens": W("many_tokens", T=20000, H=128, E=64, k=8, I=128, bias_std=0.5),
    # more than 128 experts: the router kernel's 256-wide tile (8 experts a lane)
    # and the router weight gradient's split-K path (the cluster kernel takes
    # at most 128 experts); exactly 128 and 256 at the limits
    "experts_200": W("experts_200", T=700, H=192, E=200, k=6, I=128, bias_std=0.5),
    "experts_128": W("experts_128", T=300, H=320, E=128, k=8, I=128, bias_std=0.5),
    "experts_256": W("experts_256", T=400, H=128, E=256, k=8, I=128, bias_std=0.5),
}


def _run(w, seed=7, **layer_kw):
    di = U.DeviceInputs(w, seed=seed, with_grad=True)
    layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True, save_logits=True, **layer_kw)
    layer.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                  di.w_sh_down)
    grads = layer.alloc_grads(with_bias=w.bias_std > 0)
    layer.backward(di.grad_out, di.x, di.w_router, di.w_gate_up, di.w_down, grads,
                   di.w_sh_gate_up, di.w_sh_down)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(layer.workspace) == 0
    return di, layer, grads


def _check_all(di, layer, grads, capacity=None, aux_coef=None, gu_layer=None):
    """Routing bit-exact, out and every gradient against the oracle.  gu_layer:
    the layer whose saved (g, u) the bias check uses (default: this one)."""
    w = di.w
    idx = layer.topk_idx.cpu().numpy()
    off, perm, inv = O.permute(idx, w.E)
    keep = O.keep_slots(idx, w.E, capacity)
    assert np.array_equal(layer.expert_offsets.cpu().numpy(), off)
    assert np.array_equal(layer.perm_slot.cpu().numpy(), perm)
    assert np.array_equal(layer.slot_perm.cpu().numpy(), np.where(keep.ravel(), inv, -1))
    f = U.oracle_forward(di, topk_idx=idx, capacity=capacity)
    U.check_close(layer.out, f["out"], "out")
    b = O.layer_backward(f, di.f64("grad_out"), di.f64("x"), di.f64("w_router"),
                         di.f64("w_gate_up"), di.f64("w_down"), w.k,
                         w_sh_gu=di.f64("w_sh_gate_up"), w_sh_down=di.f64("w_sh_down"),
                         aux_coef=aux_coef)
    for key, got in grads.items():
        if got is None:
            continue
        ref = b[key]
        if not np.any(ref):          # e.g. the router gradient of a one-expert layer
            assert torch.count_nonzero(got) == 0, key
        elif key == "grad_router_bias":
            gu = (gu_layer or layer).gu_saved
            U.check_bias_grad(got, di, f, gu, aux_coef=aux_coef)
        else:
            U.check_close(got, ref, key)
    return f, b


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_shapes_forward_backward(name):
    di, layer, grads = _run(EDGE[name])
    f, b = _check_all(di, layer, grads)
    w = di.w
    counts = np.diff(layer.expert_offsets.cpu().numpy())
    if name == "one_expert":
        assert counts.tolist() == [w.T]
    if name == "k_equals_E":
        assert np.array_equal(counts, np.full(w.E, w.T))
    if name == "one_hot_expert":
        assert counts.max() >= 0.4 * w.T * w.k   # one expert takes most slots (several row tiles)


def test_capacity_with_auxiliary_loss():
    w = W("cap_aux", T=300, H=192, E=6, k=3, I=320, bias_std=0.8)
    C = M.expert_capacity(w.T, w.k, w.E, 0.7)
    alpha = w.T / 4.0
    di, layer, grads = _run(w, capacity=C, aux_alpha=alpha)
    idx = layer.topk_idx.cpu().numpy()
    p_dev = O.softmax(U.to_f64(layer.logits))
    L_ref, c_ref = O.aux_loss(p_dev, idx, alpha)       # counts before dropping
    assert abs(float(layer.aux_loss.item()) - L_ref) <= 1e-5 * max(1.0, abs(L_ref))
    _check_all(di, layer, grads, capacity=C, aux_coef=c_ref)


def test_recompute_with_capacity_and_shared_expert():
    w = W("rc_cap_sh", T=260, H=128, E=5, k=2, I=192, I_shared=256, bias_std=0.8)
    C = M.expert_capacity(w.T, w.k, w.E, 0.8)
    di, layer, grads = _run(w, capacity=C, recompute=True)
    assert layer.gu_saved is None
    # the saved-pre-activation run with the same capacity gives the (g, u)
    # that the recompute forms again
    _, layer2, grads2 = _run(w, capacity=C)
    _check_all(di, layer, grads, capacity=C, gu_layer=layer2)
    # and bit-identical to that run's backward
    for key, v in grads.items():
        if v is not None:
            assert torch.equal(v, grads2[key]), key
