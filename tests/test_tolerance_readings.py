"""Why the router bias gradient is compared on the device's own (g, u) (no GPU).

The bias gradient db[e] = sum_t dlogit[t, e] cancels twice (within each
token's k selected slots, then across tokens), so a single bf16 rounding of
the gate/up pre-activations, which the device saves and differentiates
through, can move it by more than the common bf16 tolerance while every other
gradient stays far inside it.  These tests show that on the oracle alone and
check that the helper the GPU tests use adds no arithmetic of its own: given
the oracle's own (g, u) it reproduces the oracle's backward exactly.
"""

import numpy as np
import torch

import gpu_util as U
from grouped_expert_gemm_top_b300 import inputs as G
from oracle import moe_oracle as O

# a case whose bias gradient is small against its terms (seed 2 of the ragged
# shared-expert parity case)
W = G.Workload("ragged_shared", T=200, H=128, E=5, k=2, I=192, I_shared=320, bias_std=0.5)
SEED = 2


class HostInputs(U.DeviceInputs):
    """The seeded inputs' float64 copies only (no device upload)."""

    def __init__(self, w, seed):
        self.w = w
        self.np = G.make_inputs(w, seed, True)
        self._f64 = {}


def _oracle(di):
    f = U.oracle_forward(di)
    b = O.layer_backward(f, di.f64("grad_out"), di.f64("x"), di.f64("w_router"),
                         di.f64("w_gate_up"), di.f64("w_down"), di.w.k,
                         w_sh_gu=di.f64("w_sh_gate_up"), w_sh_down=di.f64("w_sh_down"))
    return f, b


def test_device_gu_helper_is_the_oracle_on_exact_gu():
    di = HostInputs(W, SEED)
    f, b = _oracle(di)
    b2 = U.oracle_backward_with_device_gu(di, f, torch.from_numpy(f["gu_perm"]))
    for key, ref in b.items():
        assert np.allclose(b2[key], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), key


def test_one_bf16_rounding_of_gu_moves_only_the_bias_gradient_past_tolerance():
    di = HostInputs(W, SEED)
    f, b = _oracle(di)
    gu16 = torch.from_numpy(f["gu_perm"]).to(torch.bfloat16)
    b2 = U.oracle_backward_with_device_gu(di, f, gu16)
    rel = {key: np.linalg.norm(b2[key] - b[key]) / np.linalg.norm(b[key])
           for key in ("grad_x", "grad_w_router", "grad_w_gate_up", "grad_w_down",
                       "grad_router_bias")}
    assert rel["grad_router_bias"] > U.REL_L2, rel
    for key in ("grad_x", "grad_w_router", "grad_w_gate_up", "grad_w_down"):
        assert rel[key] < 0.5 * U.REL_L2, (key, rel)
    # the cancellation: |db| is a small fraction of sum_t |dlogit|
    dl = b["grad_logits"]
    assert np.abs(dl.sum(axis=0)).min() < 0.05 * np.abs(dl).sum(axis=0).max()


# ---------------------------------------------------------------------------
# The bound the GPU tests put on the bias gradient against the plain oracle
# (gpu_util.bias_grad_bound): it must hold for the one bf16 rounding of g, u
# the device makes, and be tight enough that plausible mistakes exceed it.

BOUND_CASES = [
    G.Workload("tiny_bias", T=256, H=256, E=8, k=2, I=512, bias_std=0.5, x_std=0.02),
    G.Workload("ragged", T=300, H=192, E=6, k=3, I=320, bias_std=0.5),
    G.Workload("ragged_shared", T=200, H=128, E=5, k=2, I=192, I_shared=320, bias_std=0.5),
    G.Workload("skewed_small", T=512, H=256, E=16, k=4, I=256, bias_std=1.5),
    G.Workload("wide_k", T=256, H=256, E=32, k=12, I=192, bias_std=0.5),
]


def _rounded_gu_case(w, seed, capacity=None, aux_alpha=None):
    di = HostInputs(w, seed)
    f = U.oracle_forward(di, capacity=capacity)
    c = None
    if aux_alpha is not None:
        _, c = O.aux_loss(f["p"], f["topk_idx"], aux_alpha)
    b = O.layer_backward(f, di.f64("grad_out"), di.f64("x"), di.f64("w_router"),
                         di.f64("w_gate_up"), di.f64("w_down"), w.k, aux_coef=c)
    gu16 = torch.from_numpy(f["gu_perm"]).to(torch.bfloat16)
    b2 = U.oracle_backward_with_device_gu(di, f, gu16, aux_coef=c)
    bound = U.bias_grad_bound(di, f, b["grad_logits"], aux_coef=c)
    return di, f, b, b2, bound


def test_bias_bound_holds_for_one_bf16_rounding_of_gu():
    worst = 0.0
    for w in BOUND_CASES:
        for seed in range(3):
            _, f, b, b2, bound = _rounded_gu_case(w, seed)
            z = np.abs(b2["grad_router_bias"] - b["grad_router_bias"]) / bound
            assert np.all(z <= 1.0), (w.name, seed, z.max())
            worst = max(worst, float(z.max()))
    # the rounding uses a small part of the bound (about 1 sigma of the 8)
    assert worst < 0.5, worst


def test_bias_bound_holds_with_capacity_and_aux_loss():
    w = BOUND_CASES[3]
    cap = O.expert_capacity(w.T, w.k, w.E, 0.8)
    for kw in (dict(capacity=cap), dict(aux_alpha=0.01), dict(capacity=cap, aux_alpha=0.01)):
        _, f, b, b2, bound = _rounded_gu_case(w, 1, **kw)
        assert np.all(np.abs(b2["grad_router_bias"] - b["grad_router_bias"]) <= bound), kw


def test_bias_bound_catches_planted_mistakes():
    """Each mistake, planted in the oracle's own bias gradient, leaves the bound."""
    for w in BOUND_CASES[1:]:
        di, f, b, _, bound = _rounded_gu_case(w, 0)
        db, idx, wts, dw = b["grad_router_bias"], f["topk_idx"], f["topk_w"], b["grad_topk_w"]
        E = w.E

        def per_expert(dl_sel):
            return np.bincount(idx.ravel(), dl_sel.ravel(), minlength=E)

        mean = np.sum(wts * dw, axis=1, keepdims=True)
        planted = {
            "sign": -db,
            "rows of the next expert": np.roll(db, 1),
            "within-token mean dropped": per_expert(wts * dw),
            "weight factor dropped": per_expert(dw - mean),
            "mean without weights": per_expert(wts * (dw - dw.mean(axis=1, keepdims=True))),
            "one slot per token lost": per_expert(np.where(np.arange(w.k)[None, :] == 0, 0.0,
                                                           wts * (dw - mean))),
        }
        for name, bad in planted.items():
            assert np.any(np.abs(bad - db) > bound), (w.name, name)
