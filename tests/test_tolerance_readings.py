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
