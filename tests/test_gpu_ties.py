"""Exact ties in the router, on the GPU, against the oracle bit for bit.

The selection rule takes the lower expert id among equal logits.  Random
logits practically never tie, so these cases make them tie on purpose:

* zero router weights: every logit is 0, so the softmax gate must pick
  experts 0 .. k-1 for every token (and weights 1/k);
* duplicated router rows (row 2m+1 = row 2m): the logits of experts 2m and
  2m+1 are equal (bit for bit on the device, which the test checks first),
  so whenever 2m+1 is chosen, 2m must have been chosen in the round before;
* zero weights and a bias of -0.0 on even experts, +0.0 on odd ones: every
  logit compares equal, ids 0 .. k-1 again;
* zero weights and a bias rounded to multiples of 0.5: many exact ties
  between experts at several levels, decided by expert id.

Each case runs under both gates at (E=128, k=8) and (E=32, k=12).  The ids
must equal the oracle's selection on the device's fp32 logits (contract 1)
and, since these ties are exact in float64 too, the oracle's selection on
its own logits with no exception.  The sort and the layer output are
checked against the oracle as well.
"""

import numpy as np
import pytest
import torch

import gpu_util as U
from grouped_expert_gemm_top_b300 import inputs as G
from grouped_expert_gemm_top_b300 import moe as M
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

SHAPES = {
    "E128_k8": G.Workload("ties_E128_k8", T=256, H=256, E=128, k=8, I=64),
    "E32_k12": G.Workload("ties_E32_k12", T=192, H=128, E=32, k=12, I=64),
}
VARIANTS = ("zero_router", "duplicated_rows", "signed_zero_bias", "quantised_bias")
GATES = {"softmax": G.GATE_SOFTMAX_TOPK, "balanced": G.GATE_BALANCED}


def _tie_inputs(w, variant, seed=0):
    di = U.DeviceInputs(w, seed=seed, with_grad=False)
    wr = di.np["w_router"].copy()          # bf16 bits [E, H]
    bias = None
    if variant == "zero_router":
        wr[:] = 0
    elif variant == "duplicated_rows":
        wr[1::2] = wr[0::2]
    elif variant == "signed_zero_bias":
        wr[:] = 0
        bias = np.where(np.arange(w.E) % 2 == 0, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
    elif variant == "quantised_bias":
        wr[:] = 0
        r = np.random.default_rng(seed + 11)
        bias = (np.round(r.normal(size=w.E) * 2.0) / 2.0).astype(np.float32)
    di.np["w_router"] = wr
    di.np["router_bias"] = bias
    di._f64.clear()
    di.w_router = U.dev_bf16(wr)
    di.router_bias = U.dev_f32(bias)
    return di


@pytest.mark.parametrize("gate", list(GATES))
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", list(SHAPES))
def test_router_ties_bit_exact(shape, variant, gate):
    w = SHAPES[shape].replace(gate=GATES[gate])
    di = _tie_inputs(w, variant)
    layer = U.run_forward(di, with_backward=False, save_logits=True)
    assert M.moe_read_device_status(layer.workspace) == 0
    logits = layer.logits.cpu().numpy()
    idx = layer.topk_idx.cpu().numpy()
    wgt = layer.topk_w.cpu().numpy().astype(np.float64)
    balanced = gate == "balanced"

    # the ties are really there, bit for bit, on the device
    if variant == "duplicated_rows":
        assert np.array_equal(logits[:, 0::2].view(np.uint32), logits[:, 1::2].view(np.uint32))
    elif variant in ("zero_router", "signed_zero_bias"):
        assert np.all(logits == 0.0)
    else:
        assert np.array_equal(logits, np.broadcast_to(di.np["router_bias"], logits.shape))

    # contract 1: the oracle's selection on the device's logits
    idx1, w1, _ = O.route(logits.astype(np.float64), w.k, balanced=balanced, decision_logits=logits)
    assert np.array_equal(idx, idx1)
    assert np.allclose(wgt, w1, rtol=2e-6, atol=1e-7)
    # the oracle's selection on its own float64 logits: the ties are exact there
    # too, so no near-tie allowance applies
    ref = O.router_logits(di.f64("x"), di.f64("w_router"), di.f64("router_bias"))
    idx2, w2, _ = O.route(ref, w.k, balanced=balanced)
    assert np.array_equal(idx, idx2)
    assert np.allclose(wgt, w2, rtol=2e-6, atol=1e-7)

    if balanced:
        assert np.array_equal(idx, O.balanced_topk(w.T, w.E, w.k))
    elif variant in ("zero_router", "signed_zero_bias"):
        assert np.array_equal(idx, np.broadcast_to(np.arange(w.k, dtype=np.int32), idx.shape))
        assert np.allclose(wgt, 1.0 / w.k, rtol=1e-6)
    elif variant == "duplicated_rows":
        # 2m+1 only ever right after 2m (lower id first at the tie)
        for t in range(w.T):
            pos = {int(e): j for j, e in enumerate(idx[t])}
            for e, j in pos.items():
                if e % 2 == 1:
                    assert pos.get(e - 1, -1) == j - 1, (t, idx[t])
    else:
        # (bias descending, id ascending) is the whole order
        b = di.np["router_bias"]
        order = np.lexsort((np.arange(w.E), -b.astype(np.float64)))[: w.k]
        assert np.array_equal(idx, np.broadcast_to(order.astype(np.int32), idx.shape))

    off, perm, inv = O.permute(idx, w.E)
    assert np.array_equal(layer.expert_offsets.cpu().numpy(), off)
    assert np.array_equal(layer.perm_slot.cpu().numpy(), perm)
    assert np.array_equal(layer.slot_perm.cpu().numpy(), inv)
    f = U.oracle_forward(di, topk_idx=idx)
    U.check_close(layer.out, f["out"], "out")
