"""GPU parity: every call of the C ABI against the CPU oracle, element by element.

Sizes are small enough for the float64 oracle to finish in seconds but span
several 128-row tiles, ragged row tails, ragged column blocks (I and H not
multiples of the 256-wide tile), empty experts, a shared expert, and both
gates.  Bit-exact for ids and the permutation; bf16 tolerance (gpu_util) for
floating outputs and gradients.
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
CASES = {
    "tiny": G.WORKLOADS["tiny"],
    "ragged": W("ragged", T=300, H=192, E=6, k=3, I=320, bias_std=0.5),
    "ragged_shared": W("ragged_shared", T=200, H=128, E=5, k=2, I=192, I_shared=320, bias_std=0.5),
    "balanced_small": W("balanced_small", T=512, H=256, E=16, k=4, I=256, gate=G.GATE_BALANCED),
    "skewed_mid": W("skewed_mid", T=1024, H=512, E=32, k=4, I=384, bias_std=1.5),
    # k > 8: the per-token kernels' wide variants (up to 32 slots a token)
    "wide_k": W("wide_k", T=256, H=256, E=32, k=12, I=192, bias_std=0.5),
}


@pytest.fixture(scope="module", params=[(n, seed) for n in CASES for seed in (0, 1, 2)],
                ids=lambda p: f"{p[0]}-seed{p[1]}")
def case(request):
    name, seed = request.param
    w = CASES[name]
    di = U.DeviceInputs(w, seed=seed, with_grad=True)
    layer = U.run_forward(di)
    assert M.moe_read_device_status(layer.workspace) == 0
    return di, layer


def test_router_logits_and_topk(case):
    di, layer = case
    x, wr, b = di.f64("x"), di.f64("w_router"), di.f64("router_bias")
    ref = O.router_logits(x, wr, b)
    got = U.to_f64(layer.logits)
    bound = di.w.H * 2.0 ** -23 * (np.abs(x) @ np.abs(wr).T) + 2.0 ** -23 * (np.abs(ref) + 1.0)
    assert np.all(np.abs(got - ref) <= bound)
    idx = layer.topk_idx.cpu().numpy()
    wgt = layer.topk_w.cpu().numpy().astype(np.float64)
    balanced = di.w.gate == G.GATE_BALANCED
    # contract 1: the oracle's selection on the device's own fp32 logits is identical
    idx1, w1, _ = O.route(got, di.w.k, balanced=balanced,
                          decision_logits=layer.logits.cpu().numpy())
    assert np.array_equal(idx, idx1)
    assert np.allclose(wgt, w1, rtol=2e-6, atol=1e-7)
    # contract 2: against the oracle's own logits, any difference is a near tie
    U.check_routing_contract2(di, layer)
    if balanced:
        assert np.array_equal(idx, O.balanced_topk(di.w.T, di.w.E, di.w.k))


def test_route_permute_equals_route_then_permute(case):
    """The fused call (router kernel counting experts + one sort pass) gives the
    same bits as moe_route then moe_permute, with and without an expert
    capacity and the probability sums."""
    di, _ = case
    w = di.w
    T, E, k = w.T, w.E, w.k
    counts = None
    for cap in (0, None):
        if cap is None:   # a capacity that drops slots of the busiest experts
            cap = max(1, int(counts.max()) - 1)
        d = M.MoeDims.of(*di.dims, capacity=cap)
        ws = torch.zeros(M.moe_workspace_size(d, False), dtype=torch.uint8, device="cuda")
        outs = []
        for fused in (False, True):
            lg = torch.empty(T, E, dtype=torch.float32, device="cuda")
            idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
            tw = torch.empty(T, k, dtype=torch.float32, device="cuda")
            ps = torch.empty(E, dtype=torch.float32, device="cuda")
            off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
            perm = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
            inv = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
            if fused:
                M.moe_route_permute(d, w.gate, di.x, di.w_router, di.router_bias, lg, idx, tw, off,
                                    perm, inv, ws, prob_sum=ps)
            else:
                M.moe_route(d, w.gate, di.x, di.w_router, di.router_bias, lg, idx, tw, ws, prob_sum=ps)
                M.moe_permute(d, idx, off, perm, inv, ws)
            torch.cuda.synchronize()
            assert M.moe_read_device_status(ws) == 0
            outs.append([t.cpu() for t in (lg, idx, tw, ps, off, perm, inv)])
        for a, b in zip(*outs):
            assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                               b.view(torch.int32) if b.dtype == torch.float32 else b)
        counts = np.diff(outs[1][4].numpy())


def test_permute_bit_exact(case):
    di, layer = case
    idx = layer.topk_idx.cpu().numpy()
    off, perm, inv = O.permute(idx, di.w.E)
    assert np.array_equal(layer.expert_offsets.cpu().numpy(), off)
    assert np.array_equal(layer.perm_slot.cpu().numpy(), perm)
    assert np.array_equal(layer.slot_perm.cpu().numpy(), inv)


def test_forward_matches_oracle(case):
    di, layer = case
    idx = layer.topk_idx.cpu().numpy()
    f = U.oracle_forward(di, topk_idx=idx)
    U.check_close(layer.gu_saved, f["gu_perm"], "gu_saved")
    U.check_close(layer.y_perm, f["y_perm"], "y_perm")
    if di.w.I_shared:
        U.check_close(layer.sh_gu_saved, f["gu_shared"], "sh_gu_saved")
        U.check_close(layer.y_shared, f["y_shared"], "y_shared")
    U.check_close(layer.out, f["out"], "out")


def test_combine_is_exact_weighted_sum_of_device_rows(case):
    """Combine alone: from the device's own bf16 y_perm, one fp32 sum + one rounding."""
    di, layer = case
    y = U.to_f64(layer.y_perm)
    ysh = U.to_f64(layer.y_shared) if di.w.I_shared else None
    ref = O.combine(y, layer.slot_perm.cpu().numpy(), layer.topk_w.cpu().numpy().astype(np.float64), ysh)
    got = U.to_f64(layer.out)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30 + 1e-6 * np.abs(ref).max())


def test_backward_matches_oracle(case):
    di, layer = case
    grads = layer.alloc_grads(with_bias=di.w.bias_std > 0)
    layer.backward(di.grad_out, di.x, di.w_router, di.w_gate_up, di.w_down, grads,
                   di.w_sh_gate_up, di.w_sh_down)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(layer.workspace) == 0
    idx = layer.topk_idx.cpu().numpy()
    f = U.oracle_forward(di, topk_idx=idx)
    b = O.layer_backward(f, di.f64("grad_out"), di.f64("x"), di.f64("w_router"),
                         di.f64("w_gate_up"), di.f64("w_down"), di.w.k,
                         w_sh_gu=di.f64("w_sh_gate_up"), w_sh_down=di.f64("w_sh_down"))
    U.check_close(grads["grad_w_down"], b["grad_w_down"], "grad_w_down")
    U.check_close(grads["grad_w_gate_up"], b["grad_w_gate_up"], "grad_w_gate_up")
    U.check_close(grads["grad_x"], b["grad_x"], "grad_x")
    U.check_close(grads["grad_w_router"], b["grad_w_router"], "grad_w_router")
    if grads["grad_router_bias"] is not None:
        U.check_bias_grad(grads["grad_router_bias"], di, f, layer.gu_saved)
    if di.w.I_shared:
        U.check_close(grads["grad_w_sh_gate_up"], b["grad_w_sh_gate_up"], "grad_w_sh_gate_up")
        U.check_close(grads["grad_w_sh_down"], b["grad_w_sh_down"], "grad_w_sh_down")
    # experts that got no token: exact zero gradients
    empty = np.nonzero(np.diff(layer.expert_offsets.cpu().numpy()) == 0)[0]
    for e in empty:
        assert torch.count_nonzero(grads["grad_w_down"][e]) == 0
        assert torch.count_nonzero(grads["grad_w_gate_up"][e]) == 0


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (5, 7, 3), (3000, 128, 8), (700, 256, 6), (2049, 3, 2),
                                   (8192, 128, 8), (9000, 64, 8), (40000, 256, 2)])
def test_permute_random_ids(T, E, k):
    r = np.random.default_rng(T * 31 + E)
    idx = r.integers(0, E, size=(T, k)).astype(np.int32)
    if E > 4:
        idx[idx == 2] = 1        # at least one empty expert
    dims = (T, 64, E, k, 64, 0)
    ws = torch.zeros(M.moe_workspace_size(dims, False), dtype=torch.uint8, device="cuda")
    d_idx = torch.from_numpy(idx).cuda()
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    M.moe_permute(dims, d_idx, off, perm, inv, ws)
    o_off, o_perm, o_inv = O.permute(idx, E)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(perm.cpu().numpy(), o_perm)
    assert np.array_equal(inv.cpu().numpy(), o_inv)
    assert M.moe_read_device_status(ws) == 0


@pytest.mark.parametrize("T,k", [(64, 2), (9000, 8)])   # one and many sort blocks
def test_out_of_range_expert_ids_are_reported_not_used(T, k):
    E = 8
    idx = np.random.default_rng(0).integers(0, E, size=(T, k)).astype(np.int32)
    idx[3, 1] = E
    idx[10, 0] = -1
    dims = (T, 64, E, k, 64, 0)
    ws = torch.zeros(M.moe_workspace_size(dims, False), dtype=torch.uint8, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    M.moe_permute(dims, torch.from_numpy(idx).cuda(), off, perm, inv, ws)
    assert M.moe_read_device_status(ws) == 5
    good = (idx >= 0) & (idx < E)
    counts = np.bincount(idx[good].ravel(), minlength=E)
    assert np.array_equal(np.diff(off.cpu().numpy()), counts)
    assert int(off[-1]) == T * k - 2
    assert M.moe_read_device_status(ws) == 0   # cleared by the previous read


def test_forward_backward_bit_identical_run_to_run():
    w = CASES["skewed_mid"]
    di = U.DeviceInputs(w, seed=1, with_grad=True)
    outs = []
    for _ in range(2):
        layer = U.run_forward(di)
        g = layer.alloc_grads(with_bias=True)
        layer.backward(di.grad_out, di.x, di.w_router, di.w_gate_up, di.w_down, g)
        torch.cuda.synchronize()
        outs.append([layer.out.clone(), layer.topk_w.clone(), g["grad_x"].clone(),
                     g["grad_w_gate_up"].clone(), g["grad_w_router"].clone()])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["ragged_shared", "skewed_mid"])
def test_backward_recompute_matches_saved(name):
    """Activation recompute: a backward that recomputes the gate/up
    pre-activations (none saved by the forward) gives the same gradients, bit
    for bit, as one reading the saved copy; and the forward's outputs match."""
    w = CASES[name]
    di = U.DeviceInputs(w, seed=1, with_grad=True)
    outs = []
    for recompute in (False, True):
        layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True, recompute=recompute)
        layer.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                      di.w_sh_down)
        assert (layer.gu_saved is None) == recompute
        grads = layer.alloc_grads(with_bias=w.bias_std > 0)
        layer.backward(di.grad_out, di.x, di.w_router, di.w_gate_up, di.w_down, grads,
                       di.w_sh_gate_up, di.w_sh_down)
        torch.cuda.synchronize()
        assert M.moe_read_device_status(layer.workspace) == 0
        outs.append((layer.out.clone(), {k: v.clone() for k, v in grads.items() if v is not None}))
        idx = layer.topk_idx.cpu().numpy()
    (o0, g0), (o1, g1) = outs
    assert torch.equal(o0, o1)
    assert g0.keys() == g1.keys()
    for key in g0:
        assert torch.equal(g0[key], g1[key]), key
    # and against the oracle (on the device's routing, as in the other tests)
    f = U.oracle_forward(di, topk_idx=idx)
    b = O.layer_backward(f, di.f64("grad_out"), di.f64("x"), di.f64("w_router"),
                         di.f64("w_gate_up"), di.f64("w_down"), w.k,
                         w_sh_gu=di.f64("w_sh_gate_up"), w_sh_down=di.f64("w_sh_down"))
    U.check_close(g1["grad_w_gate_up"], b["grad_w_gate_up"], "grad_w_gate_up (recompute)")
    U.check_close(g1["grad_x"], b["grad_x"], "grad_x (recompute)")


@pytest.mark.parametrize("name", ["ragged", "skewed_mid", "balanced_small", "ragged_shared", "wide_k"])
def test_aux_loss_forward_and_backward(name):
    """Auxiliary load-balancing loss: the probability sums, the loss and its
    coefficients against the oracle on the device's routing and fp32 logits;
    the backward with the loss's gradient against the oracle; the expert
    weight gradients (which the loss does not reach) bit-identical to a
    backward without it."""
    w = CASES[name]
    # large enough that the loss's logit gradient (~alpha E f_e / T) is of the
    # order of the main loss's, so that dropping it would fail the comparison
    alpha = w.T / 4.0
    di = U.DeviceInputs(w, seed=2, with_grad=True)
    runs = {}
    for aux in (None, alpha):
        layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True, save_logits=True,
                           aux_alpha=aux)
        layer.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                      di.w_sh_down)
        grads = layer.alloc_grads(with_bias=w.bias_std > 0)
        layer.backward(di.grad_out, di.x, di.w_router, di.w_gate_up, di.w_down, grads,
                       di.w_sh_gate_up, di.w_sh_down)
        torch.cuda.synchronize()
        assert M.moe_read_device_status(layer.workspace) == 0
        runs[aux] = (layer, {k: v.clone() for k, v in grads.items() if v is not None})
    layer, g = runs[alpha]
    _, g0 = runs[None]
    idx = layer.topk_idx.cpu().numpy()
    # forward: on the device's fp32 logits
    p_dev = O.softmax(U.to_f64(layer.logits))
    assert np.allclose(U.to_f64(layer.prob_sum), p_dev.sum(axis=0), rtol=1e-5, atol=1e-5)
    L_ref, c_ref = O.aux_loss(p_dev, idx, alpha)
    assert abs(float(layer.aux_loss.item()) - L_ref) <= 1e-5 * max(1.0, abs(L_ref))
    assert np.allclose(U.to_f64(layer.aux_coef), c_ref, rtol=1e-6, atol=0)
    # backward against the oracle with the same coefficients
    f = U.oracle_forward(di, topk_idx=idx)
    b = O.layer_backward(f, di.f64("grad_out"), di.f64("x"), di.f64("w_router"),
                         di.f64("w_gate_up"), di.f64("w_down"), w.k,
                         w_sh_gu=di.f64("w_sh_gate_up"), w_sh_down=di.f64("w_sh_down"),
                         aux_coef=c_ref)
    U.check_close(g["grad_w_router"], b["grad_w_router"], "grad_w_router (aux)")
    U.check_close(g["grad_x"], b["grad_x"], "grad_x (aux)")
    if "grad_router_bias" in g:
        U.check_bias_grad(g["grad_router_bias"], di, f, layer.gu_saved,
                          name="grad_router_bias (aux)", aux_coef=c_ref)
    for key in ("grad_w_gate_up", "grad_w_down", "grad_w_sh_gate_up", "grad_w_sh_down"):
        if key in g:
            assert torch.equal(g[key], g0[key]), key
    # with uneven routing the loss changes the router gradient; with equal
    # counts (balanced gate) c is uniform and p (c - <c, p>) vanishes
    counts = np.diff(layer.expert_offsets.cpu().numpy())
    if counts.min() != counts.max():
        assert not torch.equal(g["grad_w_router"], g0["grad_w_router"])
    else:
        assert np.allclose(U.to_f64(g["grad_w_router"]), U.to_f64(g0["grad_w_router"]),
                           rtol=1e-2, atol=1e-2 * np.abs(U.to_f64(g0["grad_w_router"])).max())


def _run_layer(di, **kw):
    w = di.w
    layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=True, save_logits=True, **kw)
    layer.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                  di.w_sh_down)
    grads = layer.alloc_grads(with_bias=w.bias_std > 0)
    layer.backward(di.grad_out, di.x, di.w_router, di.w_gate_up, di.w_down, grads,
                   di.w_sh_gate_up, di.w_sh_down)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(layer.workspace) == 0
    return layer, {k: v.clone() for k, v in grads.items() if v is not None}


@pytest.mark.parametrize("name,factor", [("ragged", 0.6), ("skewed_mid", 1.0),
                                         ("ragged_shared", 0.8), ("balanced_small", 0.75),
                                         ("tiny", None), ("wide_k", 0.7)])
def test_capacity_forward_and_backward(name, factor):
    """Expert capacity (token dropping): the full sort and the kept/dropped
    split bit-exact (slot_perm -1 on dropped slots), out, the kept slots' rows
    of y_perm and gu_saved, and every gradient against the oracle with the
    same capacity.  factor None: capacity 1, nearly every slot dropped."""
    w = CASES[name]
    C = M.expert_capacity(w.T, w.k, w.E, factor) if factor else 1
    di = U.DeviceInputs(w, seed=3, with_grad=True)
    layer, g = _run_layer(di, capacity=C)
    idx = layer.topk_idx.cpu().numpy()
    off, perm, inv = O.permute(idx, w.E)
    keep = O.keep_slots(idx, w.E, C)
    assert (~keep).any()
    assert np.array_equal(layer.expert_offsets.cpu().numpy(), off)
    assert np.array_equal(layer.perm_slot.cpu().numpy(), perm)
    assert np.array_equal(layer.slot_perm.cpu().numpy(), np.where(keep.ravel(), inv, -1))
    f = U.oracle_forward(di, topk_idx=idx, capacity=C)
    U.check_close(layer.out, f["out"], "out (capacity)")
    rows = torch.from_numpy(inv[keep.ravel()].astype(np.int64)).cuda()
    U.check_close(layer.y_perm[rows], f["y_perm"][inv[keep.ravel()]], "y_perm (kept rows)")
    U.check_close(layer.gu_saved[rows], f["gu_perm"][inv[keep.ravel()]], "gu_saved (kept rows)")
    b = O.layer_backward(f, di.f64("grad_out"), di.f64("x"), di.f64("w_router"),
                         di.f64("w_gate_up"), di.f64("w_down"), w.k,
                         w_sh_gu=di.f64("w_sh_gate_up"), w_sh_down=di.f64("w_sh_down"))
    for key, got in g.items():
        if key == "grad_router_bias":
            U.check_bias_grad(got, di, f, layer.gu_saved, name=key + " (capacity)")
        else:
            U.check_close(got, b[key], key + " (capacity)")


@pytest.mark.parametrize("name", ["ragged", "balanced_small"])
def test_capacity_at_or_above_max_count_is_bit_identical(name):
    """A capacity no expert reaches drops nothing: outputs and gradients are
    bit-identical to the layer without a capacity."""
    w = CASES[name]
    di = U.DeviceInputs(w, seed=4, with_grad=True)
    l0, g0 = _run_layer(di)
    cmax = int(np.diff(l0.expert_offsets.cpu().numpy()).max())
    l1, g1 = _run_layer(di, capacity=cmax)
    assert torch.equal(l1.slot_perm, l0.slot_perm)
    assert torch.equal(l1.out, l0.out)
    for key in g0:
        assert torch.equal(g1[key], g0[key]), key


@pytest.mark.parametrize("name", ["ragged", "skewed_mid", "balanced_small", "ragged_shared", "wide_k"])
def test_inference_forward_matches_training_forward(name):
    """The forward without saved pre-activations (its gate/up GEMM stores h
    only and runs its own configuration) gives the training forward's bits,
    and so matches the oracle as that one does."""
    w = CASES[name]
    di = U.DeviceInputs(w, seed=11, with_grad=False)
    outs = []
    for with_backward in (True, False):
        layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=with_backward)
        layer.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                      di.w_sh_down)
        torch.cuda.synchronize()
        assert M.moe_read_device_status(layer.workspace) == 0
        outs.append((layer.out.clone(), layer.y_perm.clone(), layer.topk_idx.clone()))
    assert torch.equal(outs[0][2], outs[1][2])
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][0], outs[1][0])
    f = U.oracle_forward(di, topk_idx=outs[1][2].cpu().numpy())
    U.check_close(outs[1][0], f["out"], "out (inference)")


@pytest.mark.parametrize("name,factor", [("ragged", 0.6), ("skewed_mid", 1.0), ("ragged_shared", 0.8)])
def test_inference_forward_with_capacity_matches_training_forward(name, factor):
    """With an expert capacity the groups are the experts' first C rows, so the
    inference gate/up GEMM's tails (and its narrow units) follow the capped
    counts: y_perm and out equal the training forward's bit for bit."""
    w = CASES[name]
    C = M.expert_capacity(w.T, w.k, w.E, factor)
    di = U.DeviceInputs(w, seed=12, with_grad=False)
    outs = []
    for with_backward in (True, False):
        layer = M.MoeLayer(di.dims, gate_mode=w.gate, with_backward=with_backward, capacity=C)
        layer.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                      di.w_sh_down)
        torch.cuda.synchronize()
        assert M.moe_read_device_status(layer.workspace) == 0
        outs.append((layer.out.clone(), layer.y_perm.clone(), layer.slot_perm.clone()))
    assert torch.equal(outs[0][2], outs[1][2])
    assert (outs[1][2] < 0).any()  # the capacity drops slots
    kept = outs[1][2][outs[1][2] >= 0].long()
    assert torch.equal(outs[0][1][kept], outs[1][1][kept])
    assert torch.equal(outs[0][0], outs[1][0])
