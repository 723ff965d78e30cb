"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against a closed form, an invariant the method
fixes, a brute-force enumeration, a library routine for a special case, or
central finite differences.  The mutation tests at the end plant plausible
mistakes in the oracle and check that some pin catches each one.
"""

import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from grouped_expert_gemm_top_b300 import inputs as G

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- bf16 widening
def test_widen_bf16_closed_forms():
    bits = np.array([0x0000, 0x3F80, 0xC000, 0x3F00, 0x4049, 0x8000, 0x7F7F, 0x0001], np.uint16)
    got = O.widen_bf16(bits)
    want = [0.0, 1.0, -2.0, 0.5, 3.140625, -0.0, 3.3895313892515355e38, 2.0 ** -133]
    assert np.array_equal(got, np.array(want))


def test_generator_round_trip_matches_oracle_widening():
    b = G.normal_bf16((64, 64), 1.0, 0, "x")
    assert np.array_equal(G.bf16_bits_to_f32(b).astype(np.float64), O.widen_bf16(b))


# ---------------------------------------------------------------- router
def test_router_logits_hand_example():
    x = np.array([[1.0, 2.0], [0.5, -1.0]])
    w = np.array([[3.0, 4.0], [5.0, 6.0], [0.0, 1.0]])
    b = np.array([0.0, -1.0, 2.0])
    assert np.array_equal(O.router_logits(x, w), [[11.0, 17.0, 2.0], [-2.5, -3.5, -1.0]])
    assert np.array_equal(O.router_logits(x, w, b), [[11.0, 16.0, 4.0], [-2.5, -4.5, 1.0]])


def test_softmax_closed_form_and_shift_invariance():
    p = O.softmax(np.array([[0.0, math.log(3.0)]]))
    assert np.allclose(p, [[0.25, 0.75]], rtol=0, atol=1e-15)
    l = RNG.normal(size=(7, 13))
    assert np.allclose(O.softmax(l), O.softmax(l + 1000.0), atol=1e-14)
    assert np.allclose(O.softmax(l).sum(1), 1.0, atol=1e-14)
    assert np.allclose(O.softmax(l), torch.softmax(torch.from_numpy(l), 1).numpy(), atol=1e-15)


def _topk_by_stable_sort(vals, k):
    # brute force: full stable sort by (value descending, index ascending)
    order = np.argsort(-vals.astype(np.float64), axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


@pytest.mark.parametrize("E,k", [(8, 2), (8, 8), (128, 8), (128, 6), (5, 1)])
def test_topk_matches_full_stable_sort(E, k):
    vals = RNG.normal(size=(300, E)).astype(np.float32)
    assert np.array_equal(O.select_topk(vals, k), _topk_by_stable_sort(vals, k))
    # heavy ties: small integers
    ties = RNG.integers(-2, 3, size=(300, E)).astype(np.float32)
    assert np.array_equal(O.select_topk(ties, k), _topk_by_stable_sort(ties, k))


def test_topk_all_equal_takes_lowest_indices():
    assert np.array_equal(O.select_topk(np.zeros((3, 10), np.float32), 4), np.tile(np.arange(4), (3, 1)))
    # signed zeros compare equal
    v = np.array([[0.0, -0.0, 0.0, -0.0]], np.float32)
    assert np.array_equal(O.select_topk(v, 3), [[0, 1, 2]])


def test_topk_hand_example():
    v = np.array([[0.1, 0.7, 0.7, -3.0, 0.9]], np.float32)
    assert np.array_equal(O.select_topk(v, 3), [[4, 1, 2]])


def test_balanced_gate_exact_uniform_split_and_distinct():
    for (T, E, k) in [(4096, 128, 8), (8192, 128, 6), (256, 8, 2), (12, 6, 3)]:
        idx = O.balanced_topk(T, E, k)
        assert np.array_equal(np.bincount(idx.ravel(), minlength=E), np.full(E, T * k // E))
        assert all(len(set(r)) == k for r in idx[: min(T, 500)])
    assert np.array_equal(O.balanced_topk(3, 4, 2), [[0, 1], [2, 3], [0, 1]])


def test_renormalised_weights_closed_form():
    p = np.array([[0.1, 0.2, 0.3, 0.4]])
    w = O.renormalised_weights(p, np.array([[3, 1]]))
    assert np.allclose(w, [[2.0 / 3.0, 1.0 / 3.0]], rtol=0, atol=1e-15)
    l = RNG.normal(size=(50, 16))
    idx, w, p = O.route(l, 16)
    assert np.allclose(np.sort(w, 1), np.sort(p, 1), atol=1e-15)    # k = E: w = p
    idx, w, p = O.route(l, 5)
    assert np.allclose(w.sum(1), 1.0, atol=1e-15)
    # renormalised softmax over the chosen logits = softmax restricted to them
    rows = np.arange(50)[:, None]
    assert np.allclose(w, O.softmax(l[rows, idx]), atol=1e-15)


# ---------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k", [(256, 8, 2), (1000, 128, 8), (7, 5, 5), (1, 1, 1)])
def test_permute_is_stable_counting_sort(T, E, k):
    idx = RNG.integers(0, E, size=(T, k)).astype(np.int32)
    if E > 3:
        idx[idx == 3] = 2          # leave an empty expert
    off, perm, inv = O.permute(idx, E)
    flat = idx.ravel()
    assert np.array_equal(perm, np.argsort(flat, kind="stable"))
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert np.array_equal(perm[inv], np.arange(T * k)) and np.array_equal(inv[perm], np.arange(T * k))
    for e in range(E):
        seg = perm[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


# ---------------------------------------------------------------- expert MLP
def test_silu_closed_forms_and_library():
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert abs(O.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(O.silu(np.array([50.0]))[0] - 50.0) < 1e-12
    assert abs(O.silu(np.array([-50.0]))[0]) < 1e-19
    z = RNG.normal(size=1000) * 5
    assert np.allclose(O.silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(), atol=1e-15)


def _torch_dense_swiglu(x, wgu, wd):
    I = wd.shape[1]
    xt, wgut, wdt = (torch.from_numpy(a) for a in (x, wgu, wd))
    gu = torch.nn.functional.linear(xt, wgut)
    return torch.nn.functional.linear(torch.nn.functional.silu(gu[:, :I]) * gu[:, I:], wdt).numpy()


def _tiny(T=12, H=16, E=4, k=2, I=8, seed=0, bias=True):
    r = np.random.default_rng(seed)
    d = dict(x=r.normal(size=(T, H)), w_router=r.normal(size=(E, H)) * 0.5,
             w_gu=r.normal(size=(E, 2 * I, H)) * 0.3, w_down=r.normal(size=(E, H, I)) * 0.3,
             bias=r.normal(size=E) if bias else None)
    return d


def test_single_expert_layer_is_dense_swiglu_mlp():
    d = _tiny(E=1, k=1, H=16, I=8)
    f = O.layer_forward(d["x"], d["w_router"], d["w_gu"], d["w_down"], 1)
    assert np.allclose(f["topk_w"], 1.0)
    assert np.allclose(f["out"], _torch_dense_swiglu(d["x"], d["w_gu"][0], d["w_down"][0]), atol=1e-12)


def test_k_equals_E_identical_experts_is_dense_mlp():
    d = _tiny(E=5, k=5)
    wgu = np.repeat(d["w_gu"][:1], 5, axis=0)
    wd = np.repeat(d["w_down"][:1], 5, axis=0)
    f = O.layer_forward(d["x"], d["w_router"], wgu, wd, 5, bias=d["bias"])
    dense = _torch_dense_swiglu(d["x"], wgu[0], wd[0])
    assert np.allclose(f["out"], dense, atol=1e-12)
    # and the gradient: sum of the per-expert weight grads is the dense grad; router grad vanishes
    g = np.random.default_rng(9).normal(size=f["out"].shape)
    b = O.layer_backward(f, g, d["x"], d["w_router"], wgu, wd, 5)
    xt = torch.from_numpy(d["x"]).requires_grad_()
    wg = torch.from_numpy(wgu[0]).requires_grad_()
    wdn = torch.from_numpy(wd[0]).requires_grad_()
    I = wd.shape[2]
    gu = xt @ wg.T
    y = (torch.nn.functional.silu(gu[:, :I]) * gu[:, I:]) @ wdn.T
    (y * torch.from_numpy(g)).sum().backward()
    assert np.allclose(b["grad_x"], xt.grad.numpy(), atol=1e-10)
    assert np.allclose(b["grad_w_gate_up"].sum(0), wg.grad.numpy(), atol=1e-10)
    assert np.allclose(b["grad_w_down"].sum(0), wdn.grad.numpy(), atol=1e-10)
    assert np.allclose(b["grad_w_router"], 0.0, atol=1e-10)


def test_three_backends_agree():
    d = _tiny(T=20, H=24, E=6, k=3, I=16)
    idx, w, _ = O.route(O.router_logits(d["x"], d["w_router"], d["bias"]), 3)
    off, perm, inv = O.permute(idx, 6)
    yg, _, _ = O.experts_grouped(d["x"], off, perm, 3, d["w_gu"], d["w_down"])
    ye = O.experts_eager(d["x"], idx, d["w_gu"], d["w_down"])
    yb = O.experts_batched(d["x"], idx, d["w_gu"], d["w_down"])
    y_slot_from_grouped = yg[inv].reshape(20, 3, -1)
    assert np.allclose(ye, yb, rtol=1e-12, atol=1e-12)
    assert np.allclose(ye, y_slot_from_grouped, rtol=1e-12, atol=1e-12)
    out_g = O.combine(yg, inv, w)
    assert np.allclose(out_g, O.combine_slots(ye, w), rtol=1e-12, atol=1e-12)


def test_combine_hand_example():
    y_perm = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0], [1000.0, 2000.0]])
    slot_perm = np.array([2, 0, 3, 1])        # token0: rows 2,0; token1: rows 3,1
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    out = O.combine(y_perm, slot_perm, w, y_shared=np.array([[1.0, 1.0], [0.0, -1.0]]))
    assert np.array_equal(out, [[25.0 + 0.75 + 1, 50.0 + 1.5 + 1], [505.0, 1010.0 - 1]])


# ---------------------------------------------------------------- backward
def _loss_and_grads(d, k, G_, balanced=False, shared=None, capacity=None):
    f = O.layer_forward(d["x"], d["w_router"], d["w_gu"], d["w_down"], k, balanced=balanced,
                        bias=d["bias"], capacity=capacity, **(shared or {}))
    b = O.layer_backward(f, G_, d["x"], d["w_router"], d["w_gu"], d["w_down"], k,
                         **(shared or {}))
    return float(np.sum(f["out"] * G_)), f, b


def _fd_check(d, k, balanced=False, shared=None, n_probe=12, seed=3, capacity=None):
    T, H = d["x"].shape
    G_ = np.random.default_rng(seed).normal(size=(T, H))
    _, f0, b = _loss_and_grads(d, k, G_, balanced, shared, capacity)
    eps = 1e-6
    names = [("x", "grad_x"), ("w_router", "grad_w_router"), ("w_gu", "grad_w_gate_up"),
             ("w_down", "grad_w_down")]
    if d["bias"] is not None:
        names.append(("bias", "grad_router_bias"))
    r = np.random.default_rng(seed + 1)
    for pname, gname in names:
        arr = d[pname]
        for _ in range(n_probe):
            i = tuple(r.integers(0, s) for s in arr.shape)
            old = arr[i]
            arr[i] = old + eps
            lp, fp_, _ = _loss_and_grads(d, k, G_, balanced, shared, capacity)
            arr[i] = old - eps
            lm, fm_, _ = _loss_and_grads(d, k, G_, balanced, shared, capacity)
            arr[i] = old
            assert np.array_equal(fp_["topk_idx"], f0["topk_idx"]) and np.array_equal(fm_["topk_idx"], f0["topk_idx"])
            num = (lp - lm) / (2 * eps)
            assert abs(num - b[gname][i]) <= 1e-6 * max(1.0, abs(num)), (pname, i, num, b[gname][i])
    if shared:
        for pname, gname in [("w_sh_gu", "grad_w_sh_gate_up"), ("w_sh_down", "grad_w_sh_down")]:
            arr = shared[pname]
            for _ in range(n_probe):
                i = tuple(r.integers(0, s) for s in arr.shape)
                old = arr[i]
                arr[i] = old + eps
                lp = _loss_and_grads(d, k, G_, balanced, shared, capacity)[0]
                arr[i] = old - eps
                lm = _loss_and_grads(d, k, G_, balanced, shared, capacity)[0]
                arr[i] = old
                num = (lp - lm) / (2 * eps)
                assert abs(num - b[gname][i]) <= 1e-6 * max(1.0, abs(num)), (pname, i)


def test_backward_matches_finite_differences_softmax_topk():
    _fd_check(_tiny(T=4, H=8, E=4, k=2, I=8, seed=11), 2)


def test_backward_matches_finite_differences_balanced_gate():
    _fd_check(_tiny(T=6, H=8, E=4, k=2, I=8, seed=12), 2, balanced=True)


def test_backward_matches_finite_differences_shared_expert():
    d = _tiny(T=5, H=8, E=4, k=3, I=8, seed=13)
    r = np.random.default_rng(5)
    sh = dict(w_sh_gu=r.normal(size=(12, 8)) * 0.3, w_sh_down=r.normal(size=(8, 6)) * 0.3)
    _fd_check(d, 3, shared=sh)


def test_backward_matches_autograd_of_plain_torch_layer():
    """Autograd of an independent dense torch formulation (one-hot routing mask)."""
    T, H, E, k, I = 16, 32, 6, 3, 24
    d = _tiny(T, H, E, k, I, seed=21)
    G_ = np.random.default_rng(2).normal(size=(T, H))
    _, f, b = _loss_and_grads(d, k, G_)
    idx = torch.from_numpy(f["topk_idx"].astype(np.int64))
    x = torch.from_numpy(d["x"]).requires_grad_()
    wr = torch.from_numpy(d["w_router"]).requires_grad_()
    bias = torch.from_numpy(d["bias"]).requires_grad_()
    wgu = torch.from_numpy(d["w_gu"]).requires_grad_()
    wd = torch.from_numpy(d["w_down"]).requires_grad_()
    p = torch.softmax(x @ wr.T + bias, dim=1)
    mask = torch.zeros(T, E, dtype=torch.float64).scatter_(1, idx, 1.0)
    gate = p * mask
    gate = gate / gate.sum(1, keepdim=True)                     # [T, E], zero off the selection
    gu = torch.einsum("th,eih->tei", x, wgu)                    # every expert on every token
    hh = torch.nn.functional.silu(gu[..., :I]) * gu[..., I:]
    y = torch.einsum("tei,ehi->teh", hh, wd)
    out = torch.einsum("te,teh->th", gate, y)
    (out * torch.from_numpy(G_)).sum().backward()
    assert np.allclose(out.detach().numpy(), f["out"], atol=1e-12)
    for t_, g in [(x, "grad_x"), (wr, "grad_w_router"), (bias, "grad_router_bias"),
                  (wgu, "grad_w_gate_up"), (wd, "grad_w_down")]:
        assert np.allclose(t_.grad.numpy(), b[g], atol=1e-10), g


# ---------------------------------------------------------------- auxiliary load-balancing loss
def test_aux_loss_uniform_routing_is_alpha():
    """Equal logits (uniform p) and the balanced gate (uniform counts): L = alpha."""
    T, E, k = 12, 4, 2
    p = O.softmax(np.zeros((T, E)))
    idx = O.balanced_topk(T, E, k)
    L, c = O.aux_loss(p, idx, 0.01)
    assert abs(L - 0.01) < 1e-15
    assert np.allclose(c, 0.01 * E * (1.0 / E) / T)


def test_aux_loss_hand_example():
    p = np.array([[0.7, 0.3], [0.4, 0.6]])
    idx = np.array([[0], [0]])
    L, c = O.aux_loss(p, idx, 0.5)
    # f = [1, 0], P = [0.55, 0.45]: L = 0.5 * 2 * 0.55; c = 0.5 * 2 * f / 2
    assert abs(L - 0.55) < 1e-15
    assert np.allclose(c, [0.5, 0.0])


def _loss_and_grads_aux(d, k, G_, alpha, balanced=False):
    f = O.layer_forward(d["x"], d["w_router"], d["w_gu"], d["w_down"], k, balanced=balanced,
                        bias=d["bias"])
    L_aux, c = O.aux_loss(f["p"], f["topk_idx"], alpha)
    b = O.layer_backward(f, G_, d["x"], d["w_router"], d["w_gu"], d["w_down"], k, aux_coef=c)
    return float(np.sum(f["out"] * G_)) + L_aux, f, b


@pytest.mark.parametrize("balanced", [False, True])
def test_aux_loss_gradient_matches_finite_differences(balanced):
    """J = <G, out> + L_aux: the backward with the aux coefficients against
    central differences in x, W_r and the router bias (routing, hence the
    counts, unchanged by the probes)."""
    d = _tiny(T=6, H=8, E=4, k=2, I=8, seed=31)
    T, H = d["x"].shape
    G_ = np.random.default_rng(4).normal(size=(T, H))
    alpha = 0.7   # large, so the aux term is not hidden by the main loss
    _, f0, b = _loss_and_grads_aux(d, 2, G_, alpha, balanced)
    eps = 1e-6
    r = np.random.default_rng(6)
    for pname, gname in [("x", "grad_x"), ("w_router", "grad_w_router"), ("bias", "grad_router_bias")]:
        arr = d[pname]
        for _ in range(10):
            i = tuple(r.integers(0, s_) for s_ in arr.shape)
            old = arr[i]
            arr[i] = old + eps
            lp, fp_, _ = _loss_and_grads_aux(d, 2, G_, alpha, balanced)
            arr[i] = old - eps
            lm, fm_, _ = _loss_and_grads_aux(d, 2, G_, alpha, balanced)
            arr[i] = old
            assert np.array_equal(fp_["topk_idx"], f0["topk_idx"]) and np.array_equal(fm_["topk_idx"], f0["topk_idx"])
            num = (lp - lm) / (2 * eps)
            assert abs(num - b[gname][i]) <= 1e-6 * max(1.0, abs(num)), (pname, i, num, b[gname][i])


def test_aux_loss_gradient_matches_autograd():
    """Autograd of L_aux = alpha E sum_e f_e mean_t p[t, e] written in torch,
    with the counts f as constants, plus the main loss."""
    T, H, E, k, I = 10, 16, 5, 2, 8
    d = _tiny(T, H, E, k, I, seed=41)
    G_ = np.random.default_rng(3).normal(size=(T, H))
    alpha = 0.3
    _, f, b = _loss_and_grads_aux(d, k, G_, alpha)
    b0 = O.layer_backward(f, G_, d["x"], d["w_router"], d["w_gu"], d["w_down"], k)
    x = torch.from_numpy(d["x"]).requires_grad_()
    wr = torch.from_numpy(d["w_router"]).requires_grad_()
    bias = torch.from_numpy(d["bias"]).requires_grad_()
    p = torch.softmax(x @ wr.T + bias, dim=1)
    counts = torch.zeros(E, dtype=torch.float64)
    counts.index_add_(0, torch.from_numpy(f["topk_idx"].ravel().astype(np.int64)),
                      torch.ones(T * k, dtype=torch.float64))
    l_aux = alpha * E * torch.sum(counts / (T * k) * p.mean(dim=0))
    l_aux.backward()
    for t_, g in [(x, "grad_x"), (wr, "grad_w_router"), (bias, "grad_router_bias")]:
        assert np.allclose(t_.grad.numpy(), b[g] - b0[g], atol=1e-12), g


def test_mutation_aux_coefficients_without_token_mean_is_caught(monkeypatch):
    good = O.aux_loss

    def bad(p, topk_idx, alpha):
        L, c = good(p, topk_idx, alpha)
        return L, c * p.shape[0]   # forgets the 1/T of the token mean

    monkeypatch.setattr(O, "aux_loss", bad)
    assert _pins_fail(lambda: test_aux_loss_gradient_matches_finite_differences(False))


# ---------------------------------------------------------------- whole workloads
# ---------------------------------------------------------------- expert capacity
def test_expert_capacity_closed_forms():
    assert O.expert_capacity(4096, 8, 128, 1.0) == 256
    assert O.expert_capacity(4096, 8, 128, 1.25) == 320
    assert O.expert_capacity(10, 2, 3, 1.0) == 7          # ceil(20 / 3)
    assert O.expert_capacity(10, 2, 3, 0.5) == 4          # ceil(10 / 3)
    assert O.expert_capacity(8, 1, 4, 0.0) == 0
    assert O.expert_capacity(100, 1, 10, 1.1) == 11     # 1.1 * 100 / 10, not 11.000000000000002


def test_keep_slots_hand_example():
    # slots in order: s0 t0->0, s1 t0->1, s2 t1->0, s3 t1->2, s4 t2->0, s5 t2->1,
    # s6 t3->1, s7 t3->0.  Capacity 2: expert 0 keeps s0, s2 (drops s4, s7),
    # expert 1 keeps s1, s5 (drops s6), expert 2 keeps s3.
    idx = np.array([[0, 1], [0, 2], [0, 1], [1, 0]])
    keep = O.keep_slots(idx, 3, 2)
    assert np.array_equal(keep, [[True, True], [True, True], [False, True], [False, False]])
    assert O.keep_slots(idx, 3, None).all()
    assert not O.keep_slots(idx, 3, 0).any()
    assert np.array_equal(O.keep_slots(idx, 3, 1), [[True, True], [False, True], [False, False],
                                                    [False, False]])


@pytest.mark.parametrize("T,E,k,C", [(50, 4, 2, 10), (200, 8, 3, 1), (64, 16, 4, 17), (9, 3, 3, 3)])
def test_keep_slots_brute_force_rank(T, E, k, C):
    """Kept iff the number of earlier slots with the same expert (counted one
    by one) is below C; every expert keeps min(count, C) slots."""
    idx = np.random.default_rng(T + C).integers(0, E, size=(T, k))
    flat = idx.ravel()
    rank = np.array([int(np.sum(flat[:s] == flat[s])) for s in range(flat.size)])
    keep = O.keep_slots(idx, E, C)
    assert np.array_equal(keep.ravel(), rank < C)
    for e in range(E):
        assert keep.ravel()[flat == e].sum() == min(int(np.sum(flat == e)), C)


def test_capacity_at_or_above_max_count_drops_nothing():
    d = _tiny(T=16, H=16, E=4, k=2, I=8, seed=51)
    G_ = np.random.default_rng(2).normal(size=d["x"].shape)
    _, f0, b0 = _loss_and_grads(d, 2, G_)
    cmax = int(np.diff(f0["expert_offsets"]).max())
    for C in (cmax, cmax + 5):
        _, f1, b1 = _loss_and_grads(d, 2, G_, capacity=C)
        assert f1["keep"].all()
        assert np.array_equal(f1["out"], f0["out"])
        for key in b0:
            assert np.array_equal(b1[key], b0[key]), key


def test_capacity_zero_leaves_the_shared_expert_only():
    """Every slot dropped: out is the shared expert (a dense SwiGLU MLP, torch),
    the routed experts and the router get no gradient, grad_x is the shared
    expert's input gradient (torch autograd)."""
    d = _tiny(T=10, H=16, E=4, k=2, I=8, seed=52)
    r = np.random.default_rng(5)
    sh = dict(w_sh_gu=r.normal(size=(24, 16)) * 0.2, w_sh_down=r.normal(size=(16, 12)) * 0.2)
    G_ = r.normal(size=d["x"].shape)
    _, f, b = _loss_and_grads(d, 2, G_, shared=sh, capacity=0)
    xt = torch.from_numpy(d["x"]).requires_grad_()
    wg = torch.from_numpy(sh["w_sh_gu"]).requires_grad_()
    wdn = torch.from_numpy(sh["w_sh_down"]).requires_grad_()
    gu = xt @ wg.T
    y = (torch.nn.functional.silu(gu[:, :12]) * gu[:, 12:]) @ wdn.T
    (y * torch.from_numpy(G_)).sum().backward()
    assert np.allclose(f["out"], y.detach().numpy(), atol=1e-12)
    assert np.allclose(b["grad_x"], xt.grad.numpy(), atol=1e-12)
    assert np.allclose(b["grad_w_sh_gate_up"], wg.grad.numpy(), atol=1e-12)
    for key in ("grad_w_gate_up", "grad_w_down", "grad_w_router", "grad_router_bias",
                "grad_topk_w", "grad_logits"):
        assert not np.any(b[key]), key


def test_capacity_forward_matches_eager_backend_with_dropped_slots():
    """The grouped path with drops equals the eager for-loop backend over the
    kept slots, with the router's weights as they are (not renormalised)."""
    T, E, k = 30, 5, 3
    d = _tiny(T=T, H=16, E=E, k=k, I=8, seed=53)
    f = O.layer_forward(d["x"], d["w_router"], d["w_gu"], d["w_down"], k, bias=d["bias"],
                        capacity=10)
    assert 0 < (~f["keep"]).sum() < T * k
    idx, w, _ = O.route(O.router_logits(d["x"], d["w_router"], d["bias"]), k)
    ye = O.experts_eager(d["x"], idx, d["w_gu"], d["w_down"])
    flat = idx.ravel()
    rank = np.array([int(np.sum(flat[:s] == flat[s])) for s in range(flat.size)]).reshape(T, k)
    out = O.combine_slots(ye * (rank < 10)[:, :, None], w)
    assert np.allclose(f["out"], out, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("C", [1, 3])
def test_capacity_backward_matches_finite_differences(C):
    d = _tiny(T=10, H=8, E=3, k=2, I=8, seed=54)
    f = O.layer_forward(d["x"], d["w_router"], d["w_gu"], d["w_down"], 2, bias=d["bias"],
                        capacity=C)
    assert 0 < (~f["keep"]).sum()
    _fd_check(d, 2, n_probe=8, seed=11, capacity=C)


def test_tiny_workload_forward_invariants():
    w = G.WORKLOADS["tiny"]
    inp = G.make_inputs(w, 0)
    x, wr = O.widen_bf16(inp["x"]), O.widen_bf16(inp["w_router"])
    wgu, wd = O.widen_bf16(inp["w_gate_up"]), O.widen_bf16(inp["w_down"])
    f = O.layer_forward(x, wr, wgu, wd, w.k)
    assert f["expert_offsets"][-1] == w.S
    assert np.allclose(f["topk_w"].sum(1), 1.0)
    assert np.isfinite(f["out"]).all() and np.abs(f["out"]).max() > 0


def test_balanced_qwen_shape_routing():
    w = G.WORKLOADS["qwen3_30b_a3b_balanced"]
    idx = O.balanced_topk(w.T, w.E, w.k)
    off, perm, inv = O.permute(idx, w.E)
    assert np.array_equal(np.diff(off), np.full(w.E, 256))


# ---------------------------------------------------------------- mutations
def _pins_fail(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_mutation_wrong_swiglu_halves_is_caught(monkeypatch):
    def bad(xr, w_gu, w_down):
        I = w_down.shape[1]
        gu = xr @ w_gu.T
        h = O.silu(gu[:, I:]) * gu[:, :I]          # gate/up swapped
        return h @ w_down.T, gu, h
    monkeypatch.setattr(O, "swiglu_mlp", bad)
    assert _pins_fail(test_single_expert_layer_is_dense_swiglu_mlp)


def test_mutation_dropped_silu_derivative_term_is_caught(monkeypatch):
    orig = O.swiglu_mlp_backward

    def bad(xr, gu, w_gu, w_down, dy):
        I = w_down.shape[1]
        g, u = gu[:, :I], gu[:, I:]
        s = O.sigmoid(g)
        dh = dy @ w_down
        dgu = np.concatenate([dh * u * s, dh * g * s], axis=1)   # (1 + g(1-s)) dropped
        return dgu @ w_gu, dgu.T @ xr, dy.T @ (g * s * u)
    monkeypatch.setattr(O, "swiglu_mlp_backward", bad)
    assert _pins_fail(test_backward_matches_finite_differences_softmax_topk)
    monkeypatch.setattr(O, "swiglu_mlp_backward", orig)


def test_mutation_router_sign_is_caught(monkeypatch):
    orig = O.layer_backward

    def bad(*a, **kw):
        r = orig(*a, **kw)
        r["grad_w_router"] = -r["grad_w_router"]
        return r
    monkeypatch.setattr(O, "layer_backward", bad)
    assert _pins_fail(test_backward_matches_finite_differences_softmax_topk)


def test_mutation_tie_break_to_higher_index_is_caught(monkeypatch):
    def bad(v, k):
        return np.argsort(-v.astype(np.float64)[:, ::-1], axis=1, kind="stable")[:, :k].astype(np.int32)
    monkeypatch.setattr(O, "select_topk", lambda v, k: (v.shape[1] - 1 - bad(v, k)).astype(np.int32))
    assert _pins_fail(test_topk_all_equal_takes_lowest_indices)


def test_mutation_unstable_permutation_is_caught(monkeypatch):
    orig = O.permute

    def bad(idx, E):
        off, perm, inv = orig(idx, E)
        perm = perm.copy()
        for e in range(E):                           # reverse order inside each group
            perm[off[e]:off[e + 1]] = perm[off[e]:off[e + 1]][::-1]
        inv = np.empty_like(perm)
        inv[perm] = np.arange(perm.size)
        return off, perm, inv
    monkeypatch.setattr(O, "permute", bad)
    assert _pins_fail(lambda: test_permute_is_stable_counting_sort(256, 8, 2))


def test_mutation_transposed_down_weight_is_caught(monkeypatch):
    def bad(xr, w_gu, w_down):
        I = w_down.shape[1]
        gu = xr @ w_gu.T
        h = O.silu(gu[:, :I]) * gu[:, I:]
        return h @ w_down.reshape(w_down.shape[1], w_down.shape[0]), gu, h   # [H,I] read as [I,H]
    monkeypatch.setattr(O, "swiglu_mlp", bad)
    assert _pins_fail(test_single_expert_layer_is_dense_swiglu_mlp)


def test_mutation_combine_without_weights_is_caught(monkeypatch):
    def bad(y_perm, slot_perm, topk_w, y_shared=None):
        T, k = topk_w.shape
        return y_perm[slot_perm.reshape(T, k)].mean(1) + (0 if y_shared is None else y_shared)
    monkeypatch.setattr(O, "combine", bad)
    assert _pins_fail(test_combine_hand_example)


def test_mutation_capacity_keeps_last_slots_is_caught(monkeypatch):
    orig = O.keep_slots

    def bad(idx, E, C):
        return orig(idx[::-1, ::-1], E, C)[::-1, ::-1]
    monkeypatch.setattr(O, "keep_slots", bad)
    assert _pins_fail(test_keep_slots_hand_example)


def test_mutation_capacity_renormalised_weights_is_caught(monkeypatch):
    orig = O.combine

    def bad(y_perm, slot_perm, topk_w, y_shared=None, keep=None):
        if keep is not None:
            kw = np.where(keep, topk_w, 0.0)
            topk_w = kw / np.maximum(kw.sum(axis=1, keepdims=True), 1e-300)
        return orig(y_perm, slot_perm, topk_w, y_shared, keep)
    monkeypatch.setattr(O, "combine", bad)
    assert _pins_fail(test_capacity_forward_matches_eager_backend_with_dropped_slots)


def test_mutation_capacity_ignored_in_backward_is_caught(monkeypatch):
    orig = O.layer_backward

    def bad(fwd, *a, **kw):
        f2 = dict(fwd)
        f2["keep"] = None
        return orig(f2, *a, **kw)
    monkeypatch.setattr(O, "layer_backward", bad)
    assert _pins_fail(lambda: test_capacity_backward_matches_finite_differences(1))


# ---------------------------------------------------------------- page facts
def test_workloads_and_oracle_follow_the_pages_printed_facts():
    """tests/golden/pages_facts.json: the Qwen3-shaped workloads have the
    expert count the pages print; experts are fused 3-D tensors (the oracle
    and the generator take W_gu [E, 2I, H], W_down [E, H, I]); sharding the
    expert dimension 8 ways leaves each GPU 1/8 of the expert weights, as the
    pages' 55 GiB -> 6.8 GiB states (to the pages' rounding)."""
    import json
    import os
    facts = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_facts.json")))["facts"]
    E = facts["qwen3_moe_experts"]["value"]
    for name in ("qwen3_30b_a3b_balanced", "qwen3_30b_a3b_skewed", "qwen3_30b_a3b_balanced_fwd_bwd"):
        assert G.WORKLOADS[name].E == E
    w = G.WORKLOADS["tiny"]
    inp = G.make_inputs(w, 0, with_grad=False)
    assert facts["experts_as_fused_3d_tensors"]["value"]
    assert inp["w_gate_up"].shape == (w.E, 2 * w.I, w.H) and inp["w_down"].shape == (w.E, w.H, w.I)
    ep = facts["expert_parallel_size"]["value"]
    mem = facts["expert_memory_per_gpu_at_ep8"]["value"]
    assert abs(mem["total_gib"] / ep - mem["per_gpu_gib"]) < 0.1
    # the balanced gate at that expert count splits the slots exactly evenly
    w = G.WORKLOADS["qwen3_30b_a3b_balanced"]
    idx = O.balanced_topk(w.T, E, w.k)
    assert np.array_equal(np.bincount(idx.ravel(), minlength=E), np.full(E, w.T * w.k // E))
