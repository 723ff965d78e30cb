"""Pins of the oracle's expert-parallel dispatch / combine (no GPU).

Expert parallelism splits the experts over the ranks (Shard(0) on the expert
dimension) while each rank keeps its own tokens; the layer's result must not
depend on the split.  Pinned against what fixes it independently of the
oracle's own EP code:

* the expert ranges are torch's chunking of the expert dimension;
* a source's send counts are brute-force counts of its slots per rank;
* every expert's grouped rows on its receiving rank are the global stable
  sort's rows of that expert (the single-rank permute of all ranks' slots,
  tokens numbered rank by rank), in the same order;
* the n-rank layer equals the one-rank layer on all tokens, and one rank is
  the plain layer;
* a planted mistake (receive rows grouped by source instead of by expert)
  breaks the layer.
"""

import numpy as np
import pytest
import torch

from grouped_expert_gemm_top_b300 import inputs as G
from oracle import moe_oracle as O


def _weights(E, H, I, seed=0):
    r = np.random.default_rng(seed)
    return (r.normal(0, 0.05, (E, H)), r.normal(0, 0.05, (E, 2 * I, H)), r.normal(0, 0.05, (E, H, I)))


@pytest.mark.parametrize("E,n", [(128, 8), (8, 2), (6, 4), (5, 3), (7, 8), (1, 1), (16, 1)])
def test_expert_ranges_are_torch_chunks(E, n):
    b = O.ep_expert_ranges(E, n)
    chunks = torch.arange(E).chunk(n)
    for r in range(n):
        got = list(range(int(b[r]), int(b[r + 1])))
        want = chunks[r].tolist() if r < len(chunks) else []
        assert got == want, (r, got, want)
    assert b[0] == 0 and b[n] == E


def test_send_counts_brute_force():
    r = np.random.default_rng(1)
    for E, n, T, k in [(16, 4, 50, 3), (6, 4, 20, 2), (9, 2, 33, 4)]:
        idx = np.stack([r.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        off, perm, inv, send, counts = O.ep_dispatch(idx, E, n)
        b = O.ep_expert_ranges(E, n)
        for q in range(n):
            assert send[q] == sum(1 for e in idx.ravel() if b[q] <= e < b[q + 1])
        assert send.sum() == T * k
        assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
        # the sorted order is rank-major: rows of rank q's block go to q's experts
        flat = idx.ravel()
        start = 0
        for q in range(n):
            rows = perm[start:start + send[q]]
            assert np.all((flat[rows] >= b[q]) & (flat[rows] < b[q + 1]))
            start += send[q]


def test_receive_layout_matches_the_global_sort():
    r = np.random.default_rng(2)
    for E, n, Ts, k in [(16, 4, [10, 0, 7, 12], 3), (6, 4, [5, 5, 5, 5], 2), (8, 2, [40, 31], 4)]:
        ids = [np.array([r.choice(E, size=k, replace=False) for _ in range(T)],
                        dtype=np.int32).reshape(T, k) for T in Ts]
        plans = [O.ep_dispatch(i, E, n) for i in ids]
        b = O.ep_expert_ranges(E, n)
        # global sort of all ranks' slots, tokens numbered rank by rank
        g_off, g_perm, _ = O.permute(np.concatenate(ids, axis=0), E)
        starts = np.cumsum([0] + [T * k for T in Ts])
        for q in range(n):
            loc_off, recv_perm = O.ep_receive([p[4] for p in plans], int(b[q]), int(b[q + 1]))
            R = sum(int(p[3][q]) for p in plans)
            assert np.array_equal(np.sort(recv_perm), np.arange(R))        # a bijection
            # receive row -> (source, position in the source's block)
            src_of, slot_of = [], []
            for s, p in enumerate(plans):
                off_s, perm_s = p[0], p[1]
                blk = perm_s[int(off_s[b[q]]):int(off_s[b[q + 1]])]
                src_of += [s] * len(blk)
                slot_of += [int(starts[s]) + int(x) for x in blk]
            src_of, slot_of = np.array(src_of, dtype=np.int64), np.array(slot_of, dtype=np.int64)
            for e in range(int(b[q]), int(b[q + 1])):
                rows = recv_perm[loc_off[e - b[q]]:loc_off[e - b[q] + 1]]
                want = g_perm[g_off[e]:g_off[e + 1]]
                assert np.array_equal(slot_of[rows], want), (q, e)


@pytest.mark.parametrize("E,n,Ts,k", [(8, 2, [24, 17], 2), (6, 4, [9, 0, 11, 8], 3),
                                      (16, 4, [12, 12, 12, 12], 4), (5, 3, [7, 3, 10], 5)])
def test_ep_layer_equals_one_rank_layer(E, n, Ts, k):
    H, I = 16, 12
    wr, wgu, wd = _weights(E, H, I, seed=E + n)
    r = np.random.default_rng(E * n)
    xs = [r.normal(0, 1, (T, H)) for T in Ts]
    outs = O.ep_layer_forward(xs, wr, wgu, wd, k)
    ref = O.layer_forward(np.concatenate(xs, axis=0), wr, wgu, wd, k)
    got = np.concatenate([o["out"] for o in outs], axis=0)
    assert np.allclose(got, ref["out"], rtol=1e-13, atol=1e-15)
    # every source holds its rows' outputs in its own sorted order
    start = 0
    for o, T in zip(outs, Ts):
        tok_rows = ref["slot_perm"][start * k:(start + T) * k]
        assert np.allclose(o["y_sorted"][o["slot_perm"]], ref["y_perm"][tok_rows], rtol=1e-13,
                           atol=1e-15)
        start += T


def test_one_rank_is_the_plain_layer():
    E, H, I, T, k = 8, 16, 12, 30, 3
    wr, wgu, wd = _weights(E, H, I, seed=3)
    x = np.random.default_rng(3).normal(0, 1, (T, H))
    (o,) = O.ep_layer_forward([x], wr, wgu, wd, k)
    ref = O.layer_forward(x, wr, wgu, wd, k)
    assert np.array_equal(o["out"], ref["out"])
    assert np.array_equal(o["y_sorted"], ref["y_perm"])


def test_grouping_rows_by_source_is_caught():
    """Planted in the oracle: the receiver takes its rows source-major (as they
    arrived) instead of expert-major; the experts then see other experts' rows."""
    E, n, Ts, k, H, I = 8, 2, [20, 20], 2, 16, 12
    wr, wgu, wd = _weights(E, H, I, seed=5)
    xs = [np.random.default_rng(5 + i).normal(0, 1, (T, H)) for i, T in enumerate(Ts)]
    outs = O.ep_layer_forward(xs, wr, wgu, wd, k)
    o = outs[0]
    wrong = np.arange(len(o["recv_perm"]), dtype=np.int32)       # receive order as is
    assert not np.array_equal(wrong, o["recv_perm"])
    b = O.ep_expert_ranges(E, n)
    y_ok = O.experts_grouped(o["x_recv"], o["local_offsets"], o["recv_perm"], 1, wgu[b[0]:b[1]],
                             wd[b[0]:b[1]])[0]
    y_bad = O.experts_grouped(o["x_recv"], o["local_offsets"], wrong, 1, wgu[b[0]:b[1]],
                              wd[b[0]:b[1]])[0]
    assert not np.allclose(y_ok, y_bad)


def test_ep_layer_on_the_seeded_inputs():
    """The seeded small workload split over 2 ranks, against the one-rank layer."""
    w = G.Workload("ep_small", T=64, H=128, E=8, k=2, I=64, bias_std=0.5)
    n_ = G.make_inputs(w, 0, False)
    f = O.widen_bf16
    x = f(n_["x"])
    bias = n_["router_bias"].astype(np.float64)
    outs = O.ep_layer_forward([x[:40], x[40:]], f(n_["w_router"]), f(n_["w_gate_up"]),
                              f(n_["w_down"]), w.k, bias=bias)
    ref = O.layer_forward(x, f(n_["w_router"]), f(n_["w_gate_up"]), f(n_["w_down"]), w.k, bias=bias)
    assert np.allclose(np.concatenate([o["out"] for o in outs]), ref["out"], rtol=1e-13, atol=1e-16)


@pytest.mark.parametrize("E,n,Ts,k", [(8, 2, [24, 17], 2), (6, 4, [9, 0, 11, 8], 3),
                                      (16, 4, [12, 12, 12, 12], 4), (5, 3, [7, 3, 10], 5)])
def test_ep_backward_equals_one_rank_backward(E, n, Ts, k):
    """Every gradient of the n-rank backward equals the one-rank layer_backward
    (pinned by finite differences): grad_x rank by rank, the local experts'
    weight gradients chunk by chunk, and the router's summed over the ranks.
    The router step here (dl from w and dL/dw only) is a different formula from
    layer_backward's (through the softmax p), so their equality also pins it."""
    H, I = 16, 12
    wr, wgu, wd = _weights(E, H, I, seed=E + n + 1)
    r = np.random.default_rng(E * n + 1)
    xs = [r.normal(0, 1, (T, H)) for T in Ts]
    gos = [r.normal(0, 1, (T, H)) for T in Ts]
    fwd = O.ep_layer_forward(xs, wr, wgu, wd, k)
    got = O.ep_layer_backward(fwd, gos, xs, wr, wgu, wd)
    x_all = np.concatenate(xs, axis=0)
    ref_f = O.layer_forward(x_all, wr, wgu, wd, k)
    ref = O.layer_backward(ref_f, np.concatenate(gos, axis=0), x_all, wr, wgu, wd, k)
    tol = dict(rtol=1e-11, atol=1e-13)
    assert np.allclose(np.concatenate([g["grad_x"] for g in got], axis=0), ref["grad_x"], **tol)
    assert np.allclose(sum(g["grad_w_router"] for g in got), ref["grad_w_router"], **tol)
    assert np.allclose(sum(g["grad_router_bias"] for g in got), ref["grad_router_bias"], **tol)
    b = O.ep_expert_ranges(E, n)
    for q in range(n):
        assert np.allclose(got[q]["grad_w_gate_up"], ref["grad_w_gate_up"][b[q]:b[q + 1]], **tol)
        assert np.allclose(got[q]["grad_w_down"], ref["grad_w_down"][b[q]:b[q + 1]], **tol)
    # each source's slots' dL/dw, back in its sorted order, are layer_backward's
    start = 0
    for g, o, T in zip(got, fwd, Ts):
        dw_slot = g["dw_sorted"][o["slot_perm"].astype(np.int64)].reshape(T, k)
        assert np.allclose(dw_slot, ref["grad_topk_w"][start:start + T], **tol)
        start += T


def test_router_backward_is_zero_off_the_chosen_experts():
    """dl vanishes at every expert a token did not choose, and its row sums are
    zero (the renormalised weights sum to one whatever the logits)."""
    r = np.random.default_rng(9)
    T, E, k, H = 20, 10, 3, 8
    idx = np.stack([r.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = r.random((T, k)); w /= w.sum(axis=1, keepdims=True)
    dl, _, _, _ = O.router_backward(r.normal(0, 1, (T, H)), r.normal(0, 1, (E, H)), idx, w,
                                    r.normal(0, 1, (T, k)))
    chosen = np.zeros((T, E), dtype=bool)
    chosen[np.repeat(np.arange(T), k), idx.ravel()] = True
    assert np.all(dl[~chosen] == 0.0)
    assert np.allclose(dl.sum(axis=1), 0.0, atol=1e-14)


def test_returning_dx_unsorted_is_caught():
    """Planted in the oracle: the source takes the returned dx rows in slot
    order instead of its sorted order; grad_x then no longer matches."""
    E, n, Ts, k, H, I = 8, 2, [20, 20], 2, 16, 12
    wr, wgu, wd = _weights(E, H, I, seed=6)
    xs = [np.random.default_rng(6 + i).normal(0, 1, (T, H)) for i, T in enumerate(Ts)]
    gos = [np.random.default_rng(60 + i).normal(0, 1, (T, H)) for i, T in enumerate(Ts)]
    fwd = O.ep_layer_forward(xs, wr, wgu, wd, k)
    got = O.ep_layer_backward(fwd, gos, xs, wr, wgu, wd)
    g, o = got[0], fwd[0]
    right = g["dx_sorted"][o["slot_perm"].astype(np.int64)].reshape(Ts[0], k, H).sum(axis=1)
    wrong = g["dx_sorted"].reshape(Ts[0], k, H).sum(axis=1)
    assert not np.allclose(right, wrong)
