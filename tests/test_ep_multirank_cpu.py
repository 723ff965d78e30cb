"""The expert-parallel forward's and backward's host logic over real process
groups (gloo, world size 2 and 3, CPU).

ExpertParallelMoe drives the exchanges: the expert counts, the token rows
rank by rank, and the outputs back.  Here its compute steps are the oracle's
(float64, injected by this test as OracleOps; the product path always uses
the library's kernels), so the test checks the exchange logic and the
layouts around it against the one-rank oracle layer, and each rank's
exchanged buffers against the oracle's own expert-parallel simulation.
"""

import os
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = {
    # E, world, tokens per rank, k, H, I
    "E8_w2": (8, 2, [24, 17], 2, 16, 12),
    "E6_w3": (6, 3, [9, 0, 11], 3, 16, 12),     # a rank without tokens
    "E5_w3": (5, 3, [7, 5, 10], 2, 16, 12),     # uneven expert chunks (2, 2, 1)
}


class OracleOps:
    """Float64 stand-ins for the compute steps, from the oracle."""

    def __init__(self, O, k, E, w_router, w_gu, w_down):
        self.O, self.k, self.E = O, k, E
        self.w_router, self.w_gu, self.w_down = w_router, w_gu, w_down

    def route_permute(self, x, w_router, router_bias):
        O = self.O
        logits = O.router_logits(x.numpy(), self.w_router)
        idx, w, _ = O.route(logits, self.k)
        off, perm, inv = O.permute(idx, self.E)
        t = torch.from_numpy
        return (t(idx.astype(np.int32)), t(w), t(off.astype(np.int32)), t(perm.astype(np.int32)),
                t(inv.astype(np.int32)))

    def gather_rows(self, src, idx, div):
        return src[idx.long() // div]

    def receive_layout(self, counts):
        n, E_loc = counts.shape
        full = np.zeros((n, E_loc), dtype=np.int64)
        full[:, :] = counts.numpy()
        loc_off, recv_perm = self.O.ep_receive(list(full), 0, E_loc)
        inv = np.empty_like(recv_perm)
        inv[recv_perm] = np.arange(recv_perm.size, dtype=recv_perm.dtype)
        t = torch.from_numpy
        return t(loc_off), t(recv_perm), t(inv)

    def experts(self, x_recv, loc_off, recv_perm, w_gu_local, w_down_local, gu_out=None):
        y = self.O.experts_grouped(x_recv.numpy(), loc_off.numpy(), recv_perm.numpy(), 1,
                                   w_gu_local.numpy(), w_down_local.numpy())[0]
        return torch.from_numpy(y)

    def gather_scalars(self, src, idx, div):
        return src.reshape(-1)[idx.long() // div]

    def experts_bwd(self, go_recv, x_recv, w_recv, loc_off, recv_perm, recv_inv, w_gu_local,
                    w_down_local, gu_saved):
        dx, dw, dW_gu, dW_down = self.O.ep_experts_backward(
            x_recv.numpy(), go_recv.numpy(), w_recv.numpy(), loc_off.numpy(), recv_perm.numpy(),
            w_gu_local.numpy(), w_down_local.numpy())
        t = torch.from_numpy
        return t(dx), t(dw), t(dW_gu), t(dW_down)

    def router_bwd(self, x, w_router, idx, w, off, perm, inv, dx_sorted, dw_sorted, with_bias):
        T = x.shape[0]
        k = self.k
        H = x.shape[1]
        inv_n = inv.numpy().astype(np.int64)
        dx_slot = dx_sorted.numpy()[inv_n].reshape(T, k, H)
        dw = dw_sorted.numpy()[inv_n].reshape(T, k)
        _, dx_router, dW_r, db = self.O.router_backward(x.numpy(), self.w_router, idx.numpy(),
                                                        w.numpy(), dw)
        t = torch.from_numpy
        return t(dx_slot.sum(axis=1) + dx_router), t(dW_r), (t(db) if with_bias else None)

    def combine(self, y_sorted, slot_perm, topk_w):
        return torch.from_numpy(self.O.combine(y_sorted.numpy(), slot_perm.numpy(), topk_w.numpy()))


def _inputs(E, Ts, H, I, seed):
    r = np.random.default_rng(seed)
    return ([r.normal(0, 1, (T, H)) for T in Ts], r.normal(0, 0.1, (E, H)),
            r.normal(0, 0.1, (E, 2 * I, H)), r.normal(0, 0.1, (E, H, I)))


def _worker(rank, world, port, name, out):
    sys.path.insert(0, ROOT)
    from grouped_expert_gemm_top_b300 import ep
    from oracle import moe_oracle as O
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        E, _, Ts, k, H, I = CASES[name]
        xs, wr, wgu, wd = _inputs(E, Ts, H, I, seed=E * world)
        b = ep.expert_ranges(E, world)
        lo, hi = b[rank], b[rank + 1]
        ops = OracleOps(O, k, E, wr, wgu, wd)
        layer = ep.ExpertParallelMoe((Ts[rank], H, E, k, I), rank, world, ep.DistExchange(),
                                     device="cpu", ops=ops)
        y = layer.forward(torch.from_numpy(xs[rank]), None, torch.from_numpy(wgu[lo:hi]),
                          torch.from_numpy(wd[lo:hi]))
        L = layer.last
        out[rank] = dict(out=y.numpy(), send_rows=list(L["send_rows"]),
                         recv_rows=list(L["recv_rows"]), x_recv=L["x_recv"].numpy(),
                         y_sorted=L["y_sorted"].numpy())
    finally:
        dist.destroy_process_group()


def _worker_bwd(rank, world, port, name, out):
    sys.path.insert(0, ROOT)
    from grouped_expert_gemm_top_b300 import ep
    from oracle import moe_oracle as O
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        E, _, Ts, k, H, I = CASES[name]
        xs, wr, wgu, wd = _inputs(E, Ts, H, I, seed=E * world)
        gos = _grad_outs(Ts, H, seed=E * world + 1)
        b = ep.expert_ranges(E, world)
        lo, hi = b[rank], b[rank + 1]
        ops = OracleOps(O, k, E, wr, wgu, wd)
        layer = ep.ExpertParallelMoe((Ts[rank], H, E, k, I), rank, world, ep.DistExchange(),
                                     device="cpu", ops=ops, with_backward=True)
        layer.forward(torch.from_numpy(xs[rank]), None, torch.from_numpy(wgu[lo:hi]),
                      torch.from_numpy(wd[lo:hi]))
        g = layer.backward(torch.from_numpy(gos[rank]), torch.from_numpy(xs[rank]), None,
                           torch.from_numpy(wgu[lo:hi]), torch.from_numpy(wd[lo:hi]),
                           with_bias=True)
        out[rank] = {key: (v.numpy() if v is not None else None) for key, v in g.items()}
    finally:
        dist.destroy_process_group()


def _grad_outs(Ts, H, seed):
    r = np.random.default_rng(seed)
    return [r.normal(0, 1, (T, H)) for T in Ts]


@pytest.mark.parametrize("name", list(CASES))
def test_expert_parallel_backward_matches_one_rank(name):
    """The backward's exchanges (grad_out rows and weights out, dx and dL/dw
    back) over gloo, its compute steps the oracle's: every rank's grad_x, the
    local experts' weight gradients and the router's summed over the ranks
    against the one-rank oracle backward."""
    sys.path.insert(0, ROOT)
    from oracle import moe_oracle as O
    E, world, Ts, k, H, I = CASES[name]
    port = 29700 + (os.getpid() + 7 * list(CASES).index(name)) % 200
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker_bwd, args=(world, port, name, out), nprocs=world, join=True)
        res = {r: dict(v) for r, v in out.items()}
    xs, wr, wgu, wd = _inputs(E, Ts, H, I, seed=E * world)
    gos = _grad_outs(Ts, H, seed=E * world + 1)
    x_all = np.concatenate(xs, axis=0)
    f = O.layer_forward(x_all, wr, wgu, wd, k)
    ref = O.layer_backward(f, np.concatenate(gos, axis=0), x_all, wr, wgu, wd, k)
    tol = dict(rtol=1e-11, atol=1e-13)
    got_x = np.concatenate([res[r]["grad_x"] for r in range(world)], axis=0)
    assert np.allclose(got_x, ref["grad_x"], **tol)
    assert np.allclose(sum(res[r]["grad_w_router"] for r in range(world)), ref["grad_w_router"], **tol)
    assert np.allclose(sum(res[r]["grad_router_bias"] for r in range(world)),
                       ref["grad_router_bias"], **tol)
    from grouped_expert_gemm_top_b300 import ep
    b = ep.expert_ranges(E, world)
    for r in range(world):
        assert np.allclose(res[r]["grad_w_gate_up"], ref["grad_w_gate_up"][b[r]:b[r + 1]], **tol)
        assert np.allclose(res[r]["grad_w_down"], ref["grad_w_down"][b[r]:b[r + 1]], **tol)


@pytest.mark.parametrize("name", list(CASES))
def test_expert_parallel_forward_matches_one_rank(name):
    sys.path.insert(0, ROOT)
    from oracle import moe_oracle as O
    E, world, Ts, k, H, I = CASES[name]
    port = 29600 + (os.getpid() + 7 * list(CASES).index(name)) % 300
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, name, out), nprocs=world, join=True)
        res = {r: dict(v) for r, v in out.items()}
    xs, wr, wgu, wd = _inputs(E, Ts, H, I, seed=E * world)
    ref = O.layer_forward(np.concatenate(xs, axis=0), wr, wgu, wd, k)
    got = np.concatenate([res[r]["out"] for r in range(world)], axis=0)
    assert np.allclose(got, ref["out"], rtol=1e-13, atol=1e-15)
    sim = O.ep_layer_forward(xs, wr, wgu, wd, k)
    for r in range(world):
        assert res[r]["send_rows"] == [int(v) for v in sim[r]["send_counts"]]
        assert res[r]["recv_rows"] == [int(v) for v in sim[r]["recv_counts"]]
        assert np.array_equal(res[r]["x_recv"], sim[r]["x_recv"])
        assert np.allclose(res[r]["y_sorted"], sim[r]["y_sorted"], rtol=1e-13, atol=1e-15)
