"""The expert-parallel forward's kernels on the GPU, with the ranks emulated as
threads of one process on the one GPU.

Each thread is one rank of ExpertParallelMoe with the library's kernels
(DeviceOps); ThreadExchange moves the exchanged buffers between the threads
on the host side of the GPU's stream order (every rank's work is complete
before its buffer is read, and kernels never wait on one another).  Checks:

* bit-exact: the ranks' outputs equal the one-GPU path (moe_permute,
  moe_grouped_mlp_fwd, moe_unpermute_combine) run on all ranks' tokens with
  the ranks' own routing: the dispatch, the receive layout and the return
  trip move rows without touching their bits, and an expert meets its rows
  in the same order as on one GPU;
* every source's returned rows equal the one-GPU y_perm rows of its slots;
* the outputs match the float64 oracle layer at the bf16 tolerance;
* the receive layout kernel against the oracle's, exactly.
"""

import threading

import numpy as np
import pytest
import torch

import gpu_util as U
from grouped_expert_gemm_top_b300 import ep
from grouped_expert_gemm_top_b300 import inputs as G
from grouped_expert_gemm_top_b300 import moe as M
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu


class ThreadExchange:
    """all_to_all_single among the threads of one process (one per rank)."""

    def __init__(self, world):
        self.world = world
        self.barrier = threading.Barrier(world, timeout=120)
        self.box = [None] * world
        self.device = torch.device("cuda")

    def rank_view(self, rank):
        ex = self

        class View:
            device = ex.device

            def all_to_all_single(self, out, inp, out_splits, in_splits):
                torch.cuda.synchronize()            # this rank's input is complete
                ex.box[rank] = (inp, list(in_splits))
                ex.barrier.wait()
                pos = 0
                for s in range(ex.world):
                    src, splits = ex.box[s]
                    n = splits[rank]
                    assert n == out_splits[s], (rank, s, n, out_splits)
                    start = sum(splits[:rank])
                    out[pos:pos + n].copy_(src[start:start + n])
                    pos += n
                torch.cuda.synchronize()            # every copy out of the inputs is done
                ex.barrier.wait()

        return View()


CASES = {
    # name: (E, world, tokens per rank, k, H, I, bias std)
    "E16_w2": (16, 2, [300, 212], 4, 256, 128, 0.5),
    "E6_w4_uneven": (6, 4, [64, 0, 100, 37], 2, 128, 192, 1.0),   # chunks 2,2,2,0; a rank without tokens
    "qwen3_like_w4": (128, 4, [1024, 1024, 1024, 1024], 8, 2048, 768, 1.5),
}


def _run_ep(name, seed=0):
    E, world, Ts, k, H, I, bs = CASES[name]
    w = G.Workload(name, T=sum(Ts), H=H, E=E, k=k, I=I, bias_std=bs)
    di = U.DeviceInputs(w, seed=seed, with_grad=False)
    b = ep.expert_ranges(E, world)
    ex = ThreadExchange(world)
    starts = np.cumsum([0] + Ts)
    layers = [ep.ExpertParallelMoe((Ts[r], H, E, k, I), r, world, ex.rank_view(r)) for r in range(world)]
    outs, errs = [None] * world, []

    def run(r):
        try:
            xr = di.x[int(starts[r]):int(starts[r + 1])].contiguous()
            outs[r] = layers[r].forward(xr, di.w_router, di.w_gate_up[b[r]:b[r + 1]].contiguous(),
                                        di.w_down[b[r]:b[r + 1]].contiguous(), di.router_bias)
            torch.cuda.synchronize()
        except Exception as e:   # surfaced below
            errs.append(e)
            ex.barrier.abort()

    th = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    if errs:
        raise errs[0]
    for L in layers:
        assert L.ops.status() == 0
    return di, w, layers, outs


def _one_gpu_with_ranks_routing(di, w, layers):
    """The one-GPU path on all tokens, routed as the ranks routed them."""
    idx = torch.cat([L.last["topk_idx"] for L in layers]).contiguous()
    tw = torch.cat([L.last["topk_w"] for L in layers]).contiguous()
    dims = (w.T, w.H, w.E, w.k, w.I, 0)
    ws = torch.zeros(M.moe_workspace_size(dims, False), dtype=torch.uint8, device="cuda")
    S = w.T * w.k
    off = torch.empty(w.E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(S, dtype=torch.int32, device="cuda")
    inv = torch.empty(S, dtype=torch.int32, device="cuda")
    M.moe_permute(dims, idx, off, perm, inv, ws)
    y = torch.empty(S, w.H, dtype=torch.bfloat16, device="cuda")
    M.moe_grouped_mlp_fwd(dims, di.x, off, perm, di.w_gate_up, di.w_down, None, y, None, None, None,
                          None, ws)
    out = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    M.moe_unpermute_combine(dims, y, inv, tw, None, out)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(ws) == 0
    return idx, tw, y, inv, out


@pytest.mark.parametrize("name", list(CASES))
def test_expert_parallel_forward_bit_exact_against_one_gpu(name):
    di, w, layers, outs = _run_ep(name)
    idx, tw, y, inv, out = _one_gpu_with_ranks_routing(di, w, layers)
    got = torch.cat(outs)
    assert torch.equal(got.view(torch.int16), out.view(torch.int16))
    # each source holds its slots' expert outputs in its own sorted order
    Ts = CASES[name][2]
    s0 = 0
    for L, T in zip(layers, Ts):
        if T:
            rows = inv[s0 * w.k:(s0 + T) * w.k].long()
            mine = L.last["y_sorted"][L.last["slot_perm"].long()]
            assert torch.equal(mine.view(torch.int16), y[rows].view(torch.int16))
        s0 += T
    if w.T * w.H <= 1 << 20:
        # against the float64 oracle layer, routed as the ranks routed
        f = U.oracle_forward(di, topk_idx=idx.cpu().numpy())
        U.check_close(got, f["out"], "out (expert parallel)")


def test_receive_layout_kernel_matches_oracle():
    r = np.random.default_rng(4)
    for n_src, E_loc in [(1, 1), (2, 8), (4, 16), (8, 128), (3, 5)]:
        counts = r.integers(0, 40, size=(n_src, E_loc)).astype(np.int32)
        counts[r.random(size=counts.shape) < 0.2] = 0          # empty (source, expert) cells
        R = int(counts.sum())
        full = [np.concatenate([np.zeros(0, np.int64), c.astype(np.int64)]) for c in counts]
        loc_ref, perm_ref = O.ep_receive(full, 0, E_loc)
        d_counts = torch.from_numpy(counts).cuda()
        loc = torch.empty(E_loc + 1, dtype=torch.int32, device="cuda")
        perm = torch.empty(R, dtype=torch.int32, device="cuda")
        inv = torch.empty(R, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        M.moe_ep_receive_layout(d_counts, loc, perm, inv, device_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(loc.cpu().numpy(), loc_ref)
        assert np.array_equal(perm.cpu().numpy(), perm_ref)
        pi = perm.cpu().numpy().astype(np.int64)
        assert np.array_equal(inv.cpu().numpy()[pi], np.arange(R))


def test_gather_rows_kernel():
    src = torch.randn(50, 264, device="cuda").to(torch.bfloat16)
    idx = torch.tensor([0, 7, 7, 49, 12, 3], dtype=torch.int32, device="cuda")
    dst = torch.empty(6, 264, dtype=torch.bfloat16, device="cuda")
    M.moe_gather_rows(src, idx, 1, dst)
    assert torch.equal(dst.view(torch.int16), src[idx.long()].view(torch.int16))
    idx3 = torch.tensor([5, 148, 0, 2], dtype=torch.int32, device="cuda")     # div 3: rows 1, 49, 0, 0
    dst3 = torch.empty(4, 264, dtype=torch.bfloat16, device="cuda")
    M.moe_gather_rows(src, idx3, 3, dst3)
    assert torch.equal(dst3.view(torch.int16), src[(idx3 // 3).long()].view(torch.int16))
    # a row index outside the source: zero row, reported
    bad = torch.tensor([1, 50], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dstb = torch.full((2, 264), 1.0, dtype=torch.bfloat16, device="cuda")
    M.moe_gather_rows(src, bad, 1, dstb, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5
    assert torch.equal(dstb[0], src[1]) and torch.count_nonzero(dstb[1]) == 0


def _run_ep_train(name, seed=0):
    """Forward and backward of the expert-parallel layer, ranks as threads."""
    E, world, Ts, k, H, I, bs = CASES[name]
    w = G.Workload(name, T=sum(Ts), H=H, E=E, k=k, I=I, bias_std=bs)
    di = U.DeviceInputs(w, seed=seed, with_grad=True)
    b = ep.expert_ranges(E, world)
    ex = ThreadExchange(world)
    starts = np.cumsum([0] + Ts)
    layers = [ep.ExpertParallelMoe((Ts[r], H, E, k, I), r, world, ex.rank_view(r), with_backward=True)
              for r in range(world)]
    grads, errs = [None] * world, []

    def run(r):
        try:
            sl = slice(int(starts[r]), int(starts[r + 1]))
            xr = di.x[sl].contiguous()
            wgu, wd = di.w_gate_up[b[r]:b[r + 1]].contiguous(), di.w_down[b[r]:b[r + 1]].contiguous()
            layers[r].forward(xr, di.w_router, wgu, wd, di.router_bias)
            grads[r] = layers[r].backward(di.grad_out[sl].contiguous(), xr, di.w_router, wgu, wd,
                                          with_bias=True)
            torch.cuda.synchronize()
        except Exception as e:   # surfaced below
            errs.append(e)
            ex.barrier.abort()

    th = [threading.Thread(target=run, args=(r,)) for r in range(world)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    if errs:
        raise errs[0]
    for L in layers:
        assert L.ops.status() == 0
    return di, w, layers, grads


@pytest.mark.parametrize("name", list(CASES))
def test_expert_parallel_backward_bit_exact_against_one_gpu(name):
    """grad_x and every local expert's weight gradients equal moe_layer_bwd on
    all ranks' tokens with the ranks' routing bit for bit; the router's weight
    and bias gradients, formed by each rank over its own tokens, add up to the
    one-GPU ones within their rounding."""
    di, w, layers, grads = _run_ep_train(name)
    E, world = w.E, CASES[name][1]
    idx, tw, _, _, _ = _one_gpu_with_ranks_routing(di, w, layers)
    dims = (w.T, w.H, w.E, w.k, w.I, 0)
    ws = torch.zeros(M.moe_workspace_size(dims, True), dtype=torch.uint8, device="cuda")
    S = w.T * w.k
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(S, dtype=torch.int32, device="cuda")
    inv = torch.empty(S, dtype=torch.int32, device="cuda")
    M.moe_permute(dims, idx, off, perm, inv, ws)
    y = torch.empty(S, w.H, dtype=torch.bfloat16, device="cuda")
    gu = torch.empty(S, 2 * w.I, dtype=torch.bfloat16, device="cuda")
    M.moe_grouped_mlp_fwd(dims, di.x, off, perm, di.w_gate_up, di.w_down, gu, y, None, None, None,
                          None, ws)
    gx = torch.empty(w.T, w.H, dtype=torch.bfloat16, device="cuda")
    gwr = torch.empty(E, w.H, dtype=torch.bfloat16, device="cuda")
    gb = torch.empty(E, dtype=torch.float32, device="cuda")
    gwgu = torch.empty_like(di.w_gate_up)
    gwd = torch.empty_like(di.w_down)
    M.moe_layer_bwd(dims, di.grad_out, di.x, di.w_router, idx, tw, off, perm, inv, di.w_gate_up,
                    di.w_down, gu, None, None, None, gx, gwr, gb, gwgu, gwd, None, None, ws)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(ws) == 0
    got_x = torch.cat([g["grad_x"] for g in grads])
    assert torch.equal(got_x.view(torch.int16), gx.view(torch.int16))
    b = ep.expert_ranges(E, world)
    for r in range(world):
        assert torch.equal(grads[r]["grad_w_gate_up"].view(torch.int16),
                           gwgu[b[r]:b[r + 1]].view(torch.int16)), r
        assert torch.equal(grads[r]["grad_w_down"].view(torch.int16),
                           gwd[b[r]:b[r + 1]].view(torch.int16)), r
    # router: per-rank bf16 parts against the one-GPU bf16 whole
    parts = [g["grad_w_router"].double().cpu() for g in grads]
    one = gwr.double().cpu()
    err = (sum(parts) - one).abs()
    bound = 2.0 ** -7 * (sum(p.abs() for p in parts) + one.abs()) + 1e-6 * float(one.abs().max())
    assert bool((err <= bound).all()), float((err - bound).max())
    bsum = sum(g["grad_router_bias"].double().cpu() for g in grads)
    assert torch.allclose(bsum, gb.double().cpu(), rtol=1e-4, atol=1e-6 * float(gb.abs().max()))
