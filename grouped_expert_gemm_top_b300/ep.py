"""Expert-parallel forward of the MoE layer: dispatch to the experts' ranks,
local grouped experts, combine back.

NeMo AutoModel blog, "专家并行与 DeepEP": expert parallelism is a mesh
dimension of its own beside data parallelism; every rank trains on its own
tokens and holds 1/ep of the experts, split along the expert dimension
(DTensor Shard(0)); DeepEP dispatches the tokens to the ranks of their
experts and combines the outputs back (all-to-all).

Per rank, one forward:

1. route and sort its own tokens over all E experts (``moe_route_permute``);
   expert order is rank order (each rank's experts are contiguous, the
   Shard(0) chunks), so the sorted slots form one block per destination;
2. send every rank its expert counts, then the token rows of its block
   (``moe_gather_rows`` lays them out in sorted order);
3. group what it received by local expert (``moe_ep_receive_layout``) and run
   its experts on it (``moe_grouped_mlp_fwd``: T = rows received, k = 1,
   E = local experts, perm_slot = the grouping);
4. put the outputs back in receive order (``moe_gather_rows``) and send each
   source its rows; the source now holds its slots' outputs in its own sorted
   order and combines them (``moe_unpermute_combine``).

The rows of an expert meet on its rank in global slot order (sources in rank
order, each in its slot order), as on one GPU, so with tokens numbered rank
by rank the result equals the one-GPU layer's.

The backward (``ExpertParallelMoe.backward``, for a layer built with
``with_backward=True``) is the reverse trip: each source sends its slots'
grad_out rows (``moe_gather_rows``) and routing weights
(``moe_gather_scalars``) in its sorted order, as it sent the token rows; the
experts' rank runs ``moe_experts_bwd`` on them (the saved pre-activations of
its forward) and sends each row's dx and dL/dw back; the source runs
``moe_router_bwd``.  Every gradient equals the one-GPU ``moe_layer_bwd``'s
bit for bit except the router's, which each rank forms over its own tokens:
the caller sums it over the ranks, as data parallelism sums any replicated
parameter's gradient.

The exchange is an object with ``all_to_all_single(out, inp, out_splits,
in_splits)`` along dim 0 (a torch.distributed process group wrapper, see
``DistExchange``); bf16 rows travel as int16 words.  The compute steps are the
library's kernels (``DeviceOps``); every step runs on the device, and the
split sizes come to the host once per exchange, as all-to-all needs them.
"""

from __future__ import annotations

import torch

from . import moe as M


def expert_ranges(E: int, world: int) -> list[int]:
    """Rank r owns experts bounds[r] .. bounds[r+1]-1: chunks of ceil(E / world)
    in rank order, as Shard(0) splits the expert dimension."""
    c = -(-E // world)
    return [min(r * c, E) for r in range(world + 1)]


class DistExchange:
    """all_to_all_single over a torch.distributed process group; `device` is
    where the group's tensors live (the current GPU for NCCL, the host for gloo)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist, self.group = dist, group
        nccl = dist.get_backend(group) == "nccl"
        self.device = torch.device("cuda", torch.cuda.current_device()) if nccl else torch.device("cpu")

    def all_to_all_single(self, out, inp, out_splits, in_splits):
        self.dist.all_to_all_single(out, inp, list(out_splits), list(in_splits), group=self.group)


class DeviceOps:
    """The forward's compute steps, each one or two library kernels on the device."""

    def __init__(self, dims, gate_mode, device, with_backward=False):
        self.dims = M.MoeDims.of(*M._dims(dims).as_tuple())
        self.gate_mode = gate_mode
        self.device = torch.device(device)
        # a rank without tokens still takes part in the exchanges (routes nothing)
        nbytes = M.moe_workspace_size(self.dims, with_backward) if self.dims.T > 0 else 256
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        self._loc_ws = None

    def route_permute(self, x, w_router, router_bias):
        T, H, E, k, I, _ = self.dims.as_tuple()
        dev, i32, f32 = self.device, torch.int32, torch.float32
        idx = torch.empty(T, k, dtype=i32, device=dev)
        w = torch.empty(T, k, dtype=f32, device=dev)
        off = torch.zeros(E + 1, dtype=i32, device=dev)
        perm = torch.empty(T * k, dtype=i32, device=dev)
        inv = torch.empty(T * k, dtype=i32, device=dev)
        if T > 0:
            M.moe_route_permute(self.dims, self.gate_mode, x, w_router, router_bias, None, idx, w,
                                off, perm, inv, self.ws)
        return idx, w, off, perm, inv

    def gather_rows(self, src, idx, div):
        dst = torch.empty(idx.numel(), src.shape[1], dtype=src.dtype, device=self.device)
        M.moe_gather_rows(src, idx, div, dst, device_status=self.ws.view(torch.int32)[:1])
        return dst

    def receive_layout(self, counts):
        n_src, E_loc = counts.shape
        R = int(counts.sum().item()) if counts.numel() else 0
        i32 = torch.int32
        loc_off = torch.empty(E_loc + 1, dtype=i32, device=self.device)
        recv_perm = torch.empty(R, dtype=i32, device=self.device)
        recv_inv = torch.empty(R, dtype=i32, device=self.device)
        M.moe_ep_receive_layout(counts.to(self.device, torch.int32).contiguous(), loc_off,
                                recv_perm, recv_inv, device_status=self.ws.view(torch.int32)[:1])
        return loc_off, recv_perm, recv_inv

    def _local_ws(self, d, with_backward):
        need = M.moe_workspace_size(d, with_backward)
        if self._loc_ws is None or self._loc_ws.numel() < need:
            self._loc_ws = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self._loc_ws

    def experts(self, x_recv, loc_off, recv_perm, w_gate_up_local, w_down_local, gu_out=None):
        R, H = x_recv.shape
        E_loc = w_gate_up_local.shape[0]
        I = w_down_local.shape[2]
        y = torch.empty(R, H, dtype=torch.bfloat16, device=self.device)
        d = M.MoeDims.of(R, H, E_loc, 1, I, 0)
        M.moe_grouped_mlp_fwd(d, x_recv, loc_off, recv_perm, w_gate_up_local, w_down_local, gu_out,
                              y, None, None, None, None, self._local_ws(d, gu_out is not None))
        return y

    def gather_scalars(self, src, idx, div):
        dst = torch.empty(idx.numel(), dtype=src.dtype, device=self.device)
        M.moe_gather_scalars(src, idx, div, dst, device_status=self.ws.view(torch.int32)[:1])
        return dst

    def experts_bwd(self, go_recv, x_recv, w_recv, loc_off, recv_perm, recv_inv, w_gate_up_local,
                    w_down_local, gu_saved):
        """Each received row's dx and dL/dw (receive order) and the local
        experts' weight gradients."""
        R, H = x_recv.shape
        E_loc = w_gate_up_local.shape[0]
        I = w_down_local.shape[2]
        d = M.MoeDims.of(R, H, E_loc, 1, I, 0)
        dx = torch.empty(R, H, dtype=torch.bfloat16, device=self.device)
        dw = torch.empty(R, dtype=torch.float32, device=self.device)
        gwgu = torch.empty_like(w_gate_up_local)
        gwd = torch.empty_like(w_down_local)
        M.moe_experts_bwd(d, go_recv, x_recv, w_recv, loc_off, recv_perm, recv_inv, w_gate_up_local,
                          w_down_local, gu_saved, dx, dw, gwgu, gwd, self._local_ws(d, True))
        return dx, dw, gwgu, gwd

    def router_bwd(self, x, w_router, idx, w, off, perm, inv, dx_sorted, dw_sorted, with_bias):
        T, H = x.shape
        E = w_router.shape[0]
        gx = torch.empty(T, H, dtype=torch.bfloat16, device=self.device)
        gwr = torch.zeros(E, H, dtype=torch.bfloat16, device=self.device)
        gb = torch.zeros(E, dtype=torch.float32, device=self.device) if with_bias else None
        if T > 0:
            M.moe_router_bwd(self.dims, x, w_router, idx, w, off, perm, inv, dx_sorted, dw_sorted,
                             gx, gwr, gb, self.ws)
        return gx, gwr, gb

    def combine(self, y_sorted, slot_perm, topk_w):
        T, H = self.dims.T, self.dims.H
        out = torch.empty(T, H, dtype=torch.bfloat16, device=self.device)
        if T > 0:
            M.moe_unpermute_combine(self.dims, y_sorted, slot_perm, topk_w, None, out)
        return out

    def status(self) -> int:
        return M.moe_read_device_status(self.ws)


class ExpertParallelMoe:
    """One rank of the expert-parallel layer (forward).

    dims = (T, H, E, k, I) of this rank's tokens and the global expert count;
    the rank holds w_gate_up / w_down of its experts only ([E_local, 2I, H] and
    [E_local, H, I], the Shard(0) chunk) and the whole router.
    """

    def __init__(self, dims, rank: int, world: int, exchange, gate_mode=M.MOE_GATE_SOFTMAX_TOPK,
                 device="cuda", ops=None, with_backward=False):
        T, H, E, k, I = dims[:5]
        self.T, self.H, self.E, self.k, self.I = T, H, E, k, I
        self.rank, self.world = rank, world
        self.bounds = expert_ranges(E, world)
        self.lo, self.hi = self.bounds[rank], self.bounds[rank + 1]
        self.exchange = exchange
        self.with_backward = with_backward
        self.ops = ops if ops is not None else DeviceOps((T, H, E, k, I, 0), gate_mode, device,
                                                         with_backward)
        self.last = {}

    def _xdev(self):
        return getattr(self.exchange, "device", torch.device("cpu"))

    def _a2a_rows(self, rows, in_splits, out_splits):
        """Rows [n, H] (bf16) to the ranks, block q to rank q; returns what arrives."""
        xdev = self._xdev()
        src = rows if rows.device == xdev else rows.to(xdev)
        out = torch.empty(sum(out_splits), rows.shape[1], dtype=rows.dtype, device=xdev)
        if rows.dtype == torch.bfloat16:
            self.exchange.all_to_all_single(out.view(torch.int16), src.view(torch.int16),
                                            out_splits, in_splits)
        else:
            self.exchange.all_to_all_single(out, src, out_splits, in_splits)
        return out if out.device == rows.device else out.to(rows.device)

    def _a2a_vec(self, v, in_splits, out_splits):
        """One value a row (fp32), block q to rank q; returns what arrives."""
        xdev = self._xdev()
        src = v if v.device == xdev else v.to(xdev)
        out = torch.empty(sum(out_splits), dtype=v.dtype, device=xdev)
        self.exchange.all_to_all_single(out, src, out_splits, in_splits)
        return out if out.device == v.device else out.to(v.device)

    def forward(self, x, w_router, w_gate_up_local, w_down_local, router_bias=None):
        ops, b, n = self.ops, self.bounds, self.world
        assert w_gate_up_local.shape[0] == self.hi - self.lo
        # 1. route and sort this rank's tokens over all experts
        idx, w, off, perm, inv = ops.route_permute(x, w_router, router_bias)
        off_h = off.cpu().tolist()
        counts = torch.tensor([off_h[e + 1] - off_h[e] for e in range(self.E)], dtype=torch.int32)
        send_rows = [off_h[b[q + 1]] - off_h[b[q]] for q in range(n)]
        # 2. every rank learns how many rows of each of its experts this rank sends
        e_splits = [b[q + 1] - b[q] for q in range(n)]
        E_loc = self.hi - self.lo
        xdev = self._xdev()
        recv_counts = torch.empty(n * E_loc, dtype=torch.int32, device=xdev)
        self.exchange.all_to_all_single(recv_counts, counts.to(xdev), [E_loc] * n, e_splits)
        recv_counts = recv_counts.view(n, E_loc).cpu()
        recv_rows = [int(v) for v in recv_counts.sum(dim=1).tolist()] if E_loc else [0] * n
        # 3. the token rows, in sorted order, block q to rank q
        x_send = ops.gather_rows(x, perm, self.k)
        x_recv = self._a2a_rows(x_send, send_rows, recv_rows)
        # 4. the local experts on the rows grouped by expert
        R = sum(recv_rows)
        gu = None
        if E_loc and R:
            loc_off, recv_perm, recv_inv = ops.receive_layout(recv_counts)
            if self.with_backward:   # the experts' pre-activations, for the backward
                gu = torch.empty(R, 2 * self.I, dtype=torch.bfloat16, device=x_recv.device)
            y_grouped = ops.experts(x_recv, loc_off, recv_perm, w_gate_up_local, w_down_local, gu)
            y_recv = ops.gather_rows(y_grouped, recv_inv, 1)
        else:
            loc_off = recv_perm = recv_inv = None
            y_recv = torch.empty(0, self.H, dtype=x_send.dtype, device=x_send.device)
        # 5. outputs back to their sources, then the weighted combine
        y_sorted = self._a2a_rows(y_recv, recv_rows, send_rows)
        out = ops.combine(y_sorted, inv, w)
        self.last = dict(topk_idx=idx, topk_w=w, expert_offsets=off, perm_slot=perm, slot_perm=inv,
                         send_rows=send_rows, recv_rows=recv_rows, recv_counts=recv_counts,
                         x_recv=x_recv, local_offsets=loc_off, recv_perm=recv_perm,
                         recv_inv=recv_inv, y_sorted=y_sorted, gu_saved=gu)
        return out

    def backward(self, grad_out, x, w_router, w_gate_up_local, w_down_local, with_bias=False):
        """Gradients of the last forward (built with with_backward=True).

        Returns grad_x [T, H] (this rank's tokens), grad_w_gate_up /
        grad_w_down of the local experts, and grad_w_router (and
        grad_router_bias with with_bias) over this rank's tokens: sum those
        over the ranks.
        """
        if not self.with_backward:
            raise RuntimeError("the layer was built without with_backward=True")
        ops, L = self.ops, self.last
        send_rows, recv_rows = L["send_rows"], L["recv_rows"]
        perm = L["perm_slot"]
        # 1. this rank's slots' grad_out rows and weights, in its sorted order
        go_send = ops.gather_rows(grad_out, perm, self.k)
        w_send = ops.gather_scalars(L["topk_w"].reshape(-1), perm, 1)
        go_recv = self._a2a_rows(go_send, send_rows, recv_rows)
        w_recv = self._a2a_vec(w_send, send_rows, recv_rows)
        # 2. the local experts: each received row's dx and dL/dw, the weight gradients
        E_loc = self.hi - self.lo
        R = sum(recv_rows)
        if E_loc and R:
            dx_recv, dw_recv, gwgu, gwd = ops.experts_bwd(
                go_recv, L["x_recv"], w_recv, L["local_offsets"], L["recv_perm"], L["recv_inv"],
                w_gate_up_local, w_down_local, L["gu_saved"])
        else:   # no rows: exact-zero weight gradients
            dx_recv = torch.empty(0, self.H, dtype=go_send.dtype, device=go_send.device)
            dw_recv = torch.empty(0, dtype=w_send.dtype, device=w_send.device)
            gwgu, gwd = torch.zeros_like(w_gate_up_local), torch.zeros_like(w_down_local)
        # 3. back to their sources, then the router's backward there
        dx_sorted = self._a2a_rows(dx_recv, recv_rows, send_rows)
        dw_sorted = self._a2a_vec(dw_recv, recv_rows, send_rows)
        gx, gwr, gb = ops.router_bwd(x, w_router, L["topk_idx"], L["topk_w"], L["expert_offsets"],
                                     perm, L["slot_perm"], dx_sorted, dw_sorted, with_bias)
        self.last.update(go_recv=go_recv, w_recv=w_recv, dx_recv=dx_recv, dw_recv=dw_recv,
                         dx_sorted=dx_sorted, dw_sorted=dw_sorted)
        return dict(grad_x=gx, grad_w_router=gwr, grad_router_bias=gb, grad_w_gate_up=gwgu,
                    grad_w_down=gwd)
