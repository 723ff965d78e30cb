"""Host-fed layer steps with the host<->device copies overlapped.

A forward+backward step whose inputs (x, grad_out) arrive from pinned host
memory and whose results (out, grad_x) go back to it.  Two device slots hold
each step's inputs and read-back results.  The host-to-device copies of step
i+1 run on one stream and the device-to-host copies of step i-1 on another,
while step i computes on the caller's stream, ordered by CUDA events:

  * slot s's inputs are overwritten only after the step that last read them
    (two steps earlier) has finished computing;
  * a step writes its out/grad_x into slot s only after the read-back of the
    step that last used the slot has finished.

Within a step the forward and the backward are ordered separately: the
forward waits only for x, the backward for grad_out, and out goes back as
soon as the forward has written it, so a step's grad_out copy and out
read-back overlap its own compute (this matters for the first and last steps
of a run, which have no neighbours to hide behind).

Every copy still happens once per step; only their overlap with compute
changes.  This is stream plumbing: the copies are cudaMemcpyAsync (through
torch), and every step of the layer runs in the library's kernels.
"""

from __future__ import annotations

import torch


class HostStepPipeline:
    """Runs MoeLayer forward+backward steps fed from pinned host buffers.

    layer: a MoeLayer built with_backward=True; grads: its alloc_grads()
    dict (weight gradients stay on the device, overwritten every step);
    weights: dict with w_router, w_gate_up, w_down and optionally
    router_bias, w_sh_gate_up, w_sh_down (device tensors).  use_graph: run
    each slot's step as a captured CUDA graph (one per slot, captured here
    after an eager warm-up step) instead of call by call.
    """

    def __init__(self, layer, grads, weights, slots: int = 2, use_graph: bool = True):
        self.layer, self.grads, self.w = layer, grads, weights
        T, H = layer.out.shape
        dev = layer.out.device
        bf = torch.bfloat16
        self.n = slots
        # zeroed: the graph capture's warm-up step reads them before any data
        self.x = [torch.zeros(T, H, dtype=bf, device=dev) for _ in range(slots)]
        self.go = [torch.zeros(T, H, dtype=bf, device=dev) for _ in range(slots)]
        self.out = [torch.empty(T, H, dtype=bf, device=dev) for _ in range(slots)]
        self.gx = [torch.empty(T, H, dtype=bf, device=dev) for _ in range(slots)]
        self.h2d = torch.cuda.Stream(device=dev)
        self.d2h = torch.cuda.Stream(device=dev)
        ev = lambda: [torch.cuda.Event() for _ in range(slots)]
        self.x_ready, self.go_ready = ev(), ev()
        self.fwd_done, self.computed = ev(), ev()
        self.out_back, self.gx_back = ev(), ev()
        self.used = [False] * slots
        self.i = 0
        self.graphs = None
        if use_graph:
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                for s in range(slots):
                    self._forward(s)
                    self._backward(s)
            torch.cuda.current_stream(dev).wait_stream(side)
            self.graphs = []
            for s in range(slots):
                gf, gb = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.graph(gf):
                    self._forward(s)
                with torch.cuda.graph(gb):
                    self._backward(s)
                self.graphs.append((gf, gb))

    def _forward(self, s):
        w = self.w
        self.layer.forward(self.x[s], w["w_router"], w["w_gate_up"], w["w_down"],
                           w.get("router_bias"), w.get("w_sh_gate_up"), w.get("w_sh_down"),
                           out=self.out[s])

    def _backward(self, s):
        w = self.w
        g = dict(self.grads)
        g["grad_x"] = self.gx[s]
        self.layer.backward(self.go[s], self.x[s], w["w_router"], w["w_gate_up"], w["w_down"], g,
                            w.get("w_sh_gate_up"), w.get("w_sh_down"))

    def step(self, x_host, go_host, out_host, gx_host):
        """Enqueue one step: x_host, go_host in; out_host, gx_host written back.

        Asynchronous: out_host/gx_host are valid after drain() (or a device
        synchronize); a host buffer handed to a later step is not read
        before this step's copies have been issued."""
        s = self.i % self.n
        compute = torch.cuda.current_stream(self.x[s].device)
        with torch.cuda.stream(self.h2d):
            if self.used[s]:
                self.h2d.wait_event(self.computed[s])   # the step that last read slot s
            self.x[s].copy_(x_host, non_blocking=True)
            self.x_ready[s].record(self.h2d)
            self.go[s].copy_(go_host, non_blocking=True)
            self.go_ready[s].record(self.h2d)
        compute.wait_event(self.x_ready[s])
        if self.used[s]:
            compute.wait_event(self.out_back[s])        # slot s's out was read back
        if self.graphs is not None:
            self.graphs[s][0].replay()
        else:
            self._forward(s)
        self.fwd_done[s].record(compute)
        compute.wait_event(self.go_ready[s])
        if self.used[s]:
            compute.wait_event(self.gx_back[s])         # slot s's grad_x was read back
        if self.graphs is not None:
            self.graphs[s][1].replay()
        else:
            self._backward(s)
        self.computed[s].record(compute)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.fwd_done[s])
            out_host.copy_(self.out[s], non_blocking=True)
            self.out_back[s].record(self.d2h)
            self.d2h.wait_event(self.computed[s])
            gx_host.copy_(self.gx[s], non_blocking=True)
            self.gx_back[s].record(self.d2h)
        self.used[s] = True
        self.i += 1

    def drain(self):
        """Make the caller's stream wait for every copy issued so far."""
        compute = torch.cuda.current_stream(self.x[0].device)
        for s in range(self.n):
            if self.used[s]:
                compute.wait_event(self.out_back[s])
                compute.wait_event(self.gx_back[s])

    @property
    def h2d_bytes_per_step(self) -> int:
        return (self.x[0].numel() + self.go[0].numel()) * 2

    @property
    def d2h_bytes_per_step(self) -> int:
        return (self.out[0].numel() + self.gx[0].numel()) * 2


class StepGraph:
    """One forward+backward step of a MoeLayer captured as a CUDA graph.

    The step reads its inputs from the caller's device buffers x and
    grad_out (copy new data into them before each replay) and writes
    layer.out and grads as the eager step does; with grad_out None (and
    grads None) it is the forward alone.  replay() launches every
    kernel of the step at once from the graph instead of one call at a time
    from the host.  The library's calls are stream-ordered and never
    synchronise, so they capture as they are; the eager warm-up steps before
    the capture make every one-time host set-up happen outside it.
    """

    def __init__(self, layer, grads, weights, x, grad_out=None, warmup: int = 2):
        self.layer, self.grads, self.w = layer, grads, weights
        self.x, self.grad_out = x, grad_out
        side = torch.cuda.Stream(device=x.device)
        side.wait_stream(torch.cuda.current_stream(x.device))
        with torch.cuda.stream(side):
            for _ in range(warmup):
                self._step()
        torch.cuda.current_stream(x.device).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._step()

    def _step(self):
        w = self.w
        self.layer.forward(self.x, w["w_router"], w["w_gate_up"], w["w_down"], w.get("router_bias"),
                           w.get("w_sh_gate_up"), w.get("w_sh_down"))
        if self.grad_out is None:
            return
        self.layer.backward(self.grad_out, self.x, w["w_router"], w["w_gate_up"], w["w_down"],
                            self.grads, w.get("w_sh_gate_up"), w.get("w_sh_down"))

    def replay(self):
        self.graph.replay()
