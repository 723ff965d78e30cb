"""Helpers shared by the GPU parity tests: device upload of the seeded inputs,
running the layer through the C ABI, and the bf16 tolerance check.

Tolerance (bf16 outputs and gradients, fp32 accumulation): relative L2 error
<= 1e-2 and max-abs error <= 2e-2 * max|reference|.  The absolute bound is
scaled by the reference magnitude because the tiny workload's outputs are
~1e-4 (an unscaled 2e-2 would accept anything there) while summed weight
gradients reach magnitudes where one bf16 rounding alone exceeds 2e-2.
"""

from __future__ import annotations

import numpy as np
import torch

from grouped_expert_gemm_top_b300 import inputs as G
from grouped_expert_gemm_top_b300 import moe as M
from oracle import moe_oracle as O

REL_L2 = 1e-2
MAX_ABS_FRAC = 2e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(a) -> torch.Tensor | None:
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_close(got, ref, name, rel_l2=REL_L2, frac=MAX_ABS_FRAC):
    got = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    diff = got - ref
    nref = np.linalg.norm(ref)
    rl2 = np.linalg.norm(diff) / (nref if nref > 0 else 1.0)
    mabs = float(np.abs(diff).max()) if diff.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    if nref == 0:
        assert mabs == 0.0, f"{name}: expected exact zeros, max-abs {mabs}"
        return dict(rel_l2=0.0, max_abs=0.0)
    assert rl2 <= rel_l2, f"{name}: rel-L2 {rl2:.3e} > {rel_l2}"
    assert mabs <= frac * scale, f"{name}: max-abs {mabs:.3e} > {frac} * {scale:.3e}"
    return dict(rel_l2=rl2, max_abs=mabs)


def oracle_backward_with_device_gu(di, f, gu_dev, x=None, grad_out=None, aux_coef=None):
    """The oracle's backward from the device's own bf16 gate/up pre-activations.

    The router bias gradient db[e] = sum_t dlogit[t, e] sums terms that nearly
    cancel: dlogit_j = w_j (dw_j - sum_i w_i dw_i) cancels within a token and
    the tokens' contributions cancel again per expert (db can be ~1/500 of
    sum_t |dlogit[t, e]|).  The device forms dw = <grad_out W_down, h> from
    its saved bf16 (g, u), so that one rounding of g and u moves db by up to
    a few percent of itself while every other gradient stays far inside the
    tolerance.  As with the routing (compared on the device's fp32 logits),
    the device's (g, u) go in here and everything after them (h, y, dw, the
    logit gradient and its sums) is the oracle's, in float64.

    f: the oracle forward dict; gu_dev [S, 2I] (device tensor): the device's
    saved (g, u) in f's sorted row order (rows of dropped slots, which the
    device never writes, are ignored)."""
    w = di.w
    I = w.I
    keep = f["keep"].ravel()[f["perm_slot"]]
    kept = torch.from_numpy(keep).to(gu_dev.device)[:, None]
    gu_dev = torch.where(kept, gu_dev, torch.zeros((), dtype=gu_dev.dtype, device=gu_dev.device))
    gu_dev = gu_dev.double().cpu().numpy()
    gu = f["gu_perm"].copy()
    gu[keep] = gu_dev[keep]
    wd = di.f64("w_down")
    y = np.zeros_like(f["y_perm"])
    off = f["expert_offsets"]
    for e in range(w.E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            y[r0:r1] = (O.silu(gu[r0:r1, :I]) * gu[r0:r1, I:]) @ wd[e].T
    f2 = dict(f, gu_perm=gu, y_perm=y)
    x = di.f64("x") if x is None else x
    grad_out = di.f64("grad_out") if grad_out is None else grad_out
    return O.layer_backward(f2, grad_out, x, di.f64("w_router"), di.f64("w_gate_up"), wd, w.k,
                            w_sh_gu=di.f64("w_sh_gate_up"), w_sh_down=di.f64("w_sh_down"),
                            aux_coef=aux_coef)


def check_bias_grad(got, di, f, gu_dev, name="grad_router_bias", **kw):
    """The router bias gradient at the common tolerance against the oracle's
    backward from the device's own (g, u) (see oracle_backward_with_device_gu)."""
    b = oracle_backward_with_device_gu(di, f, gu_dev, **kw)
    return check_close(got, b["grad_router_bias"], name)


class DeviceInputs:
    """Seeded inputs on the device (bf16 tensors) plus their float64 copies."""

    def __init__(self, w: G.Workload, seed=0, with_grad=None):
        self.w = w
        self.np = G.make_inputs(w, seed, with_grad)
        self._f64 = {}
        n = self.np
        self.x = dev_bf16(n["x"])
        self.w_router = dev_bf16(n["w_router"])
        self.w_gate_up = dev_bf16(n["w_gate_up"])
        self.w_down = dev_bf16(n["w_down"])
        self.router_bias = dev_f32(n["router_bias"])
        self.w_sh_gate_up = dev_bf16(n["w_sh_gate_up"]) if n["w_sh_gate_up"] is not None else None
        self.w_sh_down = dev_bf16(n["w_sh_down"]) if n["w_sh_down"] is not None else None
        self.grad_out = dev_bf16(n["grad_out"]) if n["grad_out"] is not None else None

    def f64(self, key):
        """float64 copy of an input, widened once and kept (full-size weights are GBs)."""
        if key not in self._f64:
            v = self.np[key]
            if v is None:
                return None
            self._f64[key] = O.widen_bf16(v) if v.dtype == np.uint16 else v.astype(np.float64)
        return self._f64[key]

    @property
    def dims(self):
        w = self.w
        return (w.T, w.H, w.E, w.k, w.I, w.I_shared)


def run_forward(di: DeviceInputs, with_backward=True, save_logits=True):
    layer = M.MoeLayer(di.dims, gate_mode=di.w.gate, with_backward=with_backward,
                       save_logits=save_logits)
    layer.forward(di.x, di.w_router, di.w_gate_up, di.w_down, di.router_bias, di.w_sh_gate_up,
                  di.w_sh_down)
    torch.cuda.synchronize()
    return layer


def oracle_forward(di: DeviceInputs, topk_idx=None, capacity=None):
    return O.layer_forward(di.f64("x"), di.f64("w_router"), di.f64("w_gate_up"), di.f64("w_down"),
                           di.w.k, balanced=di.w.gate == G.GATE_BALANCED,
                           bias=di.f64("router_bias"), w_sh_gu=di.f64("w_sh_gate_up"),
                           w_sh_down=di.f64("w_sh_down"), topk_idx=topk_idx, capacity=capacity)


def logit_error_bound(x64, wr64):
    """Deterministic bound on |fp32-accumulated logit - exact logit| per (t, e):
    H * 2^-23 * sum_h |x[t,h] W[e,h]| (twice the recursive-summation bound) plus
    one rounding of the bias add."""
    H = x64.shape[1]
    return H * 2.0 ** -23 * (np.abs(x64) @ np.abs(wr64).T) + 2.0 ** -22 * (np.abs(x64) @ np.abs(wr64).T).max()
