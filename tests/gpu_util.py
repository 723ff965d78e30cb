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


BIAS_SIGMAS = 8.0


def bias_grad_bound(di, f, dl, grad_out=None, aux_coef=None):
    """Per-expert bound on |db_device[e] - db_oracle[e]| for the router bias
    gradient db[e] = sum_t dlogit[t, e], derived from the device's arithmetic.

    The device's one large error source is the bf16 rounding (relative error
    at most 2^-8, round to nearest even) of the gate/up pre-activations g, u
    it saves and differentiates through; everything else it computes in fp32.
    Slot j of token t (expert e_j, weight w_j) has
        dw_j = sum_i a_i h_i,  a = dout[t] W_down[e_j] (fp32 from exact bf16
        inputs), h = silu(g) u,
    and a rounding g -> g(1 + eg), u -> u(1 + eu) moves h_i by
    silu'(g) u g eg + silu(g) u eu.  Treating the rounding errors as
    independent, zero-mean and no wider than uniform on [-2^-8, 2^-8]
    (variance at most 2^-16 / 3):
        var(ddw_j) <= 2^-16/3 * sum_i a_i^2 ((silu'(g_i) u_i g_i)^2 + (silu(g_i) u_i)^2).
    dlogit_j = w_j (dw_j - sum_i w_i dw_i) (the renormalised weights are a
    softmax over the selected logits), so with independent slots
        var(ddl_j) = w_j^2 ((1 - w_j)^2 var_j + sum_{i != j} w_i^2 var_i),
    and a token's slots go to distinct experts, so var(ddb_e) is the sum of
    var(ddl) over e's slots.  The bound is BIAS_SIGMAS standard deviations of
    that, plus deterministic terms: the fp32 sums and the device's fp32
    routing weights (relative 1e-5 of w_j (|a.h|_1 + sum_i w_i |a.h|_1) per
    slot and of sum_t |dlogit[t, e]|), the auxiliary loss's dense term
    p_e (c_e - <c, p>) formed in fp32 (relative 1e-5 of its absolute terms),
    and a floor of 1e-9 of the largest sum_t |dlogit[t, e]| for the float64
    oracle's own noise (an expert nobody chose has db ~1e-17 there and
    exactly 0 on the device).

    f: oracle forward dict (float64 g, u in gu_perm, routing, keep mask);
    dl: the oracle's dense logit gradient [T, E]; grad_out: float64 [T, H]
    (default the inputs'); aux_coef: the auxiliary loss's c_e, if any.
    """
    w_ = di.w
    I, E, k = w_.I, w_.E, w_.k
    idx, wts = f["topk_idx"], f["topk_w"]
    off, perm = f["expert_offsets"], f["perm_slot"]
    keep = f.get("keep")
    keep = np.ones(idx.shape, dtype=bool) if keep is None else keep
    gu = f["gu_perm"]
    wd = di.f64("w_down")
    go = di.f64("grad_out") if grad_out is None else grad_out
    T = idx.shape[0]
    var = np.zeros((T, k))
    l1 = np.zeros((T, k))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        slots = perm[r0:r1].astype(np.int64)
        tok, j = slots // k, slots % k
        a = go[tok] @ wd[e]
        g, u = gu[r0:r1, :I], gu[r0:r1, I:]
        sg = 1.0 / (1.0 + np.exp(-g))
        silu = g * sg
        dsilu = sg * (1.0 + g * (1.0 - sg))
        v = 2.0 ** -16 / 3.0 * np.sum(a * a * ((dsilu * u * g) ** 2 + (silu * u) ** 2), axis=1)
        kp = keep[tok, j]
        var[tok, j] = np.where(kp, v, 0.0)
        l1[tok, j] = np.where(kp, np.sum(np.abs(a * silu * u), axis=1), 0.0)
    wsq_var = np.sum(wts ** 2 * var, axis=1, keepdims=True)
    var_dl = wts ** 2 * ((1.0 - wts) ** 2 * var + wsq_var - wts ** 2 * var)
    det_dl = 1e-5 * wts * (l1 + np.sum(wts * l1, axis=1, keepdims=True))
    var_e = np.bincount(idx.ravel(), var_dl.ravel(), minlength=E)
    det_e = np.bincount(idx.ravel(), det_dl.ravel(), minlength=E)
    dl_l1 = np.abs(dl).sum(axis=0)
    bound = BIAS_SIGMAS * np.sqrt(var_e) + det_e + 1e-5 * dl_l1 + 1e-9 * dl_l1.max()
    if aux_coef is not None:
        c = np.asarray(aux_coef, dtype=np.float64)
        p = f["p"]
        pc = np.sum(p * np.abs(c)[None, :], axis=1, keepdims=True)
        bound = bound + 1e-5 * np.sum(p * (np.abs(c)[None, :] + pc), axis=0)
    return bound


def check_bias_grad(got, di, f, gu_dev, name="grad_router_bias", x=None, grad_out=None,
                    aux_coef=None):
    """The router bias gradient against the plain float64 oracle, within the
    bound bias_grad_bound derives from the device's arithmetic (db cancels
    twice, so the common relative tolerance does not apply to it); and, as a
    second check, at the common tolerance against the oracle's backward from
    the device's own (g, u) (oracle_backward_with_device_gu)."""
    x64 = di.f64("x") if x is None else x
    go64 = di.f64("grad_out") if grad_out is None else grad_out
    b = O.layer_backward(f, go64, x64, di.f64("w_router"), di.f64("w_gate_up"), di.f64("w_down"),
                         di.w.k, aux_coef=aux_coef)
    g = to_f64(got)
    bound = bias_grad_bound(di, f, b["grad_logits"], grad_out=go64, aux_coef=aux_coef)
    err = np.abs(g - b["grad_router_bias"])
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    worst = int(np.argmax(err / bound))
    assert np.all(err <= bound), (f"{name}: expert {worst} off by {err[worst]:.3e} > bound "
                                  f"{bound[worst]:.3e} (oracle {b['grad_router_bias'][worst]:.3e})")
    b2 = oracle_backward_with_device_gu(di, f, gu_dev, x=x, grad_out=grad_out, aux_coef=aux_coef)
    return check_close(got, b2["grad_router_bias"], name + " (device g,u)")


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


def check_routing_contract2(di, layer):
    """Device top-k ids against the oracle's selection on its own float64
    logits.  The device sums its logits in fp32 in another order, so the two
    can differ only at a near tie: every token whose chosen experts (or their
    order) differ must have the differing experts' exact logits within twice
    the fp32 accumulation bound H 2^-23 sum_h |x w| + 2^-23 (|l| + 1) of each
    other.  No count of differing tokens is allowed beyond that.  Returns the
    number of tokens that differ (all of them near ties)."""
    w = di.w
    x, wr, b = di.f64("x"), di.f64("w_router"), di.f64("router_bias")
    ref = O.router_logits(x, wr, b)
    bound = w.H * 2.0 ** -23 * (np.abs(x) @ np.abs(wr).T) + 2.0 ** -23 * (np.abs(ref) + 1.0)
    idx = layer.topk_idx.cpu().numpy()
    idx2, _, _ = O.route(ref, w.k, balanced=w.gate == G.GATE_BALANCED)
    bad = np.nonzero((idx != idx2).any(axis=1))[0]
    for t in bad:
        diff_e = np.setxor1d(idx[t], idx2[t])
        if diff_e.size == 0:      # same set, order swapped by a tie
            diff_e = idx[t][idx[t] != idx2[t]]
        vals = ref[t, diff_e]
        assert vals.max() - vals.min() <= 2 * bound[t, diff_e].max(), (t, diff_e, vals)
    return int(bad.size)
