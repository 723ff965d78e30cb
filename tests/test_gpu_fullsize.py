"""Parity at the full benchmark shapes, through the same MoeLayer calls bench.py times.

* Qwen3-30B-A3B shape (4096 tokens, hidden 2048, 128 experts, top-8,
  intermediate 768): the float64 oracle runs the whole layer in seconds, so
  every output and gradient is compared in full, for the balanced gate
  (forward + backward) and the skewed softmax gate (forward).
* The shared-expert shape (8192 tokens, hidden 2688, top-6, intermediate
  1856, shared 3712) is too large for the oracle as a whole.  Its routing ids
  and sort are checked in full; the rest through exact sub-problems:
  - a token's out and grad_x depend only on its own slots, so a layer
    restricted to a sample of tokens gives their rows exactly;
  - one expert's weight gradients depend only on the tokens routed to it;
  - the backward is linear in grad_out, so a full-size backward whose
    grad_out is zero outside a token sample gives, for EVERY gradient tensor
    (router, bias, shared expert included), exactly the restricted layer's
    gradients (zeros for untouched experts and tokens).
  Plus a property that holds at any size: softmax gradients sum to zero over
  experts, so the column sums of grad_w_router and the sum of the bias
  gradient vanish up to rounding.
"""

import numpy as np
import pytest
import torch

import gpu_util as U
from grouped_expert_gemm_top_b300 import inputs as G
from grouped_expert_gemm_top_b300 import moe as M
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

GRAD_KEYS = ("grad_x", "grad_w_router", "grad_router_bias", "grad_w_gate_up", "grad_w_down",
             "grad_w_sh_gate_up", "grad_w_sh_down")


def _forward(name):
    w = G.WORKLOADS[name]
    di = U.DeviceInputs(w, seed=0, with_grad=True)
    layer = U.run_forward(di, with_backward=True, save_logits=True)
    assert M.moe_read_device_status(layer.workspace) == 0
    return di, layer


def _backward(di, layer, grad_out):
    grads = layer.alloc_grads(with_bias=di.router_bias is not None)
    layer.backward(grad_out, di.x, di.w_router, di.w_gate_up, di.w_down, grads,
                   di.w_sh_gate_up, di.w_sh_down)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(layer.workspace) == 0
    return grads


def _check_routing(di, layer):
    """Ids bit-exact against the oracle's selection on the device's fp32 logits
    (contract 1) and, for the softmax gate, equal to the selection on the
    oracle's own logits except at near ties (contract 2); sort in full."""
    w = di.w
    idx = layer.topk_idx.cpu().numpy()
    balanced = w.gate == G.GATE_BALANCED
    got = U.to_f64(layer.logits)
    idx1, w1, _ = O.route(got, w.k, balanced=balanced, decision_logits=layer.logits.cpu().numpy())
    assert np.array_equal(idx, idx1)
    assert np.allclose(layer.topk_w.cpu().numpy(), w1, rtol=2e-6, atol=1e-7)
    if balanced:
        assert np.array_equal(idx, O.balanced_topk(w.T, w.E, w.k))
    else:
        # contract 2: against the oracle's own float64 logits, near ties only
        U.check_routing_contract2(di, layer)
    off, perm, inv = O.permute(idx, w.E)
    assert np.array_equal(layer.expert_offsets.cpu().numpy(), off)
    assert np.array_equal(layer.perm_slot.cpu().numpy(), perm)
    assert np.array_equal(layer.slot_perm.cpu().numpy(), inv)
    return idx


def _sub_layer(di, tokens, idx, grad_out=True):
    """Oracle forward (+ backward) of the layer restricted to `tokens`, with their own routing."""
    x = di.f64("x")[tokens]
    wr, wgu, wd = di.f64("w_router"), di.f64("w_gate_up"), di.f64("w_down")
    sh = dict(w_sh_gu=di.f64("w_sh_gate_up"), w_sh_down=di.f64("w_sh_down"))
    f = O.layer_forward(x, wr, wgu, wd, di.w.k, bias=di.f64("router_bias"), topk_idx=idx[tokens], **sh)
    if not grad_out:
        return f, None
    b = O.layer_backward(f, di.f64("grad_out")[tokens], x, wr, wgu, wd, di.w.k, **sh)
    return f, b


def _rows(t, tokens):
    return t[torch.from_numpy(np.asarray(tokens, dtype=np.int64)).to(t.device)]


def _check_softmax_grad_sums(grads):
    """sum_e dl[t, e] = 0 for every token, hence sum_e dW_r[e, :] = 0 and sum_e db[e] = 0."""
    g = U.to_f64(grads["grad_w_router"])
    col = np.abs(g.sum(axis=0))
    assert np.all(col <= 1e-2 * np.abs(g).sum(axis=0) + 1e-30), col.max()
    if grads["grad_router_bias"] is not None:
        db = U.to_f64(grads["grad_router_bias"])
        assert abs(db.sum()) <= 1e-4 * np.abs(db).sum()


@pytest.mark.parametrize("name", ["qwen3_30b_a3b_balanced_fwd_bwd", "qwen3_30b_a3b_skewed"])
def test_qwen3_shape_full_oracle(name):
    _need_host_gb(32)
    di, layer = _forward(name)
    idx = _check_routing(di, layer)
    if di.w.gate == G.GATE_BALANCED:
        assert np.array_equal(np.diff(layer.expert_offsets.cpu().numpy()), np.full(di.w.E, 256))
    else:
        counts = np.diff(layer.expert_offsets.cpu().numpy())
        assert counts.max() > 3 * counts.mean()          # the skewed router really is ragged
    f = U.oracle_forward(di, topk_idx=idx)
    U.check_close(layer.gu_saved, f["gu_perm"], "gu_saved")
    U.check_close(layer.y_perm, f["y_perm"], "y_perm")
    U.check_close(layer.out, f["out"], "out")
    # the inference forward (h only: wide gate/up units, bench.py's forward)
    # gives the same bits at this size too
    inf = U.run_forward(di, with_backward=False, save_logits=False)
    assert M.moe_read_device_status(inf.workspace) == 0
    assert torch.equal(inf.y_perm.view(torch.int16), layer.y_perm.view(torch.int16))
    assert torch.equal(inf.out.view(torch.int16), layer.out.view(torch.int16))
    del inf
    if not di.w.backward:
        return
    grads = _backward(di, layer, di.grad_out)
    b = O.layer_backward(f, di.f64("grad_out"), di.f64("x"), di.f64("w_router"),
                         di.f64("w_gate_up"), di.f64("w_down"), di.w.k)
    for key in ("grad_w_down", "grad_w_gate_up", "grad_x", "grad_w_router"):
        _check_by_expert(grads[key], b[key], key)
    _check_softmax_grad_sums(grads)


def _need_host_gb(gb):
    with open("/proc/meminfo") as fh:
        info = dict(line.split(":", 1) for line in fh)
    avail = int(info["MemAvailable"].split()[0]) / 2**20
    if avail < gb:
        pytest.skip(f"needs ~{gb} GB of free host memory for the float64 oracle, {avail:.0f} GB free")


def _check_by_expert(got, ref, name):
    """Expert-stacked tensors one expert at a time (bounds host memory; stricter than whole)."""
    if got.dim() < 3:
        return U.check_close(got, ref, name)
    for e in range(got.shape[0]):
        U.check_close(got[e], ref[e], f"{name}[{e}]")


def test_shared_expert_shape_sampled():
    _need_host_gb(48)
    di, layer = _forward("shared_expert_skewed")
    w = di.w
    idx = _check_routing(di, layer)
    counts = np.diff(layer.expert_offsets.cpu().numpy())
    rng = np.random.default_rng(3)

    # sampled tokens: forward rows
    tokens = np.sort(rng.choice(w.T, size=32, replace=False))
    f, b = _sub_layer(di, tokens, idx)
    U.check_close(_rows(layer.out, tokens), f["out"], "out (sampled tokens)")
    U.check_close(_rows(layer.y_shared, tokens), f["y_shared"], "y_shared (sampled tokens)")
    slots = (tokens[:, None] * w.k + np.arange(w.k)[None, :]).ravel()
    rows = layer.slot_perm.cpu().numpy()[slots]
    U.check_close(_rows(layer.y_perm, rows), f["y_perm"][f["slot_perm"]], "y_perm (their rows)")
    U.check_close(_rows(layer.gu_saved, rows), f["gu_perm"][f["slot_perm"]], "gu_saved (their rows)")

    # full-size backward with grad_out zero outside the sample: every gradient tensor in full
    keep = torch.zeros(w.T, 1, dtype=torch.bfloat16, device="cuda")
    keep[torch.from_numpy(tokens).cuda()] = 1
    grads = _backward(di, layer, di.grad_out * keep)
    gx = np.zeros((w.T, w.H))
    gx[tokens] = b["grad_x"]
    U.check_close(grads["grad_x"], gx, "grad_x (grad_out on sampled tokens)")
    for key in GRAD_KEYS[1:]:
        if key == "grad_router_bias":
            sub_slots = f["perm_slot"].astype(np.int64)
            dev_rows = layer.slot_perm.cpu().numpy()[tokens[sub_slots // w.k] * w.k + sub_slots % w.k]
            U.check_bias_grad(grads[key], di, f, _rows(layer.gu_saved, dev_rows),
                              name=key + " (grad_out on sampled tokens)",
                              x=di.f64("x")[tokens], grad_out=di.f64("grad_out")[tokens])
        else:
            _check_by_expert(grads[key], b[key], key + " (grad_out on sampled tokens)")
    del grads, f, b, gx

    # the real grad_out: sampled tokens' grad_x, sampled experts' weight gradients
    grads = _backward(di, layer, di.grad_out)
    _check_softmax_grad_sums(grads)
    tokens = np.sort(rng.choice(w.T, size=32, replace=False))
    _, b = _sub_layer(di, tokens, idx)
    U.check_close(_rows(grads["grad_x"], tokens), b["grad_x"], "grad_x (sampled tokens)")
    del b
    # the median expert, one of ~3x the mean load (several ragged tiles; the busiest expert
    # holds most tokens and is covered by the masked run above), and an empty one
    experts = [int(np.argsort(counts)[w.E // 2]), int(np.argmin(np.abs(counts - 3 * counts.mean())))]
    experts += [int(e) for e in np.nonzero(counts == 0)[0][:1]]
    for e in experts:
        toks = np.nonzero((idx == e).any(axis=1))[0]
        if toks.size == 0:
            assert torch.count_nonzero(grads["grad_w_gate_up"][e]) == 0
            assert torch.count_nonzero(grads["grad_w_down"][e]) == 0
            continue
        _, be = _sub_layer(di, toks, idx)
        U.check_close(grads["grad_w_gate_up"][e], be["grad_w_gate_up"][e], f"grad_w_gate_up[{e}]")
        U.check_close(grads["grad_w_down"][e], be["grad_w_down"][e], f"grad_w_down[{e}]")
        del be
