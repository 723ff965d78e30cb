"""CPU oracle for the single-GPU MoE expert layer behind the "grouped_mm" backend.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library; both sides are
fed the same seeded bf16 inputs and nothing else.

Everything here is plain float64 numpy (bf16 inputs are widened exactly).  A
matrix product (``@``) is the only library step; there is no blocking, fusion
or reordering beyond what the definitions below state.

Sources (page title, section):

* NeMo AutoModel blog, zh-CN translation ("Accelerating Transformers
  fine-tuning with NVIDIA NeMo AutoModel"), table "专家后端 / Expert backends":
  eager = a for-loop over the selected experts (used for correctness checks);
  batched_mm = copy the expert parameters and run one batched GEMM;
  grouped_mm = sort the tokens by their assigned expert and run a single
  grouped GEMM, with no parameter copies.
* same page, "v4 死锁原因 / why v4 deadlocks" and "动态权重加载 / dynamic weight
  loading": experts are stored as fused 3-D parameter tensors, one per
  projection, not as one module per expert.
* same page, "关于路由门的说明 / note on the routing gate": the NeMo numbers use a
  balanced routing gate that forces tokens evenly across experts.
* DeepEP paragraphs of the same page and of "英伟达开源MoE新方案" (section
  "DeepEP"): the layer dispatches tokens to experts and combines the results.
* "NVIDIA NeMo AutoModel MoE 微調的 3.7 倍加速突破", closing paragraph on load
  balancing (citing the Hugging Face MoE guide): token routing is naturally
  uneven, experts can overflow, and an auxiliary loss keeps routing even; the
  routing-gate note above: a load-balancing loss drives expert utilisation
  towards uniform.

The pages fix neither the router formula, the activation, the gate's exact
rule nor any tensor shape.  Readings taken here (each also listed in the
design notes):

* router: logits = x W_r^T (+ b); p = softmax over all E; top-k chosen on the
  fp32-rounded logits, largest first, ties to the lower expert index;
  w = p[selected] / sum(p[selected]).
* balanced gate: slot (t, j) goes to expert (t*k + j) mod E; its weight is the
  router softmax renormalised over those k experts.
* permutation: stable counting sort of the slots s = t*k + j by expert.
* expert MLP: SwiGLU, h = silu(gate) * up, gate = first I rows of W_gu[e].
* combine: out[t] = sum_j w[t,j] * y[t,j] (+ shared expert, weight 1).
* auxiliary load-balancing loss (no formula on the pages; the Switch
  Transformer form the cited guide describes): L_aux = alpha * E *
  sum_e f_e P_e with f_e = the fraction of the T*k slots routed to e and
  P_e = the mean over tokens of p[t, e]; f is a count, so it passes no
  gradient.  Uniform routing and probabilities give L_aux = alpha.
* expert capacity (the pages name overflow as a risk of uneven routing and
  give no rule): an expert takes at most C slots; the ones it keeps are its
  first C in slot order s = t*k + j (the stable sort's order), the rest are
  dropped.  A dropped slot adds nothing to the output (the layer's residual
  carries the token) and its weight keeps its value, so the kept weights are
  not renormalised.  Dropping is piecewise constant in the inputs: it passes
  no gradient, the dropped slot's dL/dw is 0, and the router gradient keeps
  its formula.  The counts f of the auxiliary loss are the router's
  assignment before dropping.  C = ceil(factor * T * k / E) for a capacity
  factor; C >= max count drops nothing.

* expert parallelism (NeMo AutoModel blog, "专家并行与 DeepEP"; the pages give
  no exchange layout): the readings are stated above ``ep_expert_ranges``.

Parity status: every function below is pinned by a test in
``tests/test_oracle_pins.py`` (closed forms, invariants, brute force, library
special cases, finite differences) or, for the expert-parallel functions,
``tests/test_ep_oracle.py`` (torch's chunking, brute-force counts, the global
stable sort, equality with the one-rank layer).
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np


# --------------------------------------------------------------------------
# bf16 widening (the oracle's own; the CUDA path has its own)
# --------------------------------------------------------------------------
def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 raw bits -> float64, exactly (a bf16 is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Router (logits, softmax, top-k, renormalisation, balanced gate)
# --------------------------------------------------------------------------
def router_logits(x: np.ndarray, w_router: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * W_r[e, h] (+ bias[e]).

    The router is the linear layer in front of the experts; the pages call it
    the native router ("原生路由器", note on the routing gate).  The bias is the
    learned-style per-expert skew of the skewed workloads.
    """
    logits = x @ w_router.T
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=np.float64)[None, :]
    return logits


def softmax(logits: np.ndarray) -> np.ndarray:
    """Row softmax, p[t,e] = exp(l[t,e] - max_e l) / sum_e exp(l[t,e] - max_e l)."""
    m = logits.max(axis=1, keepdims=True)
    z = np.exp(logits - m)
    return z / z.sum(axis=1, keepdims=True)


def select_topk(decision_logits: np.ndarray, k: int) -> np.ndarray:
    """Top-k expert ids per token by repeated argmax.

    Selection j picks the largest remaining logit; among equal logits the lower
    expert index is taken first (np.argmax returns the first maximum).  The
    decision is taken on the values as given (callers pass fp32-rounded logits,
    the precision the kernel decides in).  Returns int32 [T, k] in selection
    order.  Finite logits are assumed.
    """
    T, E = decision_logits.shape
    assert 1 <= k <= E
    work = np.asarray(decision_logits, dtype=np.float64).copy()
    idx = np.empty((T, k), dtype=np.int32)
    rows = np.arange(T)
    for j in range(k):
        sel = np.argmax(work, axis=1)
        idx[:, j] = sel
        work[rows, sel] = -np.inf
    return idx


def balanced_topk(T: int, E: int, k: int) -> np.ndarray:
    """Balanced gate: slot (t, j) -> expert (t*k + j) mod E.

    Forces an even token-to-expert split (note on the routing gate): when E
    divides T*k every expert receives exactly T*k/E slots, and the k experts
    of one token are distinct whenever k <= E.
    """
    s = np.arange(T * k, dtype=np.int64).reshape(T, k)
    return (s % E).astype(np.int32)


def renormalised_weights(p: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w[t, j] = p[t, idx[t,j]] / sum_j' p[t, idx[t,j']]."""
    rows = np.arange(p.shape[0])[:, None]
    psel = p[rows, idx]
    return psel / psel.sum(axis=1, keepdims=True)


def route(logits: np.ndarray, k: int, balanced: bool = False, decision_logits=None):
    """Full router step: returns (topk_idx int32 [T,k], topk_w float64 [T,k], p).

    ``decision_logits`` (default: ``logits`` rounded to fp32) is what top-k
    compares; softmax and weights always use ``logits``.
    """
    T, E = logits.shape
    p = softmax(logits)
    if balanced:
        idx = balanced_topk(T, E, k)
    else:
        if decision_logits is None:
            decision_logits = logits.astype(np.float32)
        idx = select_topk(decision_logits, k)
    return idx, renormalised_weights(p, idx), p


# --------------------------------------------------------------------------
# Sort token-slots by expert (grouped_mm "sort the tokens by expert")
# --------------------------------------------------------------------------
def permute(topk_idx: np.ndarray, E: int):
    """Counting sort of the T*k slots by expert, stable in slot id s = t*k + j.

    Returns (expert_offsets int32 [E+1], perm_slot int32 [S], slot_perm int32 [S]):
    rows expert_offsets[e] .. expert_offsets[e+1]-1 of the sorted order belong
    to expert e; perm_slot[r] is the slot at sorted row r and slot_perm is its
    inverse.  Only token ids move; no expert weight is copied (grouped_mm row
    of the expert-backend table).
    """
    flat = np.asarray(topk_idx, dtype=np.int64).ravel()
    S = flat.size
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    perm_slot = np.empty(S, dtype=np.int64)
    for s in range(S):
        e = flat[s]
        perm_slot[fill[e]] = s
        fill[e] += 1
    slot_perm = np.empty(S, dtype=np.int64)
    slot_perm[perm_slot] = np.arange(S)
    return offsets.astype(np.int32), perm_slot.astype(np.int32), slot_perm.astype(np.int32)


def expert_capacity(T: int, k: int, E: int, factor: float) -> int:
    """Slots an expert keeps for capacity factor `factor`: ceil(factor * T * k / E),
    with the factor taken as the decimal it is written as (1.1 is 11/10)."""
    return int(math.ceil(Fraction(str(factor)) * T * k / E))


def keep_slots(topk_idx: np.ndarray, E: int, capacity: int | None) -> np.ndarray:
    """bool [T, k]: slot (t, j) is kept iff fewer than `capacity` earlier slots
    (in slot order s = t*k + j) went to the same expert.  None: keep every slot."""
    T, k = topk_idx.shape
    keep = np.ones((T, k), dtype=bool)
    if capacity is None:
        return keep
    taken = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(topk_idx[t, j])
            keep[t, j] = taken[e] < capacity
            taken[e] += 1
    return keep


# --------------------------------------------------------------------------
# Expert MLP (SwiGLU) in the three backends of the expert-backend table
# --------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


def swiglu_mlp(xr: np.ndarray, w_gu: np.ndarray, w_down: np.ndarray):
    """One expert on rows xr [n, H]: gu = xr W_gu^T, h = silu(gate) * up, y = h W_down^T.

    W_gu is [2I, H] with the gate rows first; W_down is [H, I].
    Returns (y [n,H], gu [n,2I], h [n,I]).
    """
    I = w_down.shape[1]
    gu = xr @ w_gu.T
    h = silu(gu[:, :I]) * gu[:, I:]
    return h @ w_down.T, gu, h


def experts_grouped(x, offsets, perm_slot, k, w_gu, w_down):
    """grouped_mm backend: tokens already sorted by expert, one GEMM per group.

    Returns y_perm [S, H], gu_perm [S, 2I], h_perm [S, I] in sorted-row order.
    """
    S = perm_slot.size
    E, twoI, H = w_gu.shape
    I = twoI // 2
    y = np.zeros((S, H))
    gu = np.zeros((S, twoI))
    h = np.zeros((S, I))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        tok = perm_slot[r0:r1] // k
        y[r0:r1], gu[r0:r1], h[r0:r1] = swiglu_mlp(x[tok], w_gu[e], w_down[e])
    return y, gu, h


def experts_eager(x, topk_idx, w_gu, w_down):
    """eager backend: for-loop over the selected experts, token by token.

    Returns y_slot [T, k, H] (each slot's unweighted expert output).
    """
    T, k = topk_idx.shape
    H = x.shape[1]
    y = np.zeros((T, k, H))
    for e in np.unique(topk_idx):
        for t in range(T):
            for j in range(k):
                if topk_idx[t, j] == e:
                    y[t, j] = swiglu_mlp(x[t:t + 1], w_gu[e], w_down[e])[0][0]
    return y


def experts_batched(x, topk_idx, w_gu, w_down):
    """batched_mm backend: copy each slot's expert parameters, one batched GEMM.

    Returns y_slot [T, k, H].  Memory grows with T*k*(3*I*H); tiny inputs only.
    """
    T, k = topk_idx.shape
    I = w_down.shape[2]
    flat = topk_idx.ravel()
    xs = np.repeat(x, k, axis=0)                  # [S, H]
    wg = w_gu[flat]                               # [S, 2I, H]  (parameter copies)
    wd = w_down[flat]                             # [S, H, I]
    gu = np.einsum("sh,sih->si", xs, wg)
    h = silu(gu[:, :I]) * gu[:, I:]
    y = np.einsum("si,shi->sh", h, wd)
    return y.reshape(T, k, -1)


def combine(y_perm, slot_perm, topk_w, y_shared=None, keep=None):
    """Weighted un-permute: out[t] = sum_j w[t,j] * y_perm[slot_perm[t*k+j]] (+ y_shared[t]),
    over the kept slots only when a keep mask [T, k] is given."""
    T, k = topk_w.shape
    out = np.zeros((T, y_perm.shape[1]))
    for j in range(k):
        rows = slot_perm.reshape(T, k)[:, j]
        contrib = topk_w[:, j:j + 1] * y_perm[rows]
        if keep is not None:
            contrib = np.where(keep[:, j:j + 1], contrib, 0.0)
        out += contrib
    if y_shared is not None:
        out = out + y_shared
    return out


def combine_slots(y_slot, topk_w, y_shared=None):
    """Same weighted sum for outputs already in slot order [T, k, H]."""
    out = np.einsum("tk,tkh->th", topk_w, y_slot)
    if y_shared is not None:
        out = out + y_shared
    return out


# --------------------------------------------------------------------------
# Whole layer, forward
# --------------------------------------------------------------------------
def layer_forward(x, w_router, w_gu, w_down, k, balanced=False, bias=None,
                  w_sh_gu=None, w_sh_down=None, topk_idx=None, decision_logits=None,
                  capacity=None):
    """MoE layer forward through the grouped path.

    All arrays float64 except ids.  ``topk_idx`` overrides the selection (used
    when comparing against a device whose fp32 logits sit on a near-tie).
    ``capacity``: slots each expert keeps (None: no limit); the expert outputs
    of dropped slots are still formed here (rows of y_perm) but not combined.
    Returns a dict with every intermediate the backward needs.
    """
    E = w_gu.shape[0]
    logits = router_logits(x, w_router, bias)
    idx, w, p = route(logits, k, balanced=balanced, decision_logits=decision_logits)
    if topk_idx is not None:
        idx = np.asarray(topk_idx, dtype=np.int32)
        w = renormalised_weights(p, idx)
    offsets, perm_slot, slot_perm = permute(idx, E)
    y_perm, gu_perm, h_perm = experts_grouped(x, offsets, perm_slot, k, w_gu, w_down)
    y_sh = gu_sh = None
    if w_sh_gu is not None:
        y_sh, gu_sh, _ = swiglu_mlp(x, w_sh_gu, w_sh_down)
    keep = keep_slots(idx, E, capacity)
    out = combine(y_perm, slot_perm, w, y_sh, keep=keep)
    return dict(logits=logits, p=p, topk_idx=idx, topk_w=w, expert_offsets=offsets,
                perm_slot=perm_slot, slot_perm=slot_perm, gu_perm=gu_perm, h_perm=h_perm,
                y_perm=y_perm, y_shared=y_sh, gu_shared=gu_sh, out=out, keep=keep)


# --------------------------------------------------------------------------
# Expert parallelism: dispatch to the experts' ranks and combine back
# --------------------------------------------------------------------------
# NeMo AutoModel blog (zh-CN), "专家并行与 DeepEP": expert parallelism is its
# own mesh dimension beside data parallelism; every rank trains on its own
# data shard and holds 1/ep of the experts, the expert weights being split
# along the expert dimension (DTensor Shard(0)).  DeepEP paragraphs: tokens are
# dispatched to the ranks of their experts and the results combined back
# (all-to-all).  The pages give no exchange layout; the readings here:
# * rank r owns the experts Shard(0) gives it: chunks of ceil(E / n) in rank
#   order (the last ranks may own fewer, or none);
# * a source sends its slots in its expert-sorted order (permute), which is
#   rank order because every rank's experts are contiguous; the rows for
#   rank q are the block of q's experts;
# * a receiver's buffer holds the sources' blocks in source order; its one
#   grouped GEMM takes the rows expert by expert, within an expert source by
#   source, within a source in the source's order;
# * each output row goes back to its source in the order it came, so the
#   source holds its rows' outputs in its own sorted order and combines them
#   exactly as on one rank.
# * backward (the pages time the backward but give no layout for it): the
#   reverse trip.  A source sends every slot's grad_out row and routing
#   weight in its sorted order, as it sent the token rows; the experts' rank
#   forms each row's dx and dL/dw and its experts' weight gradients, and sends
#   dx and dL/dw back; the source sums its tokens' slot gradients and runs the
#   router's backward.  The router is replicated, so each rank's router
#   gradient covers its own tokens and the ranks' gradients add up (as data
#   parallelism adds any replicated parameter's).


def ep_expert_ranges(E: int, n_ranks: int) -> np.ndarray:
    """int [n+1]: rank r owns experts bounds[r] .. bounds[r+1]-1 (Shard(0) chunks)."""
    c = -(-E // n_ranks)
    return np.minimum(np.arange(n_ranks + 1) * c, E)


def ep_dispatch(topk_idx: np.ndarray, E: int, n_ranks: int):
    """A source rank's dispatch plan from its own slots' expert ids.

    Returns (expert_offsets, perm_slot, slot_perm, send_counts [n], expert_counts
    [E]): the sort of permute; send_counts[q] = rows of the sorted order that go
    to rank q (the block expert_offsets[bounds[q]] .. expert_offsets[bounds[q+1]]);
    expert_counts[e] = the source's slots routed to e (what it tells the
    receivers so that they can lay out their buffers).
    """
    offsets, perm_slot, slot_perm = permute(topk_idx, E)
    b = ep_expert_ranges(E, n_ranks)
    send_counts = np.array([int(offsets[b[q + 1]]) - int(offsets[b[q]]) for q in range(n_ranks)])
    return offsets, perm_slot, slot_perm, send_counts, np.diff(offsets.astype(np.int64))


def ep_receive(expert_counts_from, lo: int, hi: int):
    """The receive layout of the rank owning experts lo .. hi-1.

    expert_counts_from[s]: source s's expert counts [E].  The receive buffer
    holds, source by source, that source's rows for experts lo .. hi-1 in
    expert order.  Returns (local_offsets [E_loc+1], recv_perm [R]): grouped
    row g (expert-major, then source, then the source's order) is receive row
    recv_perm[g]; local expert e owns grouped rows local_offsets[e] ..
    local_offsets[e+1]-1.
    """
    n = len(expert_counts_from)
    E_loc = hi - lo
    C = np.array([[int(expert_counts_from[s][lo + e]) for e in range(E_loc)] for s in range(n)],
                 dtype=np.int64).reshape(n, E_loc)
    seg = np.zeros((n, E_loc), dtype=np.int64)   # receive row where (source, expert) starts
    pos = 0
    for s in range(n):
        for e in range(E_loc):
            seg[s, e] = pos
            pos += C[s, e]
    local_offsets = np.zeros(E_loc + 1, dtype=np.int64)
    recv_perm = np.empty(pos, dtype=np.int64)
    g = 0
    for e in range(E_loc):
        local_offsets[e] = g
        for s in range(n):
            for i in range(C[s, e]):
                recv_perm[g] = seg[s, e] + i
                g += 1
    local_offsets[E_loc] = g
    return local_offsets.astype(np.int32), recv_perm.astype(np.int32)


def ep_layer_forward(x_ranks, w_router, w_gu, w_down, k, balanced=False, bias=None,
                     topk_idx_ranks=None):
    """The layer over n ranks with expert parallelism, every step written out.

    x_ranks[r]: rank r's tokens [T_r, H] (its data shard); the router is
    replicated; rank q runs only the experts ep_expert_ranges gives it.
    Steps: each rank routes its tokens (topk_idx_ranks overrides the
    selection) and sorts its slots (ep_dispatch); it sends the token rows of
    its sorted order, block q to rank q; rank q lays out what it received
    (ep_receive), runs its experts on the grouped rows (one grouped GEMM per
    projection), and sends every output row back to its source in the order
    it came; each source combines its rows' outputs with its weights.
    Returns a list of per-rank dicts: out, the plans, the receive layouts and
    the exchanged buffers (for the tests).
    """
    n = len(x_ranks)
    E = w_gu.shape[0]
    b = ep_expert_ranges(E, n)
    src = []
    for r in range(n):
        logits = router_logits(x_ranks[r], w_router, bias)
        idx, w, p = route(logits, k, balanced=balanced)
        if topk_idx_ranks is not None:
            idx = np.asarray(topk_idx_ranks[r], dtype=np.int32)
            w = renormalised_weights(p, idx)
        off, perm, inv, send_counts, counts = ep_dispatch(idx, E, n)
        x_send = x_ranks[r][perm.astype(np.int64) // k]
        src.append(dict(topk_idx=idx, topk_w=w, expert_offsets=off, perm_slot=perm,
                        slot_perm=inv, send_counts=send_counts, expert_counts=counts,
                        x_send=x_send))
    dst = []
    for q in range(n):
        blocks = [src[s]["x_send"][int(src[s]["expert_offsets"][b[q]]):
                                   int(src[s]["expert_offsets"][b[q + 1]])] for s in range(n)]
        x_recv = np.concatenate(blocks, axis=0)
        loc_off, recv_perm = ep_receive([src[s]["expert_counts"] for s in range(n)], int(b[q]),
                                        int(b[q + 1]))
        y_grouped = experts_grouped(x_recv, loc_off, recv_perm, 1, w_gu[b[q]:b[q + 1]],
                                    w_down[b[q]:b[q + 1]])[0]
        y_recv = np.zeros_like(x_recv)
        y_recv[recv_perm.astype(np.int64)] = y_grouped
        recv_counts = [len(bl) for bl in blocks]
        dst.append(dict(x_recv=x_recv, local_offsets=loc_off, recv_perm=recv_perm,
                        y_recv=y_recv, recv_counts=recv_counts))
    outs = []
    for s in range(n):
        back = []
        for q in range(n):
            start = int(sum(dst[q]["recv_counts"][:s]))
            back.append(dst[q]["y_recv"][start:start + dst[q]["recv_counts"][s]])
        y_sorted = np.concatenate(back, axis=0)
        out = combine(y_sorted, src[s]["slot_perm"], src[s]["topk_w"])
        outs.append(dict(src[s], y_sorted=y_sorted, out=out, **dst[s]))
    return outs


def ep_experts_backward(x_recv, go_recv, w_recv, local_offsets, recv_perm, w_gu_loc, w_down_loc):
    """The experts' rank's part of the expert-parallel backward.

    Received rows (receive order): token rows x_recv [R, H], their grad_out
    rows go_recv [R, H] and routing weights w_recv [R]; the grouping of
    ep_receive.  Per local expert e, for its rows: y = MLP_e(x), dL/dw =
    <dout, y>, the expert sees dy = w dout (as layer_backward).  Returns
    (dx_recv [R, H], dw_recv [R], dW_gu [E_loc, 2I, H], dW_down [E_loc, H, I]).
    """
    R, H = x_recv.shape
    E_loc = w_gu_loc.shape[0]
    dx = np.zeros((R, H))
    dw = np.zeros(R)
    dW_gu = np.zeros_like(w_gu_loc)
    dW_down = np.zeros_like(w_down_loc)
    for e in range(E_loc):
        rows = np.asarray(recv_perm[int(local_offsets[e]):int(local_offsets[e + 1])], dtype=np.int64)
        if rows.size == 0:
            continue
        y, gu, _ = swiglu_mlp(x_recv[rows], w_gu_loc[e], w_down_loc[e])
        dw[rows] = np.sum(go_recv[rows] * y, axis=1)
        dy = np.asarray(w_recv)[rows][:, None] * go_recv[rows]
        dx[rows], dW_gu[e], dW_down[e] = swiglu_mlp_backward(x_recv[rows], gu, w_gu_loc[e],
                                                              w_down_loc[e], dy)
    return dx, dw, dW_gu, dW_down


def router_backward(x, w_router, topk_idx, topk_w, dw):
    """The router's backward from each slot's dL/dw (no auxiliary loss).

    The renormalised weights are a softmax over the chosen logits, so the
    gradient reaches only those: dl[t, e_j] = w_j (dw_j - sum_i w_i dw_i), and
    0 at every other expert.  Returns (dl [T, E], dx_router = dl W_r,
    dW_r = dl^T x, db = sum_t dl).
    """
    T = x.shape[0]
    E = w_router.shape[0]
    w = np.asarray(topk_w, dtype=np.float64)
    dwv = np.asarray(dw, dtype=np.float64)
    dl_sel = w * (dwv - np.sum(w * dwv, axis=1, keepdims=True))
    dl = np.zeros((T, E))
    np.add.at(dl, (np.repeat(np.arange(T), topk_idx.shape[1]), np.asarray(topk_idx).ravel()),
              dl_sel.ravel())
    return dl, dl @ w_router, dl.T @ x, dl.sum(axis=0)


def ep_layer_backward(ranks, grad_out_ranks, x_ranks, w_router, w_gu, w_down):
    """The backward over n ranks with expert parallelism, every step written out.

    ranks: ep_layer_forward's per-rank dicts; grad_out_ranks[r]: rank r's
    dL/d(out) [T_r, H].  Each source gathers its slots' grad_out rows and
    weights in its sorted order and sends block q to rank q; rank q runs
    ep_experts_backward on what it received (rows in the forward's receive
    order) and sends dx and dL/dw back in the order they came; the source
    sums each token's slot gradients and adds the router's term.  Returns a
    list of per-rank dicts: grad_x, grad_w_router and grad_router_bias (over
    the rank's tokens), the rank's local expert gradients, and the exchanged
    buffers.
    """
    n = len(ranks)
    E = w_gu.shape[0]
    k = ranks[0]["topk_idx"].shape[1] if len(ranks) else 1
    b = ep_expert_ranges(E, n)
    send = []
    for r in range(n):
        perm = ranks[r]["perm_slot"].astype(np.int64)
        send.append(dict(go=grad_out_ranks[r][perm // k], w=np.asarray(ranks[r]["topk_w"]).ravel()[perm]))
    back = []
    for q in range(n):
        off = [ranks[s]["expert_offsets"] for s in range(n)]
        go_recv = np.concatenate([send[s]["go"][int(off[s][b[q]]):int(off[s][b[q + 1]])]
                                  for s in range(n)], axis=0)
        w_recv = np.concatenate([send[s]["w"][int(off[s][b[q]]):int(off[s][b[q + 1]])]
                                 for s in range(n)], axis=0)
        dx_recv, dw_recv, dW_gu, dW_down = ep_experts_backward(
            ranks[q]["x_recv"], go_recv, w_recv, ranks[q]["local_offsets"], ranks[q]["recv_perm"],
            w_gu[b[q]:b[q + 1]], w_down[b[q]:b[q + 1]])
        back.append(dict(go_recv=go_recv, w_recv=w_recv, dx_recv=dx_recv, dw_recv=dw_recv,
                         grad_w_gate_up=dW_gu, grad_w_down=dW_down))
    res = []
    for s in range(n):
        parts_dx, parts_dw = [], []
        for q in range(n):
            start = int(sum(ranks[q]["recv_counts"][:s]))
            cnt = int(ranks[q]["recv_counts"][s])
            parts_dx.append(back[q]["dx_recv"][start:start + cnt])
            parts_dw.append(back[q]["dw_recv"][start:start + cnt])
        H = x_ranks[s].shape[1]
        dx_sorted = np.concatenate(parts_dx, axis=0) if parts_dx else np.zeros((0, H))
        dw_sorted = np.concatenate(parts_dw, axis=0) if parts_dw else np.zeros(0)
        T = x_ranks[s].shape[0]
        inv = ranks[s]["slot_perm"].astype(np.int64)
        dx_slot = dx_sorted[inv].reshape(T, k, H)
        dw = dw_sorted[inv].reshape(T, k)
        _, dx_router, dW_r, db = router_backward(x_ranks[s], w_router, ranks[s]["topk_idx"],
                                                 ranks[s]["topk_w"], dw)
        res.append(dict(grad_x=dx_slot.sum(axis=1) + dx_router, grad_w_router=dW_r,
                        grad_router_bias=db, dx_sorted=dx_sorted, dw_sorted=dw_sorted,
                        **back[s]))
    return res


# --------------------------------------------------------------------------
# Whole layer, backward (hand-derived; pinned by finite differences)
# --------------------------------------------------------------------------
def swiglu_mlp_backward(xr, gu, w_gu, w_down, dy):
    """Backward of y = (silu(g) * u) W_down^T with [g|u] = xr W_gu^T.

    dy [n,H] is the gradient at y.  Returns (dx [n,H], dW_gu [2I,H], dW_down [H,I]).
    dh = dy W_down; dg = dh * u * s * (1 + g (1 - s)) with s = sigmoid(g);
    du = dh * silu(g).
    """
    I = w_down.shape[1]
    g, u = gu[:, :I], gu[:, I:]
    s = sigmoid(g)
    h = g * s * u
    dW_down = dy.T @ h
    dh = dy @ w_down
    dg = dh * u * s * (1.0 + g * (1.0 - s))
    du = dh * g * s
    dgu = np.concatenate([dg, du], axis=1)
    return dgu @ w_gu, dgu.T @ xr, dW_down


def aux_loss(p, topk_idx, alpha):
    """Auxiliary load-balancing loss and its logit-gradient coefficients.

    f_e = count_e / (T k) (slots routed to e), P_e = (1/T) sum_t p[t, e],
    L = alpha * E * sum_e f_e P_e.  With f held constant, dL/dp[t, e] =
    c_e = alpha * E * f_e / T for every token.  Returns (L, c).
    """
    T, E = p.shape
    k = topk_idx.shape[1]
    counts = np.zeros(E)
    np.add.at(counts, np.asarray(topk_idx).ravel(), 1.0)
    f = counts / (T * k)
    P = p.sum(axis=0) / T
    L = alpha * E * float(np.sum(f * P))
    c = alpha * E * f / T
    return L, c


def layer_backward(fwd: dict, grad_out, x, w_router, w_gu, w_down, k,
                   w_sh_gu=None, w_sh_down=None, aux_coef=None):
    """Gradients of the layer output w.r.t. x, W_r, router bias and every expert weight.

    Per slot (t, j) routed to e with weight w:  y = MLP_e(x[t]),
    dL/dw[t,j] = <dout[t], y>, the expert sees dy = w * dout[t].  Router:
    w = p[sel]/P, so dp[sel_j] = (dw_j - sum_i w_i dw_i) / P and every other
    dp is 0; through the softmax dl = p * (dp - <dp, p>).  dW_r = dl^T x,
    db = sum_t dl[t], and x also receives dl W_r.  Top-k selection itself is
    piecewise constant and passes no gradient.  With aux_coef = c (from
    aux_loss), the auxiliary loss adds dL_aux/dp[t, e] = c_e for every expert,
    so its logit gradient p * (c - <c, p>) is dense.  A slot the forward
    dropped (fwd["keep"] False) gets dL/dw = 0 and sends nothing to its expert.
    """
    T, H = x.shape
    E = w_gu.shape[0]
    idx, w, p = fwd["topk_idx"], fwd["topk_w"], fwd["p"]
    offsets, perm_slot = fwd["expert_offsets"], fwd["perm_slot"]
    gu_perm, y_perm = fwd["gu_perm"], fwd["y_perm"]
    keep = fwd.get("keep")
    if keep is None:
        keep = np.ones(idx.shape, dtype=bool)
    dx = np.zeros((T, H))
    dW_gu = np.zeros_like(w_gu)
    dW_down = np.zeros_like(w_down)
    dw = np.zeros((T, k))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        slots = perm_slot[r0:r1].astype(np.int64)
        tok, j = slots // k, slots % k
        dout_r = np.where(keep[tok, j][:, None], grad_out[tok], 0.0)
        dw[tok, j] = np.sum(dout_r * y_perm[r0:r1], axis=1)
        dy = w[tok, j][:, None] * dout_r
        dxr, dW_gu[e], dW_down[e] = swiglu_mlp_backward(x[tok], gu_perm[r0:r1], w_gu[e], w_down[e], dy)
        np.add.at(dx, tok, dxr)
    # router
    rows = np.arange(T)[:, None]
    P = p[rows, idx].sum(axis=1, keepdims=True)
    dp_sel = (dw - np.sum(w * dw, axis=1, keepdims=True)) / P
    dp = np.zeros_like(p)
    np.add.at(dp, (np.repeat(np.arange(T), k), idx.ravel()), dp_sel.ravel())
    if aux_coef is not None:
        dp = dp + np.asarray(aux_coef, dtype=np.float64)[None, :]
    dl = p * (dp - np.sum(dp * p, axis=1, keepdims=True))
    dW_r = dl.T @ x
    db = dl.sum(axis=0)
    dx += dl @ w_router
    res = dict(grad_x=dx, grad_w_router=dW_r, grad_router_bias=db, grad_w_gate_up=dW_gu,
               grad_w_down=dW_down, grad_topk_w=dw, grad_logits=dl)
    if w_sh_gu is not None:
        dxs, res["grad_w_sh_gate_up"], res["grad_w_sh_down"] = swiglu_mlp_backward(
            x, fwd["gu_shared"], w_sh_gu, w_sh_down, grad_out)
        res["grad_x"] = res["grad_x"] + dxs
    return res
