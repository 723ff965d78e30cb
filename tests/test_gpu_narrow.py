"""Narrow units of the inference gate/up GEMM, against the training GEMM and the oracle.

An expert whose last row tile holds at most 128 rows (its row count modulo
256 is in 1..128) would leave the odd CTA of a pair with no rows; the
inference (h-only, wide) gate/up GEMM then runs that tile with the operands'
roles swapped, the weight rows as the 256-row side and the tile's token rows
(rounded up to 32) as N.  These cases drive the grouped expert MLP directly
with expert row counts chosen to hit every kind of tail: 1 row, the 32-row
rounding edges, half a pair (64 rows per CTA), a full CTA (128), tails behind
one and two full pairs, empty experts, and experts with no narrow tile at all.
The intermediate size is not a multiple of 256, so the last unit's columns
run past I.  The h-only forward must give the training forward's bits
(y_perm equal), and both match the oracle's sorted-row expert MLP.
"""

import numpy as np
import pytest
import torch

import gpu_util as U
from grouped_expert_gemm_top_b300 import inputs as G
from grouped_expert_gemm_top_b300 import moe as M
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

# rows per expert: tails of 1..128 rows (narrow), 129..256 (a full pair), and
# multiples of 256 behind them
COUNTS = {
    "tails": [1, 17, 31, 32, 33, 0, 63, 64, 65, 96, 127, 128, 129, 255, 256, 257, 383, 384, 513, 0],
    "only_narrow": [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 110, 128],
    "none_narrow": [256, 129, 200, 512, 0, 255],
}


def _run(counts, H, I, seed, with_gu):
    E = len(counts)
    R = int(sum(counts))
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    perm = np.random.default_rng(seed).permutation(R).astype(np.int32)
    x = G.normal_bf16((R, H), 1.0, seed, "x")
    wgu = G.normal_bf16((E, 2 * I, H), H ** -0.5, seed, "w_gate_up")
    wd = G.normal_bf16((E, H, I), I ** -0.5, seed, "w_down")
    d = M.MoeDims.of(R, H, E, 1, I, 0)
    ws = torch.zeros(M.moe_workspace_size(d, 1 if with_gu else 0), dtype=torch.uint8, device="cuda")
    y = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    gu = torch.empty(R, 2 * I, dtype=torch.bfloat16, device="cuda") if with_gu else None
    M.moe_grouped_mlp_fwd(d, U.dev_bf16(x), torch.from_numpy(off).cuda(),
                          torch.from_numpy(perm).cuda(), U.dev_bf16(wgu), U.dev_bf16(wd), gu, y,
                          None, None, None, None, ws)
    torch.cuda.synchronize()
    assert M.moe_read_device_status(ws) == 0
    return y, (x, wgu, wd, off, perm)


@pytest.mark.parametrize("name", list(COUNTS))
@pytest.mark.parametrize("H,I", [(256, 320), (128, 512)])
def test_narrow_tiles_match_training_forward_and_oracle(name, H, I):
    counts = COUNTS[name]
    y_inf, (x, wgu, wd, off, perm) = _run(counts, H, I, seed=5, with_gu=False)
    y_tr, _ = _run(counts, H, I, seed=5, with_gu=True)
    assert torch.equal(y_inf, y_tr)
    y_ref, _, _ = O.experts_grouped(O.widen_bf16(x), off, perm, 1, O.widen_bf16(wgu),
                                    O.widen_bf16(wd))
    U.check_close(y_inf, y_ref, f"y_perm ({name})")
    # every expert's rows on their own as well (a tail's error cannot hide in the norm)
    for e in range(len(counts)):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 > r0:
            U.check_close(y_inf[r0:r1], y_ref[r0:r1], f"y_perm ({name}, expert {e})")
