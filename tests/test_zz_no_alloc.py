"""The allocation-free sort (moe_permute_static_scratch) against moe_permute.

Some callers cannot allocate device memory (a pre-sized memory pool, a plugin
whose host owns all allocations), so they cannot pass moe_permute's
workspace; the variant keeps its scratch in a fixed array inside the library.
Its outputs are integers, so the check is exact equality with the workspace
version, on two calls in a row (the second with a different shape, so a stale
array from the first call would show).  This file is collected last.
"""

import numpy as np
import pytest
import torch

from grouped_expert_gemm_top_b300 import moe as M

pytestmark = pytest.mark.gpu


def _both(T, E, k, seed, capacity=0, with_status=True):
    r = np.random.default_rng(seed)
    idx = r.integers(0, E, size=(T, k)).astype(np.int32)
    if E > 4:
        idx[idx == 1] = 0      # an empty expert
    dims = M.MoeDims.of(T, 64, E, k, 64, 0, capacity=capacity)
    d_idx = torch.from_numpy(idx).cuda()
    outs = []
    for variant in ("workspace", "static"):
        off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        perm = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
        inv = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
        if variant == "workspace":
            ws = torch.zeros(M.moe_workspace_size(dims, False), dtype=torch.uint8, device="cuda")
            M.moe_permute(dims, d_idx, off, perm, inv, ws)
        else:
            status = torch.zeros(1, dtype=torch.int32, device="cuda") if with_status else None
            M.moe_permute_static_scratch(dims, d_idx, off, perm, inv, status)
            torch.cuda.synchronize()
            if with_status:
                assert int(status.item()) == 0
        outs.append((off.cpu(), perm.cpu(), inv.cpu()))
    return outs


def test_static_scratch_sort_matches_workspace_sort_twice():
    for (T, E, k, seed) in [(4096, 128, 8, 0), (300, 7, 3, 1), (9000, 64, 8, 2)]:
        a, b = _both(T, E, k, seed)
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_static_scratch_sort_with_capacity_and_without_status_word():
    """Expert capacity (dropped slots get slot_perm -1) and no status word, each
    exactly equal to moe_permute on the same dims."""
    for (T, E, k, seed, cap, st) in [(4096, 128, 8, 4, 200, True), (1000, 16, 4, 5, 180, False),
                                     (300, 7, 3, 6, 1, True), (2048, 32, 2, 7, 0, False)]:
        a, b = _both(T, E, k, seed, capacity=cap, with_status=st)
        for x, y in zip(a, b):
            assert torch.equal(x, y)
        if cap:
            inv = a[2].numpy()
            counts = np.diff(a[0].numpy())
            assert (inv == -1).sum() == np.maximum(counts - cap, 0).sum() > 0


def test_static_scratch_sort_launches_are_counted():
    T, E, k = 512, 16, 2
    idx = torch.from_numpy(np.random.default_rng(8).integers(0, E, size=(T, k)).astype(np.int32)).cuda()
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    M.moe_kernel_stats(reset=True)
    M.moe_permute_static_scratch((T, 64, E, k, 64, 0), idx, off, perm, inv)
    torch.cuda.synchronize()
    st = M.moe_kernel_stats(reset=True)
    assert st["sort_histogram"][0] == 1 and st["sort_scatter"][0] == 1


def test_static_scratch_sort_rejects_oversized_shapes():
    # ceil(T*k / 1024) * E > 65536 block counts: refused before any launch
    dims = (65536, 64, 256, 8, 64, 0)
    dummy = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(M.MoeError) as e:
        M.moe_permute_static_scratch(dims, dummy, dummy, dummy, dummy)
    assert e.value.status == 2


def test_static_scratch_sort_reports_bad_expert_ids():
    T, E, k = 64, 8, 2
    idx = np.random.default_rng(3).integers(0, E, size=(T, k)).astype(np.int32)
    idx[5, 0] = E
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * k, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_permute_static_scratch((T, 64, E, k, 64, 0), torch.from_numpy(idx).cuda(), off, perm,
                                 inv, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    assert int(off[-1].item()) == T * k - 1
