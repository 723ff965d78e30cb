"""Host-side checks of the C ABI (no GPU needed, no compute calls).

The shared library must load here, export every function include/moe.h
declares, and reject bad arguments on the host with the documented status
codes before anything touches CUDA.
"""

import ctypes
import os

import pytest

from grouped_expert_gemm_top_b300 import build as B
from grouped_expert_gemm_top_b300 import moe as M


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(M.LIB_PATH):
        B.build()
    return M.load_library()


def test_header_declares_the_five_layer_calls():
    names = M.declared_functions()
    for n in ["moe_route", "moe_route_permute", "moe_permute", "moe_grouped_mlp_fwd", "moe_unpermute_combine",
              "moe_layer_bwd", "moe_workspace_size", "moe_read_device_status",
              "moe_status_string", "moe_abi_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in M.declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert M.moe_abi_version() == 12
    assert M.moe_status_string(0) == "ok"
    for s in range(1, 7):
        assert M.moe_status_string(s) not in ("ok", "unknown status")
    assert M.moe_status_string(99) == "unknown status"


def test_workspace_size_covers_intermediates(lib):
    T, H, E, k, I = 4096, 2048, 128, 8, 768
    fwd = M.moe_workspace_size((T, H, E, k, I, 0), False)
    bwd = M.moe_workspace_size((T, H, E, k, I, 0), True)
    S = T * k
    assert fwd >= S * I * 2                          # SwiGLU output h
    assert bwd > fwd + S * (2 * I + I + H) * 2        # dgu, w*h, per-slot dx
    sh = M.moe_workspace_size((8192, 2688, 128, 6, 1856, 3712), False)
    assert sh >= 8192 * 6 * 1856 * 2 + 8192 * 3712 * 2
    # activation recompute: room for the recomputed gate/up pre-activations
    rc = M.moe_workspace_size((T, H, E, k, I, 0), 2)
    assert rc >= bwd + S * 2 * I * 2
    d5 = (8192, 2688, 128, 6, 1856, 3712)
    assert M.moe_workspace_size(d5, 2) >= M.moe_workspace_size(d5, 1) + 8192 * 6 * 2 * 1856 * 2 + 8192 * 2 * 3712 * 2
    with pytest.raises(M.MoeError):
        M.moe_workspace_size((T, H, E, k, I, 0), 3)


@pytest.mark.parametrize("dims,code", [
    ((0, 256, 8, 2, 512, 0), 2),        # T = 0
    ((16, 250, 8, 2, 512, 0), 2),       # H not a multiple of 64
    ((16, 256, 8, 2, 500, 0), 2),       # I not a multiple of 64
    ((16, 256, 8, 9, 512, 0), 2),       # k > E
    ((16, 256, 300, 2, 512, 0), 2),     # E > 256
    ((16, 256, 64, 33, 512, 0), 2),     # k > 32
    ((16, 256, 8, 2, 512, 100), 2),     # I_shared not a multiple of 64
])
def test_unsupported_shapes_rejected(lib, dims, code):
    out = ctypes.c_size_t(0)
    st = lib.moe_workspace_size(ctypes.byref(M.MoeDims.of(*dims)), 0, ctypes.byref(out))
    assert st == code


def test_null_and_misaligned_arguments_rejected_before_launch(lib):
    d = M.MoeDims.of(256, 256, 8, 2, 512, 0)
    ws = ctypes.create_string_buffer(1 << 20)
    wsp = (ctypes.addressof(ws) + 255) // 256 * 256
    assert lib.moe_workspace_size(None, 0, None) == 1
    # null inputs
    assert lib.moe_route(ctypes.byref(d), 0, None, None, None, None, None, None, None, wsp, 1 << 19, None) == 1
    # bad gate enum
    assert lib.moe_route(ctypes.byref(d), 7, wsp, wsp, None, None, wsp, wsp, None, wsp, 1 << 19, None) == 1
    # misaligned x
    assert lib.moe_route(ctypes.byref(d), 0, wsp + 2, wsp, None, None, wsp, wsp, None, wsp, 1 << 19, None) == 1
    # workspace too small
    assert lib.moe_route(ctypes.byref(d), 0, wsp, wsp, None, None, wsp, wsp, None, wsp, 16, None) == 3
    assert lib.moe_permute(ctypes.byref(d), wsp, wsp, wsp, wsp, wsp, 64, None) == 3
    # router + sort in one call: null outputs, bad gate, misaligned x, small workspace
    rp = [wsp, wsp, None, None, wsp, wsp, None, wsp, wsp, wsp]   # x .. slot_perm
    assert lib.moe_route_permute(ctypes.byref(d), 0, *rp[:7], None, wsp, wsp, wsp, 1 << 19, None) == 1
    assert lib.moe_route_permute(ctypes.byref(d), 0, *rp[:9], None, wsp, 1 << 19, None) == 1
    assert lib.moe_route_permute(ctypes.byref(d), 3, *rp, wsp, 1 << 19, None) == 1
    assert lib.moe_route_permute(ctypes.byref(d), 0, wsp + 8, *rp[1:], wsp, 1 << 19, None) == 1
    assert lib.moe_route_permute(ctypes.byref(d), 0, *rp, wsp, 64, None) == 3
    args = [wsp] * 12
    assert lib.moe_grouped_mlp_fwd(ctypes.byref(d), *args[:6], None, None, None, None, None, wsp, 64, None) == 1
    assert lib.moe_unpermute_combine(ctypes.byref(d), None, wsp, wsp, None, wsp, None) == 1
    assert lib.moe_layer_bwd(ctypes.byref(d), *([None] * 23), wsp, 1 << 19, None) == 1
    # auxiliary loss: needs the probability sums, the offsets and an output
    f = ctypes.c_float(0.01)
    assert lib.moe_aux_loss(ctypes.byref(d), None, wsp, f, wsp, wsp, None) == 1
    assert lib.moe_aux_loss(ctypes.byref(d), wsp, wsp, f, None, None, None) == 1
    st = ctypes.c_int32(0)
    assert lib.moe_read_device_status(None, 0, None, 0, ctypes.byref(st)) == 1


def test_kernel_accounting_without_launches(lib):
    n = M.moe_kernel_count()
    names = [M.moe_kernel_name(i) for i in range(n)]
    assert len(set(names)) == n and "gate_up" in names and "wgrad_gate_up" in names
    assert M.moe_kernel_name(n) == "unknown"
    M.moe_timing_enable(False)
    st = M.moe_kernel_stats(reset=True)
    assert all(v == (0, 0.0) for v in M.moe_kernel_stats().values()) or st is not None


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 4)
    with pytest.raises(ValueError):
        M._ptr(x)


def test_capacity_field_validation(lib):
    d = M.MoeDims.of(64, 128, 4, 2, 128, 0, capacity=-1)
    out = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(d), 1, ctypes.byref(out)) == 1   # invalid arg
    for cap in (0, 1, 1000):
        d = M.MoeDims.of(64, 128, 4, 2, 128, 0, capacity=cap)
        assert lib.moe_workspace_size(ctypes.byref(d), 1, ctypes.byref(out)) == 0
    assert ctypes.sizeof(M.MoeDims) == 7 * 4


def test_expert_capacity_helper():
    assert M.expert_capacity(4096, 8, 128, 1.0) == 256
    assert M.expert_capacity(4096, 8, 128, 0.75) == 192
    assert M.expert_capacity(10, 2, 3, 1.0) == 7
    assert M.expert_capacity(100, 1, 10, 1.1) == 11
    with pytest.raises(ValueError):
        M.expert_capacity(8, 1, 4, 0.0)


def test_backward_argument_checks_before_launch(lib):
    """The backward refuses, before launching anything: the auxiliary loss's
    coefficients without the router logits, and recomputation (no saved g,u)
    with a workspace sized for the saved-pre-activation backward."""
    dims = (256, 256, 8, 2, 512, 0)
    d = M.MoeDims.of(*dims)
    saved = M.moe_workspace_size(dims, 1)
    recompute = M.moe_workspace_size(dims, 2)
    assert recompute > saved
    ws = ctypes.create_string_buffer(recompute + 256)
    p = (ctypes.addressof(ws) + 255) // 256 * 256

    def bwd(gu_saved, router_logits, aux_coef, nbytes):
        # grad_out, x, w_router, topk_idx, topk_w, offsets, perm_slot, slot_perm,
        # w_gate_up, w_down, gu_saved, w_sh_gate_up, w_sh_down, sh_gu_saved, grad_x,
        # grad_w_router, grad_router_bias, grad_w_gate_up, grad_w_down,
        # grad_w_sh_gate_up, grad_w_sh_down, router_logits, aux_coef
        a = [p] * 10 + [gu_saved, None, None, None, p, p, None, p, p, None, None,
                        router_logits, aux_coef]
        return lib.moe_layer_bwd(ctypes.byref(d), *a, p, nbytes, None)

    assert bwd(p, None, p, recompute) == 1          # aux coefficients, no logits
    assert bwd(None, None, None, saved) == 3        # recompute needs the larger workspace


def test_expert_parallel_calls_validate_before_launch(lib):
    ws = ctypes.create_string_buffer(4096)
    p = (ctypes.addressof(ws) + 255) // 256 * 256
    g = lib.moe_gather_rows
    assert g(p, 10, 64, p, 0, 1, p, None, None) == 0          # nothing to copy
    assert g(None, 10, 64, p, 4, 1, p, None, None) == 1       # null source
    assert g(p, 10, 64, p, 4, 0, p, None, None) == 1          # div < 1
    assert g(p, 10, 64, p, -1, 1, p, None, None) == 1         # negative count
    assert g(p + 8, 10, 64, p, 4, 1, p, None, None) == 1      # misaligned rows
    assert g(p, 10, 60, p, 4, 1, p, None, None) == 2          # H not a multiple of 8
    L = lib.moe_ep_receive_layout
    assert L(0, 4, p, 0, p, None, None, None, None) == 1      # no sources
    assert L(2, 0, p, 0, p, None, None, None, None) == 1      # no local experts
    assert L(2, 4, None, 0, p, None, None, None, None) == 1   # no counts
    assert L(2, 4, p, 8, p, None, None, None, None) == 1      # rows but no outputs
    assert L(2, 300, p, 0, p, None, None, None, None) == 2    # > 256 local experts
    assert L(64, 128, p, 0, p, None, None, None, None) == 2   # > 4096 cells
    assert "moe_gather_rows" in M.declared_functions()
    assert "moe_ep_receive_layout" in M.declared_functions()


def test_expert_parallel_backward_calls_validate_before_launch(lib):
    """The two halves of the expert-parallel backward and the scalar gather
    refuse bad arguments before launching anything."""
    dims_loc = M.MoeDims.of(64, 256, 4, 1, 512, 0)      # rows received, local experts, k = 1
    dims_src = M.MoeDims.of(32, 256, 8, 2, 512, 0)
    nbytes = max(M.moe_workspace_size(dims_loc, 1), M.moe_workspace_size(dims_src, 1))
    ws = ctypes.create_string_buffer(nbytes + 256)
    p = (ctypes.addressof(ws) + 255) // 256 * 256

    def experts(d, dx=p, dw=p, row_w=p, n=nbytes):
        # grad_out_rows, x_rows, row_w, offsets, perm_slot, slot_perm, w_gate_up, w_down,
        # gu_saved, dx_rows, dw_rows, grad_w_gate_up, grad_w_down
        a = [p, p, row_w, p, p, p, p, p, p, dx, dw, p, p]
        return lib.moe_experts_bwd(ctypes.byref(d), *a, p, n, None)

    assert experts(M.MoeDims.of(64, 256, 4, 2, 512, 0)) == 2      # k != 1
    assert experts(M.MoeDims.of(64, 256, 4, 1, 512, 128)) == 2    # a shared expert
    assert experts(dims_loc, dx=None) == 1                        # nowhere to put dx
    assert experts(dims_loc, dw=None) == 1
    assert experts(dims_loc, row_w=None) == 1                     # no routing weights
    assert experts(dims_loc, dx=p + 8) == 1                       # misaligned rows
    assert experts(dims_loc, n=256) == 3                          # workspace too small

    def router(d, dxs=p, dws=p, gx=p):
        # x, w_router, topk_idx, topk_w, offsets, perm_slot, slot_perm, dx_sorted,
        # dw_sorted, grad_x, grad_w_router, grad_router_bias
        a = [p, p, p, p, p, p, p, dxs, dws, gx, p, None]
        return lib.moe_router_bwd(ctypes.byref(d), *a, p, nbytes, None)

    assert router(M.MoeDims.of(32, 256, 8, 2, 512, 128)) == 2     # a shared expert
    assert router(dims_src, dxs=None) == 1                        # no slot gradients
    assert router(dims_src, dws=None) == 1
    assert router(dims_src, gx=None) == 1                         # nowhere to put grad_x
    assert router(dims_src, dxs=p + 8) == 1

    g = lib.moe_gather_scalars
    assert g(p, 10, p, 0, 1, p, None, None) == 0                  # nothing to copy
    assert g(None, 10, p, 4, 1, p, None, None) == 1
    assert g(p, 10, p, 4, 0, p, None, None) == 1                  # div < 1
    assert g(p, 10, p, -1, 1, p, None, None) == 1
    assert g(p + 2, 10, p, 4, 1, p, None, None) == 1              # not 4-byte aligned
    for name in ("moe_experts_bwd", "moe_router_bwd", "moe_gather_scalars"):
        assert name in M.declared_functions()
