"""Thin Python binding of the C ABI in include/moe.h (argument marshalling only).

Every function here has the name of the C call it wraps and forwards torch
tensors as raw device pointers together with the current CUDA stream.  All
computation runs in the CUDA library; if the library is missing this module
raises instead of computing anything on the CPU.

``MoeLayer`` is a small convenience on top: it allocates the routing buffers,
saved activations and the workspace with torch and runs the five calls in
order (forward, then backward).
"""

from __future__ import annotations

import ctypes
import math
import os
import re
from fractions import Fraction

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_b300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "moe.h")

MOE_GATE_SOFTMAX_TOPK = 0
MOE_GATE_BALANCED = 1

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
                3: "MOE_ERR_WORKSPACE_TOO_SMALL", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_INDEX",
                6: "MOE_ERR_TIMEOUT"}


class MoeError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {STATUS_NAMES.get(status, status)}")


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("I", ctypes.c_int32), ("I_shared", ctypes.c_int32),
                ("capacity", ctypes.c_int32)]

    @classmethod
    def of(cls, T, H, E, k, I, I_shared=0, capacity=0):
        return cls(int(T), int(H), int(E), int(k), int(I), int(I_shared), int(capacity))

    def as_tuple(self):
        """The shape (T, H, E, k, I, I_shared); capacity is a separate field."""
        return (self.T, self.H, self.E, self.k, self.I, self.I_shared)


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I32 = ctypes.c_int32
_DIMS = ctypes.POINTER(MoeDims)

_SIGS = {
    "moe_abi_version": ([], _I32),
    "moe_status_string": ([_I32], ctypes.c_char_p),
    "moe_workspace_size": ([_DIMS, _I32, ctypes.POINTER(_SZ)], _I32),
    "moe_route": ([_DIMS, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _I32),
    "moe_route_permute": ([_DIMS, _I32] + [_P] * 11 + [_SZ, _P], _I32),
    "moe_aux_loss": ([_DIMS, _P, _P, ctypes.c_float, _P, _P, _P], _I32),
    "moe_permute": ([_DIMS, _P, _P, _P, _P, _P, _SZ, _P], _I32),
    "moe_grouped_mlp_fwd": ([_DIMS, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], _I32),
    "moe_unpermute_combine": ([_DIMS, _P, _P, _P, _P, _P, _P], _I32),
    "moe_layer_bwd": ([_DIMS] + [_P] * 23 + [_P, _SZ, _P], _I32),
    "moe_read_device_status": ([_P, _SZ, _P, _I32, ctypes.POINTER(_I32)], _I32),
    "moe_permute_static_scratch": ([_DIMS, _P, _P, _P, _P, _P, _P], _I32),
    "moe_gather_rows": ([_P, ctypes.c_int64, _I32, _P, _I32, _I32, _P, _P, _P], _I32),
    "moe_ep_receive_layout": ([_I32, _I32, _P, _I32, _P, _P, _P, _P, _P], _I32),
    "moe_gather_scalars": ([_P, ctypes.c_int64, _P, _I32, _I32, _P, _P, _P], _I32),
    "moe_experts_bwd": ([_DIMS] + [_P] * 13 + [_P, _SZ, _P], _I32),
    "moe_router_bwd": ([_DIMS] + [_P] * 12 + [_P, _SZ, _P], _I32),
    "moe_kernel_count": ([], _I32),
    "moe_kernel_name": ([_I32], ctypes.c_char_p),
    "moe_timing_enable": ([_I32], _I32),
    "moe_kernel_stats": ([_I32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)], _I32),
}

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"MoE CUDA library not found at {path}; run "
                           "`python -m grouped_expert_gemm_top_b300.build` first")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def declared_functions(header: str = HEADER) -> list[str]:
    """Names of the functions declared in include/moe.h."""
    text = open(header).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(moe_\w+)\s*\(", text, re.M)))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ws(ws):
    return _ptr(ws), ws.numel() * ws.element_size()


def _check(call: str, st: int):
    if st != 0:
        raise MoeError(call, st)


def _dims(d) -> MoeDims:
    return d if isinstance(d, MoeDims) else MoeDims.of(*d)


def expert_capacity(T: int, k: int, E: int, factor: float) -> int:
    """Slots each expert keeps for a capacity factor: ceil(factor * T * k / E).

    The library takes the integer (moe_dims.capacity, 0 = no limit), so a
    factor whose capacity rounds to 0 is refused here rather than silently
    meaning "no limit"."""
    c = math.ceil(Fraction(str(factor)) * T * k / E)   # the factor as written, exactly
    if c < 1:
        raise ValueError(f"capacity factor {factor} keeps no slot per expert")
    return c


# ----------------------------------------------------------------- C-ABI calls
def moe_abi_version() -> int:
    return load_library().moe_abi_version()


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


def moe_workspace_size(dims, with_backward) -> int:
    """with_backward: 0 forward only, 1 backward with saved pre-activations,
    2 backward that recomputes them (True/False map to 1/0)."""
    out = _SZ(0)
    _check("moe_workspace_size",
           load_library().moe_workspace_size(ctypes.byref(_dims(dims)), int(with_backward), ctypes.byref(out)))
    return out.value


def moe_route(dims, gate_mode, x, w_router, router_bias, logits_out, topk_idx, topk_w, workspace,
              stream=None, prob_sum=None):
    p, n = _ws(workspace)
    _check("moe_route", load_library().moe_route(
        ctypes.byref(_dims(dims)), int(gate_mode), _ptr(x), _ptr(w_router), _ptr(router_bias),
        _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(prob_sum), p, n, _stream(stream)))


def moe_route_permute(dims, gate_mode, x, w_router, router_bias, logits_out, topk_idx, topk_w,
                      expert_offsets, perm_slot, slot_perm, workspace, stream=None, prob_sum=None):
    p, n = _ws(workspace)
    _check("moe_route_permute", load_library().moe_route_permute(
        ctypes.byref(_dims(dims)), int(gate_mode), _ptr(x), _ptr(w_router), _ptr(router_bias),
        _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(prob_sum), _ptr(expert_offsets),
        _ptr(perm_slot), _ptr(slot_perm), p, n, _stream(stream)))


def moe_aux_loss(dims, prob_sum, expert_offsets, alpha, loss, coef, stream=None):
    _check("moe_aux_loss", load_library().moe_aux_loss(
        ctypes.byref(_dims(dims)), _ptr(prob_sum), _ptr(expert_offsets), ctypes.c_float(alpha),
        _ptr(loss), _ptr(coef), _stream(stream)))


def moe_permute(dims, topk_idx, expert_offsets, perm_slot, slot_perm, workspace, stream=None):
    p, n = _ws(workspace)
    _check("moe_permute", load_library().moe_permute(
        ctypes.byref(_dims(dims)), _ptr(topk_idx), _ptr(expert_offsets), _ptr(perm_slot),
        _ptr(slot_perm), p, n, _stream(stream)))


def moe_grouped_mlp_fwd(dims, x, expert_offsets, perm_slot, w_gate_up, w_down, gu_saved, y_perm,
                        w_sh_gate_up, w_sh_down, sh_gu_saved, y_shared, workspace, stream=None):
    p, n = _ws(workspace)
    _check("moe_grouped_mlp_fwd", load_library().moe_grouped_mlp_fwd(
        ctypes.byref(_dims(dims)), _ptr(x), _ptr(expert_offsets), _ptr(perm_slot), _ptr(w_gate_up),
        _ptr(w_down), _ptr(gu_saved), _ptr(y_perm), _ptr(w_sh_gate_up), _ptr(w_sh_down),
        _ptr(sh_gu_saved), _ptr(y_shared), p, n, _stream(stream)))


def moe_unpermute_combine(dims, y_perm, slot_perm, topk_w, y_shared, out, stream=None):
    _check("moe_unpermute_combine", load_library().moe_unpermute_combine(
        ctypes.byref(_dims(dims)), _ptr(y_perm), _ptr(slot_perm), _ptr(topk_w), _ptr(y_shared),
        _ptr(out), _stream(stream)))


def moe_layer_bwd(dims, grad_out, x, w_router, topk_idx, topk_w, expert_offsets, perm_slot,
                  slot_perm, w_gate_up, w_down, gu_saved, w_sh_gate_up, w_sh_down, sh_gu_saved,
                  grad_x, grad_w_router, grad_router_bias, grad_w_gate_up, grad_w_down,
                  grad_w_sh_gate_up, grad_w_sh_down, workspace, stream=None, router_logits=None,
                  aux_coef=None):
    p, n = _ws(workspace)
    args = [grad_out, x, w_router, topk_idx, topk_w, expert_offsets, perm_slot, slot_perm,
            w_gate_up, w_down, gu_saved, w_sh_gate_up, w_sh_down, sh_gu_saved, grad_x,
            grad_w_router, grad_router_bias, grad_w_gate_up, grad_w_down, grad_w_sh_gate_up,
            grad_w_sh_down, router_logits, aux_coef]
    _check("moe_layer_bwd", load_library().moe_layer_bwd(
        ctypes.byref(_dims(dims)), *[_ptr(a) for a in args], p, n, _stream(stream)))


def moe_read_device_status(workspace, clear: bool = True, stream=None) -> int:
    p, n = _ws(workspace)
    out = _I32(0)
    _check("moe_read_device_status", load_library().moe_read_device_status(
        p, n, _stream(stream), int(clear), ctypes.byref(out)))
    return out.value


def moe_permute_static_scratch(dims, topk_idx, expert_offsets, perm_slot, slot_perm,
                               device_status=None, stream=None):
    """moe_permute without a workspace, for callers that cannot allocate device
    memory: the sort's scratch is a fixed 256 KiB array inside the library
    (shared by every call on a device, so calls must not overlap on the GPU)."""
    _check("moe_permute_static_scratch", load_library().moe_permute_static_scratch(
        ctypes.byref(_dims(dims)), _ptr(topk_idx), _ptr(expert_offsets), _ptr(perm_slot),
        _ptr(slot_perm), _ptr(device_status), _stream(stream)))


def moe_gather_rows(src, idx, div, dst, device_status=None, stream=None):
    """dst[i] = src[idx[i] // div] (bf16 rows; idx int32 [n]; dst [n, H])."""
    n = int(idx.numel())
    _check("moe_gather_rows", load_library().moe_gather_rows(
        _ptr(src) if src.numel() else None, int(src.shape[0]), int(src.shape[1]),
        _ptr(idx) if n else None, n, int(div), _ptr(dst) if n else None, _ptr(device_status),
        _stream(stream)))


def moe_ep_receive_layout(counts, local_offsets, recv_perm, recv_inv, device_status=None,
                          stream=None):
    """counts int32 [n_src, E_local] (device) -> local_offsets [E_local+1],
    recv_perm / recv_inv [R] with R = counts.sum() (given by their length)."""
    n_src, E_loc = int(counts.shape[0]), int(counts.shape[1])
    R = int(recv_perm.numel())
    _check("moe_ep_receive_layout", load_library().moe_ep_receive_layout(
        n_src, E_loc, _ptr(counts), R, _ptr(local_offsets), _ptr(recv_perm) if R else None,
        _ptr(recv_inv) if R else None, _ptr(device_status), _stream(stream)))


def moe_gather_scalars(src, idx, div, dst, device_status=None, stream=None):
    """dst[i] = src.flat[idx[i] // div] for 4-byte elements (idx int32 [n], dst [n])."""
    n = int(idx.numel())
    _check("moe_gather_scalars", load_library().moe_gather_scalars(
        _ptr(src) if src.numel() else None, int(src.numel()), _ptr(idx) if n else None, n,
        int(div), _ptr(dst) if n else None, _ptr(device_status), _stream(stream)))


def moe_experts_bwd(dims, grad_out_rows, x_rows, row_w, expert_offsets, perm_slot, slot_perm,
                    w_gate_up, w_down, gu_saved, dx_rows, dw_rows, grad_w_gate_up, grad_w_down,
                    workspace, stream=None):
    """The experts part of the expert-parallel backward (dims: T = rows received,
    k = 1, E = local experts); see include/moe.h."""
    p, n = _ws(workspace)
    args = [grad_out_rows, x_rows, row_w, expert_offsets, perm_slot, slot_perm, w_gate_up, w_down,
            gu_saved, dx_rows, dw_rows, grad_w_gate_up, grad_w_down]
    _check("moe_experts_bwd", load_library().moe_experts_bwd(
        ctypes.byref(_dims(dims)), *[_ptr(a) for a in args], p, n, _stream(stream)))


def moe_router_bwd(dims, x, w_router, topk_idx, topk_w, expert_offsets, perm_slot, slot_perm,
                   dx_sorted, dw_sorted, grad_x, grad_w_router, grad_router_bias, workspace,
                   stream=None):
    """The router part of the expert-parallel backward on the tokens' rank; see
    include/moe.h."""
    p, n = _ws(workspace)
    args = [x, w_router, topk_idx, topk_w, expert_offsets, perm_slot, slot_perm, dx_sorted,
            dw_sorted, grad_x, grad_w_router, grad_router_bias]
    _check("moe_router_bwd", load_library().moe_router_bwd(
        ctypes.byref(_dims(dims)), *[_ptr(a) for a in args], p, n, _stream(stream)))


def moe_kernel_count() -> int:
    return load_library().moe_kernel_count()


def moe_kernel_name(i: int) -> str:
    return load_library().moe_kernel_name(i).decode()


def moe_timing_enable(on: bool):
    _check("moe_timing_enable", load_library().moe_timing_enable(int(on)))


def moe_kernel_stats(reset: bool = True) -> dict:
    """{kernel name: (launches, summed event ms)} since the last reset."""
    n = moe_kernel_count()
    launches = (ctypes.c_int64 * n)()
    ms = (ctypes.c_double * n)()
    _check("moe_kernel_stats", load_library().moe_kernel_stats(int(reset), launches, ms))
    return {moe_kernel_name(i): (int(launches[i]), float(ms[i])) for i in range(n)}


# ----------------------------------------------------------------- convenience
class MoeLayer:
    """Buffers + call sequence for one layer shape on one device.

    Weights are passed in (bf16 torch tensors on the device); all activations,
    routing buffers and the workspace are allocated once here with torch.
    """

    def __init__(self, dims, gate_mode=MOE_GATE_SOFTMAX_TOPK, device="cuda", with_backward=True,
                 save_logits=False, recompute=False, aux_alpha=None, capacity=0):
        """recompute: the forward keeps no gate/up pre-activations; the
        backward recomputes them (activation recompute).  aux_alpha: add the
        auxiliary load-balancing loss with this coefficient (its value lands
        in self.aux_loss after forward; its gradient is added in backward).
        capacity: slots each expert keeps (0: no limit); the others are
        dropped (slot_perm -1; their rows of y_perm / gu_saved are not written)."""
        self.dims = MoeDims.of(*_dims(dims).as_tuple(), capacity=capacity)
        T, H, E, k, I, Is = self.dims.as_tuple()
        S = T * k
        self.gate_mode = gate_mode
        dev = torch.device(device)
        bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        self.aux_alpha = aux_alpha
        aux = aux_alpha is not None
        self.logits = torch.empty(T, E, dtype=f32, device=dev) if (save_logits or aux) else None
        self.prob_sum = torch.empty(E, dtype=f32, device=dev) if aux else None
        self.aux_loss = torch.zeros(1, dtype=f32, device=dev) if aux else None
        self.aux_coef = torch.empty(E, dtype=f32, device=dev) if aux else None
        self.topk_idx = torch.empty(T, k, dtype=i32, device=dev)
        self.topk_w = torch.empty(T, k, dtype=f32, device=dev)
        self.expert_offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.perm_slot = torch.empty(S, dtype=i32, device=dev)
        self.slot_perm = torch.empty(S, dtype=i32, device=dev)
        keep = with_backward and not recompute
        self.gu_saved = torch.empty(S, 2 * I, dtype=bf, device=dev) if keep else None
        self.y_perm = torch.empty(S, H, dtype=bf, device=dev)
        self.sh_gu_saved = torch.empty(T, 2 * Is, dtype=bf, device=dev) if (Is and keep) else None
        self.y_shared = torch.empty(T, H, dtype=bf, device=dev) if Is else None
        self.out = torch.empty(T, H, dtype=bf, device=dev)
        nbytes = moe_workspace_size(self.dims, (2 if recompute else 1) if with_backward else 0)
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def forward(self, x, w_router, w_gate_up, w_down, router_bias=None, w_sh_gate_up=None,
                w_sh_down=None, stream=None, out=None):
        """out: bf16 [T, H] to write the layer output into (default: self.out)."""
        d, ws = self.dims, self.workspace
        out = self.out if out is None else out
        moe_route_permute(d, self.gate_mode, x, w_router, router_bias, self.logits, self.topk_idx,
                          self.topk_w, self.expert_offsets, self.perm_slot, self.slot_perm, ws,
                          stream, prob_sum=self.prob_sum)
        if self.aux_alpha is not None:
            moe_aux_loss(d, self.prob_sum, self.expert_offsets, self.aux_alpha, self.aux_loss,
                         self.aux_coef, stream)
        moe_grouped_mlp_fwd(d, x, self.expert_offsets, self.perm_slot, w_gate_up, w_down,
                            self.gu_saved, self.y_perm, w_sh_gate_up, w_sh_down, self.sh_gu_saved,
                            self.y_shared, ws, stream)
        moe_unpermute_combine(d, self.y_perm, self.slot_perm, self.topk_w, self.y_shared, out, stream)
        return out

    def alloc_grads(self, with_bias=False):
        T, H, E, k, I, Is = self.dims.as_tuple()
        dev = self.out.device
        bf = torch.bfloat16
        g = dict(grad_x=torch.empty(T, H, dtype=bf, device=dev),
                 grad_w_router=torch.empty(E, H, dtype=bf, device=dev),
                 grad_router_bias=torch.empty(E, dtype=torch.float32, device=dev) if with_bias else None,
                 grad_w_gate_up=torch.empty(E, 2 * I, H, dtype=bf, device=dev),
                 grad_w_down=torch.empty(E, H, I, dtype=bf, device=dev),
                 grad_w_sh_gate_up=torch.empty(2 * Is, H, dtype=bf, device=dev) if Is else None,
                 grad_w_sh_down=torch.empty(H, Is, dtype=bf, device=dev) if Is else None)
        return g

    def backward(self, grad_out, x, w_router, w_gate_up, w_down, grads, w_sh_gate_up=None,
                 w_sh_down=None, stream=None):
        moe_layer_bwd(self.dims, grad_out, x, w_router, self.topk_idx, self.topk_w,
                      self.expert_offsets, self.perm_slot, self.slot_perm, w_gate_up, w_down,
                      self.gu_saved, w_sh_gate_up, w_sh_down, self.sh_gu_saved, grads["grad_x"],
                      grads["grad_w_router"], grads["grad_router_bias"], grads["grad_w_gate_up"],
                      grads["grad_w_down"], grads["grad_w_sh_gate_up"], grads["grad_w_sh_down"],
                      self.workspace, stream, router_logits=self.logits if self.aux_coef is not None else None,
                      aux_coef=self.aux_coef)
        return grads
