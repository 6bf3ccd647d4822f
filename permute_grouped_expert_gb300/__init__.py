"""GB300-native (sm_103a) single-GPU MoE dispatch -> grouped expert MLP -> combine.

A thin ctypes binding over ``libmoe_gb300.so``, whose C ABI is declared in
``include/moe.h``.  The binding only marshals arguments: torch tensors become
device pointers, shapes become the C structs, and the current torch CUDA stream
becomes the ``stream`` argument.  Every step of the path runs in the library's
CUDA kernels; there is no CPU fallback.  If the library has not been built the
import fails with an explicit error.

The four calls of one MoE layer forward keep their C names:
``moe_preprocess``, ``moe_dispatch_permute``, ``moe_grouped_mlp`` and
``moe_combine_unpermute``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

# --------------------------------------------------------------- C mirrors

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_RING_EARLY_REUSE = 5
MOE_ERR_RING_DOUBLE_RELEASE = 6

ROUTING_DENSE_I16 = 0
ROUTING_SPARSE_BOOL = 1

DTYPE_BF16 = 0
DTYPE_FP8_E4M3_B128 = 1
DTYPE_BF16_TO_FP8 = 2
DTYPE_NVFP4 = 3
DTYPE_BF16_TO_NVFP4 = 4

COMBINE_BF16 = 0
COMBINE_MXFP8 = 1
COMBINE_MXFP4 = 2

DEV_ERR_BAD_EXPERT = 1
DEV_ERR_TOO_MANY_ROUTES = 2
DEV_ERR_TIMEOUT = 4
DEV_ERR_BOUNDS = 8  # bounds-checked builds only


class _Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("E", ctypes.c_int64), ("K", ctypes.c_int64),
                ("I", ctypes.c_int64)]


class _Layout(ctypes.Structure):
    _fields_ = [("pad_multiple", ctypes.c_int64), ("capacity", ctypes.c_int64)]


class _Routing(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("map", ctypes.c_void_p), ("probs", ctypes.c_void_p)]


class _HandleDev(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("tokens_per_expert", "padded_offsets", "row_of", "token_of",
                                               "slot_of", "total_rows", "overflow", "status")]


class _Nvfp4Globals(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("fc1_input_scale", "fc2_input_scale", "w13_scale_2",
                                               "w2_scale_2")]


# Every symbol include/moe.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SIGNATURES = {
    "moe_capacity": [_I64, ctypes.c_double, _I64, ctypes.POINTER(_I64)],
    "moe_routing_map_bytes": [ctypes.c_int32, _I64, _I64, _I64, ctypes.POINTER(ctypes.c_size_t)],
    "moe_decode_bucket": [_I64, ctypes.POINTER(_I64), ctypes.c_int32, ctypes.POINTER(_I64)],
    "moe_last_cuda_error": [],
    "moe_status_string": [ctypes.c_int],
    "moe_preprocess_workspace_size": [ctypes.POINTER(_Shape), ctypes.POINTER(ctypes.c_size_t)],
    "moe_preprocess": [ctypes.POINTER(_Routing), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                       ctypes.POINTER(_HandleDev), _P, ctypes.c_size_t, _P],
    "moe_preprocess_noalloc": [ctypes.POINTER(_Routing), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                               ctypes.POINTER(_HandleDev), _P],
    "moe_dispatch_permute": [ctypes.POINTER(_HandleDev), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                             ctypes.c_int32, _P, _P, ctypes.POINTER(_Routing), _P, _P, _P, _P],
    "moe_combine_unpermute": [ctypes.POINTER(_HandleDev), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                              _P, _P, _P, _P],
    "moe_combine_backward": [ctypes.POINTER(_HandleDev), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                             _P, _P, _P, _P, _P, _P],
    "moe_dispatch_backward": [ctypes.POINTER(_HandleDev), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                              ctypes.c_int32, _P, _P, _P, _P, _P],
    "moe_grouped_mlp_workspace_size": [ctypes.POINTER(_Shape), ctypes.POINTER(_Layout), ctypes.c_int32,
                                       ctypes.POINTER(ctypes.c_size_t)],
    "moe_grouped_mlp": [ctypes.POINTER(_HandleDev), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                        ctypes.c_int32, _P, _P, _P, _P, _P, _P, ctypes.POINTER(_Nvfp4Globals), _P,
                        ctypes.c_size_t, _P, _P],
    "moe_grouped_mlp_ex": [ctypes.POINTER(_HandleDev), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                           ctypes.c_int32, _P, _P, _P, _P, _P, _P, ctypes.POINTER(_Nvfp4Globals), _P,
                           ctypes.c_size_t, ctypes.c_int32, _P, _P, _P, _P],
    "moe_combine_unpermute_fmt": [ctypes.POINTER(_HandleDev), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                                  ctypes.c_int32, _P, _P, _P, _P, _P],
    "moe_quantize_mx_rows": [_P, _I64, _I64, ctypes.c_int32, _P, _P, _P],
    "moe_grouped_mlp_kernel_count": [ctypes.POINTER(_Shape), ctypes.POINTER(_Layout), ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_int32)],
    "moe_profile_next_grouped_mlp": [_P, _P, _P],
    "moe_debug_next_grouped_mlp_silent_token_tile": [_I64],
    "moe_debug_preprocess_silent_tile": [ctypes.POINTER(_Routing), ctypes.POINTER(_Shape), ctypes.POINTER(_Layout),
                                         ctypes.POINTER(_HandleDev), _P, ctypes.c_size_t, ctypes.c_int64, _P],
    "moe_quantize_fp8_blocks": [_P, _I64, _I64, _I64, _P, _P, _P],
    "moe_quantize_nvfp4_rows": [_P, _I64, _I64, _P, _P, _P, _P],
    "moe_ring_create": [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_P)],
    "moe_ring_acquire": [_P, _P, ctypes.POINTER(ctypes.c_int32)],
    "moe_ring_release": [_P, ctypes.c_int32, _P],
    "moe_ring_destroy": [_P],
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(nvcc, sm_103a) before using permute_grouped_expert_gb300")
    lib = ctypes.CDLL(LIB_PATH)
    for name, args in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name in ("moe_last_cuda_error", "moe_status_string") else ctypes.c_int
    return lib


_lib = _load()


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        msg = _lib.moe_status_string(status).decode()
        if status == MOE_ERR_CUDA:
            msg += " (" + _lib.moe_last_cuda_error().decode() + ")"
        super().__init__(f"{what}: {msg}")
        self.status = status


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ------------------------------------------------------------ public types

@dataclasses.dataclass(frozen=True)
class Shape:
    T: int
    H: int
    E: int
    K: int
    I: int = 0

    def c(self):
        return _Shape(self.T, self.H, self.E, self.K, self.I)


@dataclasses.dataclass(frozen=True)
class Layout:
    pad_multiple: int
    capacity: int

    def c(self):
        return _Layout(self.pad_multiple, self.capacity)


@dataclasses.dataclass
class Routing:
    """format: ROUTING_DENSE_I16 (map int16 [T, K], probs float [T, K]) or
    ROUTING_SPARSE_BOOL (map uint8 [T, E], probs float [T, E]); probs optional."""
    format: int
    map: torch.Tensor
    probs: Optional[torch.Tensor] = None

    def c(self):
        return _Routing(self.format, _ptr(self.map), _ptr(self.probs))


@dataclasses.dataclass
class Handle:
    """The device arrays moe_preprocess fills (see moe_handle_dev in moe.h)."""
    tokens_per_expert: torch.Tensor
    padded_offsets: torch.Tensor
    row_of: torch.Tensor
    token_of: torch.Tensor
    slot_of: torch.Tensor
    total_rows: torch.Tensor
    overflow: torch.Tensor
    status: torch.Tensor

    @staticmethod
    def empty(shape: Shape, layout: Layout, device="cuda") -> "Handle":
        i32 = dict(dtype=torch.int32, device=device)
        return Handle(
            tokens_per_expert=torch.empty(shape.E, **i32), padded_offsets=torch.empty(shape.E + 1, **i32),
            row_of=torch.empty(max(shape.T * shape.K, 1), **i32), token_of=torch.empty(max(layout.capacity, 1), **i32),
            slot_of=torch.empty(max(layout.capacity, 1), **i32), total_rows=torch.empty(1, **i32),
            overflow=torch.empty(1, **i32), status=torch.empty(1, **i32))

    def c(self):
        return _HandleDev(*(_ptr(getattr(self, f.name)) for f in dataclasses.fields(self)))


@dataclasses.dataclass
class Nvfp4Globals:
    fc1_input_scale: torch.Tensor  # float [1]
    fc2_input_scale: torch.Tensor  # float [1]
    w13_scale_2: torch.Tensor      # float [E]
    w2_scale_2: torch.Tensor       # float [E]

    def c(self):
        return _Nvfp4Globals(_ptr(self.fc1_input_scale), _ptr(self.fc2_input_scale), _ptr(self.w13_scale_2),
                             _ptr(self.w2_scale_2))


# --------------------------------------------------------------- host calls

def moe_capacity(rows: int, factor: float, align: int = 4) -> int:
    out = _I64()
    _check(_lib.moe_capacity(rows, factor, align, ctypes.byref(out)), "moe_capacity")
    return out.value


def moe_decode_bucket(tokens: int, ladder) -> int:
    """Smallest bucket of ``ladder`` (ascending token counts) that holds ``tokens``."""
    arr = (_I64 * len(ladder))(*ladder)
    out = _I64()
    _check(_lib.moe_decode_bucket(tokens, arr, len(ladder), ctypes.byref(out)), "moe_decode_bucket")
    return out.value


def moe_routing_map_bytes(fmt: int, T: int, E: int, K: int) -> int:
    out = ctypes.c_size_t()
    _check(_lib.moe_routing_map_bytes(fmt, T, E, K, ctypes.byref(out)), "moe_routing_map_bytes")
    return out.value


def moe_preprocess_workspace_size(shape: Shape) -> int:
    out = ctypes.c_size_t()
    _check(_lib.moe_preprocess_workspace_size(ctypes.byref(shape.c()), ctypes.byref(out)),
           "moe_preprocess_workspace_size")
    return out.value


def moe_grouped_mlp_workspace_size(shape: Shape, layout: Layout, w_dtype: int) -> int:
    out = ctypes.c_size_t()
    _check(_lib.moe_grouped_mlp_workspace_size(ctypes.byref(shape.c()), ctypes.byref(layout.c()), w_dtype,
                                               ctypes.byref(out)), "moe_grouped_mlp_workspace_size")
    return out.value


def moe_grouped_mlp_kernel_count(shape: Shape, layout: Layout, w_dtype: int) -> int:
    out = ctypes.c_int32()
    _check(_lib.moe_grouped_mlp_kernel_count(ctypes.byref(shape.c()), ctypes.byref(layout.c()), w_dtype,
                                             ctypes.byref(out)), "moe_grouped_mlp_kernel_count")
    return out.value


# ------------------------------------------------------------- device calls

def moe_preprocess(routing: Routing, shape: Shape, layout: Layout, handle: Handle, workspace: torch.Tensor,
                   stream=None) -> None:
    _check(_lib.moe_preprocess(ctypes.byref(routing.c()), ctypes.byref(shape.c()), ctypes.byref(layout.c()),
                               ctypes.byref(handle.c()), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_preprocess")


def moe_preprocess_noalloc(routing: Routing, shape: Shape, layout: Layout, handle: Handle, stream=None) -> None:
    """moe_preprocess without a caller workspace: for callers that cannot
    allocate device memory (a plugin whose host application owns all device
    memory, a loop that must not call cudaMalloc).  Uses the library's fixed
    scratch array; see moe_preprocess_noalloc in moe.h for its limits."""
    _check(_lib.moe_preprocess_noalloc(ctypes.byref(routing.c()), ctypes.byref(shape.c()), ctypes.byref(layout.c()),
                                       ctypes.byref(handle.c()), _stream(stream)), "moe_preprocess_noalloc")


def moe_dispatch_permute(handle: Handle, shape: Shape, layout: Layout, in_dtype: int, x: torch.Tensor,
                         x_scales: Optional[torch.Tensor], routing: Routing, out_tokens: torch.Tensor,
                         out_probs: Optional[torch.Tensor] = None, out_scales: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    _check(_lib.moe_dispatch_permute(ctypes.byref(handle.c()), ctypes.byref(shape.c()),
                                     ctypes.byref(layout.c()), in_dtype, _ptr(x), _ptr(x_scales),
                                     ctypes.byref(routing.c()), _ptr(out_tokens), _ptr(out_probs),
                                     _ptr(out_scales), _stream(stream)), "moe_dispatch_permute")


def moe_grouped_mlp(handle: Handle, shape: Shape, layout: Layout, w_dtype: int, perm_tokens: torch.Tensor,
                    perm_scales: Optional[torch.Tensor], w13: torch.Tensor, w13_scales: Optional[torch.Tensor],
                    w2: torch.Tensor, w2_scales: Optional[torch.Tensor], globals_: Optional[Nvfp4Globals],
                    workspace: torch.Tensor, out_fc2: torch.Tensor, stream=None) -> None:
    g = ctypes.byref(globals_.c()) if globals_ is not None else None
    _check(_lib.moe_grouped_mlp(ctypes.byref(handle.c()), ctypes.byref(shape.c()), ctypes.byref(layout.c()),
                                w_dtype, _ptr(perm_tokens), _ptr(perm_scales), _ptr(w13), _ptr(w13_scales),
                                _ptr(w2), _ptr(w2_scales), g, _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(out_fc2), _stream(stream)),
           "moe_grouped_mlp")


def moe_grouped_mlp_ex(handle: Handle, shape: Shape, layout: Layout, w_dtype: int, perm_tokens: torch.Tensor,
                       perm_scales: Optional[torch.Tensor], w13: torch.Tensor, w13_scales: Optional[torch.Tensor],
                       w2: torch.Tensor, w2_scales: Optional[torch.Tensor], globals_: Optional[Nvfp4Globals],
                       workspace: torch.Tensor, out_format: int, out_fc2: torch.Tensor,
                       out_fc2_scales: Optional[torch.Tensor] = None, fc2_row_probs: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    g = ctypes.byref(globals_.c()) if globals_ is not None else None
    _check(_lib.moe_grouped_mlp_ex(ctypes.byref(handle.c()), ctypes.byref(shape.c()), ctypes.byref(layout.c()),
                                   w_dtype, _ptr(perm_tokens), _ptr(perm_scales), _ptr(w13), _ptr(w13_scales),
                                   _ptr(w2), _ptr(w2_scales), g, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), out_format, _ptr(out_fc2),
                                   _ptr(out_fc2_scales), _ptr(fc2_row_probs), _stream(stream)),
           "moe_grouped_mlp_ex")


def moe_combine_unpermute_fmt(handle: Handle, shape: Shape, layout: Layout, in_format: int,
                              expert_out: torch.Tensor, expert_out_scales: Optional[torch.Tensor],
                              perm_probs: Optional[torch.Tensor], y: torch.Tensor, stream=None) -> None:
    _check(_lib.moe_combine_unpermute_fmt(ctypes.byref(handle.c()), ctypes.byref(shape.c()),
                                          ctypes.byref(layout.c()), in_format, _ptr(expert_out),
                                          _ptr(expert_out_scales), _ptr(perm_probs), _ptr(y), _stream(stream)),
           "moe_combine_unpermute_fmt")


def moe_quantize_mx_rows(x: torch.Tensor, fmt: int, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    H = x.shape[-1]
    R = x.numel() // H
    _check(_lib.moe_quantize_mx_rows(_ptr(x), R, H, fmt, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_quantize_mx_rows")


def moe_combine_unpermute(handle: Handle, shape: Shape, layout: Layout, expert_out: torch.Tensor,
                          perm_probs: Optional[torch.Tensor], y: torch.Tensor, stream=None) -> None:
    _check(_lib.moe_combine_unpermute(ctypes.byref(handle.c()), ctypes.byref(shape.c()), ctypes.byref(layout.c()),
                                      _ptr(expert_out), _ptr(perm_probs), _ptr(y), _stream(stream)),
           "moe_combine_unpermute")


def moe_combine_backward(handle: Handle, shape: Shape, layout: Layout, grad_y: torch.Tensor,
                         expert_out: Optional[torch.Tensor], perm_probs: Optional[torch.Tensor],
                         grad_expert_out: torch.Tensor, grad_perm_probs: Optional[torch.Tensor] = None,
                         stream=None) -> None:
    _check(_lib.moe_combine_backward(ctypes.byref(handle.c()), ctypes.byref(shape.c()), ctypes.byref(layout.c()),
                                     _ptr(grad_y), _ptr(expert_out), _ptr(perm_probs), _ptr(grad_expert_out),
                                     _ptr(grad_perm_probs), _stream(stream)), "moe_combine_backward")


def moe_dispatch_backward(handle: Handle, shape: Shape, layout: Layout, routing_format: int,
                          grad_perm_tokens: torch.Tensor, grad_perm_probs: Optional[torch.Tensor],
                          grad_x: torch.Tensor, grad_probs: Optional[torch.Tensor] = None, stream=None) -> None:
    _check(_lib.moe_dispatch_backward(ctypes.byref(handle.c()), ctypes.byref(shape.c()), ctypes.byref(layout.c()),
                                      routing_format, _ptr(grad_perm_tokens), _ptr(grad_perm_probs), _ptr(grad_x),
                                      _ptr(grad_probs), _stream(stream)), "moe_dispatch_backward")


def moe_profile_next_grouped_mlp(ev_before_fc1, ev_after_fc1, ev_after_fc2) -> None:
    """Record three torch.cuda.Event objects around FC1 / FC2 of the next moe_grouped_mlp call."""
    handles = [ctypes.c_void_p(e.cuda_event) if e is not None else None
               for e in (ev_before_fc1, ev_after_fc1, ev_after_fc2)]
    _check(_lib.moe_profile_next_grouped_mlp(*handles), "moe_profile_next_grouped_mlp")


def moe_debug_next_grouped_mlp_silent_token_tile(token_tile: int) -> None:
    """Testing hook: the next fused bf16 grouped MLP call lets token tile
    `token_tile`'s FC1 tiles withhold their completion publication (-1 cancels)."""
    _check(_lib.moe_debug_next_grouped_mlp_silent_token_tile(token_tile),
           "moe_debug_next_grouped_mlp_silent_token_tile")


def moe_debug_preprocess_silent_tile(routing: Routing, shape: Shape, layout: Layout, handle: Handle,
                                     workspace: torch.Tensor, silent_tile: int, stream=None) -> None:
    """Testing hook: preprocess with one tile withholding its lookback publication (see moe.h)."""
    _check(_lib.moe_debug_preprocess_silent_tile(ctypes.byref(routing.c()), ctypes.byref(shape.c()),
                                                 ctypes.byref(layout.c()), ctypes.byref(handle.c()), _ptr(workspace),
                                                 workspace.numel() * workspace.element_size(), silent_tile,
                                                 _stream(stream)), "moe_debug_preprocess_silent_tile")


def moe_quantize_fp8_blocks(w: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    G, N, Kd = w.shape
    _check(_lib.moe_quantize_fp8_blocks(_ptr(w), G, N, Kd, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_quantize_fp8_blocks")


def moe_quantize_nvfp4_rows(x: torch.Tensor, global_scale: torch.Tensor, packed: torch.Tensor,
                            scales: torch.Tensor, stream=None) -> None:
    Kd = x.shape[-1]
    R = x.numel() // Kd
    _check(_lib.moe_quantize_nvfp4_rows(_ptr(x), R, Kd, _ptr(global_scale), _ptr(packed), _ptr(scales),
                                        _stream(stream)), "moe_quantize_nvfp4_rows")


class Ring:
    """Host-side ring of caller-owned output slots (moe_ring_* in moe.h)."""

    def __init__(self, n_slots: int, use_events: bool = True):
        self._r = ctypes.c_void_p()
        _check(_lib.moe_ring_create(n_slots, 1 if use_events else 0, ctypes.byref(self._r)), "moe_ring_create")

    def acquire(self, stream=None) -> int:
        slot = ctypes.c_int32()
        s = _stream(stream) if torch.cuda.is_available() else None
        _check(_lib.moe_ring_acquire(self._r, s, ctypes.byref(slot)), "moe_ring_acquire")
        return slot.value

    def release(self, slot: int, stream=None) -> None:
        s = _stream(stream) if torch.cuda.is_available() else None
        _check(_lib.moe_ring_release(self._r, slot, s), "moe_ring_release")

    def close(self) -> None:
        if self._r:
            _check(_lib.moe_ring_destroy(self._r), "moe_ring_destroy")
            self._r = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def library():
    """The loaded ctypes library (for symbol checks)."""
    return _lib


def exported_symbols():
    return list(_SIGNATURES)
