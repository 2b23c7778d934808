"""Python binding of the GB300 W4A16 MoE expert library (ctypes over the C ABI).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels (``csrc/``, built for sm_103a into ``_build/libw4a16_moe.so``).  There is
no CPU fallback: if the library is missing or fails to load, every call raises.
PyTorch provides device memory and streams; calls are enqueued on the current
torch CUDA stream.

The C ABI is declared, with argument meaning, layouts and error behaviour, in
``include/w4a16_moe.h``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "load", "library_path", "align_capacity", "moe_align", "PackedWeights", "pack_weights",
    "Routing", "pack_weights_nvfp4", "moe_gemm", "gather_rows", "contiguous_gemm", "masked_gemm", "topk_sum", "moe_layer", "layer_workspace_size", "plan_block_m",
    "plan_gemm", "debug_dequant", "gemm_workspace_size", "EPILOGUE_NONE", "EPILOGUE_SILU_MUL",
    "A_ROWS_SORTED", "C_ROWS_SORTED", "C_FP32", "PACK_GATE_UP_PAIRED", "LibraryError",
]

EPILOGUE_NONE = 0
EPILOGUE_SILU_MUL = 1
A_ROWS_SORTED = 0x1
C_ROWS_SORTED = 0x2
C_FP32 = 0x4
PACK_GATE_UP_PAIRED = 0x1
PACK_NVFP4 = 0x2
LAYER_FUSED_TOPK = 0x1
LAYER_FUSED = 0x2
LAYER_DEBUG_WAIT_TIMEOUT = 0x80000000  # test hook: the fused layer's cross-CTA waits run out
PACK_MAGIC = 0x3631413457454F4D
PACK_VERSION = 2

DEVERR_BAD_EXPERT_ID = 0x1
DEVERR_CAPACITY = 0x2
DEVERR_TIMEOUT = 0x4
DEVERR_BAD_HEADER = 0x8

_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "bad packed weight",
           4: "workspace too small", 5: "CUDA error"}


class LibraryError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn}: {_STATUS.get(status, status)} ({detail})")
        self.status = status


class PackedDesc(ctypes.Structure):
    _fields_ = [("magic", ctypes.c_uint64), ("version", ctypes.c_uint32), ("flags", ctypes.c_uint32),
                ("E", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
                ("group", ctypes.c_int32), ("bytes", ctypes.c_uint64), ("data", ctypes.c_void_p)]


class RoutingDesc(ctypes.Structure):
    _fields_ = [("sorted_ids", ctypes.c_void_p), ("expert_ids", ctypes.c_void_p),
                ("num_tokens_padded", ctypes.c_void_p), ("capacity", ctypes.c_int64),
                ("block_m", ctypes.c_int32), ("total_slots", ctypes.c_int32)]


class ScheduleDesc(ctypes.Structure):
    _fields_ = [("split_k", ctypes.c_int32), ("num_ctas", ctypes.c_int32), ("cta_pairs", ctypes.c_int32),
                ("tile_group", ctypes.c_int32)]


class PlanDesc(ctypes.Structure):
    _fields_ = [("block_m", ctypes.c_int32), ("split_k", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("est_units", ctypes.c_int32), ("cta_pairs", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()

_VP, _I32, _I64, _U32, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
_P = ctypes.POINTER
_SIGNATURES = {
    "w4a16_status_string": (ctypes.c_char_p, [_I32]),
    "w4a16_last_error_detail": (ctypes.c_char_p, []),
    "w4a16_align_capacity": (_I64, [_I32, _I32, _I32, _I32]),
    "w4a16_moe_align": (_I32, [_VP, _I32, _I32, _I32, _I32, _VP, _VP, _VP, _I64, _I32, _VP, _VP]),
    "w4a16_packed_bytes": (_SZ, [_I32, _I32, _I32, _I32, _U32]),
    "w4a16_pack_weights": (_I32, [_VP, _VP, _I32, _I32, _I32, _I32, _U32, _VP, _SZ, _P(PackedDesc), _VP]),
    "w4a16_pack_weights_nvfp4": (_I32, [_VP, _VP, _I32, _I32, _I32, _U32, _VP, _SZ, _P(PackedDesc), _VP]),
    "w4a16_gemm_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "w4a16_workspace_clear": (_I32, [_VP, _SZ, _VP]),
    "w4a16_moe_gemm": (_I32, [_VP, _I64, _I32, _P(PackedDesc), _P(RoutingDesc), _I32, _U32, _VP, _I64,
                              _VP, _SZ, _I32, _P(ScheduleDesc), _VP, _VP]),
    "w4a16_topk_sum": (_I32, [_VP, _VP, _VP, _I32, _I32, _I32, _VP, _VP]),
    "w4a16_gather_rows": (_I32, [_VP, _I64, _I32, _I32, _P(RoutingDesc), _VP, _I64, _VP]),
    "w4a16_moe_gemm_static_scratch": (_I32, [_VP, _I64, _I32, _P(PackedDesc), _P(RoutingDesc), _I32,
                                             _U32, _VP, _I64, _I32, _P(ScheduleDesc), _VP, _VP]),
    "w4a16_contiguous_workspace_size": (_SZ, [_I64]),
    "w4a16_contiguous_gemm": (_I32, [_VP, _I64, _I64, _VP, _P(PackedDesc), _I32, _VP, _I64, _VP, _SZ,
                                     _VP, _VP]),
    "w4a16_masked_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "w4a16_masked_gemm": (_I32, [_VP, _I64, _I32, _I32, _VP, _I32, _P(PackedDesc), _I32, _VP, _I64,
                                 _VP, _SZ, _VP, _VP]),
    "w4a16_plan_block_m": (_I32, [_I32, _I32, _I32, _I32]),
    "w4a16_layer_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32, _I32]),
    "w4a16_moe_layer": (_I32, [_VP, _P(PackedDesc), _P(PackedDesc), _VP, _VP, _I32, _I32, _I32, _I32,
                               _VP, _VP, _SZ, _VP, _VP]),
    "w4a16_moe_layer_ex": (_I32, [_VP, _P(PackedDesc), _P(PackedDesc), _VP, _VP, _I32, _I32, _I32, _I32,
                                  _U32, _VP, _VP, _SZ, _VP, _VP]),
    "w4a16_plan_gemm": (_I32, [_I32, _I32, _I32, _I32, _I32, _I32, _I32, _P(PlanDesc)]),
    "w4a16_debug_dequant": (_I32, [_P(PackedDesc), _I32, _VP, _VP]),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load the CUDA library (building it first if asked and needed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                if not build_if_missing:
                    raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
                _build.build()
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        detail = load().w4a16_last_error_detail().decode(errors="replace")
        raise LibraryError(fn, status, detail)


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _cuda(t: torch.Tensor, dtype: torch.dtype, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ---- routing -------------------------------------------------------------------------------

def align_capacity(T: int, top_k: int, E: int, block_m: int) -> int:
    return int(load().w4a16_align_capacity(T, top_k, E, block_m))


@dataclass
class Routing:
    sorted_ids: torch.Tensor
    expert_ids: torch.Tensor
    num_tokens_padded: torch.Tensor
    block_m: int
    total_slots: int

    @property
    def capacity(self) -> int:
        return self.sorted_ids.numel()

    def desc(self) -> RoutingDesc:
        return RoutingDesc(self.sorted_ids.data_ptr(), self.expert_ids.data_ptr(),
                           self.num_tokens_padded.data_ptr(), self.capacity, self.block_m,
                           self.total_slots)


def moe_align(topk_ids: torch.Tensor, E: int, block_m: int, capacity: Optional[int] = None,
              validate: bool = False, dev_err: Optional[torch.Tensor] = None) -> Routing:
    _cuda(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    cap = align_capacity(T, k, E, block_m) if capacity is None else capacity
    dev = topk_ids.device
    sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
    expert_ids = torch.empty(cap // block_m, dtype=torch.int32, device=dev)
    ntp = torch.empty(1, dtype=torch.int32, device=dev)
    _check("w4a16_moe_align", load().w4a16_moe_align(
        _ptr(topk_ids), T, k, E, block_m, _ptr(sorted_ids), _ptr(expert_ids), _ptr(ntp), cap,
        1 if validate else 0, _ptr(dev_err), _stream()))
    return Routing(sorted_ids, expert_ids, ntp, block_m, T * k)


# ---- weights -------------------------------------------------------------------------------

class PackedWeights:
    """A packed weight blob in device memory plus its host descriptor."""

    def __init__(self, blob: torch.Tensor, desc: PackedDesc):
        self.blob = blob
        self.desc = desc

    @property
    def E(self):
        return self.desc.E

    @property
    def N(self):
        return self.desc.N

    @property
    def K(self):
        return self.desc.K

    @property
    def paired(self) -> bool:
        return bool(self.desc.flags & PACK_GATE_UP_PAIRED)

    @property
    def nbytes(self) -> int:
        return int(self.desc.bytes)

    def clone(self) -> "PackedWeights":
        """A second device copy of the same packed weights (a device-to-device copy of the blob)."""
        blob = self.blob.clone()
        desc = PackedDesc()
        ctypes.memmove(ctypes.byref(desc), ctypes.byref(self.desc), ctypes.sizeof(PackedDesc))
        desc.data = blob.data_ptr()
        return PackedWeights(blob, desc)


def packed_bytes(E: int, N: int, K: int, paired: bool = False) -> int:
    return int(load().w4a16_packed_bytes(E, N, K, 32, PACK_GATE_UP_PAIRED if paired else 0))


def pack_weights(qweight: torch.Tensor, scales: torch.Tensor, paired: bool = False) -> PackedWeights:
    """Repack canonical int32 [E, N, K/8] codes and BF16 [E, N, K/32] scales for the GEMM."""
    _cuda(qweight, torch.int32, "qweight")
    _cuda(scales, torch.bfloat16, "scales")
    E, N, K8 = qweight.shape
    K = K8 * 8
    if tuple(scales.shape) != (E, N, K // 32):
        raise ValueError(f"scales must be [E, N, K/32] = {(E, N, K // 32)}, got {tuple(scales.shape)}")
    flags = PACK_GATE_UP_PAIRED if paired else 0
    nbytes = int(load().w4a16_packed_bytes(E, N, K, 32, flags))
    if nbytes == 0:
        raise LibraryError("w4a16_packed_bytes", 2, f"unsupported shape E={E} N={N} K={K}")
    blob = torch.empty(nbytes, dtype=torch.uint8, device=qweight.device)
    desc = PackedDesc()
    _check("w4a16_pack_weights", load().w4a16_pack_weights(
        _ptr(qweight), _ptr(scales), E, N, K, 32, flags, _ptr(blob), nbytes, ctypes.byref(desc),
        _stream()))
    return PackedWeights(blob, desc)


def pack_weights_nvfp4(codes: torch.Tensor, scales: torch.Tensor, paired: bool = False) -> PackedWeights:
    """Repack NVFP4 weights: uint8 [E, N, K/2] E2M1 codes (element 2j in the low nibble) and
    uint8 [E, N, K/16] E4M3 scales, for the same GEMM and layer calls as INT4 weights."""
    _cuda(codes, torch.uint8, "codes")
    _cuda(scales, torch.uint8, "scales")
    E, N, K2 = codes.shape
    K = K2 * 2
    if tuple(scales.shape) != (E, N, K // 16):
        raise ValueError(f"scales must be [E, N, K/16] = {(E, N, K // 16)}, got {tuple(scales.shape)}")
    flags = PACK_GATE_UP_PAIRED if paired else 0
    nbytes = int(load().w4a16_packed_bytes(E, N, K, 16, flags | PACK_NVFP4))
    if nbytes == 0:
        raise LibraryError("w4a16_packed_bytes", 2, f"unsupported shape E={E} N={N} K={K}")
    blob = torch.empty(nbytes, dtype=torch.uint8, device=codes.device)
    desc = PackedDesc()
    _check("w4a16_pack_weights_nvfp4", load().w4a16_pack_weights_nvfp4(
        _ptr(codes), _ptr(scales), E, N, K, flags, _ptr(blob), nbytes, ctypes.byref(desc), _stream()))
    return PackedWeights(blob, desc)


def debug_dequant(W: PackedWeights, expert: int) -> torch.Tensor:
    out = torch.empty((W.N, W.K), dtype=torch.bfloat16, device=W.blob.device)
    _check("w4a16_debug_dequant", load().w4a16_debug_dequant(
        ctypes.byref(W.desc), expert, _ptr(out), _stream()))
    return out


# ---- GEMM ----------------------------------------------------------------------------------

def gemm_workspace_size(total_slots: int, E: int, N: int, K: int, block_m: int) -> int:
    return int(load().w4a16_gemm_workspace_size(total_slots, E, N, K, block_m))


def gemm_workspace(total_slots: int, E: int, N: int, K: int, block_m: int, device) -> torch.Tensor:
    """A zeroed workspace (its counters must start at zero; calls leave them zero)."""
    return torch.zeros(gemm_workspace_size(total_slots, E, N, K, block_m), dtype=torch.uint8,
                       device=device)


def moe_gemm(A: torch.Tensor, a_row_div: int, W: PackedWeights, routing: Routing,
             epilogue: int = EPILOGUE_NONE, row_flags: int = 0, out: Optional[torch.Tensor] = None,
             out_rows: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
             expected_rows_per_expert: int = 0, split_k: int = 0, num_ctas: int = 0,
             dev_err: Optional[torch.Tensor] = None, cta_pairs: int = 0,
             tile_group: int = 0) -> torch.Tensor:
    """The indexed W4A16 GEMM (``w4a16_moe_gemm``).  ``split_k``, ``num_ctas``, ``cta_pairs``
    and ``tile_group`` override the planner for measurements (0 = planner; cta_pairs 1 = one
    CTA per 128-row tile, 2 = one M = 256 MMA over two CTAs; tile_group 1 = one tile per work
    unit, 2 or 4 = that many tiles of a block per unit)."""
    _cuda(A, torch.bfloat16, "A")
    width = W.N // 2 if epilogue == EPILOGUE_SILU_MUL else W.N
    if out is None:
        rows = out_rows if out_rows is not None else (
            routing.capacity if row_flags & C_ROWS_SORTED else routing.total_slots)
        out = torch.zeros((rows, width), dtype=torch.float32 if row_flags & C_FP32 else torch.bfloat16,
                          device=A.device)
    _cuda(out, torch.float32 if row_flags & C_FP32 else torch.bfloat16, "out")
    if workspace is None:
        workspace = gemm_workspace(routing.total_slots, W.E, W.N, W.K, routing.block_m, A.device)
    sched = ScheduleDesc(split_k, num_ctas, cta_pairs, tile_group)
    rd = routing.desc()
    _check("w4a16_moe_gemm", load().w4a16_moe_gemm(
        _ptr(A), A.stride(0), a_row_div, ctypes.byref(W.desc), ctypes.byref(rd), epilogue, row_flags,
        _ptr(out), out.stride(0), _ptr(workspace), workspace.numel(), expected_rows_per_expert,
        ctypes.byref(sched), _ptr(dev_err), _stream()))
    return out


def gather_rows(x: torch.Tensor, a_row_div: int, routing: Routing,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Activation rows in aligned order: out[p] = x[sorted_ids[p] // a_row_div] (routed p)."""
    _cuda(x, torch.bfloat16, "x")
    K = x.shape[1]
    if out is None:
        out = torch.zeros((routing.capacity, K), dtype=torch.bfloat16, device=x.device)
    _cuda(out, torch.bfloat16, "out")
    rd = routing.desc()
    _check("w4a16_gather_rows", load().w4a16_gather_rows(
        _ptr(x), x.stride(0), K, a_row_div, ctypes.byref(rd), _ptr(out), out.stride(0), _stream()))
    return out


def moe_gemm_static_scratch(A: torch.Tensor, a_row_div: int, W: PackedWeights, routing: Routing,
                            epilogue: int = EPILOGUE_NONE, row_flags: int = 0,
                            out: Optional[torch.Tensor] = None, expected_rows_per_expert: int = 0,
                            split_k: int = 0, num_ctas: int = 0,
                            dev_err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The indexed GEMM for callers that cannot allocate: its K-split scratch is a device array
    owned by the library (shared by all calls, so calls must not overlap on the GPU).  The
    output tensor is the caller's; pass ``out`` to make the call allocate nothing at all."""
    _cuda(A, torch.bfloat16, "A")
    width = W.N // 2 if epilogue == EPILOGUE_SILU_MUL else W.N
    if out is None:
        rows = routing.capacity if row_flags & C_ROWS_SORTED else routing.total_slots
        out = torch.zeros((rows, width), dtype=torch.float32 if row_flags & C_FP32 else torch.bfloat16,
                          device=A.device)
    _cuda(out, torch.float32 if row_flags & C_FP32 else torch.bfloat16, "out")
    sched = ScheduleDesc(split_k, num_ctas, 0)
    rd = routing.desc()
    _check("w4a16_moe_gemm_static_scratch", load().w4a16_moe_gemm_static_scratch(
        _ptr(A), A.stride(0), a_row_div, ctypes.byref(W.desc), ctypes.byref(rd), epilogue, row_flags,
        _ptr(out), out.stride(0), expected_rows_per_expert, ctypes.byref(sched), _ptr(dev_err),
        _stream()))
    return out


def contiguous_gemm(A: torch.Tensor, W: PackedWeights, m_indices: torch.Tensor,
                    epilogue: int = EPILOGUE_NONE, out: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None,
                    dev_err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Contiguous grouped layout: A [m, K] rows concatenated by expert (groups padded to 128
    rows), m_indices int32 [m] (-1 for padding) -> C [m, N or N/2]."""
    _cuda(A, torch.bfloat16, "A")
    _cuda(m_indices, torch.int32, "m_indices")
    m = A.shape[0]
    width = W.N // 2 if epilogue == EPILOGUE_SILU_MUL else W.N
    if out is None:
        out = torch.empty((m, width), dtype=torch.bfloat16, device=A.device)
    _cuda(out, torch.bfloat16, "out")
    need = int(load().w4a16_contiguous_workspace_size(m))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=A.device)
    _check("w4a16_contiguous_gemm", load().w4a16_contiguous_gemm(
        _ptr(A), A.stride(0), m, _ptr(m_indices), ctypes.byref(W.desc), epilogue, _ptr(out),
        out.stride(0), _ptr(workspace), workspace.numel(), _ptr(dev_err), _stream()))
    return out


def masked_gemm(A: torch.Tensor, W: PackedWeights, masked_m: torch.Tensor, expected_m: int,
                epilogue: int = EPILOGUE_NONE, out: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None,
                dev_err: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Masked grouped layout: A [G, max_m, K] or [G * max_m, K], masked_m int32 [G] valid rows
    -> flat C [G * max_m, N or N/2] (rows past each expert's count are left as they are)."""
    _cuda(A, torch.bfloat16, "A")
    _cuda(masked_m, torch.int32, "masked_m")
    G = masked_m.numel()
    A2 = A.reshape(-1, A.shape[-1])
    max_m = A2.shape[0] // max(G, 1)
    width = W.N // 2 if epilogue == EPILOGUE_SILU_MUL else W.N
    if out is None:
        out = torch.zeros((G * max_m, width), dtype=torch.bfloat16, device=A.device)
    _cuda(out, torch.bfloat16, "out")
    need = int(load().w4a16_masked_workspace_size(G, max_m, expected_m))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=A.device)
    _check("w4a16_masked_gemm", load().w4a16_masked_gemm(
        _ptr(A2), A2.stride(0), G, max_m, _ptr(masked_m), expected_m, ctypes.byref(W.desc),
        epilogue, _ptr(out), out.stride(0), _ptr(workspace), workspace.numel(), _ptr(dev_err),
        _stream()))
    return out


def topk_sum(Y: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
             out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _cuda(Y, torch.float32, "Y")
    _cuda(topk_ids, torch.int32, "topk_ids")
    _cuda(topk_weights, torch.float32, "topk_weights")
    T, k = topk_ids.shape
    H = Y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=Y.device)
    _check("w4a16_topk_sum", load().w4a16_topk_sum(
        _ptr(Y), _ptr(topk_ids), _ptr(topk_weights), T, k, H, _ptr(out), _stream()))
    return out


# ---- layer ---------------------------------------------------------------------------------

def plan_block_m(T: int, top_k: int, E: int, E_global: int = 0) -> int:
    return int(load().w4a16_plan_block_m(T, top_k, E, E_global))


def layer_workspace_size(T: int, top_k: int, E: int, H: int, I: int, E_global: int = 0,
                         block_m: int = 0) -> int:
    return int(load().w4a16_layer_workspace_size(T, top_k, E, E_global, H, I, block_m))


def moe_layer(x: torch.Tensor, w13: PackedWeights, w2: PackedWeights, topk_ids: torch.Tensor,
              topk_weights: torch.Tensor, E_global: int = 0, block_m: int = 0,
              out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
              dev_err: Optional[torch.Tensor] = None, fused_topk: bool = False,
              fused: bool = False, debug_wait_timeout: bool = False) -> torch.Tensor:
    """The whole layer; ``fused_topk`` merges the top-k outputs inside the down GEMM
    (atomic FP32 sums: within the tolerance, not bitwise reproducible); ``fused`` also runs
    gate_up and down as one persistent kernel (and implies ``fused_topk``).
    ``debug_wait_timeout`` (with ``fused``; tests only) makes every cross-CTA wait of the down
    units run out after a short limit (``W4A16_LAYER_DEBUG_WAIT_TIMEOUT``)."""
    _cuda(x, torch.bfloat16, "x")
    _cuda(topk_ids, torch.int32, "topk_ids")
    _cuda(topk_weights, torch.float32, "topk_weights")
    T, H = x.shape
    k = topk_ids.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    need = layer_workspace_size(T, k, w13.E, H, w13.N // 2, E_global, block_m)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check("w4a16_moe_layer_ex", load().w4a16_moe_layer_ex(
        _ptr(x), ctypes.byref(w13.desc), ctypes.byref(w2.desc), _ptr(topk_ids), _ptr(topk_weights),
        T, k, E_global, block_m, (LAYER_FUSED if fused else 0) | (LAYER_FUSED_TOPK if fused_topk else 0)
        | (LAYER_DEBUG_WAIT_TIMEOUT if debug_wait_timeout else 0),
        _ptr(out), _ptr(workspace),
        workspace.numel(), _ptr(dev_err), _stream()))
    return out


# ---- host planner --------------------------------------------------------------------------

def plan_gemm(total_slots: int, E: int, N: int, K: int, block_m: int, num_sms: int,
              expected_rows_per_expert: int = 0) -> dict:
    p = PlanDesc()
    _check("w4a16_plan_gemm", load().w4a16_plan_gemm(
        total_slots, E, N, K, block_m, expected_rows_per_expert, num_sms, ctypes.byref(p)))
    return {f: getattr(p, f) for f, _ in PlanDesc._fields_}
