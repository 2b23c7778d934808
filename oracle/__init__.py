"""CPU oracle for the W4A16 MoE expert path (test infrastructure only).

The oracle is the plain, single-threaded C++ reference in
``w4a16_oracle.cpp``; this module builds it with the host compiler and wraps
it with ctypes.  Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this package.  It shares no code with the CUDA
library: inputs come from ``w4a16_moe_expert_gb300.workloads`` (which holds
no arithmetic of the method) and everything is computed here on the host.

Every function cites, in the C++ source, the passage it follows.  Each one is
pinned in ``tests/test_oracle_pins.py`` against something other than itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libw4a16_oracle.so")
_lib = None
_lock = threading.Lock()

CFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (skipped when up to date)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cxx = os.environ.get("CXX", "g++")
    subprocess.check_call([cxx, *CFLAGS, "-o", tmp, _SRC])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
            sig = {
                "w4a16_oracle_float_to_bf16": (None, [vp, i64, vp]),
                "w4a16_oracle_double_to_bf16": (None, [vp, i64, vp]),
                "w4a16_oracle_align_capacity": (i64, [i32, i32, i32, i32]),
                "w4a16_oracle_align": (i32, [vp, i32, i32, i32, i32, i64, vp, vp, vp]),
                "w4a16_oracle_dequant": (None, [vp, vp, i64, i32, i32, vp]),
                "w4a16_oracle_gemm_rows": (None, [vp, i32, i32, vp, vp, i32, i32, vp, vp, i64, vp, vp]),
                "w4a16_oracle_moe_gemm": (i32, [vp, i32, i32, vp, vp, i32, i32, vp, vp, i32, i32,
                                                i32, i32, i32, vp, vp]),
                "w4a16_oracle_contiguous_gemm": (i32, [vp, i64, i32, vp, vp, i32, i32, i32, vp, vp,
                                                       vp]),
                "w4a16_oracle_masked_gemm": (i32, [vp, i32, i32, i32, vp, vp, i32, i32, vp, vp, vp]),
                "w4a16_oracle_nvfp4_dequant": (None, [vp, vp, i64, i32, vp]),
                "w4a16_oracle_nvfp4_moe_gemm": (i32, [vp, i32, i32, vp, vp, i32, vp, vp, i32, i32,
                                                      i32, i32, i32, vp, vp]),
                "w4a16_oracle_silu_mul": (None, [vp, i64, i32, vp]),
                "w4a16_oracle_topk_sum": (None, [vp, vp, vp, i32, i32, i32, vp]),
                "w4a16_oracle_moe_layer": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                 i32, i32, i32, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


# ---- array helpers -------------------------------------------------------------------

def _np(t, dtype):
    """Contiguous numpy view of a CPU tensor / array with the given storage dtype."""
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        t = t.numpy()
    a = np.ascontiguousarray(t)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_tensor(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)


def float_to_bf16_bits(x) -> np.ndarray:
    a = _np(np.asarray(x, dtype=np.float32), np.float32)
    out = np.empty(a.shape, np.uint16)
    lib().w4a16_oracle_float_to_bf16(_ptr(a), a.size, _ptr(out))
    return out


def double_to_bf16_bits(x) -> np.ndarray:
    a = _np(np.asarray(x, dtype=np.float64), np.float64)
    out = np.empty(a.shape, np.uint16)
    lib().w4a16_oracle_double_to_bf16(_ptr(a), a.size, _ptr(out))
    return out


# ---- the method's steps ---------------------------------------------------------------

def align_capacity(T: int, top_k: int, E: int, block_m: int) -> int:
    return int(lib().w4a16_oracle_align_capacity(T, top_k, E, block_m))


def moe_align(topk_ids, E: int, block_m: int, capacity: int | None = None):
    """Returns (sorted_ids int32 [cap], expert_ids int32 [cap/block_m], ntp int)."""
    ids = _np(topk_ids, np.int32)
    T, k = ids.shape
    cap = align_capacity(T, k, E, block_m) if capacity is None else capacity
    sorted_ids = np.empty(cap, np.int32)
    expert_ids = np.empty(cap // block_m, np.int32)
    ntp = np.zeros(1, np.int32)
    rc = lib().w4a16_oracle_align(_ptr(ids), T, k, E, block_m, cap, _ptr(sorted_ids),
                                  _ptr(expert_ids), _ptr(ntp))
    if rc:
        raise ValueError(f"oracle align failed with code {rc}")
    return sorted_ids, expert_ids, int(ntp[0])


def dequant(qweight, scales, group: int = 32) -> torch.Tensor:
    """qweight int32 [..., N, K/8], scales bf16 [..., N, K/group] -> bf16 [..., N, K]."""
    q = _np(qweight, np.int32)
    s = _np(scales, np.uint16)
    K = q.shape[-1] * 8
    rows = q.size // (K // 8)
    out = np.empty(q.shape[:-1] + (K,), np.uint16)
    lib().w4a16_oracle_dequant(_ptr(q), _ptr(s), rows, K, group, _ptr(out))
    return _bf16_tensor(out)


def gemm_rows(A, a_row_div: int, qweight, scales, slots, experts, group: int = 32,
              out_f32: bool = False, threads: int = 1) -> torch.Tensor:
    """out[r] = A[slots[r] // a_row_div] @ dequant(W[experts[r]]).T: bf16 [len(slots), N], or the
    unrounded FP32 sums with ``out_f32``.

    With ``threads > 1`` the same single-threaded function runs over disjoint row ranges on
    that many host threads; every output element has the same arithmetic, so the result is
    identical.
    """
    a = _np(A, np.uint16)
    q = _np(qweight, np.int32)
    s = _np(scales, np.uint16)
    sl = _np(np.asarray(slots), np.int32)
    ex = _np(np.asarray(experts), np.int32)
    K = a.shape[-1]
    N = q.shape[-2]
    out = np.empty((sl.size, N), np.float32 if out_f32 else np.uint16)
    L = lib()

    def run(lo, hi):
        if hi <= lo:
            return
        L.w4a16_oracle_gemm_rows(_ptr(a), a_row_div, K, _ptr(q), _ptr(s), N, group,
                                 _ptr(sl[lo:hi]), _ptr(ex[lo:hi]), hi - lo,
                                 None if out_f32 else _ptr(out[lo:hi]),
                                 _ptr(out[lo:hi]) if out_f32 else None)

    threads = max(1, min(threads, sl.size))
    if threads == 1:
        run(0, sl.size)
    else:
        cuts = np.linspace(0, sl.size, threads + 1).astype(np.int64)
        with ThreadPoolExecutor(threads) as pool:
            list(pool.map(lambda lh: run(int(lh[0]), int(lh[1])), zip(cuts[:-1], cuts[1:])))
    return torch.from_numpy(out) if out_f32 else _bf16_tensor(out)


def moe_gemm(A, a_row_div: int, qweight, scales, sorted_ids, expert_ids, ntp: int, block_m: int,
             total_slots: int, group: int = 32, threads: int = 1, out_f32: bool = False) -> torch.Tensor:
    """Indexed grouped GEMM; returns C [total_slots, N] (unrouted rows are 0), BF16, or
    the unrounded FP32 sums with ``out_f32``.

    With ``threads > 1`` the same single-threaded function runs over disjoint
    expert ranges on that many host threads; every output element has the
    same arithmetic, so the result is identical.
    """
    a = _np(A, np.uint16)
    q = _np(qweight, np.int32)
    s = _np(scales, np.uint16)
    si = _np(sorted_ids, np.int32)
    ei = _np(expert_ids, np.int32)
    K = a.shape[-1]
    E, N = q.shape[0], q.shape[1]
    C = np.zeros((total_slots, N), np.float32 if out_f32 else np.uint16)
    L = lib()

    def run(lo, hi):
        rc = L.w4a16_oracle_moe_gemm(_ptr(a), a_row_div, K, _ptr(q), _ptr(s), N, group, _ptr(si),
                                     _ptr(ei), ntp, block_m, total_slots, lo, hi,
                                     None if out_f32 else _ptr(C), _ptr(C) if out_f32 else None)
        if rc:
            raise ValueError(f"oracle moe_gemm failed with code {rc}")

    if threads <= 1:
        run(0, E)
    else:
        # balance by routed rows per expert
        valid = ei[: ntp // block_m]
        rows_per_e = np.bincount(valid[valid >= 0], minlength=E).astype(np.float64) + 1e-3
        cuts = np.searchsorted(np.cumsum(rows_per_e), np.linspace(0, rows_per_e.sum(), threads + 1)[1:-1])
        bounds = [0, *[int(c) + 1 for c in cuts], E]
        bounds = sorted(set(min(max(b, 0), E) for b in bounds))
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            list(ex.map(lambda lh: run(*lh), zip(bounds[:-1], bounds[1:])))
    return torch.from_numpy(C) if out_f32 else _bf16_tensor(C)


def nvfp4_dequant(codes, scales) -> torch.Tensor:
    """NVFP4 codes uint8 [..., N, K/2] (element 2j in the low nibble), E4M3 scales uint8
    [..., N, K/16] -> bf16 [..., N, K] (each weight the exact product)."""
    c = _np(codes, np.uint8)
    s = _np(scales, np.uint8)
    K = c.shape[-1] * 2
    rows = c.size // (K // 2)
    out = np.empty(c.shape[:-1] + (K,), np.uint16)
    lib().w4a16_oracle_nvfp4_dequant(_ptr(c), _ptr(s), rows, K, _ptr(out))
    return _bf16_tensor(out)


def nvfp4_moe_gemm(A, a_row_div: int, codes, scales, sorted_ids, expert_ids, ntp: int,
                   block_m: int, total_slots: int, threads: int = 1,
                   out_f32: bool = False) -> torch.Tensor:
    """The indexed grouped GEMM with NVFP4 weights (codes [E, N, K/2], scales [E, N, K/16])."""
    a = _np(A, np.uint16)
    c = _np(codes, np.uint8)
    s = _np(scales, np.uint8)
    si = _np(sorted_ids, np.int32)
    ei = _np(expert_ids, np.int32)
    K = a.shape[-1]
    E, N = c.shape[0], c.shape[1]
    C = np.zeros((total_slots, N), np.float32 if out_f32 else np.uint16)
    L = lib()

    def run(lo, hi):
        rc = L.w4a16_oracle_nvfp4_moe_gemm(_ptr(a), a_row_div, K, _ptr(c), _ptr(s), N, _ptr(si),
                                           _ptr(ei), ntp, block_m, total_slots, lo, hi,
                                           None if out_f32 else _ptr(C), _ptr(C) if out_f32 else None)
        if rc:
            raise ValueError(f"oracle nvfp4_moe_gemm failed with code {rc}")

    if threads <= 1:
        run(0, E)
    else:
        bounds = np.linspace(0, E, threads + 1).astype(int)
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda lh: run(*lh), zip(bounds[:-1], bounds[1:])))
    return torch.from_numpy(C) if out_f32 else _bf16_tensor(C)


def contiguous_gemm(A, qweight, scales, m_indices, group: int = 32,
                    out_f32: bool = False) -> torch.Tensor:
    """Contiguous grouped layout: C[r] = A[r] @ dequant(W[m_indices[r]]).T, padding rows 0;
    BF16, or the unrounded FP32 sums with ``out_f32``."""
    a = _np(A, np.uint16)
    q = _np(qweight, np.int32)
    s = _np(scales, np.uint16)
    mi = _np(m_indices, np.int32)
    m, K = a.shape
    E, N = q.shape[0], q.shape[1]
    C = np.zeros((m, N), np.float32 if out_f32 else np.uint16)
    rc = lib().w4a16_oracle_contiguous_gemm(_ptr(a), m, K, _ptr(q), _ptr(s), E, N, group,
                                            _ptr(mi), None if out_f32 else _ptr(C),
                                            _ptr(C) if out_f32 else None)
    if rc:
        raise ValueError(f"oracle contiguous_gemm failed with code {rc}")
    return torch.from_numpy(C) if out_f32 else _bf16_tensor(C)


def masked_gemm(A, qweight, scales, masked_m, max_m: int, group: int = 32,
                out_f32: bool = False) -> torch.Tensor:
    """Masked grouped layout over A [G * max_m, K]: rows g*max_m + r, r < masked_m[g], of the
    flat [G * max_m, N] output; the other rows are returned as 0 (undefined by the contract).
    BF16, or the unrounded FP32 sums with ``out_f32``."""
    a = _np(A, np.uint16).reshape(-1, _np(A, np.uint16).shape[-1])
    q = _np(qweight, np.int32)
    s = _np(scales, np.uint16)
    mm = _np(masked_m, np.int32)
    G = q.shape[0]
    N = q.shape[1]
    K = a.shape[-1]
    C = np.zeros((G * max_m, N), np.float32 if out_f32 else np.uint16)
    rc = lib().w4a16_oracle_masked_gemm(_ptr(a), G, max_m, K, _ptr(q), _ptr(s), N, group,
                                        _ptr(mm), None if out_f32 else _ptr(C),
                                        _ptr(C) if out_f32 else None)
    if rc:
        raise ValueError(f"oracle masked_gemm failed with code {rc}")
    return torch.from_numpy(C) if out_f32 else _bf16_tensor(C)


def silu_mul(C) -> torch.Tensor:
    """C [rows, 2I] gate_up sums -> h bf16 [rows, I], h = bf16(silu(gate) * up).  The sums are
    meant unrounded (FP32, e.g. ``gemm_rows(..., out_f32=True)``); BF16 input is widened
    exactly."""
    if isinstance(C, torch.Tensor):
        C = C.detach().cpu().float()
    c = _np(C, np.float32)
    rows, two_i = c.shape
    h = np.empty((rows, two_i // 2), np.uint16)
    lib().w4a16_oracle_silu_mul(_ptr(c), rows, two_i // 2, _ptr(h))
    return _bf16_tensor(h)


def topk_sum(Y, topk_ids, topk_weights) -> torch.Tensor:
    """Y fp32 [T*k, H] (per-slot down outputs) -> bf16 [T, H]."""
    if isinstance(Y, torch.Tensor) and Y.dtype == torch.bfloat16:
        Y = Y.float()
    y = _np(Y, np.float32)
    ids = _np(topk_ids, np.int32)
    w = _np(topk_weights, np.float32)
    T, k = ids.shape
    H = y.shape[-1]
    out = np.empty((T, H), np.uint16)
    lib().w4a16_oracle_topk_sum(_ptr(y), _ptr(ids), _ptr(w), T, k, H, _ptr(out))
    return _bf16_tensor(out)


def moe_layer(x, w13_q, w13_s, w2_q, w2_s, topk_ids, topk_weights, block_m: int = 16,
              group: int = 32) -> torch.Tensor:
    """Whole layer in one single-threaded call: align, gate_up, silu_mul, down, topk_sum."""
    xa = _np(x, np.uint16)
    q13, s13 = _np(w13_q, np.int32), _np(w13_s, np.uint16)
    q2, s2 = _np(w2_q, np.int32), _np(w2_s, np.uint16)
    ids = _np(topk_ids, np.int32)
    w = _np(topk_weights, np.float32)
    T, H = xa.shape
    E, two_i = q13.shape[0], q13.shape[1]
    k = ids.shape[1]
    out = np.empty((T, H), np.uint16)
    rc = lib().w4a16_oracle_moe_layer(_ptr(xa), _ptr(q13), _ptr(s13), _ptr(q2), _ptr(s2), _ptr(ids),
                                      _ptr(w), T, H, two_i // 2, E, k, group, block_m, _ptr(out))
    if rc:
        raise ValueError(f"oracle moe_layer failed with code {rc}")
    return _bf16_tensor(out)


def moe_layer_parallel(x, w13_q, w13_s, w2_q, w2_s, topk_ids, topk_weights, block_m: int = 16,
                       threads: int | None = None) -> torch.Tensor:
    """The same layer, its two GEMMs spread over host threads by expert range."""
    threads = threads or os.cpu_count() or 1
    ids = _np(topk_ids, np.int32)
    T, k = ids.shape
    E = int(_np(w13_q, np.int32).shape[0])
    sorted_ids, expert_ids, ntp = moe_align(ids, E, block_m)
    c13 = moe_gemm(x, k, w13_q, w13_s, sorted_ids, expert_ids, ntp, block_m, T * k, threads=threads,
                   out_f32=True)
    h = silu_mul(c13)
    y = moe_gemm(h, 1, w2_q, w2_s, sorted_ids, expert_ids, ntp, block_m, T * k, threads=threads,
                 out_f32=True)
    return topk_sum(y, ids, topk_weights)
