"""Shared helpers for the parity tests (CUDA path vs the CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerance for BF16 outputs: |gpu - ref| <= REL * |ref| + ABS_RMS * rms(ref), per element,
# rms over the valid elements of that output.
REL = 1e-2
ABS_RMS = 1e-2


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.detach().cpu().contiguous().view(torch.int16)


def assert_close_bf16(gpu: torch.Tensor, ref: torch.Tensor, what: str = "output"):
    g = gpu.detach().cpu().float()
    r = ref.detach().cpu().float()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if r.numel() == 0:
        return
    assert torch.isfinite(g).all(), f"{what}: non-finite values in the CUDA result"
    rms = float(torch.sqrt(torch.mean(r.double() ** 2)))
    err = (g - r).abs()
    bound = REL * r.abs() + ABS_RMS * rms
    bad = err > bound
    if bad.any():
        idx = torch.nonzero(bad)[:5].tolist()
        worst = float((err / bound.clamp_min(1e-30)).max())
        raise AssertionError(f"{what}: {int(bad.sum())} of {r.numel()} elements outside tolerance "
                             f"(worst err/bound {worst:.3g}); first at {idx}")


def routed_rows(topk_ids: torch.Tensor) -> torch.Tensor:
    """Flat slot indices with a local expert."""
    return torch.nonzero(topk_ids.reshape(-1) >= 0).reshape(-1)


def ensure_cuda_lib():
    import w4a16_moe_expert_gb300 as lib
    lib.load()
    return lib


def to_dev(*ts, device="cuda"):
    return [t.to(device) for t in ts]


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    if T <= n:
        return np.arange(T)
    return np.sort(rng.choice(T, size=n, replace=False))


def tile_modes(W) -> torch.Tensor:
    """The packed blob's mode byte per (expert, 128-row tile): 1 = scales stored times 2^133
    (multiply-add conversion), 0 = scales as given (subtract-then-multiply conversion)."""
    n_tiles, n_kb = W.N // 128, W.K // 64
    off = 256 + W.E * n_tiles * n_kb * 4608
    return W.blob[off:off + W.E * n_tiles].cpu().reshape(W.E, n_tiles)
