"""Grouped contracts on the GPU ("Grouped SM90 kernels": contiguous prefill, masked decode)
against the CPU oracle, through the C ABI."""
from __future__ import annotations

import pytest
import torch

import oracle
from parity_util import assert_close_bf16, bits, ensure_cuda_lib
from w4a16_moe_expert_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    return ensure_cuda_lib()


def contiguous_layout(group_rows, seed, K):
    """Rows concatenated by expert, each group padded to 128 rows (m_indices -1 there)."""
    ids = []
    for e, rows in group_rows:
        ids += [e] * rows + [-1] * ((-rows) % 128)
    mi = torch.tensor(ids, dtype=torch.int32)
    x = workloads.draw_activations(mi.numel(), K, seed=seed)
    return x, mi


@pytest.mark.parametrize("epilogue", [0, 1])
def test_contiguous_matches_oracle(lib, epilogue):
    E, N, K = 8, 512, 256
    qw, sc = workloads.draw_weights(E, N, K, seed=31)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=True)
    x, mi = contiguous_layout([(0, 5), (3, 128), (1, 200), (7, 300), (2, 1)], seed=31, K=K)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = lib.contiguous_gemm(x.to(DEV), W, mi.to(DEV), epilogue=epilogue, dev_err=err).cpu()
    ref = oracle.contiguous_gemm(x, qw, sc, mi, out_f32=bool(epilogue))
    if epilogue:
        ref = oracle.silu_mul(ref)
    valid = mi >= 0
    assert int(err.item()) == 0
    assert_close_bf16(out[valid], ref[valid], "contiguous valid rows")
    assert torch.all(out[~valid].float() == 0), "padding rows of a block with valid rows are zeros"


def test_contiguous_qwen_shape_from_a_routing(lib):
    # The rows of a top-8 routing of 512 tokens over 128 experts, grouped by expert
    wl = workloads.WORKLOADS["qwen3_30b_a3b"]
    qw, sc = workloads.draw_weights(wl.E, 2 * wl.I, wl.H, seed=32)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=True)
    ids, _ = workloads.draw_routing(512, wl.E, wl.top_k, seed=32)
    counts = torch.bincount(ids.reshape(-1), minlength=wl.E).tolist()
    x, mi = contiguous_layout([(e, c) for e, c in enumerate(counts) if c], seed=32, K=wl.H)
    out = lib.contiguous_gemm(x.to(DEV), W, mi.to(DEV), epilogue=1).cpu()
    rows = torch.nonzero(mi >= 0).reshape(-1)[::7]  # a sample of the valid rows
    ref = oracle.silu_mul(oracle.gemm_rows(x, 1, qw, sc, rows.numpy(), mi[rows].numpy(),
                                           out_f32=True))
    assert_close_bf16(out[rows], ref, "contiguous qwen rows")


@pytest.mark.parametrize("expected_m", [4, 40, 100])
def test_masked_matches_oracle_and_leaves_other_rows(lib, expected_m):
    G, N, K, max_m = 48, 256, 512, 96
    qw, sc = workloads.draw_weights(G, N, K, seed=33)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))
    x = workloads.draw_activations(G * max_m, K, seed=33).reshape(G, max_m, K)
    g = torch.Generator().manual_seed(33)
    mm = torch.randint(0, max_m + 1, (G,), generator=g, dtype=torch.int32)
    mm[0], mm[1], mm[2] = 0, max_m, 1
    out = torch.full((G * max_m, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.masked_gemm(x.to(DEV), W, mm.to(DEV), expected_m, out=out, dev_err=err)
    out = out.cpu()
    ref = oracle.masked_gemm(x, qw, sc, mm, max_m)
    valid = (torch.arange(max_m)[None, :] < mm[:, None].long()).reshape(-1)
    assert int(err.item()) == 0
    assert_close_bf16(out[valid], ref[valid], "masked valid rows")
    assert torch.isnan(out[~valid].float()).all(), "rows past masked_m are left untouched"


def test_masked_silu_and_two_calls_identical(lib):
    G, N, K, max_m = 16, 512, 256, 32
    qw, sc = workloads.draw_weights(G, N, K, seed=34)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=True)
    x = workloads.draw_activations(G * max_m, K, seed=34)
    mm = torch.arange(G, dtype=torch.int32) * 2
    a = lib.masked_gemm(x.to(DEV), W, mm.to(DEV), 8, epilogue=1).cpu()
    b = lib.masked_gemm(x.to(DEV), W, mm.to(DEV), 8, epilogue=1).cpu()
    ref = oracle.silu_mul(oracle.masked_gemm(x, qw, sc, mm, max_m, out_f32=True))
    valid = (torch.arange(max_m)[None, :] < mm[:, None].long()).reshape(-1)
    assert_close_bf16(a[valid], ref[valid], "masked silu")
    assert torch.equal(bits(a[valid]), bits(b[valid]))


def test_grouped_mode_and_argument_checks(lib):
    E, N, K = 4, 256, 128
    qw, sc = workloads.draw_weights(E, N, K, seed=35)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))  # not gate/up paired
    x, mi = contiguous_layout([(0, 10)], seed=35, K=K)
    with pytest.raises(lib.LibraryError, match="bad packed weight"):
        lib.contiguous_gemm(x.to(DEV), W, mi.to(DEV), epilogue=1)
    with pytest.raises(lib.LibraryError, match="invalid argument"):
        lib.contiguous_gemm(x[:100].contiguous().to(DEV), W, mi[:100].contiguous().to(DEV))
    mm = torch.ones(E + 1, dtype=torch.int32)
    xm = workloads.draw_activations((E + 1) * 8, K, seed=35)
    with pytest.raises(lib.LibraryError, match="invalid argument"):
        lib.masked_gemm(xm.to(DEV), W, mm.to(DEV), 1)


def test_grouped_device_side_flags(lib):
    E, N, K = 4, 256, 128
    qw, sc = workloads.draw_weights(E, N, K, seed=36)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))
    x, mi = contiguous_layout([(0, 10), (1, 20)], seed=36, K=K)
    mi[5] = 2  # a second expert inside the first 128-row block
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.contiguous_gemm(x.to(DEV), W, mi.to(DEV), dev_err=err)
    assert int(err.item()) & lib.DEVERR_BAD_EXPERT_ID
    mm = torch.tensor([3, 99, 0, 8], dtype=torch.int32)  # 99 > max_m = 8
    xm = workloads.draw_activations(E * 8, K, seed=36)
    err.zero_()
    out = lib.masked_gemm(xm.to(DEV), W, mm.to(DEV), 4, dev_err=err).cpu()
    assert int(err.item()) & lib.DEVERR_CAPACITY
    ref = oracle.masked_gemm(xm, qw, sc, torch.clamp(mm, 0, 8), 8)  # clamped to max_m
    valid = (torch.arange(8)[None, :] < torch.clamp(mm, 0, 8)[:, None].long()).reshape(-1)
    assert_close_bf16(out[valid], ref[valid], "masked clamped")
