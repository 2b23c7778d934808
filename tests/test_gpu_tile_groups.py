"""Tile groups: for short-K calls (K <= 512, e.g. the Kimi-K2 TP8 down projection, K = 256) a
work unit covers 2 or 4 consecutive 128-row weight tiles of one block, which share the block's
activation stages.  Each tile's products are summed in the same K order as with one tile per
unit, so results are bitwise identical to that schedule; both are checked against the oracle."""
from __future__ import annotations

import pytest
import torch

import oracle
from parity_util import assert_close_bf16, bits, ensure_cuda_lib, routed_rows
from w4a16_moe_expert_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    return ensure_cuda_lib()


def _case(lib, T, k, E, N, K, bm, seed, paired=False):
    qw, sc = workloads.draw_weights(E, N, K, seed=seed)
    x = workloads.draw_activations(T, K, seed=seed)
    ids, _ = workloads.draw_routing(T, E, k, seed=seed)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=paired)
    r = lib.moe_align(ids.to(DEV), E, bm)
    s, e, ntp = oracle.moe_align(ids, E, bm)
    return qw, sc, x, ids, W, r, (s, e, ntp)


@pytest.mark.parametrize("bm,group", [(16, 4), (16, 2), (32, 2), (16, 0), (32, 0)])
@pytest.mark.parametrize("K", [256, 512])
def test_groups_match_oracle_and_one_tile_per_unit(lib, bm, group, K):
    # gathered activation rows (a_row_div = top_k), BF16 output by slot
    T, k, E, N = 40, 4, 12, 1024
    qw, sc, x, ids, W, r, (s, e, ntp) = _case(lib, T, k, E, N, K, bm, 61 + K)
    one = lib.moe_gemm(x.to(DEV), k, W, r, tile_group=1, split_k=1).cpu()  # whole K, one tile
    grp = lib.moe_gemm(x.to(DEV), k, W, r, tile_group=group, split_k=1).cpu()
    ref = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, bm, T * k)
    rows = routed_rows(ids)
    assert_close_bf16(grp[rows], ref[rows], f"tile group {group}, bm {bm}, K {K}")
    assert torch.equal(bits(grp[rows]), bits(one[rows]))


@pytest.mark.parametrize("bm", [16, 32])
def test_groups_down_projection_layout_fp32(lib, bm):
    # the layer's down projection: sorted BF16 rows in, FP32 rows out by slot (K = 256)
    T, k, E, N, K = 64, 8, 24, 2048, 256
    qw, sc, x, ids, W, r, (s, e, ntp) = _case(lib, T, k, E, N, K, bm, 62)
    h = lib.gather_rows(x.to(DEV), k, r)
    flags = lib.A_ROWS_SORTED | lib.C_FP32
    one = lib.moe_gemm(h, 1, W, r, row_flags=flags, tile_group=1, split_k=1).cpu()
    grp = lib.moe_gemm(h, 1, W, r, row_flags=flags, split_k=1).cpu()  # planner's group
    assert torch.equal(one.view(torch.int32), grp.view(torch.int32))
    ref = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, bm, T * k, out_f32=True)
    rows = routed_rows(ids)
    assert_close_bf16(grp[rows], ref[rows], f"down layout, bm {bm}")


def test_groups_with_silu_epilogue_and_sorted_output(lib):
    T, k, E, N, K = 30, 2, 10, 1024, 256
    qw, sc, x, ids, W, r, (s, e, ntp) = _case(lib, T, k, E, N, K, 16, 63, paired=True)
    kw = dict(epilogue=lib.EPILOGUE_SILU_MUL, row_flags=lib.C_ROWS_SORTED)
    one = lib.moe_gemm(x.to(DEV), k, W, r, tile_group=1, split_k=1, **kw).cpu()
    grp = lib.moe_gemm(x.to(DEV), k, W, r, tile_group=4, **kw).cpu()
    assert torch.equal(bits(one[:ntp]), bits(grp[:ntp]))
    ref = oracle.silu_mul(oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 16, T * k, out_f32=True))
    for p in range(ntp):
        i = int(s[p])
        if i < T * k:
            assert_close_bf16(grp[p:p + 1], ref[i:i + 1], f"sorted row {p}")


def test_tile_count_not_a_multiple_falls_back_and_bad_groups_are_rejected(lib):
    # N = 384: three tiles, so the planner keeps one tile per unit; K = 448 (seven 64-wide
    # blocks, not whole stages) and K = 1024 (four stages) are never grouped
    T, k, E = 20, 2, 6
    qw, sc, x, ids, W, r, (s, e, ntp) = _case(lib, T, k, E, 384, 256, 16, 64)
    a = lib.moe_gemm(x.to(DEV), k, W, r, split_k=1).cpu()
    b = lib.moe_gemm(x.to(DEV), k, W, r, tile_group=1, split_k=1).cpu()
    assert torch.equal(bits(a), bits(b))
    with pytest.raises(lib.LibraryError):
        lib.moe_gemm(x.to(DEV), k, W, r, tile_group=2)
    for K in (448, 1024):
        qw, sc, x, ids, W, r, _ = _case(lib, T, k, E, 512, K, 16, 65)
        with pytest.raises(lib.LibraryError):
            lib.moe_gemm(x.to(DEV), k, W, r, tile_group=4)
    qw, sc, x, ids, W, r, _ = _case(lib, T, k, E, 512, 256, 64, 66)
    with pytest.raises(lib.LibraryError):  # 64-token blocks: one tile per unit only
        lib.moe_gemm(x.to(DEV), k, W, r, tile_group=2)
    with pytest.raises(lib.LibraryError):
        lib.moe_gemm(x.to(DEV), k, W, r, tile_group=3)
