"""The C-ABI library builds, loads and exports every symbol include/w4a16_moe.h declares.

No device work happens here: only the host-side calls (sizes, status strings,
the planner) are exercised, so this runs on a machine without a GPU.
"""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import w4a16_moe_expert_gb300 as lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16_moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    return lib.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("w4a16_moe_align", "w4a16_pack_weights", "w4a16_moe_gemm", "w4a16_moe_layer"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    assert os.path.exists(lib.library_path())


def test_status_strings(L):
    for code in range(6):
        assert L.w4a16_status_string(code)
    assert b"unknown" in L.w4a16_status_string(99)


def test_sizes_and_capacity(L):
    assert lib.align_capacity(16, 2, 8, 16) == 32 + 8 * 15 + (16 - (32 + 8 * 15) % 16) % 16
    assert lib.align_capacity(3, 2, 3, 2) == 10
    # header, 4608-byte chunks, then one mode byte per (expert, tile) padded to 16 bytes
    assert lib.packed_bytes(8, 512, 256) == 256 + 8 * 4 * 4 * 4608 + 32
    assert lib.packed_bytes(3, 128, 64) == 256 + 3 * 4608 + 16
    assert lib.packed_bytes(8, 500, 256) == 0  # N % 128 != 0 is unsupported
    assert L.w4a16_packed_bytes(1, 128, 64, 64, 0) == 0  # group must be 32
    assert lib.gemm_workspace_size(64, 128, 1536, 2048, 16) > 16 << 20
    assert lib.gemm_workspace_size(64, 128, 1536, 2048, 24) == 0
    assert lib.layer_workspace_size(16, 2, 8, 256, 256, block_m=16) > 0
    assert lib.layer_workspace_size(16, 2, 8, 256, 256, block_m=48) == 0


def test_block_m_planner():
    assert lib.plan_block_m(1, 8, 128) == 16          # decode
    assert lib.plan_block_m(512, 8, 128) == 64        # 32 rows per expert: room for the spread
    assert lib.plan_block_m(4096, 8, 128) == 128      # prefill
    assert lib.plan_block_m(256, 8, 48, 384) == 16    # EP rank: rows per local expert ~5
    assert lib.plan_block_m(16384, 8, 48, 384) == 128


def test_gemm_planner_grid_and_split():
    # decode, K = 2048 (32 blocks of 64) is never split (a slice keeps at least 24 blocks):
    # 8 routed rows over 128 experts -> ~8 blocks x 12 tiles = 96 units, one CTA each
    p = lib.plan_gemm(8, 128, 1536, 2048, 16, num_sms=148)
    assert p["split_k"] == 1 and p["num_ctas"] == 96 and p["est_units"] == 96
    # Kimi-K2 gate_up, K = 7168 (112 blocks): the device may take up to 4 slices, so the grid
    # is one CTA per SM
    p = lib.plan_gemm(8, 48, 4096, 7168, 16, num_sms=148)
    assert p["split_k"] == 4 and p["num_ctas"] == 148
    # at most 8 slices
    assert lib.plan_gemm(8, 48, 4096, 16384, 16, num_sms=148)["split_k"] == 8
    # K = 768 (12 blocks) is never split: the grid covers the estimated units
    p = lib.plan_gemm(8, 128, 2048, 768, 16, num_sms=148)
    assert p["split_k"] == 1 and p["num_ctas"] == min(148, p["est_units"]) == 128
    # prefill: thousands of tiles, a persistent grid of one CTA per SM
    p = lib.plan_gemm(32768, 128, 1536, 2048, 128, num_sms=148)
    assert p["num_ctas"] == 148
    assert p["stages"] >= 4
    with pytest.raises(lib.LibraryError):
        lib.plan_gemm(8, 128, 1536, 2000, 16, num_sms=148)


def test_gemm_planner_cta_pairs():
    # CTA pairs only for 128-token blocks whose rows are long (K >= 4096) and shared by at most
    # four tiles: Kimi-K2 TP8 gate_up (N 512 = 4 tiles, K 7168) at T=8192
    assert lib.plan_gemm(65536, 384, 512, 7168, 128, num_sms=148)["cta_pairs"] == 2
    # its down projection (56 tiles, K 256), Qwen3 and Kimi-K2 EP8 prefill gate_up (12 and 32
    # tiles), and decode blocks: one CTA per tile
    assert lib.plan_gemm(65536, 384, 7168, 256, 128, num_sms=148)["cta_pairs"] == 1
    assert lib.plan_gemm(32768, 128, 1536, 2048, 128, num_sms=148)["cta_pairs"] == 1
    assert lib.plan_gemm(65536, 48, 4096, 7168, 128, num_sms=148)["cta_pairs"] == 1
    assert lib.plan_gemm(256, 384, 512, 7168, 16, num_sms=148)["cta_pairs"] == 1
    # short K at 128-token blocks: one CTA per tile
    assert lib.plan_gemm(65536, 384, 512, 2048, 128, num_sms=148)["cta_pairs"] == 1


def test_planner_rejects_bad_arguments(L):
    plan = lib.PlanDesc()
    assert L.w4a16_plan_gemm(8, 0, 128, 64, 16, 0, 148, ctypes.byref(plan)) == 1
    assert L.w4a16_plan_gemm(8, 4, 128, 64, 16, 0, 0, ctypes.byref(plan)) == 1
