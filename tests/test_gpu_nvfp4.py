"""NVFP4 weights on the GPU (E2M1 codes with an E4M3 scale per 16 K elements, BF16
activations) against the CPU oracle, through the C ABI: the dequantised weights bit-exact,
GEMM and layer outputs within the BF16 tolerance."""
from __future__ import annotations

import numpy as np
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


def _same_bits_nan_aware(gpu: torch.Tensor, ref: torch.Tensor):
    g, r = gpu.cpu(), ref.cpu()
    gn, rn = torch.isnan(g.float()), torch.isnan(r.float())
    assert torch.equal(gn, rn), "NaN positions differ"
    assert torch.equal(bits(g[~gn]), bits(r[~rn]))


@pytest.mark.parametrize("paired", [False, True])
def test_nvfp4_dequant_exhaustive_bit_exact(lib, paired):
    # 256 rows, one per E4M3 scale byte (NaN bytes included), the first 16-block of every row
    # holding all 16 codes; the other blocks random
    N, K = 256, 128
    codes, _ = workloads.draw_nvfp4_weights(1, N, K, seed=51)
    codes = codes.clone()
    for j in range(8):
        codes[0, :, j] = (2 * j) | ((2 * j + 1) << 4)
    scales = torch.arange(256, dtype=torch.uint8).reshape(1, N, 1).repeat(1, 1, K // 16)
    W = lib.pack_weights_nvfp4(codes.to(DEV), scales.to(DEV), paired=paired)
    got = lib.debug_dequant(W, 0)
    _same_bits_nan_aware(got, oracle.nvfp4_dequant(codes, scales)[0])


def test_nvfp4_dequant_random_experts_bit_exact(lib):
    codes, scales = workloads.draw_nvfp4_weights(4, 384, 512, seed=52)
    W = lib.pack_weights_nvfp4(codes.to(DEV), scales.to(DEV))
    ref = oracle.nvfp4_dequant(codes, scales)
    for e in range(4):
        assert torch.equal(bits(lib.debug_dequant(W, e)), bits(ref[e]))


def test_nvfp4_one_hot_gemm_reads_back_the_weights_exactly(lib):
    E, N, K = 2, 128, 128
    codes, scales = workloads.draw_nvfp4_weights(E, N, K, seed=53)
    W = lib.pack_weights_nvfp4(codes.to(DEV), scales.to(DEV))
    x = torch.eye(K, dtype=torch.bfloat16)
    wd = oracle.nvfp4_dequant(codes, scales)
    for e in range(E):
        ids = torch.full((K, 1), e, dtype=torch.int32)
        r = lib.moe_align(ids.to(DEV), E, 16)
        C = lib.moe_gemm(x.to(DEV), 1, W, r)
        # equal values; the E2M1 code for -0 dequantises to -0, while the dot product adds
        # +0 terms and returns +0 there, so signed zeros are compared as values
        assert torch.equal(C.cpu().float(), wd[e].T.contiguous().float())


@pytest.mark.parametrize("bm", [16, 64, 128])
@pytest.mark.parametrize("epilogue", [0, 1])
def test_nvfp4_gemm_matches_oracle(lib, bm, epilogue):
    E, N, K, T, k = 8, 512, 256, 40, 2
    codes, scales = workloads.draw_nvfp4_weights(E, N, K, seed=54)
    x = workloads.draw_activations(T, K, seed=54)
    ids, _ = workloads.draw_routing(T, E, k, seed=54, empty_experts=(5,))
    W = lib.pack_weights_nvfp4(codes.to(DEV), scales.to(DEV), paired=True)
    r = lib.moe_align(ids.to(DEV), E, bm)
    got = lib.moe_gemm(x.to(DEV), k, W, r, epilogue=epilogue).cpu()
    s, e, ntp = oracle.moe_align(ids, E, bm)
    ref = oracle.nvfp4_moe_gemm(x, k, codes, scales, s, e, ntp, bm, T * k, out_f32=bool(epilogue))
    if epilogue:
        ref = oracle.silu_mul(ref)
    rows = routed_rows(ids)
    assert_close_bf16(got[rows], ref[rows], f"nvfp4 gemm bm={bm}")


def _oracle_nvfp4_layer(x, w13, w2, ids, tw, bm):
    T, k = ids.shape
    E = w13[0].shape[0]
    s, e, ntp = oracle.moe_align(ids, E, bm)
    c13 = oracle.nvfp4_moe_gemm(x, k, *w13, s, e, ntp, bm, T * k, out_f32=True)
    h = oracle.silu_mul(c13)
    y = oracle.nvfp4_moe_gemm(h, 1, *w2, s, e, ntp, bm, T * k, out_f32=True)
    return oracle.topk_sum(y, ids, tw)


def test_nvfp4_layer_tiny_matches_oracle(lib):
    E, H, I, T, k = 8, 256, 256, 16, 2
    w13 = workloads.draw_nvfp4_weights(E, 2 * I, H, seed=55)
    w2 = workloads.draw_nvfp4_weights(E, H, I, seed=56)
    x = workloads.draw_activations(T, H, seed=57)
    ids, tw = workloads.draw_routing(T, E, k, seed=57, empty_experts=(E - 1,))
    W13 = lib.pack_weights_nvfp4(w13[0].to(DEV), w13[1].to(DEV), paired=True)
    W2 = lib.pack_weights_nvfp4(w2[0].to(DEV), w2[1].to(DEV))
    out = lib.moe_layer(x.to(DEV), W13, W2, ids.to(DEV), tw.to(DEV), block_m=16).cpu()
    assert_close_bf16(out, _oracle_nvfp4_layer(x, w13, w2, ids, tw, 16), "nvfp4 layer")


def test_nvfp4_qwen_shape_sampled_tokens(lib):
    wl = workloads.WORKLOADS["qwen3_30b_a3b"]
    T = 64
    w13 = workloads.draw_nvfp4_weights(wl.E, 2 * wl.I, wl.H, seed=58)
    w2 = workloads.draw_nvfp4_weights(wl.E, wl.H, wl.I, seed=59)
    x, ids, tw = workloads.draw_layer_routing(wl, T)
    W13 = lib.pack_weights_nvfp4(w13[0].to(DEV), w13[1].to(DEV), paired=True)
    W2 = lib.pack_weights_nvfp4(w2[0].to(DEV), w2[1].to(DEV))
    bm = lib.plan_block_m(T, wl.top_k, wl.E)
    out = lib.moe_layer(x.to(DEV), W13, W2, ids.to(DEV), tw.to(DEV), block_m=bm).cpu()
    toks = np.arange(0, T, 8)
    ref = _oracle_nvfp4_layer(x[toks], w13, w2, ids[toks], tw[toks], 16)
    assert_close_bf16(out[toks], ref, "nvfp4 qwen sampled tokens")


def test_nvfp4_descriptor_checks(lib):
    codes, scales = workloads.draw_nvfp4_weights(2, 128, 64, seed=60)
    W = lib.pack_weights_nvfp4(codes.to(DEV), scales.to(DEV))
    assert W.desc.flags & lib.PACK_NVFP4 and W.desc.group == 16
    W.desc.group = 32  # an NVFP4 blob claiming INT4 group size fails loudly
    x = workloads.draw_activations(4, 64, seed=60)
    r = lib.moe_align(torch.zeros((4, 1), dtype=torch.int32, device=DEV), 2, 16)
    with pytest.raises(lib.LibraryError, match="bad packed weight"):
        lib.moe_gemm(x.to(DEV), 1, W, r)
    with pytest.raises(lib.LibraryError, match="bad packed weight"):
        lib.moe_gemm(x.to(DEV), 1, W, r, epilogue=1)
