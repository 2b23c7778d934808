"""The packer's two INT4 conversions on the GPU, against the CPU oracle.

A tile whose scales all lie in (0, 2^-5) is converted with one fused multiply-add per pair
(scales stored times 2^133); every other tile subtracts the zero point and multiplies.  Both
must give bf16_rne((q - 8) * s) ("vLLM x Novita AI: Chord, Faster INT4 MoE for Kimi K2.x",
"H200 and Blackwell indexed decode": subtract, then scale, one rounding), bit for bit.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from parity_util import assert_close_bf16, bits, ensure_cuda_lib, tile_modes
from w4a16_moe_expert_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALED_MAX = 0x3CFF  # largest BF16 scale bit pattern of a multiply-add tile (just under 2^-5)


@pytest.fixture(scope="module")
def lib():
    return ensure_cuda_lib()


def _all_codes(E, N, K):
    # every group of 32 elements holds all 16 codes twice
    words = torch.tensor([0x76543210, 0xFEDCBA98 - (1 << 32)] * (K // 16), dtype=torch.int64)
    return words.to(torch.int32).reshape(1, 1, K // 8).expand(E, N, K // 8).contiguous()


def test_every_in_range_scale_takes_the_fused_conversion_bit_exact(lib):
    # the 15615 positive BF16 patterns below 2^-5 (subnormals included), 256 per expert
    E, N, K = 61, 128, 64
    pat = torch.arange(1, E * N * 2 + 1, dtype=torch.int32).clamp(max=SCALED_MAX)
    scales = pat.to(torch.int16).view(torch.bfloat16).reshape(E, N, 2).contiguous()
    qw = _all_codes(E, N, K)
    W = lib.pack_weights(qw.to(DEV), scales.to(DEV))
    assert torch.all(tile_modes(W) == 1)
    ref = oracle.dequant(qw, scales)
    for e in range(E):
        assert torch.equal(bits(lib.debug_dequant(W, e)), bits(ref[e])), f"expert {e}"


def test_modes_follow_the_scale_range(lib):
    # tile t of expert e gets one out-of-range scale per case below; the rest stay in range
    E, N, K = 2, 512, 128
    qw, sc = workloads.draw_weights(E, N, K, seed=41)
    bad = {(0, 1): 0.5, (0, 3): -0.01, (1, 0): 0.0, (1, 2): 0.03125}  # 2^-5 itself is out
    for (e, t), v in bad.items():
        sc[e, 128 * t + 7, 1] = v
    sc[1, 128 * 1 + 5, 0] = 0.0311  # just below 2^-5 (bits 0x3CFF): stays fused
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))
    want = torch.ones(E, N // 128, dtype=torch.uint8)
    for e, t in bad:
        want[e, t] = 0
    assert torch.equal(tile_modes(W), want)
    ref = oracle.dequant(qw, sc)
    for e in range(E):
        assert torch.equal(bits(lib.debug_dequant(W, e)), bits(ref[e])), f"expert {e}"


@pytest.mark.parametrize("paired", [False, True])
def test_gemm_exact_and_close_on_mixed_tiles(lib, paired):
    E, N, K = 3, 512, 256
    qw, sc = workloads.draw_weights(E, N, K, seed=42)
    sc[0, 130, 3] = 0.75   # a large scale: that tile converts by subtract-then-multiply
    sc[2, 400, 0] = -0.02  # a negative one: likewise
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=paired)
    modes = tile_modes(W)
    assert int(modes.sum()) == E * (N // 128) - 2
    ref = oracle.dequant(qw, sc)
    # one-hot rows read the dequantised weights back exactly through the tensor cores
    x = torch.eye(K, dtype=torch.bfloat16)
    for e in range(E):
        ids = torch.full((K, 1), e, dtype=torch.int32)
        r = lib.moe_align(ids.to(DEV), E, 16)
        C = lib.moe_gemm(x.to(DEV), 1, W, r)
        # values, not bits: a -0 weight (q = 8, s < 0) sums to +0 like every zero product
        assert torch.equal(C.cpu().float(), ref[e].T.contiguous().float()), f"expert {e}"
    # and a routed GEMM agrees with the oracle within the tolerance
    ids, _ = workloads.draw_routing(40, E, 2, seed=42)
    xa = workloads.draw_activations(40, K, seed=42)
    r = lib.moe_align(ids.to(DEV), E, 16)
    out = lib.moe_gemm(xa.to(DEV), 2, W, r).cpu()
    rows = torch.nonzero(ids.reshape(-1) >= 0).reshape(-1)
    want = oracle.gemm_rows(xa, 2, qw, sc, rows.numpy(), ids.reshape(-1)[rows].numpy())
    assert_close_bf16(out[rows], want, "mixed-tile gemm")


def test_nvfp4_blobs_carry_plain_modes(lib):
    codes, scales = workloads.draw_nvfp4_weights(2, 256, 128, seed=43)
    W = lib.pack_weights_nvfp4(codes.to(DEV), scales.to(DEV))
    assert torch.all(tile_modes(W) == 0)
