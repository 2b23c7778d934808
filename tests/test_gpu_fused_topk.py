"""The layer with the top-k merge fused into the down GEMM (atomic FP32 token sums) against
the CPU oracle, through the C ABI."""
from __future__ import annotations

import pytest
import torch

import oracle
from parity_util import assert_close_bf16, ensure_cuda_lib, sample_tokens
from w4a16_moe_expert_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    return ensure_cuda_lib()


def _run(lib, inp, packed=None, **kw):
    if packed is None:
        packed = (lib.pack_weights(inp.w13_q.to(DEV), inp.w13_s.to(DEV), paired=True),
                  lib.pack_weights(inp.w2_q.to(DEV), inp.w2_s.to(DEV)))
    return lib.moe_layer(inp.x.to(DEV), packed[0], packed[1], inp.topk_ids.to(DEV),
                         inp.topk_weights.to(DEV), fused_topk=True, **kw).cpu()


@pytest.mark.parametrize("block_m", [16, 32, 64, 128])
def test_fused_topk_tiny_layer(lib, block_m):
    inp = workloads.draw_layer(workloads.WORKLOADS["tiny"], 16)
    out = _run(lib, inp, block_m=block_m)
    ref = oracle.moe_layer(inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, inp.topk_ids,
                           inp.topk_weights)
    assert_close_bf16(out, ref, "fused top-k tiny layer")


@pytest.mark.parametrize("T", [1, 64, 4096])
def test_fused_topk_qwen3_sampled_tokens(lib, T):
    wl = workloads.WORKLOADS["qwen3_30b_a3b"]
    inp = workloads.draw_layer(wl, T)
    out = _run(lib, inp)
    sub = torch.from_numpy(sample_tokens(T, 16, seed=T))
    ref = oracle.moe_layer_parallel(inp.x[sub], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                                    inp.topk_ids[sub], inp.topk_weights[sub])
    assert_close_bf16(out[sub], ref, f"fused top-k qwen3 T={T}")


def test_fused_topk_ep_rank_drops_slots_and_zero_rows(lib):
    wl = workloads.WORKLOADS["kimi_k2_ep8_decode"]
    inp = workloads.draw_layer(wl, 64)
    out = _run(lib, inp, E_global=wl.E_global)
    sub = torch.from_numpy(sample_tokens(64, 6, seed=3))
    ref = oracle.moe_layer_parallel(inp.x[sub], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                                    inp.topk_ids[sub], inp.topk_weights[sub])
    assert_close_bf16(out[sub], ref, "fused top-k kimi ep8 T=64")
    none_local = (inp.topk_ids < 0).all(dim=1)
    assert torch.all(out[none_local].float() == 0)


def test_fused_topk_repeated_calls_reuse_the_workspace(lib):
    inp = workloads.draw_layer(workloads.WORKLOADS["tiny"], 16)
    packed = (lib.pack_weights(inp.w13_q.to(DEV), inp.w13_s.to(DEV), paired=True),
              lib.pack_weights(inp.w2_q.to(DEV), inp.w2_s.to(DEV)))
    ws = torch.full((lib.layer_workspace_size(16, 2, 8, 256, 256, 0, 16),), 0x7F,
                    dtype=torch.uint8, device=DEV)  # garbage: the sums must be zeroed per call
    a = _run(lib, inp, packed=packed, block_m=16, workspace=ws)
    b = _run(lib, inp, packed=packed, block_m=16, workspace=ws)
    ref = oracle.moe_layer(inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, inp.topk_ids,
                           inp.topk_weights)
    assert_close_bf16(a, ref, "first call")
    assert_close_bf16(b, ref, "second call")
