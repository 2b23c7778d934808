"""The single-kernel layer (gate_up and down in one persistent cooperative launch, top-k merge
in the down epilogue) against the CPU oracle, through the C ABI."""
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


def _pack(lib, inp):
    return (lib.pack_weights(inp.w13_q.to(DEV), inp.w13_s.to(DEV), paired=True),
            lib.pack_weights(inp.w2_q.to(DEV), inp.w2_s.to(DEV)))


def _run(lib, inp, packed=None, **kw):
    packed = packed or _pack(lib, inp)
    return lib.moe_layer(inp.x.to(DEV), packed[0], packed[1], inp.topk_ids.to(DEV),
                         inp.topk_weights.to(DEV), fused=True, **kw).cpu()


@pytest.mark.parametrize("block_m", [16, 32, 64, 128])
def test_fused_layer_tiny(lib, block_m):
    inp = workloads.draw_layer(workloads.WORKLOADS["tiny"], 16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, inp, block_m=block_m, dev_err=err)
    ref = oracle.moe_layer(inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, inp.topk_ids,
                           inp.topk_weights)
    assert int(err.item()) == 0
    assert_close_bf16(out, ref, f"fused layer tiny bm={block_m}")


@pytest.mark.parametrize("T", [1, 8, 64, 512, 4096])
def test_fused_layer_qwen3_sampled_tokens(lib, T):
    wl = workloads.WORKLOADS["qwen3_30b_a3b"]
    inp = workloads.draw_layer(wl, T)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, inp, dev_err=err)
    assert int(err.item()) == 0
    sub = torch.from_numpy(sample_tokens(T, 16, seed=T))
    ref = oracle.moe_layer_parallel(inp.x[sub], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                                    inp.topk_ids[sub], inp.topk_weights[sub])
    assert_close_bf16(out[sub], ref, f"fused layer qwen3 T={T}")


@pytest.mark.parametrize("name,T", [("kimi_k2_ep8_decode", 64), ("kimi_k2_tp8", 32)])
def test_fused_layer_kimi_sampled_tokens(lib, name, T):
    wl = workloads.WORKLOADS[name]
    inp = workloads.draw_layer(wl, T)
    out = _run(lib, inp, E_global=wl.E_global)
    sub = torch.from_numpy(sample_tokens(T, 6, seed=5))
    ref = oracle.moe_layer_parallel(inp.x[sub], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                                    inp.topk_ids[sub], inp.topk_weights[sub])
    assert_close_bf16(out[sub], ref, f"fused layer {name} T={T}")
    none_local = (inp.topk_ids < 0).all(dim=1)
    assert torch.all(out[none_local].float() == 0)


def test_fused_layer_no_local_slot_gives_zeros(lib):
    inp = workloads.draw_layer(workloads.WORKLOADS["tiny"], 16)
    inp.topk_ids[:] = -1
    out = _run(lib, inp, block_m=16)
    assert torch.all(out.float() == 0)


def test_fused_layer_reuses_a_garbage_workspace_and_replays_in_a_graph(lib):
    inp = workloads.draw_layer(workloads.WORKLOADS["tiny"], 16)
    packed = _pack(lib, inp)
    ws = torch.full((lib.layer_workspace_size(16, 2, 8, 256, 256, 0, 16),), 0x7F,
                    dtype=torch.uint8, device=DEV)  # sums and block counts are zeroed per call
    ref = oracle.moe_layer(inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, inp.topk_ids,
                           inp.topk_weights)
    a = _run(lib, inp, packed=packed, block_m=16, workspace=ws)
    b = _run(lib, inp, packed=packed, block_m=16, workspace=ws)
    assert_close_bf16(a, ref, "first call")
    assert_close_bf16(b, ref, "second call")
    x, ids, w = inp.x.to(DEV), inp.topk_ids.to(DEV), inp.topk_weights.to(DEV)
    out = torch.empty_like(x)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lib.moe_layer(x, packed[0], packed[1], ids, w, block_m=16, out=out, workspace=ws, fused=True)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lib.moe_layer(x, packed[0], packed[1], ids, w, block_m=16, out=out, workspace=ws, fused=True)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert_close_bf16(out.cpu(), ref, "graph replay")
