"""The layer call captured once in a CUDA graph and replayed on new inputs, in the manner the
call is used in serving: between replays the activations and the routing (which experts,
how many rows each) are rewritten in place and the whole workspace is poisoned with 0xFF; every
replay must match the oracle for its own inputs and give the same bits when repeated, and
replaying allocates no device memory.
The schedule (K slices, tile groups, block walk) is decided on the device from the routing of
each replay, so this covers the graph-capturable contract of every decode and prefill path:
Qwen3 T=8 (16-token blocks, rows gathered in the GEMM), Kimi-K2 EP8 T=1 (the gate_up tiles cut
into K slices; routings with no local slot), Kimi-K2 TP8 T=32 (tile groups of the K = 256 down
projection) and Qwen3 T=512 (64-token blocks, the row-gather kernel, TMA rows)."""
from __future__ import annotations

import pytest
import torch

import oracle
from parity_util import assert_close_bf16, ensure_cuda_lib
from w4a16_moe_expert_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    return ensure_cuda_lib()


@pytest.mark.parametrize("name,T", [("qwen3_30b_a3b", 8), ("kimi_k2_ep8_decode", 1),
                                    ("kimi_k2_tp8", 32), ("qwen3_30b_a3b", 512)])
def test_layer_graph_replays_with_new_inputs_and_poisoned_workspace(lib, name, T):
    wl = workloads.WORKLOADS[name]
    w13_q, w13_s, w2_q, w2_s = workloads.draw_layer_weights(wl)
    w13 = lib.pack_weights(w13_q.to(DEV), w13_s.to(DEV), paired=True)
    w2 = lib.pack_weights(w2_q.to(DEV), w2_s.to(DEV))
    k = wl.top_k
    bm = lib.plan_block_m(T, k, wl.E, wl.E_global)
    # input buffers the graph reads, rewritten in place before every replay
    x = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    out = torch.empty((T, wl.H), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(lib.layer_workspace_size(T, k, wl.E, wl.H, wl.I, wl.E_global, bm),
                     dtype=torch.uint8, device=DEV)

    def draw(seed):
        xi = workloads.draw_activations(T, wl.H, seed)
        ii, wi = workloads.draw_routing(T, wl.E_global, k, seed, wl.routing, wl.local_lo, wl.E,
                                        wl.empty_experts, wl.zipf_s)
        return xi, ii, wi

    def call():
        lib.moe_layer(x, w13, w2, ids, tw, E_global=wl.E_global, block_m=bm, out=out,
                      workspace=ws)

    xi, ii, wi = draw(1)
    x.copy_(xi), ids.copy_(ii), tw.copy_(wi)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    for seed in ((2, 3, 4, 5) if T <= 32 else (2, 3)):
        xi, ii, wi = draw(1000 + 17 * seed + T)
        x.copy_(xi), ids.copy_(ii), tw.copy_(wi)
        ws.fill_(0xFF)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = out.cpu()
        ref = oracle.moe_layer_parallel(xi, w13_q, w13_s, w2_q, w2_s, ii, wi)
        assert_close_bf16(got, ref, f"{name} T={T} replay {seed}")
        assert torch.all(got[(ii < 0).all(dim=1)].float() == 0)
        # the same inputs again, workspace poisoned again: the same bits (every sum runs in a
        # fixed order, K slices included)
        ws.fill_(0xFF)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.cpu().view(torch.int16), got.view(torch.int16))
    assert torch.cuda.memory_allocated() == alloc0
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "a replay allocated device memory"
