"""The GEMM entry point that allocates nothing, checked against the regular one.

Callers such as inference-engine plugins (their enqueue hook gets only input and output
buffers) or serving loops that must not call cudaMalloc after start-up cannot pass a
workspace; w4a16_moe_gemm_static_scratch keeps the K-split scratch in a library-owned device
array instead.  This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import pytest
import torch

from w4a16_moe_expert_gb300 import workloads
from parity_util import assert_close_bf16, bits, routed_rows

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.mark.parametrize("block_m", [16, 32, 64, 128])
def test_static_scratch_gemm_matches_workspace_gemm_twice(block_m):
    import w4a16_moe_expert_gb300 as lib
    lib.load()
    E, N, K, T, k = 64, 512, 2048, 24 if block_m <= 32 else 300, 4
    qw, sc = workloads.draw_weights(E, N, K, seed=77)
    x = workloads.draw_activations(T, K, seed=77).to(DEV)
    ids, _ = workloads.draw_routing(T, E, k, seed=77)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=True)
    r = lib.moe_align(ids.to(DEV), E, block_m)
    rows = routed_rows(ids)
    for epilogue, split in ((lib.EPILOGUE_SILU_MUL, 3), (lib.EPILOGUE_NONE, 2)):
        ref = lib.moe_gemm(x, k, W, r, epilogue=epilogue, split_k=split)
        outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        # one warm-up call (the first call on a device looks up the array's address, and the
        # first launch of a kernel may load its module)
        lib.moe_gemm_static_scratch(x, k, W, r, epilogue=epilogue, out=outs[0], split_k=split,
                                    dev_err=err)
        torch.cuda.synchronize()
        for call in range(2):  # the shared scratch must be reusable call after call
            outs[call].fill_(float("nan"))
            torch.cuda.synchronize()
            free0, _ = torch.cuda.mem_get_info()
            alloc0 = torch.cuda.memory_allocated()
            lib.moe_gemm_static_scratch(x, k, W, r, epilogue=epilogue, out=outs[call],
                                        split_k=split, dev_err=err)
            torch.cuda.synchronize()
            free1, _ = torch.cuda.mem_get_info()
            assert free1 == free0, f"device memory changed by {free0 - free1} bytes during the call"
            assert torch.cuda.memory_allocated() == alloc0
            assert int(err.item()) == 0
            out = outs[call]
            assert_close_bf16(out.cpu()[rows], ref.cpu()[rows], f"static scratch call {call}")
            assert torch.equal(bits(out[rows.to(DEV)]), bits(ref[rows.to(DEV)]))
