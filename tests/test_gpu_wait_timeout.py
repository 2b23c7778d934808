"""The bounded-wait error path, on the GPU, without a fault.

Every spin-wait of the kernels is bounded; when one runs out, the CTA sets its abort flag, the
caller's error word gets W4A16_DEVERR_TIMEOUT, every role leaves its loop, in-flight copies are
drained with bounded waits and tensor memory is freed, so the call returns and the context stays
usable.  The single-kernel layer's down units wait on a per-block count of finished gate_up
tiles; the test hook W4A16_LAYER_DEBUG_WAIT_TIMEOUT makes them wait for one tile more than
exists, with a limit of 2^20 cycles, so every such wait runs out (a count that nothing
reaches).  A regular call on the same context afterwards must still match the oracle.
"""
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


@pytest.mark.parametrize("block_m", [16, 64])
def test_fused_layer_wait_runs_out_and_reports_timeout(lib, block_m):
    wl = workloads.WORKLOADS["tiny"]
    inp = workloads.draw_layer(wl, 16)
    w13 = lib.pack_weights(inp.w13_q.to(DEV), inp.w13_s.to(DEV), paired=True)
    w2 = lib.pack_weights(inp.w2_q.to(DEV), inp.w2_s.to(DEV))
    x, ids, tw = inp.x.to(DEV), inp.topk_ids.to(DEV), inp.topk_weights.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.moe_layer(x, w13, w2, ids, tw, block_m=block_m, fused=True, dev_err=err,
                  debug_wait_timeout=True)
    torch.cuda.synchronize()  # the call returned and its kernels finished without a fault
    assert int(err.item()) & lib.DEVERR_TIMEOUT

    # the context is still usable: a regular fused call matches the oracle, with no error bit
    err.zero_()
    out = lib.moe_layer(x, w13, w2, ids, tw, block_m=block_m, fused=True, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.moe_layer(inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, inp.topk_ids,
                           inp.topk_weights)
    assert_close_bf16(out.cpu(), ref, "fused layer after a timed-out call")


def test_debug_wait_timeout_needs_the_single_kernel_layer(lib):
    wl = workloads.WORKLOADS["tiny"]
    inp = workloads.draw_layer(wl, 16)
    w13 = lib.pack_weights(inp.w13_q.to(DEV), inp.w13_s.to(DEV), paired=True)
    w2 = lib.pack_weights(inp.w2_q.to(DEV), inp.w2_s.to(DEV))
    with pytest.raises(lib.LibraryError):
        lib.moe_layer(inp.x.to(DEV), w13, w2, inp.topk_ids.to(DEV), inp.topk_weights.to(DEV),
                      debug_wait_timeout=True)
