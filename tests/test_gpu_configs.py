"""Every configuration and token count of the benchmarked workloads against the CPU oracle, at
full size, through the C ABI, in the launch configuration the layer call and the benchmark use
(the planner's block_m and schedule):

* routing (sorted_ids, expert_ids, num_tokens_padded) bit-exact;
* the gate_up GEMM with SiLU-and-mul and the down GEMM (FP32 per-slot rows), element by element,
  on every routed row where the oracle finishes in seconds, else on a stratified sample that
  takes the first, the last and a random routed row of every aligned block, so that every
  (block, 128-row weight tile) unit of the persistent walk is read (each row spans every tile);
  the down GEMM is fed the CUDA path's own gate_up output, so each projection is checked alone;
* the layer output of sampled tokens (among them the tokens of the last rows of the busiest
  expert) against the oracle's whole layer.

The tolerance is the stated one, |gpu - ref| <= 1e-2 |ref| + 1e-2 rms(ref), with rms taken over
the compared rows.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_close_bf16, ensure_cuda_lib
from w4a16_moe_expert_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
THREADS = os.cpu_count() or 1
# compare every routed row when the two projections' oracle work stays below this many MACs
FULL_MACS = 6e9

POINTS = [(name, T) for name in ("qwen3_30b_a3b", "kimi_k2_ep8_decode", "kimi_k2_ep8_prefill",
                                 "kimi_k2_tp8", "kimi_k2_tp8_zipf")
          for T in workloads.WORKLOADS[name].tokens]


@pytest.fixture(scope="module")
def lib():
    return ensure_cuda_lib()


_weights = {}


def _packed_weights(lib, wl):
    """Draw and pack one workload's weights (one set held at a time)."""
    key = (wl.cfg_id, wl.E, wl.H, wl.I)
    if key not in _weights:
        _weights.clear()
        torch.cuda.empty_cache()
        w = workloads.draw_layer_weights(wl)
        packed = (lib.pack_weights(w[0].to(DEV), w[1].to(DEV), paired=True),
                  lib.pack_weights(w[2].to(DEV), w[3].to(DEV)))
        _weights[key] = (w, packed)
    return _weights[key]


def _positions(sorted_ids, ntp, bm, n_slots, full, rng):
    """Aligned positions to compare: every routed one, or first/last/random per block."""
    pos = []
    for b in range(ntp // bm):
        seg = sorted_ids[b * bm:(b + 1) * bm]
        routed = np.nonzero(seg < n_slots)[0]
        assert routed.size > 0, f"block {b} holds no routed row"
        if full:
            pick = routed
        else:
            pick = sorted({int(routed[0]), int(routed[-1]), int(rng.choice(routed))})
        pos.extend(b * bm + int(p) for p in pick)
    return np.asarray(pos, dtype=np.int64)


@pytest.mark.parametrize("name,T", POINTS)
def test_config_point_against_oracle(lib, name, T):
    wl = workloads.WORKLOADS[name]
    (w13_q, w13_s, w2_q, w2_s), (w13, w2) = _packed_weights(lib, wl)
    x, ids, tw = workloads.draw_layer_routing(wl, T)
    k, E, H, I = wl.top_k, wl.E, wl.H, wl.I
    n_slots = T * k
    bm = lib.plan_block_m(T, k, E, wl.E_global)
    hint = max(1, round(n_slots / wl.E_global))
    xd, idsd, twd = x.to(DEV), ids.to(DEV), tw.to(DEV)

    # routing, bit-exact
    r = lib.moe_align(idsd, E, bm)
    s_ref, e_ref, ntp_ref = oracle.moe_align(ids, E, bm)
    s_gpu, e_gpu = r.sorted_ids.cpu().numpy(), r.expert_ids.cpu().numpy()
    assert int(r.num_tokens_padded.item()) == ntp_ref
    assert np.array_equal(s_gpu, np.asarray(s_ref))
    assert np.array_equal(e_gpu, np.asarray(e_ref))

    # the two projections, called as the layer calls them
    if bm >= 64:
        xs = lib.gather_rows(xd, k, r)
        h = lib.moe_gemm(xs, 1, w13, r, epilogue=lib.EPILOGUE_SILU_MUL,
                         row_flags=lib.A_ROWS_SORTED | lib.C_ROWS_SORTED,
                         expected_rows_per_expert=hint)
        del xs
    else:
        h = lib.moe_gemm(xd, k, w13, r, epilogue=lib.EPILOGUE_SILU_MUL, row_flags=lib.C_ROWS_SORTED,
                         expected_rows_per_expert=hint)
    y = lib.moe_gemm(h, 1, w2, r, row_flags=lib.A_ROWS_SORTED | lib.C_FP32,
                     expected_rows_per_expert=hint)
    out = lib.moe_layer(xd, w13, w2, idsd, twd, E_global=wl.E_global)
    torch.cuda.synchronize()

    n_routed = int((s_gpu[:ntp_ref] < n_slots).sum())
    full = n_routed * 3 * I * H <= FULL_MACS
    rng = np.random.default_rng(T)
    pos = _positions(s_gpu, ntp_ref, bm, n_slots, full, rng)
    if pos.size:
        slots = s_gpu[pos]
        experts = e_gpu[pos // bm]
        # gate_up + SiLU-and-mul
        h_ref = oracle.silu_mul(oracle.gemm_rows(x, k, w13_q, w13_s, slots, experts,
                                                 out_f32=True, threads=THREADS))
        h_pos = h[torch.from_numpy(pos).to(DEV)].cpu()
        assert_close_bf16(h_pos, h_ref, f"{name} T={T} gate_up rows ({pos.size} of {n_routed})")
        # down, on the CUDA path's own gate_up rows
        y_ref = oracle.gemm_rows(h_pos, 1, w2_q, w2_s, np.arange(pos.size), experts,
                                 out_f32=True, threads=THREADS)
        y_pos = y[torch.from_numpy(slots.astype(np.int64)).to(DEV)].cpu()
        assert_close_bf16(y_pos, y_ref, f"{name} T={T} down rows ({pos.size} of {n_routed})")
    del h, y

    # the layer on sampled tokens, among them those of the busiest expert's last rows
    if T <= 16:
        tok = np.arange(T)
    else:
        ex_all = ids.reshape(-1).numpy()
        busiest = int(np.bincount(ex_all[ex_all >= 0], minlength=E).argmax()) if (ex_all >= 0).any() else 0
        hot = np.nonzero((ids.numpy() == busiest).any(axis=1))[0][-4:]
        rest = rng.choice(T, size=12, replace=False)
        tok = np.unique(np.concatenate([hot, rest]))
    sub = torch.from_numpy(tok)
    ref = oracle.moe_layer_parallel(x[sub], w13_q, w13_s, w2_q, w2_s, ids[sub], tw[sub],
                                    threads=THREADS)
    got = out.cpu()
    assert_close_bf16(got[sub], ref, f"{name} T={T} layer ({tok.size} tokens)")
    none_local = (ids < 0).all(dim=1)
    assert torch.all(got[none_local].float() == 0)
