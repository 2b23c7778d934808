"""CTA pairs against the CPU oracle and against the one-CTA schedule, through the C ABI: mode 2
(tcgen05 cta_group::2: one M = 256 MMA over two CTAs' 128-row weight tiles, each CTA holding
half of a 128-token block's activation rows)."""
from __future__ import annotations

import pytest
import torch

import oracle
from parity_util import assert_close_bf16, bits, ensure_cuda_lib, routed_rows
from w4a16_moe_expert_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
MODES = [2]


@pytest.fixture(scope="module")
def lib():
    return ensure_cuda_lib()


def _case(lib, T, k, E, N, K, seed, paired=False):
    qw, sc = workloads.draw_weights(E, N, K, seed=seed)
    x = workloads.draw_activations(T, K, seed=seed)
    ids, _ = workloads.draw_routing(T, E, k, seed=seed)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=paired)
    r = lib.moe_align(ids.to(DEV), E, 128)
    xs = lib.gather_rows(x.to(DEV), k, r)
    s, e, ntp = oracle.moe_align(ids, E, 128)
    return qw, sc, x, ids, W, r, xs, (s, e, ntp)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("paired,epilogue", [(False, 0), (True, 0), (True, 1)])
def test_pairs_match_oracle_and_single_cta(lib, mode, paired, epilogue):
    T, k, E, N, K = 200, 4, 6, 512, 384
    qw, sc, x, ids, W, r, xs, (s, e, ntp) = _case(lib, T, k, E, N, K, 51, paired)
    kw = dict(epilogue=epilogue, row_flags=lib.A_ROWS_SORTED)
    one = lib.moe_gemm(xs, 1, W, r, cta_pairs=1, **kw).cpu()
    two = lib.moe_gemm(xs, 1, W, r, cta_pairs=mode, **kw).cpu()
    ref = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 128, T * k, out_f32=bool(epilogue))
    if epilogue:
        ref = oracle.silu_mul(ref)
    rows = routed_rows(ids)
    assert_close_bf16(two[rows], ref[rows], "pairs")
    # the same products summed in the same K order: identical to the one-CTA schedule
    assert torch.equal(bits(two[rows]), bits(one[rows]))


@pytest.mark.parametrize("mode", MODES)
def test_pairs_odd_k_tail(lib, mode):
    # K = 448: seven 64-wide K blocks, so the last stage holds one
    T, k, E, N, K = 150, 4, 5, 512, 448
    qw, sc, x, ids, W, r, xs, (s, e, ntp) = _case(lib, T, k, E, N, K, 56, True)
    kw = dict(epilogue=1, row_flags=lib.A_ROWS_SORTED)
    one = lib.moe_gemm(xs, 1, W, r, cta_pairs=1, **kw).cpu()
    two = lib.moe_gemm(xs, 1, W, r, cta_pairs=mode, **kw).cpu()
    ref = oracle.silu_mul(oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 128, T * k, out_f32=True))
    rows = routed_rows(ids)
    assert_close_bf16(two[rows], ref[rows], f"pairs mode {mode}, K tail")
    assert torch.equal(bits(two[rows]), bits(one[rows]))


@pytest.mark.parametrize("mode", MODES)
def test_pairs_fp32_rows_and_grid_sizes(lib, mode):
    T, k, E, N, K = 300, 8, 16, 768, 256
    qw, sc, x, ids, W, r, xs, (s, e, ntp) = _case(lib, T, k, E, N, K, 52)
    base = lib.moe_gemm(xs, 1, W, r, row_flags=lib.A_ROWS_SORTED | lib.C_FP32, cta_pairs=1).cpu()
    rows = routed_rows(ids)
    for ctas in (2, 6, 64, 152):
        got = lib.moe_gemm(xs, 1, W, r, row_flags=lib.A_ROWS_SORTED | lib.C_FP32, cta_pairs=mode,
                           num_ctas=ctas).cpu()
        assert torch.equal(got[rows].view(torch.int32), base[rows].view(torch.int32)), f"grid {ctas}"


@pytest.mark.parametrize("mode", MODES)
def test_pairs_one_hot_reads_weights_back_exactly(lib, mode):
    E, N, K = 2, 256, 128
    qw, sc = workloads.draw_weights(E, N, K, seed=53)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))
    ref = oracle.dequant(qw, sc)
    x = torch.eye(K, dtype=torch.bfloat16)
    for ex in range(E):
        ids = torch.full((K, 1), ex, dtype=torch.int32)
        r = lib.moe_align(ids.to(DEV), E, 128)
        xs = lib.gather_rows(x.to(DEV), 1, r)
        C = lib.moe_gemm(xs, 1, W, r, row_flags=lib.A_ROWS_SORTED, cta_pairs=mode).cpu()
        assert torch.equal(bits(C), bits(ref[ex].T.contiguous())), f"expert {ex}"


@pytest.mark.parametrize("mode", MODES)
def test_pairs_qwen3_prefill_sampled_rows(lib, mode):
    wl = workloads.WORKLOADS["qwen3_30b_a3b"]
    T = 4096
    qw, sc = workloads.draw_weights(wl.E, 2 * wl.I, wl.H, seed=54)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=True)
    x = workloads.draw_activations(T, wl.H, seed=54)
    ids, _ = workloads.draw_routing(T, wl.E, wl.top_k, seed=54)
    r = lib.moe_align(ids.to(DEV), wl.E, 128)
    xs = lib.gather_rows(x.to(DEV), wl.top_k, r)
    s, e, ntp = oracle.moe_align(ids, wl.E, 128)
    C = lib.moe_gemm(xs, 1, W, r, epilogue=1, row_flags=lib.A_ROWS_SORTED | lib.C_ROWS_SORTED,
                     cta_pairs=mode).cpu()
    pos = torch.nonzero(torch.from_numpy(s[:ntp]) < T * wl.top_k).reshape(-1)[::97]
    slots = torch.from_numpy(s[pos.numpy()]).long()
    experts = torch.from_numpy(e[(pos // 128).numpy()]).long()
    ref = oracle.silu_mul(oracle.gemm_rows(x, wl.top_k, qw, sc, slots.numpy(), experts.numpy(),
                                           out_f32=True))
    assert_close_bf16(C[pos], ref, f"qwen3 T=4096 pairs mode {mode}")


@pytest.mark.parametrize("mode", MODES)
def test_pairs_with_nothing_routed(lib, mode):
    # every slot dropped: no block to compute, the output stays as it was
    E, N, K, T, k = 4, 256, 128, 40, 2
    qw, sc = workloads.draw_weights(E, N, K, seed=57)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))
    ids = torch.full((T, k), -1, dtype=torch.int32)
    r = lib.moe_align(ids.to(DEV), E, 128)
    xs = torch.zeros((r.capacity, K), dtype=torch.bfloat16, device=DEV)
    out = torch.full((T * k, N), 7.0, dtype=torch.float32, device=DEV)
    lib.moe_gemm(xs, 1, W, r, row_flags=lib.A_ROWS_SORTED | lib.C_FP32, out=out, cta_pairs=mode)
    assert int(r.num_tokens_padded.item()) == 0
    assert torch.all(out.cpu() == 7.0)


@pytest.mark.parametrize("mode", MODES)
def test_pairs_rejected_where_they_cannot_run(lib, mode):
    E, N, K = 4, 256, 128
    qw, sc = workloads.draw_weights(E, N, K, seed=55)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))
    x = workloads.draw_activations(20, K, seed=55)
    ids, _ = workloads.draw_routing(20, E, 2, seed=55)
    r64 = lib.moe_align(ids.to(DEV), E, 64)
    with pytest.raises(lib.LibraryError, match="invalid argument"):
        lib.moe_gemm(x.to(DEV), 2, W, r64, cta_pairs=mode)  # 64-token blocks, gathered rows
    r = lib.moe_align(ids.to(DEV), E, 128)
    with pytest.raises(lib.LibraryError, match="invalid argument"):
        lib.moe_gemm(x.to(DEV), 2, W, r, cta_pairs=mode)  # rows not in sorted order
    xs = lib.gather_rows(x.to(DEV), 2, r)
    with pytest.raises(lib.LibraryError, match="invalid argument"):
        lib.moe_gemm(xs, 1, W, r, row_flags=lib.A_ROWS_SORTED, cta_pairs=mode, split_k=2)


def test_planner_default_pairs_long_k_few_tiles(lib):
    """128-token blocks with 4 tiles (N 512) and K 4096: the planner's default is the pair
    schedule.  Its rows match the oracle and, bit for bit, the explicit pair and one-CTA
    schedules (results never depend on the schedule)."""
    T, k, E, N, K = 240, 4, 6, 512, 4096
    assert lib.plan_gemm(T * k, E, N, K, 128, num_sms=148)["cta_pairs"] == 2
    qw, sc, x, ids, W, r, xs, (s, e, ntp) = _case(lib, T, k, E, N, K, 58, True)
    kw = dict(epilogue=1, row_flags=lib.A_ROWS_SORTED)
    dflt = lib.moe_gemm(xs, 1, W, r, **kw).cpu()
    two = lib.moe_gemm(xs, 1, W, r, cta_pairs=2, **kw).cpu()
    one = lib.moe_gemm(xs, 1, W, r, cta_pairs=1, **kw).cpu()
    rows = routed_rows(ids)
    assert torch.equal(bits(dflt[rows]), bits(two[rows]))
    assert torch.equal(bits(dflt[rows]), bits(one[rows]))
    sample = rows[::7]
    ref = oracle.silu_mul(oracle.gemm_rows(x, k, qw, sc, sample.numpy(),
                                           ids.reshape(-1)[sample].numpy().astype("int64"),
                                           out_f32=True))
    assert_close_bf16(dflt[sample], ref, "planner-default pairs, K 4096")
