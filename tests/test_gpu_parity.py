"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on a GB300.

Bit-exact: routing (sorted_ids, expert_ids, num_tokens_padded) and dequantised
weights.  BF16 outputs: |gpu - ref| <= 1e-2*|ref| + 1e-2*rms(ref) per element.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from w4a16_moe_expert_gb300 import workloads
from parity_util import assert_close_bf16, bits, ensure_cuda_lib, routed_rows, sample_tokens

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    return ensure_cuda_lib()


def _ids(T, E_global, k, seed, kind="softmax", E=None, empty=()):
    ids, w = workloads.draw_routing(T, E_global, k, seed, kind, 0, E, empty)
    return ids, w


# ---- align --------------------------------------------------------------------------------

ALIGN_CASES = [
    # (T, k, E_global, E_local, block_m, kind)
    (16, 2, 8, 8, 16, "softmax"),
    (0, 8, 128, 128, 16, "softmax"),
    (1, 8, 384, 48, 16, "softmax"),
    (37, 3, 17, 17, 32, "softmax"),
    (513, 8, 128, 128, 64, "softmax"),
    (4096, 8, 128, 128, 128, "softmax"),
    (16384, 8, 384, 48, 128, "zipf"),
    (8192, 8, 384, 384, 128, "zipf"),
    (1000, 6, 1024, 1024, 16, "softmax"),
    # decode routings of at most 32 slots (sorted by one warp in registers)
    (2, 8, 128, 128, 16, "softmax"),
    (3, 8, 128, 128, 32, "softmax"),
    (4, 8, 128, 128, 64, "softmax"),
    (4, 8, 16, 16, 128, "softmax"),
    (4, 8, 384, 48, 16, "zipf"),
    (31, 1, 4, 4, 16, "softmax"),
]


@pytest.mark.parametrize("T,k,Eg,E,bm,kind", ALIGN_CASES)
def test_align_bit_exact(lib, T, k, Eg, E, bm, kind):
    ids, _ = workloads.draw_routing(T, Eg, k, seed=T + 7 * bm, kind=kind, local_lo=0, E_local=E)
    r = lib.moe_align(ids.to(DEV), E, bm)
    s, e, ntp = oracle.moe_align(ids, E, bm)
    assert int(r.num_tokens_padded.item()) == ntp
    assert torch.equal(r.sorted_ids.cpu(), torch.from_numpy(s))
    assert torch.equal(r.expert_ids.cpu(), torch.from_numpy(e))


def test_align_validation_flags_bad_ids(lib):
    ids, _ = workloads.draw_routing(40, 8, 4, seed=3)
    bad = ids.clone()
    bad[3, 1] = 9
    bad[7, 0] = -5
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    r = lib.moe_align(bad.to(DEV), 8, 16, validate=True, dev_err=err)
    assert int(err.item()) & lib.DEVERR_BAD_EXPERT_ID
    cleaned = bad.clone()
    cleaned[3, 1] = -1
    cleaned[7, 0] = -1
    s, e, ntp = oracle.moe_align(cleaned, 8, 16)
    assert torch.equal(r.sorted_ids.cpu(), torch.from_numpy(s))
    assert int(r.num_tokens_padded.item()) == ntp


@pytest.mark.parametrize("T,k", [(40, 4), (4, 8)])
def test_align_validation_flags_bad_ids_any_size(lib, T, k):
    ids, _ = workloads.draw_routing(T, 8, k, seed=5)
    bad = ids.clone()
    bad[1, 1] = 9
    bad[2, 0] = -5
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    r = lib.moe_align(bad.to(DEV), 8, 16, validate=True, dev_err=err)
    assert int(err.item()) & lib.DEVERR_BAD_EXPERT_ID
    cleaned = bad.clone()
    cleaned[1, 1] = -1
    cleaned[2, 0] = -1
    s, e, ntp = oracle.moe_align(cleaned, 8, 16)
    assert torch.equal(r.sorted_ids.cpu(), torch.from_numpy(s))
    assert torch.equal(r.expert_ids.cpu(), torch.from_numpy(e))
    assert int(r.num_tokens_padded.item()) == ntp
    # without validation nothing is flagged
    err.zero_()
    lib.moe_align(bad.to(DEV), 8, 16, validate=False, dev_err=err)
    assert int(err.item()) == 0


def test_align_runs_twice_identically(lib):
    ids, _ = workloads.draw_routing(3000, 384, 8, seed=11, kind="zipf", E_local=48)
    a = lib.moe_align(ids.to(DEV), 48, 32)
    b = lib.moe_align(ids.to(DEV), 48, 32)
    assert torch.equal(a.sorted_ids, b.sorted_ids) and torch.equal(a.expert_ids, b.expert_ids)


# ---- pack + dequant ---------------------------------------------------------------------------

@pytest.mark.parametrize("E,N,K,paired", [(8, 512, 256, True), (8, 256, 256, False),
                                          (3, 1536, 2048, True), (2, 2048, 768, False)])
def test_debug_dequant_bit_exact(lib, E, N, K, paired):
    qw, sc = workloads.draw_weights(E, N, K, seed=E * 31 + N)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=paired)
    ref = oracle.dequant(qw, sc)
    for e in range(E):
        got = lib.debug_dequant(W, e)
        assert torch.equal(bits(got), bits(ref[e])), f"expert {e}"


def test_dequant_exhaustive_every_code_and_scale(lib):
    # 256 experts x 128 rows x 2 groups = 65536 scale slots, one per BF16 bit pattern;
    # every group of 32 elements holds all 16 codes twice.
    E, N, K = 256, 128, 64
    scales = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(E, N, 2)
    words = torch.tensor([0x76543210, 0xFEDCBA98 - (1 << 32)] * 4, dtype=torch.int64).to(torch.int32)
    qw = words.reshape(1, 1, 8).expand(E, N, 8).contiguous()
    W = lib.pack_weights(qw.to(DEV), scales.contiguous().to(DEV))
    ref = oracle.dequant(qw, scales)
    for e in range(E):
        got = bits(lib.debug_dequant(W, e))
        want = bits(ref[e])
        nan = torch.isnan(ref[e].float())
        assert torch.equal(got[~nan], want[~nan]), f"expert {e}"
        assert torch.isnan(lib.debug_dequant(W, e).float().cpu()[nan]).all()


def test_gemm_one_hot_reads_back_dequantised_weights(lib):
    # x = unit rows: C[t, n] = wd[e][n][t] exactly (one nonzero product per output)
    E, N, K = 3, 256, 128
    qw, sc = workloads.draw_weights(E, N, K, seed=5)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))
    x = torch.eye(K, dtype=torch.bfloat16)
    ref = oracle.dequant(qw, sc)
    for bm in (16, 32, 64, 128):
        for e in range(E):
            ids = torch.full((K, 1), e, dtype=torch.int32)
            r = lib.moe_align(ids.to(DEV), E, bm)
            C = lib.moe_gemm(x.to(DEV), 1, W, r)
            assert torch.equal(bits(C), bits(ref[e].T.contiguous())), f"bm {bm} expert {e}"
            for split in (2, 3):
                C2 = lib.moe_gemm(x.to(DEV), 1, W, r, split_k=split)
                assert torch.equal(bits(C2), bits(ref[e].T.contiguous())), f"split {split}"


# ---- GEMM parity ------------------------------------------------------------------------------

def _gemm_case(lib, T, k, E, N, K, bm, seed, paired=False, empty=(), kind="softmax"):
    qw, sc = workloads.draw_weights(E, N, K, seed=seed)
    x = workloads.draw_activations(T, K, seed=seed)
    ids, _ = workloads.draw_routing(T, E, k, seed=seed, kind=kind, empty_experts=empty)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV), paired=paired)
    r = lib.moe_align(ids.to(DEV), E, bm)
    s, e, ntp = oracle.moe_align(ids, E, bm)
    return qw, sc, x, ids, W, r, (s, e, ntp)


@pytest.mark.parametrize("bm", [16, 32, 64, 128])
def test_gemm_gate_up_parity_tiny(lib, bm):
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 16, 2, 8, 512, 256, bm, 1, empty=(7,))
    C = lib.moe_gemm(x.to(DEV), 2, W, r)
    ref = oracle.moe_gemm(x, 2, qw, sc, s, e, ntp, bm, 32)
    rows = routed_rows(ids)
    assert_close_bf16(C.cpu()[rows], ref[rows], "gate_up")


@pytest.mark.parametrize("paired", [True, False])
def test_gemm_silu_and_none_epilogues_with_paired_layout(lib, paired):
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 40, 4, 6, 512, 512, 16, 2, paired=True)
    rows = routed_rows(ids)
    ref_c = oracle.moe_gemm(x, 4, qw, sc, s, e, ntp, 16, 160)
    # NONE on a paired layout writes canonical column order
    C = lib.moe_gemm(x.to(DEV), 4, W, r)
    assert_close_bf16(C.cpu()[rows], ref_c[rows], "gate_up (paired, NONE)")
    H = lib.moe_gemm(x.to(DEV), 4, W, r, epilogue=lib.EPILOGUE_SILU_MUL)
    ref_h = oracle.silu_mul(oracle.moe_gemm(x, 4, qw, sc, s, e, ntp, 16, 160, out_f32=True))
    assert_close_bf16(H.cpu()[rows], ref_h[rows], "gate_up + SiLU-mul")


def test_gemm_ragged_many_tiles(lib):
    # 300 tokens, top-3 over 37 experts, N=384 (3 tiles), K=448 (7 K blocks), ragged blocks
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 300, 3, 37, 384, 448, 32, 9)
    C = lib.moe_gemm(x.to(DEV), 3, W, r)
    ref = oracle.moe_gemm(x, 3, qw, sc, s, e, ntp, 32, 900, threads=4)
    rows = routed_rows(ids)
    assert_close_bf16(C.cpu()[rows], ref[rows], "ragged gemm")


@pytest.mark.parametrize("split", [1, 2, 4, 7])
def test_gemm_split_k_parity_and_determinism(lib, split):
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 8, 8, 128, 1536, 2048, 16, 21)
    ref = oracle.moe_gemm(x, 8, qw, sc, s, e, ntp, 16, 64, threads=4)
    rows = routed_rows(ids)
    C1 = lib.moe_gemm(x.to(DEV), 8, W, r, split_k=split)
    C2 = lib.moe_gemm(x.to(DEV), 8, W, r, split_k=split)
    assert_close_bf16(C1.cpu()[rows], ref[rows], f"split {split}")
    assert torch.equal(bits(C1), bits(C2)), "same schedule must be bitwise reproducible"


@pytest.mark.parametrize("epilogue", [0, 1])
def test_gemm_device_picked_split_for_few_long_tiles(lib, epilogue):
    # One routed row on a wide, long-K weight: 32 tiles of K = 6144 leave most SMs idle, so the
    # device slices K until the units fill one wave (at most 8 slices of >= 24 K blocks).  The
    # result matches the oracle and, bit for bit, the same split fixed by the schedule.
    E, N, K = 4, 4096, 6144
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 1, 1, E, N, K, 16, 41, paired=True)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units1 = (ntp // 16) * (N // 128)
    split = min(8, sms // units1)
    while split > 1 and K // 64 < 24 * split:
        split -= 1
    assert split > 1
    auto = lib.moe_gemm(x.to(DEV), 1, W, r, epilogue=epilogue)
    fixed = lib.moe_gemm(x.to(DEV), 1, W, r, epilogue=epilogue, split_k=split, num_ctas=sms)
    ref = oracle.moe_gemm(x, 1, qw, sc, s, e, ntp, 16, 1, out_f32=bool(epilogue))
    if epilogue:
        ref = oracle.silu_mul(ref)
    assert_close_bf16(auto.cpu(), ref, f"device-picked split ({split})")
    assert torch.equal(bits(auto), bits(fixed))


def test_gemm_units_filling_the_grid_are_not_split(lib):
    # 64 tokens x 8 slots over 128 experts: hundreds of (block, tile) units, so no K split
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 64, 8, 128, 1536, 2048, 16, 42)
    auto = lib.moe_gemm(x.to(DEV), 8, W, r)
    one = lib.moe_gemm(x.to(DEV), 8, W, r, split_k=1,
                       num_ctas=torch.cuda.get_device_properties(0).multi_processor_count)
    assert torch.equal(bits(auto), bits(one))


def test_gemm_grid_sizes_do_not_change_results(lib):
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 64, 8, 128, 512, 512, 16, 23)
    outs = [lib.moe_gemm(x.to(DEV), 8, W, r, num_ctas=n, split_k=1) for n in (1, 7, 64, 1000)]
    for o in outs[1:]:
        assert torch.equal(bits(o), bits(outs[0]))


def test_gemm_sorted_rows_modes(lib):
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 20, 2, 4, 256, 256, 16, 31)
    ref = oracle.moe_gemm(x, 2, qw, sc, s, e, ntp, 16, 40)
    Cs = lib.moe_gemm(x.to(DEV), 2, W, r, row_flags=lib.C_ROWS_SORTED).cpu()
    for p in range(ntp):
        i = int(s[p])
        if i < 40:
            assert torch.equal(bits(Cs[p]), bits(lib.moe_gemm(x.to(DEV), 2, W, r).cpu()[i]))
        else:
            assert torch.all(Cs[p].float() == 0)
    # A rows already in sorted order: gather x rows by hand
    xs = torch.zeros((r.capacity, 256), dtype=torch.bfloat16)
    for p in range(ntp):
        i = int(s[p])
        if i < 40:
            xs[p] = x[i // 2]
    C2 = lib.moe_gemm(xs.to(DEV), 1, W, r, row_flags=lib.A_ROWS_SORTED)
    rows = routed_rows(ids)
    assert_close_bf16(C2.cpu()[rows], ref[rows], "A rows sorted")


def test_gather_rows_bit_exact_and_sorted_gemm(lib):
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 50, 4, 8, 256, 512, 32, 33)
    xs = lib.gather_rows(x.to(DEV), 4, r).cpu()
    for p in range(ntp):
        i = int(s[p])
        if i < 200:
            assert torch.equal(bits(xs[p]), bits(x[i // 4]))
    C = lib.moe_gemm(xs.to(DEV), 1, W, r, row_flags=lib.A_ROWS_SORTED)
    ref = oracle.moe_gemm(x, 4, qw, sc, s, e, ntp, 32, 200)
    rows = routed_rows(ids)
    assert_close_bf16(C.cpu()[rows], ref[rows], "gathered + sorted-row GEMM")


def test_gemm_edge_cases(lib):
    E, N, K = 4, 128, 128
    qw, sc = workloads.draw_weights(E, N, K, seed=41)
    W = lib.pack_weights(qw.to(DEV), sc.to(DEV))
    # all slots dropped: nothing written
    ids = torch.full((5, 2), -1, dtype=torch.int32)
    r = lib.moe_align(ids.to(DEV), E, 16)
    assert int(r.num_tokens_padded.item()) == 0
    C = torch.full((10, N), 7.0, dtype=torch.bfloat16, device=DEV)
    lib.moe_gemm(torch.zeros((5, K), dtype=torch.bfloat16, device=DEV), 2, W, r, out=C)
    assert torch.all(C.float() == 7.0)
    # one expert receives every row (max rows for one expert)
    x = workloads.draw_activations(700, K, seed=42)
    ids = torch.full((700, 1), 2, dtype=torch.int32)
    r = lib.moe_align(ids.to(DEV), E, 128)
    C = lib.moe_gemm(x.to(DEV), 1, W, r)
    wd = oracle.dequant(qw, sc)[2]
    assert_close_bf16(C.cpu(), torch.matmul(x.float(), wd.float().T).to(torch.bfloat16), "one expert")
    # all-zero codes (q = 8) give exact zeros
    q8 = torch.full_like(qw, int(np.uint32(0x88888888).view(np.int32)))
    W8 = lib.pack_weights(q8.to(DEV), sc.to(DEV))
    assert torch.all(lib.moe_gemm(x.to(DEV), 1, W8, r).float() == 0)


def test_dev_err_stays_clear_and_bad_descriptors_rejected(lib):
    qw, sc, x, ids, W, r, _ = _gemm_case(lib, 16, 2, 8, 256, 256, 16, 51)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.moe_gemm(x.to(DEV), 2, W, r, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    W.desc.magic ^= 1
    with pytest.raises(lib.LibraryError):
        lib.moe_gemm(x.to(DEV), 2, W, r)
    W.desc.magic ^= 1
    with pytest.raises(lib.LibraryError):  # SiLU-and-mul needs a paired layout
        lib.moe_gemm(x.to(DEV), 2, W, r, epilogue=lib.EPILOGUE_SILU_MUL)


def test_gemm_fp32_output_mode(lib):
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, 24, 4, 8, 384, 512, 32, 61)
    ref = oracle.moe_gemm(x, 4, qw, sc, s, e, ntp, 32, 96, out_f32=True)
    C = lib.moe_gemm(x.to(DEV), 4, W, r, row_flags=lib.C_FP32)
    assert C.dtype == torch.float32
    rows = routed_rows(ids)
    g, rf = C.cpu()[rows], ref[rows]
    rms = float(rf.pow(2).mean().sqrt())
    assert float((g - rf).abs().max()) <= 1e-3 * rms  # FP32 sums in another order
    assert torch.equal(bits(C.to(torch.bfloat16)), bits(lib.moe_gemm(x.to(DEV), 4, W, r)))


@pytest.mark.parametrize("bm", [16, 128])
@pytest.mark.parametrize("K", [64, 128, 192, 320])
def test_sorted_rows_shorter_than_a_stage(lib, bm, K):
    # sorted activation rows come as one tensor copy per pipeline stage (4 K blocks of 64 at
    # 16-token blocks, 2 at 128-token blocks); K shorter than a stage, or a short last stage,
    # makes the copy reach past K (those blocks are zero-filled and not multiplied)
    T, k, E, N = 48, 4, 6, 256
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, T, k, E, N, K, bm, 70 + K)
    xs = lib.gather_rows(x.to(DEV), k, r)
    C = lib.moe_gemm(xs, 1, W, r, row_flags=lib.A_ROWS_SORTED | lib.C_FP32).cpu()
    ref = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, bm, T * k, out_f32=True)
    rows = routed_rows(ids)
    g, rf = C[rows], ref[rows]
    rms = float(rf.pow(2).mean().sqrt())
    assert float((g - rf).abs().max()) <= 1e-3 * rms, f"bm {bm}, K {K}"  # FP32 sums


@pytest.mark.parametrize("split", [2, 3, 5])
def test_sorted_rows_with_k_slices(lib, split):
    # K = 768 (12 blocks, three 4-block stages) cut into slices that end inside a stage: the
    # stage's copy loads blocks past the slice end, which the slice must not multiply
    T, k, E, N, K = 40, 4, 6, 256, 768
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, T, k, E, N, K, 16, 80 + split)
    xs = lib.gather_rows(x.to(DEV), k, r)
    flags = lib.A_ROWS_SORTED | lib.C_FP32
    whole = lib.moe_gemm(xs, 1, W, r, row_flags=flags, split_k=1).cpu()
    sliced = lib.moe_gemm(xs, 1, W, r, row_flags=flags, split_k=split).cpu()
    ref = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 16, T * k, out_f32=True)
    rows = routed_rows(ids)
    rms = float(ref[rows].pow(2).mean().sqrt())
    assert float((sliced[rows] - ref[rows]).abs().max()) <= 1e-3 * rms, f"split {split}"
    assert float((sliced[rows] - whole[rows]).abs().max()) <= 1e-3 * rms  # FP32 sums, other order


# ---- top-k sum and the whole layer --------------------------------------------------------------

def test_topk_sum_parity(lib):
    rng = np.random.default_rng(8)
    T, k, H = 33, 8, 2048
    Y = torch.from_numpy(rng.standard_normal((T * k, H)).astype(np.float32) * 10)
    ids = torch.from_numpy(rng.integers(-1, 5, (T, k)).astype(np.int32))
    w = torch.from_numpy(rng.random((T, k)).astype(np.float32))
    out = lib.topk_sum(Y.to(DEV), ids.to(DEV), w.to(DEV))
    assert_close_bf16(out.cpu(), oracle.topk_sum(Y, ids, w), "topk_sum")


def _layer_gpu(lib, inp, E_global=0, block_m=0, packed=None):
    if packed is None:
        packed = (lib.pack_weights(inp.w13_q.to(DEV), inp.w13_s.to(DEV), paired=True),
                  lib.pack_weights(inp.w2_q.to(DEV), inp.w2_s.to(DEV)))
    w13, w2 = packed
    return lib.moe_layer(inp.x.to(DEV), w13, w2, inp.topk_ids.to(DEV), inp.topk_weights.to(DEV),
                         E_global=E_global, block_m=block_m)


@pytest.mark.parametrize("block_m", [0, 16, 32, 64, 128])
def test_layer_tiny(lib, block_m):
    inp = workloads.draw_layer(workloads.WORKLOADS["tiny"], 16)
    out = _layer_gpu(lib, inp, block_m=block_m)
    ref = oracle.moe_layer(inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, inp.topk_ids,
                           inp.topk_weights)
    assert_close_bf16(out.cpu(), ref, "tiny layer")
    out2 = _layer_gpu(lib, inp, block_m=block_m)
    assert torch.equal(bits(out), bits(out2))


@pytest.fixture(scope="module")
def qwen_weights(lib):
    wl = workloads.WORKLOADS["qwen3_30b_a3b"]
    w = workloads.draw_layer_weights(wl)
    packed = (lib.pack_weights(w[0].to(DEV), w[1].to(DEV), paired=True),
              lib.pack_weights(w[2].to(DEV), w[3].to(DEV)))
    return wl, w, packed


@pytest.mark.parametrize("T", [1, 8, 64, 512, 4096])
def test_layer_qwen3_sampled_tokens(lib, qwen_weights, T):
    wl, w, packed = qwen_weights
    inp = workloads.draw_layer(wl, T, weights=w)
    out = _layer_gpu(lib, inp, packed=packed).cpu()
    # each token's output depends only on its own routing: check a sample of tokens exactly
    tok = sample_tokens(T, 24, seed=T)
    sub = torch.from_numpy(tok)
    ref = oracle.moe_layer_parallel(inp.x[sub], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                                    inp.topk_ids[sub], inp.topk_weights[sub])
    assert_close_bf16(out[sub], ref, f"qwen3 layer T={T}")


@pytest.mark.parametrize("name,T", [("kimi_k2_ep8_decode", 1), ("kimi_k2_ep8_decode", 256),
                                    ("kimi_k2_ep8_prefill", 2048), ("kimi_k2_tp8", 32),
                                    ("kimi_k2_tp8_zipf", 1024)])
def test_layer_kimi_sampled_tokens(lib, name, T):
    wl = workloads.WORKLOADS[name]
    inp = workloads.draw_layer(wl, T)
    out = _layer_gpu(lib, inp, E_global=wl.E_global).cpu()
    tok = sample_tokens(T, 6, seed=T)
    sub = torch.from_numpy(tok)
    ref = oracle.moe_layer_parallel(inp.x[sub], inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s,
                                    inp.topk_ids[sub], inp.topk_weights[sub])
    assert_close_bf16(out[sub], ref, f"{name} T={T}")
    none_local = (inp.topk_ids < 0).all(dim=1)
    assert torch.all(out[none_local].float() == 0)


@pytest.mark.parametrize("bm,split", [(16, 1), (32, 1), (64, 1), (128, 1), (16, 3), (128, 2)])
def test_gemm_fp32_sorted_rows_equal_slot_rows(lib, bm, split):
    # FP32 sums in sorted rows: the same values, bit for bit, as FP32 rows by slot; padding
    # positions are zeros, rows past the last block untouched
    T, k, E, N, K = 90, 4, 9, 768, 512
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, T, k, E, N, K, bm, 71)
    xs = lib.gather_rows(x.to(DEV), k, r)
    flags = lib.A_ROWS_SORTED | lib.C_FP32
    by_slot = lib.moe_gemm(xs, 1, W, r, row_flags=flags, split_k=split).cpu()
    out = torch.full((r.capacity, N), float("nan"), dtype=torch.float32, device=DEV)
    lib.moe_gemm(xs, 1, W, r, row_flags=flags | lib.C_ROWS_SORTED, out=out, split_k=split)
    got = out.cpu()
    for p in range(ntp):
        i = int(s[p])
        if i < T * k:
            assert torch.equal(got[p].view(torch.int32), by_slot[i].view(torch.int32)), p
        else:
            assert torch.all(got[p] == 0), p
    assert torch.isnan(got[ntp:]).all()
    ref = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, bm, T * k, out_f32=True)
    rows = routed_rows(ids)
    assert_close_bf16(by_slot[rows], ref[rows], f"FP32 rows bm={bm} split={split}")


@pytest.mark.parametrize("epilogue,flags", [(0, 0), (1, 0), (0, 4)])
def test_gemm_last_partial_wave_sliced(lib, epilogue, flags):
    # 4 blocks x 12 tiles = 48 units on 40 CTAs: one full wave of whole tiles, then the last 8
    # tiles cut into K slices (4 of 24 K blocks each, summed in slice order by the tile's last
    # CTA) so the partial wave fills the grid.  Checked against the oracle; two calls are
    # bitwise equal, and the tiles of the full wave equal the unsliced schedule bit for bit.
    T, k, E, N, K = 8, 4, 4, 1536, 6144
    qw, sc, x, ids, W, r, (s, e, ntp) = _gemm_case(lib, T, k, E, N, K, 16, 81, paired=bool(epilogue))
    assert ntp // 16 == 4
    kw = dict(epilogue=epilogue, row_flags=flags, num_ctas=40)
    a = lib.moe_gemm(x.to(DEV), k, W, r, **kw).cpu()
    b = lib.moe_gemm(x.to(DEV), k, W, r, **kw).cpu()
    whole = lib.moe_gemm(x.to(DEV), k, W, r, split_k=1, **kw).cpu()
    f32 = bool(flags & lib.C_FP32)
    view = (lambda t: t.view(torch.int32)) if f32 else bits
    assert torch.equal(view(a), view(b))
    ref = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 16, T * k, out_f32=bool(epilogue) or f32,
                          threads=4)
    if epilogue:
        ref = oracle.silu_mul(ref)
    rows = routed_rows(ids)
    assert_close_bf16(a[rows], ref[rows], "sliced last wave")
    # the sliced tiles really were summed in a different order somewhere
    assert not torch.equal(view(a), view(whole))
    # units 0..39 are whole tiles: blocks 0..2 (tiles 0..35) and block 3's tiles 0..3
    tile_cols = 64 if epilogue else 128
    first_tiles = 4  # of block 3
    for p in range(ntp):
        i = int(s[p])
        if i >= T * k:
            continue
        blk = p // 16
        if blk < 3:
            assert torch.equal(view(a[i]), view(whole[i])), (p, i)
        else:
            if epilogue:
                # paired SiLU output: tile j writes columns 64j .. 64j + 63
                cols = slice(0, first_tiles * tile_cols)
            else:
                cols = slice(0, first_tiles * tile_cols)
            assert torch.equal(view(a[i, cols]), view(whole[i, cols])), (p, i)
