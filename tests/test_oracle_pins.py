"""Pins for the CPU oracle: each check ties it to something other than itself.

Kinds of pin used here: the worked product printed on the pages (golden
fixture), a hand-worked routing example, exhaustive enumeration (every uint4
code times every BF16 scale bit pattern), library routines (torch's
float->bf16 conversion, torch.matmul, scipy's logistic function), brute force
on tiny inputs written independently in numpy/Python, and invariants that a
dropped term, a wrong sign or index, or a transposed operand would break.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from w4a16_moe_expert_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- independent helpers (numpy / torch only) -------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def unpack_codes_np(qweight: np.ndarray) -> np.ndarray:
    """uint4 codes [..., K] from int32 words [..., K/8], low nibble first."""
    w = qweight.view(np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    codes = (w[..., None] >> shifts) & 0xF
    return codes.reshape(*w.shape[:-1], w.shape[-1] * 8).astype(np.int64)


def dequant_np(qweight, scales) -> np.ndarray:
    """Independent dequant: float64 product, BF16 by torch's RNE, as float64."""
    q = unpack_codes_np(np.asarray(qweight))
    s = bf16_bits_to_f64(np.asarray(scales).view(np.uint16))
    s_full = np.repeat(s, 32, axis=-1)
    prod = (q - 8).astype(np.float64) * s_full
    return bf16_bits_to_f64(torch_bf16_bits(prod.astype(np.float32)))


def bf16_np(t: torch.Tensor) -> np.ndarray:
    return bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


# ---- BF16 rounding helpers -------------------------------------------------------

def test_float_to_bf16_matches_torch_rne():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        (rng.standard_normal(200_000) * 10.0 ** rng.integers(-30, 30, 200_000)).astype(np.float32),
        rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 1e-40, -1e-45], np.float32),
    ])
    ours = oracle.float_to_bf16_bits(x)
    ref = torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(bf16_bits_to_f64(ours[nan])))


def _nearest_even_bf16(x: float) -> int:
    """Brute force: the BF16 bit pattern nearest to x (ties to even mantissa)."""
    f = Fraction(x)
    cand = torch_bf16_bits(np.array([x], np.float32))[0]  # a near neighbour to start from
    best = None
    for d in range(-2, 3):
        b = int(cand) + d
        if not 0 <= b < 0x10000:
            continue
        v = bf16_bits_to_f64(np.array([b], np.uint16))[0]
        if not math.isfinite(v):
            continue
        err = abs(Fraction(v) - f)
        key = (err, b & 1)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def test_double_to_bf16_is_single_rounding():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(3000) * 10.0 ** rng.integers(-20, 20, 3000)
    # values just off a BF16 tie, where double->float->bf16 would round twice
    ties = np.array([1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 2.0 ** -8 - 2.0 ** -40,
                     -(3.0 + 2.0 ** -7 + 2.0 ** -35), 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8])
    subnormal = rng.standard_normal(500) * 2.0 ** -128  # BF16 subnormal range (quantum 2^-133)
    x = np.concatenate([x, subnormal, ties])
    ours = oracle.double_to_bf16_bits(x)
    for xi, oi in zip(x, ours):
        assert oi == _nearest_even_bf16(float(xi)), xi
    # the first tie-breaker case: a float round trip would give 1.0 (0x3f80)
    assert ours[-5] == 0x3f81 and ours[-4] == 0x3f80
    assert ours[-2] == 0x3f80 and ours[-1] == 0x3f82


# ---- dequant ----------------------------------------------------------------------

def test_dequant_worked_product_from_the_pages():
    # humans& page, "BF16 preserves each local product": 1.5 * 1.125 = 1.6875, exact in BF16.
    with open(os.path.join(GOLDEN, "bf16_exact_product.txt")) as f:
        row = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")][0]
    a, b, prod, pbits = float(row[0]), float(row[1]), float(row[2]), int(row[3], 16)
    assert a * b == prod
    # the same product as a uint4 dequant: (q - 8) * s with q - 8 = 3 and s = 1.125 / 2
    q = np.zeros((1, 1), np.int32)
    q[0, 0] = 11  # element 0 holds code 11, the others code 0
    s = torch.tensor([[b / 2]], dtype=torch.bfloat16)
    w = oracle.dequant(torch.from_numpy(q), s)
    assert bits(w)[0, 0] == pbits
    assert float(w[0, 0]) == prod


def test_dequant_exhaustive_codes_times_every_bf16_scale():
    # every scale bit pattern; each row holds the 16 codes twice (32 elements, one group)
    scales = np.arange(65536, dtype=np.uint16).reshape(65536, 1)
    word_lo = np.uint32(0x76543210)
    word_hi = np.uint32(0xFEDCBA98)
    q = np.tile(np.array([word_lo, word_hi, word_lo, word_hi], np.uint32), (65536, 1)).view(np.int32)
    out = bits(oracle.dequant(torch.from_numpy(q), torch.from_numpy(scales.view(np.int16)).view(torch.bfloat16)))
    codes = np.tile(np.arange(16), 2)
    s = bf16_bits_to_f64(scales[:, 0])
    with np.errstate(invalid="ignore", over="ignore"):
        prod64 = (codes[None, :] - 8).astype(np.float64) * s[:, None]
        prod32 = prod64.astype(np.float32)
    in_range = np.isfinite(prod64) & (np.abs(prod64) <= np.finfo(np.float32).max)
    assert np.array_equal(prod32[in_range].astype(np.float64), prod64[in_range])  # exact in FP32
    ref = torch_bf16_bits(prod32)
    nan = np.isnan(prod64)
    assert np.array_equal(out[~nan], ref[~nan])
    assert np.all(np.isnan(bf16_bits_to_f64(out[nan])))
    # code 8 is zero for every finite scale
    fin_s = np.isfinite(s)
    assert np.all(bf16_bits_to_f64(out[fin_s][:, 8]) == 0.0)


def test_dequant_nibble_order_low_first():
    # word 0x76543210 holds codes 0..7 for elements 0..7; s = 1 -> values -8..-1
    q = np.array([[0x76543210, 0x0FEDCBA9]], np.uint32).view(np.int32)
    s = torch.ones((1, 1), dtype=torch.bfloat16)
    w = oracle.dequant(torch.from_numpy(q.copy()), s)
    want = [c - 8 for c in range(8)] + [c - 8 for c in (9, 10, 11, 12, 13, 14, 15, 0)]
    assert [float(v) for v in w[0]] == want


def test_dequant_matches_independent_numpy_on_random_weights():
    qw, sc = workloads.draw_weights(3, 40, 128, seed=7)
    ours = bf16_np(oracle.dequant(qw, sc))
    ref = dequant_np(qw.numpy(), sc.view(torch.int16).numpy())
    assert np.array_equal(ours, ref)


# ---- align --------------------------------------------------------------------------

def _align_brute(ids: np.ndarray, E: int, bm: int):
    """Per-expert scan that appends slots in order (no counting sort)."""
    flat = ids.reshape(-1)
    n = flat.size
    sorted_ids, expert_ids = [], []
    for e in range(E):
        rows = [i for i in range(n) if flat[i] == e]
        if not rows:
            continue
        nb = -(-len(rows) // bm)
        rows += [n] * (nb * bm - len(rows))
        sorted_ids += rows
        expert_ids += [e] * nb
    return sorted_ids, expert_ids, len(sorted_ids)


def test_align_hand_worked_example():
    vals = {}
    with open(os.path.join(GOLDEN, "align_hand_example.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, *v = ln.split()
                vals[k] = [int(x) for x in v]
    T, k, E, bm = vals["T"][0], vals["top_k"][0], vals["E"][0], vals["block_m"][0]
    ids = np.array(vals["topk_ids"], np.int32).reshape(T, k)
    assert oracle.align_capacity(T, k, E, bm) == vals["capacity"][0]
    s, e, ntp = oracle.moe_align(ids, E, bm)
    assert s.tolist() == vals["sorted_ids"]
    assert e.tolist() == vals["expert_ids"]
    assert ntp == vals["num_tokens_padded"][0]


@pytest.mark.parametrize("seed", range(12))
def test_align_brute_force_and_invariants(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(0, 40))
    k = int(rng.integers(1, 5))
    E = int(rng.integers(1, 9))
    bm = int(rng.choice([1, 2, 3, 4, 8, 16]))
    ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    s, e, ntp = oracle.moe_align(ids, E, bm)
    bs, be, bntp = _align_brute(ids, E, bm)
    assert ntp == bntp
    assert s[:ntp].tolist() == bs
    assert e[: ntp // bm].tolist() == be
    n = T * k
    cap = s.size
    assert cap % bm == 0 and ntp <= cap and ntp % bm == 0
    assert np.all(s[ntp:] == n) and np.all(e[ntp // bm:] == -1)
    valid = s[s < n]
    flat = ids.reshape(-1)
    assert sorted(valid.tolist()) == [i for i in range(n) if flat[i] >= 0]  # each slot once
    for b in range(ntp // bm):  # every row of a block belongs to its expert
        blk = s[b * bm:(b + 1) * bm]
        assert np.all(flat[blk[blk < n]] == e[b])
        assert np.any(blk < n)  # no all-padding block: empty experts give no rows
    for ex in range(E):
        if not np.any(flat == ex):
            assert ex not in e.tolist()


def test_align_rejects_bad_ids_and_small_capacity():
    with pytest.raises(ValueError):
        oracle.moe_align(np.array([[5]], np.int32), 3, 4)
    with pytest.raises(ValueError):
        oracle.moe_align(np.array([[0, 1]], np.int32), 2, 4, capacity=4)


# ---- gemm ---------------------------------------------------------------------------

def _tiny_problem(seed, T=12, k=2, E=4, N=48, K=96, empty=()):
    qw, sc = workloads.draw_weights(E, N, K, seed=seed)
    x = workloads.draw_activations(T, K, seed=seed)
    ids, w = workloads.draw_routing(T, E, k, seed=seed, empty_experts=empty)
    return qw, sc, x, ids, w


def test_gemm_single_expert_equals_torch_matmul():
    qw, sc = workloads.draw_weights(1, 64, 256, seed=3)
    x = workloads.draw_activations(20, 256, seed=3)
    ids = torch.zeros((20, 1), dtype=torch.int32)
    s, e, ntp = oracle.moe_align(ids, 1, 16)
    C = oracle.moe_gemm(x, 1, qw, sc, s, e, ntp, 16, 20)
    wd = oracle.dequant(qw, sc)[0]
    ref = torch.matmul(x.float(), wd.float().T)  # library GEMM in FP32
    ours = C.float()
    err = (ours - ref).abs()
    assert torch.all(err <= torch.from_numpy(ulp_bf16(ref.numpy())).float() * 1.0 + 1e-6)
    assert (ours == ref.to(torch.bfloat16).float()).float().mean() > 0.97


def test_gemm_brute_force_per_token_without_align():
    qw, sc, x, ids, _ = _tiny_problem(5, empty=(3,))
    T, k = ids.shape
    s, e, ntp = oracle.moe_align(ids, 4, 4)
    C = bf16_np(oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 4, T * k))
    wd = dequant_np(qw.numpy(), sc.view(torch.int16).numpy())
    xa = bf16_np(x)
    for t in range(T):
        for j in range(k):
            ex = int(ids[t, j])
            ref = wd[ex] @ xa[t]  # float64 sum of exact products
            got = C[t * k + j]
            assert np.all(np.abs(got - ref) <= ulp_bf16(ref) + 1e-12)


def test_gemm_one_hot_rows_read_back_dequantised_weights_exactly():
    E, N, K = 3, 32, 64
    qw, sc = workloads.draw_weights(E, N, K, seed=11)
    x = torch.eye(K, dtype=torch.bfloat16)  # token t = unit vector e_t
    for ex in range(E):
        ids = torch.full((K, 1), ex, dtype=torch.int32)
        s, e, ntp = oracle.moe_align(ids, E, 16)
        C = oracle.moe_gemm(x, 1, qw, sc, s, e, ntp, 16, K)
        wd = oracle.dequant(qw, sc)[ex]
        assert np.array_equal(bits(C), bits(wd.T.contiguous()))


def test_gemm_invariants():
    qw, sc, x, ids, _ = _tiny_problem(9)
    T, k = ids.shape
    s, e, ntp = oracle.moe_align(ids, 4, 8)
    base = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 8, T * k)
    # all codes 8 -> zero output
    q8 = torch.full_like(qw, int(np.uint32(0x88888888).view(np.int32)))
    assert torch.all(oracle.moe_gemm(x, k, q8, sc, s, e, ntp, 8, T * k).float() == 0)
    # x = 0 -> zero output
    assert torch.all(oracle.moe_gemm(torch.zeros_like(x), k, qw, sc, s, e, ntp, 8, T * k).float() == 0)
    # doubling every scale doubles every output exactly
    dbl = oracle.moe_gemm(x, k, qw, (sc.float() * 2).to(torch.bfloat16), s, e, ntp, 8, T * k)
    assert torch.equal(dbl.float(), base.float() * 2)
    # permuting tokens (routing alongside) permutes the output rows, bit for bit
    perm = torch.from_numpy(np.random.default_rng(2).permutation(T))
    ids_p = ids[perm]
    s2, e2, ntp2 = oracle.moe_align(ids_p, 4, 8)
    out_p = oracle.moe_gemm(x[perm], k, qw, sc, s2, e2, ntp2, 8, T * k)
    slot_perm = (perm[:, None] * k + torch.arange(k)[None, :]).reshape(-1)
    assert torch.equal(bits_t(out_p), bits_t(base[slot_perm]))


def bits_t(t):
    return t.contiguous().view(torch.int16)


def test_gemm_rows_matches_indexed_gemm():
    qw, sc, x, ids, _ = _tiny_problem(13)
    T, k = ids.shape
    s, e, ntp = oracle.moe_align(ids, 4, 4)
    C = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 4, T * k)
    slots = np.arange(T * k)
    rows = oracle.gemm_rows(x, k, qw, sc, slots, ids.reshape(-1).numpy())
    assert torch.equal(bits_t(rows), bits_t(C))


def test_gemm_rows_fp32_within_the_sequential_summation_bound():
    # FP32 rows against an exact float64 dot of the same BF16 operands: a left-to-right FP32
    # sum of K exactly representable products is within (K - 1) * 2^-24 * sum|p| of the truth;
    # rounded to BF16 they are the BF16 rows bit for bit; host threads change nothing
    qw, sc, x, ids, _ = _tiny_problem(23, T=12, E=4)
    T, k = ids.shape
    slots = np.arange(T * k)
    experts = ids.reshape(-1).numpy()
    r32 = oracle.gemm_rows(x, k, qw, sc, slots, experts, out_f32=True)
    r16 = oracle.gemm_rows(x, k, qw, sc, slots, experts)
    assert r32.dtype == torch.float32
    assert torch.equal(bits_t(r32.to(torch.bfloat16)), bits_t(r16))
    wd = dequant_np(qw.numpy(), sc.view(torch.int16).numpy())
    xa = bf16_np(x)
    K = xa.shape[1]
    for i in range(T * k):
        prods = wd[experts[i]] * xa[i // k][None, :]
        exact = prods.sum(axis=1)
        bound = (K - 1) * 2.0 ** -24 * np.abs(prods).sum(axis=1)
        assert np.all(np.abs(r32[i].numpy().astype(np.float64) - exact) <= bound + 1e-30)
    r32t = oracle.gemm_rows(x, k, qw, sc, slots, experts, out_f32=True, threads=5)
    assert torch.equal(r32t, r32)


def test_gemm_fp32_output_rounds_to_the_bf16_output():
    qw, sc, x, ids, _ = _tiny_problem(19)
    T, k = ids.shape
    s, e, ntp = oracle.moe_align(ids, 4, 4)
    c16 = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 4, T * k)
    c32 = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 4, T * k, out_f32=True)
    assert c32.dtype == torch.float32
    assert torch.equal(bits_t(c32.to(torch.bfloat16)), bits_t(c16))


def test_gemm_threaded_partition_is_identical():
    qw, sc, x, ids, _ = _tiny_problem(17, T=30, E=4)
    T, k = ids.shape
    s, e, ntp = oracle.moe_align(ids, 4, 4)
    a = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 4, T * k, threads=1)
    b = oracle.moe_gemm(x, k, qw, sc, s, e, ntp, 4, T * k, threads=3)
    assert torch.equal(bits_t(a), bits_t(b))


# ---- silu_mul and topk_sum ---------------------------------------------------------

def test_silu_mul_against_scipy_and_odd_identity():
    from scipy.special import expit
    rng = np.random.default_rng(4)
    g = torch.from_numpy(rng.standard_normal(4000).astype(np.float32) * 4).to(torch.bfloat16)
    u = torch.from_numpy(rng.standard_normal(4000).astype(np.float32)).to(torch.bfloat16)
    C = torch.stack([g, u], dim=1)  # rows of [gate | up] with I = 1
    h = bf16_np(oracle.silu_mul(C))[:, 0]
    gf, uf = bf16_np(g), bf16_np(u)
    ref = gf * expit(gf) * uf
    assert np.all(np.abs(h - ref) <= 0.5 * ulp_bf16(ref) + 1e-30)
    # silu(x) - silu(-x) = x (sigma(x) + sigma(-x) = 1); with up = 1
    one = torch.ones_like(g)
    hp = bf16_np(oracle.silu_mul(torch.stack([g, one], 1)))[:, 0]
    hn = bf16_np(oracle.silu_mul(torch.stack([-g, one], 1)))[:, 0]
    assert np.all(np.abs((hp - hn) - gf) <= ulp_bf16(hp) + ulp_bf16(hn))
    # silu(0) = 0
    z = torch.zeros((1, 2), dtype=torch.bfloat16)
    assert float(oracle.silu_mul(z)[0, 0]) == 0.0
    # FP32 gate/up sums (not BF16 values) are used as they are: one rounding, of h
    g32 = (rng.standard_normal(4000) * 4).astype(np.float32)
    u32 = rng.standard_normal(4000).astype(np.float32)
    h32 = bf16_np(oracle.silu_mul(torch.from_numpy(np.stack([g32, u32], 1))))[:, 0]
    g64, u64 = g32.astype(np.float64), u32.astype(np.float64)
    ref32 = g64 * expit(g64) * u64
    assert np.all(np.abs(h32 - ref32) <= 0.5 * ulp_bf16(ref32) + 1e-30)
    # a gate/up pair that BF16 would move: the unrounded up value decides h
    gu = torch.tensor([[1.0, 1.00390625 + 2.0 ** -10]], dtype=torch.float32)  # up between two BF16s
    assert float(oracle.silu_mul(gu)[0, 0]) == float(torch.tensor(
        0.7310585786300049 * (1.00390625 + 2.0 ** -10)).to(torch.bfloat16))


def test_topk_sum_brute_force_and_special_cases():
    rng = np.random.default_rng(6)
    T, k, H = 7, 3, 20
    Y = torch.from_numpy(rng.standard_normal((T * k, H)).astype(np.float32)).to(torch.bfloat16)
    ids = torch.from_numpy(rng.integers(-1, 4, (T, k)).astype(np.int32))
    w = torch.from_numpy(rng.random((T, k)).astype(np.float32))
    out = bf16_np(oracle.topk_sum(Y, ids, w))
    yf = bf16_np(Y)
    for t in range(T):
        for c in range(H):
            acc = Fraction(0)
            for s in range(k):
                if ids[t, s] >= 0:
                    acc += Fraction(float(w[t, s])) * Fraction(float(yf[t * k + s, c]))
            assert out[t, c] == _round_bf16_exact(acc)
    # one-hot weights pick a row exactly; all slots dropped -> zeros
    ids1 = torch.zeros((T, k), dtype=torch.int32)
    w1 = torch.zeros((T, k))
    w1[:, 1] = 1.0
    sel = oracle.topk_sum(Y, ids1, w1)
    assert torch.equal(bits_t(sel), bits_t(Y.view(T, k, H)[:, 1]))
    dropped = oracle.topk_sum(Y, torch.full((T, k), -1, dtype=torch.int32), w)
    assert torch.all(dropped.float() == 0)


def _round_bf16_exact(v: Fraction) -> float:
    """Nearest BF16 to an exact rational (ties to even), as a float."""
    if v == 0:
        return 0.0
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = math.floor(math.log2(a)) if a > 0 else 0
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = max(e - 7, -133)
    scaled = a / Fraction(2) ** q
    r = math.floor(scaled)
    rem = scaled - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    return sign * float(Fraction(r) * Fraction(2) ** q)


# ---- whole layer --------------------------------------------------------------------

def _layer_brute(inp):
    """Per-token loops in numpy float64, BF16 rounding at the SiLU-mul and final outputs (the
    gate_up sums feed SiLU-and-mul unrounded; the per-slot down outputs are summed
    unrounded)."""
    from scipy.special import expit
    wl = inp.wl
    w13 = dequant_np(inp.w13_q.numpy(), inp.w13_s.view(torch.int16).numpy())
    w2 = dequant_np(inp.w2_q.numpy(), inp.w2_s.view(torch.int16).numpy())
    xa = bf16_np(inp.x)
    T, k = inp.topk_ids.shape
    out = np.zeros((T, wl.H))

    def rb(v):  # float64 -> BF16 by way of float32 (two roundings; fine within one ulp)
        return bf16_bits_to_f64(torch_bf16_bits(np.asarray(v, np.float64).astype(np.float32)))

    for t in range(T):
        acc = np.zeros(wl.H)
        for s in range(k):
            ex = int(inp.topk_ids[t, s])
            if ex < 0:
                continue
            c = w13[ex] @ xa[t]
            g, u = c[: wl.I], c[wl.I:]
            h = rb(g * expit(g) * u)
            y = w2[ex] @ h  # per-slot down output stays unrounded until the weighted sum
            acc += float(inp.topk_weights[t, s]) * y
        out[t] = rb(acc)
    return out


def test_layer_tiny_against_brute_force_and_block_m_independence():
    wl = workloads.WORKLOADS["tiny"]
    inp = workloads.draw_layer(wl, 16)
    assert not torch.any(inp.topk_ids == 7)  # the forced-empty expert
    args = (inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, inp.topk_ids, inp.topk_weights)
    out16 = oracle.moe_layer(*args, block_m=16)
    ref = _layer_brute(inp)
    got = bf16_np(out16)
    rms = np.sqrt(np.mean(ref ** 2))
    # the brute force rounds at the same boundaries; tiny FP32/float64 order effects only
    assert np.all(np.abs(got - ref) <= 2 * ulp_bf16(ref) + 1e-3 * rms)
    assert np.mean(got == ref) > 0.9
    for bm in (1, 4, 64):
        assert torch.equal(bits_t(oracle.moe_layer(*args, block_m=bm)), bits_t(out16))
    assert torch.equal(bits_t(oracle.moe_layer_parallel(*args, block_m=16, threads=3)), bits_t(out16))


def test_layer_dropped_slots_give_zero_rows():
    wl = workloads.WORKLOADS["tiny"]
    inp = workloads.draw_layer(wl, 16)
    ids = inp.topk_ids.clone()
    ids[3] = -1  # token 3 has no local expert
    out = oracle.moe_layer(inp.x, inp.w13_q, inp.w13_s, inp.w2_q, inp.w2_s, ids, inp.topk_weights)
    assert torch.all(out[3].float() == 0)
    assert torch.any(out[2].float() != 0)


# ---- grouped contracts ("Grouped SM90 kernels": contiguous prefill, masked decode) ----------

def _contiguous_problem(seed, groups=((0, 100), (2, 128), (1, 3)), E=3, N=32, K=64):
    """Rows concatenated by expert, each group padded to a 128-row boundary with -1."""
    qw, sc = workloads.draw_weights(E, N, K, seed=seed)
    ids = []
    for e, rows in groups:
        pad = (-rows) % 128
        ids += [e] * rows + [-1] * pad
    m_indices = torch.tensor(ids, dtype=torch.int32)
    x = workloads.draw_activations(len(ids), K, seed=seed)
    return qw, sc, x, m_indices


def test_contiguous_brute_force_rows_and_zero_padding():
    qw, sc, x, mi = _contiguous_problem(21)
    C = bf16_np(oracle.contiguous_gemm(x, qw, sc, mi))
    wd = dequant_np(qw.numpy(), sc.view(torch.int16).numpy())
    xa = bf16_np(x)
    for r in range(mi.numel()):
        e = int(mi[r])
        if e < 0:
            assert np.all(C[r] == 0)
            continue
        ref = wd[e] @ xa[r]  # float64 sum of exact products
        assert np.all(np.abs(C[r] - ref) <= ulp_bf16(ref) + 1e-12)


def test_contiguous_single_expert_equals_torch_matmul():
    qw, sc = workloads.draw_weights(2, 64, 128, seed=22)
    x = workloads.draw_activations(256, 128, seed=22)
    mi = torch.ones(256, dtype=torch.int32)
    C = oracle.contiguous_gemm(x, qw, sc, mi).float()
    ref = torch.matmul(x.float(), oracle.dequant(qw, sc)[1].float().T)
    assert torch.all((C - ref).abs() <= torch.from_numpy(ulp_bf16(ref.numpy())).float() + 1e-6)


def test_contiguous_group_order_permutes_rows():
    qw, sc, x, mi = _contiguous_problem(23, groups=((0, 128), (1, 128)), E=2)
    C = oracle.contiguous_gemm(x, qw, sc, mi)
    swapped_x = torch.cat([x[128:], x[:128]])
    swapped_mi = torch.cat([mi[128:], mi[:128]])
    D = oracle.contiguous_gemm(swapped_x, qw, sc, swapped_mi)
    assert np.array_equal(bits(D), bits(torch.cat([C[128:], C[:128]])))


def test_masked_valid_rows_equal_per_expert_matmul_and_rest_untouched():
    G, N, K, max_m = 3, 32, 64, 16
    qw, sc = workloads.draw_weights(G, N, K, seed=24)
    x = workloads.draw_activations(G * max_m, K, seed=24)
    mm = torch.tensor([5, 0, 16], dtype=torch.int32)
    C = oracle.masked_gemm(x, qw, sc, mm, max_m).float()
    wd = oracle.dequant(qw, sc)
    for g in range(G):
        rows = slice(g * max_m, g * max_m + int(mm[g]))
        ref = torch.matmul(x[rows].float(), wd[g].float().T)
        assert torch.all((C[rows] - ref).abs() <= torch.from_numpy(ulp_bf16(ref.numpy())).float() + 1e-6)
        assert torch.all(C[g * max_m + int(mm[g]):(g + 1) * max_m] == 0)


def test_masked_equals_contiguous_on_the_same_rows():
    # Masked rows laid out as a contiguous problem (budget = 128 rows per expert) give the
    # same bits: both are per-row products with that row's expert.
    G, N, K, max_m = 2, 32, 64, 128
    qw, sc = workloads.draw_weights(G, N, K, seed=25)
    x = workloads.draw_activations(G * max_m, K, seed=25)
    mm = torch.tensor([100, 7], dtype=torch.int32)
    M = oracle.masked_gemm(x, qw, sc, mm, max_m)
    mi = torch.tensor([0] * 100 + [-1] * 28 + [1] * 7 + [-1] * 121, dtype=torch.int32)
    Cc = oracle.contiguous_gemm(x, qw, sc, mi)
    valid = mi >= 0
    assert np.array_equal(bits(M[valid]), bits(Cc[valid]))


# ---- NVFP4 weights ("humans& ...", "BF16 preserves each local product") ------------------

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # the E2M1 magnitudes of the OCP FP4 format


def _nvfp4_all_pairs():
    """One row per E4M3 scale byte: 16 codes x every scale, K = 16 per row."""
    codes = np.zeros((256, 8), np.uint8)
    for j in range(8):
        codes[:, j] = (2 * j) | ((2 * j + 1) << 4)  # elements 0..15 = codes 0..15
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    return codes, scales


def test_nvfp4_worked_product_from_the_pages():
    # "the product 1.5 x 1.125 equals 1.6875; BF16 represents that value exactly"
    with open(os.path.join(os.path.dirname(__file__), "golden", "bf16_exact_product.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    a, b, prod, bits_hex = rows[0][:4]
    e2m1_code = E2M1_TABLE.index(float(a))           # 1.5 -> magnitude code 3
    e4m3_byte = (7 << 3) | 1                          # 1.125 = 2^0 * (1 + 1/8)
    assert float(b) == 1.125
    codes = torch.tensor([[e2m1_code | (e2m1_code << 4)] * 8], dtype=torch.uint8)
    scales = torch.tensor([[e4m3_byte]], dtype=torch.uint8)
    wd = oracle.nvfp4_dequant(codes, scales)
    assert float(wd[0, 0]) == float(prod)
    assert int(wd.view(torch.int16)[0, 0]) & 0xFFFF == int(bits_hex, 16)


def test_nvfp4_exhaustive_codes_times_every_e4m3_scale():
    codes, scales = _nvfp4_all_pairs()
    wd = oracle.nvfp4_dequant(torch.from_numpy(codes), torch.from_numpy(scales)).float().numpy()
    s_lib = torch.from_numpy(scales.reshape(-1)).view(torch.float8_e4m3fn).float().numpy()  # library decode
    for sb in range(256):
        for c in range(16):
            v = (-1.0 if c & 8 else 1.0) * E2M1_TABLE[c & 7]
            exact = v * float(s_lib[sb])  # exact in float64
            got = wd[sb, c]
            if np.isnan(exact):
                assert np.isnan(got)
            else:
                assert got == exact, (sb, c, got, exact)  # BF16 holds every product exactly


def test_nvfp4_nibble_order_low_first_and_block_of_16():
    codes = torch.zeros((1, 16), dtype=torch.uint8)
    codes[0, 0] = 0x4 | (0x2 << 4)  # element 0 = 2.0, element 1 = 1.0
    scales = torch.tensor([[7 << 3, 8 << 3]], dtype=torch.uint8)  # 1.0 for K 0..15, 2.0 for 16..31
    codes[0, 8] = 0x2  # element 16 = 1.0 -> 2.0 after its block's scale
    wd = oracle.nvfp4_dequant(codes, scales)[0].float()
    assert wd[0] == 2.0 and wd[1] == 1.0 and wd[2] == 0.0 and wd[16] == 2.0 and wd[17] == 0.0


def test_nvfp4_gemm_single_expert_equals_torch_matmul():
    codes, scales = workloads.draw_nvfp4_weights(1, 64, 256, seed=41)
    x = workloads.draw_activations(20, 256, seed=41)
    ids = torch.zeros((20, 1), dtype=torch.int32)
    s, e, ntp = oracle.moe_align(ids, 1, 16)
    C = oracle.nvfp4_moe_gemm(x, 1, codes, scales, s, e, ntp, 16, 20).float()
    ref = torch.matmul(x.float(), oracle.nvfp4_dequant(codes, scales)[0].float().T)
    assert torch.all((C - ref).abs() <= torch.from_numpy(ulp_bf16(ref.numpy())).float() + 1e-6)


def test_nvfp4_gemm_brute_force_per_token():
    codes, scales = workloads.draw_nvfp4_weights(4, 48, 64, seed=42)
    x = workloads.draw_activations(12, 64, seed=42)
    ids, _ = workloads.draw_routing(12, 4, 2, seed=42)
    s, e, ntp = oracle.moe_align(ids, 4, 4)
    C = bf16_np(oracle.nvfp4_moe_gemm(x, 2, codes, scales, s, e, ntp, 4, 24))
    # independent numpy decode of the codes and scales
    c = codes.numpy()
    nib = np.stack([c & 15, c >> 4], axis=-1).reshape(4, 48, 64)
    mag = np.array(E2M1_TABLE)[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    sc = torch.from_numpy(scales.numpy().reshape(-1)).view(torch.float8_e4m3fn).double().numpy().reshape(4, 48, 4)
    wd = mag * np.repeat(sc, 16, axis=-1)
    xa = bf16_np(x)
    for t in range(12):
        for j in range(2):
            ref = wd[int(ids[t, j])] @ xa[t]
            assert np.all(np.abs(C[t * 2 + j] - ref) <= ulp_bf16(ref) + 1e-12)
