// Plain CPU oracle for the W4A16 mixture-of-experts expert path.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
// reference that the CUDA library is checked against.  Only the test suite,
// the smoke check and the benchmark's CPU-baseline leg may load it; the
// library itself never calls it, and the two share no code, header, table or
// helper.  Single-threaded; compiled with -ffp-contract=off so that every
// FP32 operation below is one correctly rounded IEEE operation on every host.
//
// What it computes (sources are the pages' titles and sections):
//
//  * align -- "vLLM x Novita AI: Chord, Faster INT4 MoE for Kimi K2.x",
//    "Two kernel families" and "vLLM integration": indexed routing consumes
//    sorted_ids / expert_ids / num_tokens_padded built by vLLM's
//    moe_align_block_size, whose over-allocated buffers carry padding
//    sentinels.  Read here as a stable counting sort of the flat slot index
//    i = t*top_k + s by expert id, each expert's run padded to a multiple of
//    block_m with the sentinel T*top_k; expert_ids[b] names the expert of
//    block b, -1 past num_tokens_padded.
//  * dequant -- same page, "H200 and Blackwell indexed decode":
//    subtract-then-scale, w = (q - 8) * s, one BF16 scale per 32 K
//    elements, rounded once to BF16 (the product is exact in FP32).
//    "humans& Beats FlashInfer's Best MoE Kernel by 25% on Blackwell GPUs",
//    "BF16 preserves each local product": the dequantised weight is a BF16
//    value.
//  * gemm -- Chord page, "Two kernel families": for every sorted position
//    p < num_tokens_padded whose slot i = sorted_ids[p] is not a sentinel,
//    C[i, :] = A[i / a_row_div] . dequant(W[expert_ids[p / block_m]])^T,
//    a plain FP32 dot product over k ascending, rounded once to BF16.
//  * silu_mul -- SiLU(gate) * up with gate = C[:, :I], up = C[:, I:], on the
//    unrounded FP32 gate_up sums (the SiLU-and-mul is fused between the two
//    GEMMs, so no BF16 gate_up tensor exists on the path; rounding gate and
//    up to BF16 first and then h again stacks two order-dependent roundings,
//    up to 1.5% of |h| at the top of a binade, beyond the stated output
//    tolerance); evaluated in double, rounded once to BF16.
//  * topk_sum -- out[t, :] = sum over valid slots s (ascending) of
//    topk_weights[t, s] * Y[t*top_k + s, :]; double, rounded once to BF16.
//    The per-slot down outputs Y stay FP32 (the pages fix no precision for
//    them; rounding them to BF16 first would add up to half a BF16 ulp of the
//    largest per-slot value, an error as large as the stated output
//    tolerance, so the reading that fits that tolerance keeps them in FP32).
//  * layer -- align, gate_up gemm (FP32 out), silu_mul, down gemm (FP32 out),
//    topk_sum in that
//    order (Chord page, "Measurements": the per-layer time is gate_up plus
//    down; "humans& ..." page: FC1, FC2 and the top-K merge).
//
// Parity pins for every function live in the CPU test suite (brute force on
// tiny inputs, exhaustive dequant, library-routine special cases and
// invariants).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

float bf16_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

// IEEE float -> BF16, round to nearest, ties to even.  NaN stays NaN (quiet).
uint16_t float_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  const uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7fffu + keep_lsb;  // adds half an ulp, or a hair less on an even tie
  return static_cast<uint16_t>(u >> 16);
}

// double -> BF16, round to nearest, ties to even, in one rounding: the value
// is rounded to BF16's grid (8 significant bits, quantum 2^-133 at the
// subnormal end) with nearbyint, then it is exactly representable in float.
uint16_t double_to_bf16(double x) {
  if (std::isnan(x)) return 0x7fc0u;
  const bool neg = std::signbit(x);
  const double a = std::fabs(x);
  uint16_t mag;
  if (std::isinf(a)) {
    mag = 0x7f80u;
  } else if (a == 0.0) {
    mag = 0x0000u;
  } else {
    int e = 0;
    std::frexp(a, &e);  // a = m * 2^e with m in [0.5, 1)
    int q = e - 8;      // quantum of an 8-significant-bit value in [2^(e-1), 2^e)
    if (q < -133) q = -133;
    const double r = std::nearbyint(std::ldexp(a, -q));  // default mode: ties to even
    const double v = std::ldexp(r, q);
    if (v >= 0x1p128) {
      mag = 0x7f80u;
    } else {
      const float f = static_cast<float>(v);  // exact
      uint32_t u;
      std::memcpy(&u, &f, sizeof u);
      mag = static_cast<uint16_t>(u >> 16);
    }
  }
  return neg ? static_cast<uint16_t>(mag | 0x8000u) : mag;
}

// Element k of one weight row: w = bf16((q - 8) * s).
float dequant_one(const int32_t* qrow, const uint16_t* srow, int k, int group) {
  const uint32_t word = static_cast<uint32_t>(qrow[k / 8]);
  const int q = static_cast<int>((word >> (4 * (k % 8))) & 0xFu);
  const float prod = static_cast<float>(q - 8) * bf16_to_float(srow[k / group]);
  return bf16_to_float(float_to_bf16(prod));
}

// C[row] for one (slot, expert) pair: FP32 dot over k ascending, BF16 out (or the FP32
// sum itself when out_f32 is given).
void gemm_one_row(const uint16_t* a, int K, const int32_t* qweight, const uint16_t* scales,
                  int N, int group, int e, uint16_t* out_row, float* out_f32 = nullptr) {
  for (int n = 0; n < N; ++n) {
    const int32_t* qrow = qweight + (static_cast<int64_t>(e) * N + n) * (K / 8);
    const uint16_t* srow = scales + (static_cast<int64_t>(e) * N + n) * (K / group);
    float acc = 0.0f;
    for (int k = 0; k < K; ++k) {
      const float p = bf16_to_float(a[k]) * dequant_one(qrow, srow, k, group);
      acc = acc + p;
    }
    if (out_f32)
      out_f32[n] = acc;
    else
      out_row[n] = float_to_bf16(acc);
  }
}

// ---- NVFP4 ("humans& Beats FlashInfer's Best MoE Kernel by 25% on Blackwell GPUs", "BF16
// preserves each local product"): blocks of 16 E2M1 values along K share one E4M3 scale and a
// weight is the product of the two, which BF16 represents exactly.

// E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0 is subnormal.
double e2m1_value(unsigned code) {
  const unsigned e = (code >> 1) & 3u, m = code & 1u;
  const double mag = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, static_cast<int>(e) - 1);
  return (code & 8u) ? -mag : mag;
}

// E4M3 (the finite-only variant): sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0;
// exponent 0 is subnormal, 0x7f / 0xff are NaN.
double e4m3_value(unsigned byte) {
  const unsigned e = (byte >> 3) & 15u, m = byte & 7u;
  if (e == 15 && m == 7) return std::nan("");
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, static_cast<int>(e) - 7);
  return (byte & 0x80u) ? -mag : mag;
}

// Element k of one NVFP4 weight row (codes: two per byte, element 2j in the low nibble).
float nvfp4_dequant_one(const uint8_t* crow, const uint8_t* srow, int k) {
  const unsigned code = (crow[k / 2] >> (4 * (k % 2))) & 0xFu;
  return bf16_to_float(double_to_bf16(e2m1_value(code) * e4m3_value(srow[k / 16])));
}

void gemm_one_row_nvfp4(const uint16_t* a, int K, const uint8_t* codes, const uint8_t* scales,
                        int N, int e, uint16_t* out_row, float* out_f32) {
  for (int n = 0; n < N; ++n) {
    const uint8_t* crow = codes + (static_cast<int64_t>(e) * N + n) * (K / 2);
    const uint8_t* srow = scales + (static_cast<int64_t>(e) * N + n) * (K / 16);
    float acc = 0.0f;
    for (int k = 0; k < K; ++k) {
      const float p = bf16_to_float(a[k]) * nvfp4_dequant_one(crow, srow, k);
      acc = acc + p;
    }
    if (out_f32)
      out_f32[n] = acc;
    else
      out_row[n] = float_to_bf16(acc);
  }
}

}  // namespace

extern "C" {

// ---- scalar helpers exposed for the tests' pins --------------------------------

void w4a16_oracle_float_to_bf16(const float* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = float_to_bf16(x[i]);
}

void w4a16_oracle_double_to_bf16(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(x[i]);
}

// ---- align ---------------------------------------------------------------------

int64_t w4a16_oracle_align_capacity(int T, int top_k, int E, int block_m) {
  const int64_t raw = static_cast<int64_t>(T) * top_k + static_cast<int64_t>(E) * (block_m - 1);
  return (raw + block_m - 1) / block_m * block_m;
}

// Returns 0 on success; -1 on an expert id outside [-1, E); -2 when the
// padded rows exceed capacity; -3 on bad sizes.
int w4a16_oracle_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                       int64_t capacity, int32_t* sorted_ids, int32_t* expert_ids,
                       int32_t* num_tokens_padded) {
  if (T < 0 || top_k <= 0 || E <= 0 || block_m <= 0 || capacity < 0 || capacity % block_m)
    return -3;
  const int64_t n = static_cast<int64_t>(T) * top_k;
  const int32_t sentinel = static_cast<int32_t>(n);
  std::vector<int64_t> count(E, 0);
  for (int64_t i = 0; i < n; ++i) {
    const int32_t e = topk_ids[i];
    if (e == -1) continue;
    if (e < 0 || e >= E) return -1;
    ++count[e];
  }
  std::vector<int64_t> start(E + 1, 0);  // padded, exclusive prefix in expert order
  for (int e = 0; e < E; ++e)
    start[e + 1] = start[e] + (count[e] + block_m - 1) / block_m * block_m;
  const int64_t ntp = start[E];
  if (ntp > capacity) return -2;

  for (int64_t p = 0; p < capacity; ++p) sorted_ids[p] = sentinel;
  for (int64_t b = 0; b < capacity / block_m; ++b) expert_ids[b] = -1;
  std::vector<int64_t> cursor(start.begin(), start.end() - 1);
  for (int64_t i = 0; i < n; ++i) {  // ascending i keeps the sort stable
    const int32_t e = topk_ids[i];
    if (e < 0) continue;
    sorted_ids[cursor[e]++] = static_cast<int32_t>(i);
  }
  for (int e = 0; e < E; ++e)
    for (int64_t b = start[e] / block_m; b < start[e + 1] / block_m; ++b) expert_ids[b] = e;
  *num_tokens_padded = static_cast<int32_t>(ntp);
  return 0;
}

// ---- dequant -------------------------------------------------------------------

// qweight int32 [rows, K/8], scales bf16 [rows, K/group] -> out bf16 [rows, K]
void w4a16_oracle_dequant(const int32_t* qweight, const uint16_t* scales, int64_t rows, int K,
                          int group, uint16_t* out) {
  for (int64_t r = 0; r < rows; ++r) {
    const int32_t* qrow = qweight + r * (K / 8);
    const uint16_t* srow = scales + r * (K / group);
    for (int k = 0; k < K; ++k) out[r * K + k] = float_to_bf16(dequant_one(qrow, srow, k, group));
  }
}

// ---- gemm ----------------------------------------------------------------------

// out[r, :] = A[slots[r] / a_row_div] . dequant(W[experts[r]])^T for r < nrows: BF16 rows in
// out, or the unrounded FP32 sums in out_f32 when it is not NULL.
void w4a16_oracle_gemm_rows(const uint16_t* A, int a_row_div, int K, const int32_t* qweight,
                            const uint16_t* scales, int N, int group, const int32_t* slots,
                            const int32_t* experts, int64_t nrows, uint16_t* out,
                            float* out_f32) {
  for (int64_t r = 0; r < nrows; ++r) {
    const uint16_t* a = A + static_cast<int64_t>(slots[r] / a_row_div) * K;
    gemm_one_row(a, K, qweight, scales, N, group, experts[r], out_f32 ? nullptr : out + r * N,
                 out_f32 ? out_f32 + r * N : nullptr);
  }
}

// Indexed grouped GEMM over the aligned routing.  Writes C[i, :] for every
// routed slot i whose expert lies in [e_lo, e_hi); other rows are untouched.
// C is BF16, or FP32 (the unrounded sums) when C_f32 is not NULL.
int w4a16_oracle_moe_gemm(const uint16_t* A, int a_row_div, int K, const int32_t* qweight,
                          const uint16_t* scales, int N, int group, const int32_t* sorted_ids,
                          const int32_t* expert_ids, int num_tokens_padded, int block_m,
                          int total_slots, int e_lo, int e_hi, uint16_t* C, float* C_f32) {
  if (a_row_div <= 0 || K % 8 || K % group || block_m <= 0) return -3;
  for (int64_t p = 0; p < num_tokens_padded; ++p) {
    const int32_t i = sorted_ids[p];
    if (i >= total_slots) continue;  // padding sentinel
    const int32_t e = expert_ids[p / block_m];
    if (e < e_lo || e >= e_hi) continue;
    const uint16_t* a = A + static_cast<int64_t>(i / a_row_div) * K;
    const int64_t row = static_cast<int64_t>(i) * N;
    gemm_one_row(a, K, qweight, scales, N, group, e, C_f32 ? nullptr : C + row,
                 C_f32 ? C_f32 + row : nullptr);
  }
  return 0;
}

// ---- activation and combine -----------------------------------------------------

// C fp32 [rows, 2I] (the unrounded gate_up sums) -> h bf16 [rows, I]:
// h = bf16(silu(gate) * up).
void w4a16_oracle_silu_mul(const float* C, int64_t rows, int I, uint16_t* h) {
  for (int64_t r = 0; r < rows; ++r) {
    for (int j = 0; j < I; ++j) {
      const double g = C[r * 2 * I + j];
      const double u = C[r * 2 * I + I + j];
      const double silu = g / (1.0 + std::exp(-g));
      h[r * I + j] = double_to_bf16(silu * u);
    }
  }
}

// Y fp32 [T*top_k, H] -> out bf16 [T, H]; slots with id -1 are skipped.
void w4a16_oracle_topk_sum(const float* Y, const int32_t* topk_ids, const float* topk_weights,
                           int T, int top_k, int H, uint16_t* out) {
  for (int64_t t = 0; t < T; ++t) {
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int s = 0; s < top_k; ++s) {
        const int64_t i = t * top_k + s;
        if (topk_ids[i] < 0) continue;
        acc += static_cast<double>(topk_weights[i]) * static_cast<double>(Y[i * H + c]);
      }
      out[t * H + c] = double_to_bf16(acc);
    }
  }
}

// ---- NVFP4 weights ----------------------------------------------------------------

// codes uint8 [rows, K/2], scales E4M3 [rows, K/16] -> BF16 [rows, K].
void w4a16_oracle_nvfp4_dequant(const uint8_t* codes, const uint8_t* scales, int64_t rows, int K,
                                uint16_t* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int k = 0; k < K; ++k)
      out[r * K + k] = float_to_bf16(nvfp4_dequant_one(codes + r * (K / 2), scales + r * (K / 16), k));
}

// The indexed grouped GEMM of w4a16_oracle_moe_gemm with NVFP4 weights.
int w4a16_oracle_nvfp4_moe_gemm(const uint16_t* A, int a_row_div, int K, const uint8_t* codes,
                                const uint8_t* scales, int N, const int32_t* sorted_ids,
                                const int32_t* expert_ids, int num_tokens_padded, int block_m,
                                int total_slots, int e_lo, int e_hi, uint16_t* C, float* C_f32) {
  if (a_row_div <= 0 || K % 16 || block_m <= 0) return -3;
  for (int64_t p = 0; p < num_tokens_padded; ++p) {
    const int32_t i = sorted_ids[p];
    if (i >= total_slots) continue;  // padding sentinel
    const int32_t e = expert_ids[p / block_m];
    if (e < e_lo || e >= e_hi) continue;
    const uint16_t* a = A + static_cast<int64_t>(i / a_row_div) * K;
    const int64_t row = static_cast<int64_t>(i) * N;
    gemm_one_row_nvfp4(a, K, codes, scales, N, e, C_f32 ? nullptr : C + row,
                       C_f32 ? C_f32 + row : nullptr);
  }
  return 0;
}

// ---- grouped contracts -------------------------------------------------------------
// "Grouped SM90 kernels" (vLLM x Novita AI: Chord): the contiguous prefill layout has its rows
// concatenated by expert, each group padded to a 128-row boundary, with m_indices[r] the
// expert of row r or -1 for padding; the output row r is A[r] times the dequantised weight of
// that expert.  Padding rows are zero here.
// C is BF16, or FP32 (the unrounded sums) when C_f32 is not NULL.
int w4a16_oracle_contiguous_gemm(const uint16_t* A, int64_t m, int K, const int32_t* qweight,
                                 const uint16_t* scales, int E, int N, int group,
                                 const int32_t* m_indices, uint16_t* C, float* C_f32) {
  if (K % 8 || K % group || m % 128) return -3;
  for (int64_t r = 0; r < m; ++r) {
    const int32_t e = m_indices[r];
    uint16_t* out = C_f32 ? nullptr : C + r * N;
    float* out_f32 = C_f32 ? C_f32 + r * N : nullptr;
    if (e < 0 || e >= E) {
      for (int n = 0; n < N; ++n) {
        if (out) out[n] = 0;
        if (out_f32) out_f32[n] = 0.0f;
      }
      continue;
    }
    gemm_one_row(A + r * K, K, qweight, scales, N, group, e, out, out_f32);
  }
  return 0;
}

// Same page, masked decode layout: a fixed budget of max_m rows per expert g (rows
// g * max_m .. g * max_m + max_m - 1 of A and of the flat output), of which the first
// masked_m[g] are valid; only those output rows are defined (the others are left as they are).
int w4a16_oracle_masked_gemm(const uint16_t* A, int G, int max_m, int K, const int32_t* qweight,
                             const uint16_t* scales, int N, int group, const int32_t* masked_m,
                             uint16_t* C, float* C_f32) {
  if (K % 8 || K % group || max_m <= 0) return -3;
  for (int g = 0; g < G; ++g) {
    const int valid = masked_m[g] < 0 ? 0 : (masked_m[g] > max_m ? max_m : masked_m[g]);
    for (int r = 0; r < valid; ++r) {
      const int64_t row = static_cast<int64_t>(g) * max_m + r;
      gemm_one_row(A + row * K, K, qweight, scales, N, group, g, C_f32 ? nullptr : C + row * N,
                   C_f32 ? C_f32 + row * N : nullptr);
    }
  }
  return 0;
}

// ---- whole layer -----------------------------------------------------------------

int w4a16_oracle_moe_layer(const uint16_t* x, const int32_t* w13_q, const uint16_t* w13_s,
                           const int32_t* w2_q, const uint16_t* w2_s, const int32_t* topk_ids,
                           const float* topk_weights, int T, int H, int I, int E, int top_k,
                           int group, int block_m, uint16_t* out) {
  const int64_t cap = w4a16_oracle_align_capacity(T, top_k, E, block_m);
  const int64_t slots = static_cast<int64_t>(T) * top_k;
  std::vector<int32_t> sorted_ids(cap), expert_ids(cap / block_m);
  int32_t ntp = 0;
  int rc = w4a16_oracle_align(topk_ids, T, top_k, E, block_m, cap, sorted_ids.data(),
                              expert_ids.data(), &ntp);
  if (rc) return rc;
  std::vector<float> c13(slots * 2 * I, 0.0f), y(slots * H, 0.0f);
  std::vector<uint16_t> h(slots * I, 0);
  rc = w4a16_oracle_moe_gemm(x, top_k, H, w13_q, w13_s, 2 * I, group, sorted_ids.data(),
                             expert_ids.data(), ntp, block_m, static_cast<int>(slots), 0, E,
                             nullptr, c13.data());
  if (rc) return rc;
  w4a16_oracle_silu_mul(c13.data(), slots, I, h.data());
  rc = w4a16_oracle_moe_gemm(h.data(), 1, I, w2_q, w2_s, H, group, sorted_ids.data(),
                             expert_ids.data(), ntp, block_m, static_cast<int>(slots), 0, E,
                             nullptr, y.data());
  if (rc) return rc;
  w4a16_oracle_topk_sum(y.data(), topk_ids, topk_weights, T, top_k, H, out);
  return 0;
}

}  // extern "C"
