// Indexed W4A16 grouped GEMM for sm_103a: tcgen05 MMAs with dequantised weights in TMEM.
//
// What it computes ("vLLM x Novita AI: Chord, Faster INT4 MoE for Kimi K2.x", "Two kernel
// families"): for every aligned row position p with slot i = sorted_ids[p] (not a sentinel)
// and expert e = expert_ids[p / block_m], C[i, :] = A[i / a_row_div, :] . dequant(W[e])^T,
// with w = bf16((q - 8) * s) ("H200 and Blackwell indexed decode": subtract-then-scale fused
// into nibble extraction keeps the unfused BF16 rounding).
//
// How (GB300 design; prior art: the indexed decode kernel swaps operands so dequantised
// weights fill MMA-M, same page; "humans& Beats FlashInfer's Best MoE Kernel by 25% on
// Blackwell GPUs", "Blackwell hides the conversion work" and "Dedicated warps keep the
// pipeline busy": TMEM holds accumulators and dequantised weights, single-thread TMA/MMA
// issue, dequant-only warpgroups, dependent launch, L2 hints):
//   * the weight tile (128 rows of W[e] = MMA M) is the A operand, read from TMEM; tokens of
//     one aligned block (block_m = MMA N) are the B operand, in 128-byte-swizzled shared
//     memory; the FP32 accumulator is in TMEM;
//   * warp 0 streams the packed weights, one 1-D bulk copy per stage of one or two 64-wide K
//     blocks (evict_first when weights are streamed once), and, when the activation rows are
//     already in sorted order, their 2-D tiles by tensor TMA; otherwise warps 2-3 gather the
//     rows (row = sorted_ids[p] / a_row_div) with 16-byte cp.async into the swizzled layout.
//     Weights and activations complete on separate mbarriers, so a dependent launch streams
//     and dequantises its first weights before its inputs exist;
//   * warps 8-15 (two dequant warpgroups, alternating stages) turn codes into BF16 pairs and
//     store them to TMEM with tcgen05.st (one fused multiply-add per pair for tiles whose
//     scales the packer stored pre-multiplied by 2^133, else subtract then multiply);
//     warp 1 issues tcgen05.mma from one elected lane;
//     warps 4-7 drain the double-buffered accumulator with tcgen05.ld and write the results;
//   * a persistent grid walks (block, 128-row tile, K split) units found from
//     num_tokens_padded on the device (no host read-back); K splits (decode) write FP32
//     partials and the last CTA to arrive on a per-tile counter sums them in split order,
//     so results are deterministic.
#include <algorithm>
#include <cmath>

#include "gemm.cuh"

namespace w4a16 {

constexpr int kDqGroups = 2;  // dequant warpgroups; stage it goes to group it % kDqGroups
constexpr int kGemmThreads = 256 + 128 * kDqGroups;
constexpr int kTmemCols = 512;
constexpr int kSmemBudget = 216 * 1024;
constexpr int kEpiStageBytes = 16 * 36 * 4;  // per epilogue warp: 16 tokens x (32 + 4 pad) x 4 B
constexpr int kGatherThreads = 64;  // warps 2 and 3 gather activation rows with cp.async

// NT = block_m = MMA N; KS = 64-wide K sub-blocks per pipeline stage (one weight copy of
// KS * 4608 bytes; deeper stages halve the per-byte barrier, copy and commit overhead).
// Three independent rings: packed weights in shared memory (freed once the dequant warps hold
// them in registers), activation tiles in shared memory (freed by the MMA commit), dequantised
// weights in TMEM (freed by the MMA commit).
template <int NT, int KS, bool PAIR = false, int TPU = 1>
struct GemmCfg {
  // B bytes of one sub-block (NT rows x 64; a CTA of a pair holds half the block's rows)
  static constexpr int kSubB = (PAIR ? NT / 2 : NT) * 128;
  static constexpr int kBBytes = KS * kSubB;        // one activation stage
  static constexpr int kWBytes = KS * kChunkBytes;  // one weight stage
  // activation ring: 64-96 KB (at least 4, at most 24 stages), the rest for weights.  The
  // rows arrive with multi-microsecond latency under full HBM load and each slot is held until
  // its MMAs finish, so the ring must cover that round trip.
  static constexpr int kBBudget = (NT <= 32 ? 64 : 96) * 1024;
  static constexpr int kBStagesRaw = kBBudget / kBBytes;
  static constexpr int kBStages = kBStagesRaw < 4 ? 4 : (kBStagesRaw > 24 ? 24 : kBStagesRaw);
  static constexpr int kWStagesRaw = (kSmemBudget - 4096 - kBStages * kBBytes) / kWBytes;
  static constexpr int kWStages = kWStagesRaw > 32 ? 32 : kWStagesRaw;
  // TMEM: two FP32 accumulators of TPU * NT columns (TPU tiles per unit) at the start, then as
  // many dequantised A stages of KS * 32 columns as fit (a deep A ring covers the dequant ->
  // MMA -> commit round trip).
  static constexpr int kACol0 = (2 * NT * TPU + 31) / 32 * 32;
  static constexpr int kAStagesRaw = (kTmemCols - kACol0) / (KS * 32);
  static constexpr int kAStages = kAStagesRaw > 12 ? 12 : kAStagesRaw;
  static constexpr int kBarBytes = (2 * kWStages + 2 * kBStages + 2 * kAStages + 5) * 8;
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kBStages) * kBBytes +
                                       static_cast<size_t>(kWStages) * kWBytes + kBarBytes + 64 +
                                       NT * 4 + 16 + 4 * kEpiStageBytes;
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 128, "MMA N must be 16..128 in steps of 16");
  static_assert(kACol0 + 32 * KS * kAStages <= kTmemCols, "A stages must fit in TMEM");
  static_assert(kAStages >= 2, "A ring too shallow");
  static_assert(kWStages >= 4, "weight ring too shallow");
  static_assert(kSmemBytes <= 232448, "shared memory (227 KB per block)");
};

struct Unit {
  int b, jt, split, kb0, kb1, e;
  int gi;      // which GEMM of a fused layer call (0: gate_up, 1: down); 0 otherwise
  int nsplit;  // K slices of this unit's tile (1: whole K)
  int ptile;   // index of a sliced tile among the sliced tiles (partial sums, counters)
  int64_t tile;
  bool ok;  // the block names a valid expert
};

// Which units are K slices: units [0, tail) are whole tiles 0 .. tail-1; the units from tail
// on are the remaining tiles, each cut into s K slices (unit tail + p*s + j: slice j of tile
// tail + p).  No slicing: tail past the last unit.
struct SplitMap {
  uint32_t tail;
  uint32_t s;
};
__device__ __forceinline__ SplitMap no_split() { return SplitMap{0xFFFFFFFFu, 1u}; }

// Unit u -> (block, tile, slice).  Every role decodes every unit, so the divisions are 32-bit
// (the host keeps unit counts below 2^31) and the one by the tiles per block uses a
// precomputed multiply-shift: q = (umulhi(n, m) + n) >> s with m = ceil(2^(32+s) / d) - 2^32
// and s = ceil(log2 d), exact for n < 2^31 (round-up reciprocal method).
__device__ __forceinline__ uint32_t unit_tile(const SplitMap& sm, uint32_t u) {
  return u < sm.tail ? u : sm.tail + (u - sm.tail) / sm.s;
}

__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, const SplitMap& sm, int64_t u64) {
  const uint32_t u = static_cast<uint32_t>(u64);
  Unit t;
  uint32_t tile;
  if (u < sm.tail) {
    tile = u;
    t.split = 0;
    t.nsplit = 1;
    t.ptile = 0;
    t.kb0 = 0;
    t.kb1 = a.n_kb * a.tpu;  // a tile group's tiles are consecutive chunks of one strip
  } else {
    const uint32_t v = u - sm.tail;
    const uint32_t pt = v / sm.s;
    t.split = static_cast<int>(v - pt * sm.s);
    t.nsplit = static_cast<int>(sm.s);
    t.ptile = static_cast<int>(pt);
    tile = sm.tail + pt;
    t.kb0 = t.split * a.n_kb / t.nsplit;
    t.kb1 = (t.split + 1) * a.n_kb / t.nsplit;
  }
  const uint32_t b = (__umulhi(tile, a.nt_magic) + tile) >> a.nt_shift;
  t.tile = tile;
  t.b = static_cast<int>(b);
  t.jt = static_cast<int>(tile - b * static_cast<uint32_t>(a.n_tg)) * a.tpu;
  t.e = __ldg(a.expert_ids + t.b);
  t.ok = t.e >= 0 && t.e < a.E;
  t.gi = 0;
  return t;
}

// The aligned block of unit u (plain calls): the block part of decode_unit, without the loads.
__device__ __forceinline__ uint32_t unit_block(const GemmArgs& a, const SplitMap& sm, int64_t u64) {
  const uint32_t tile = unit_tile(sm, static_cast<uint32_t>(u64));
  return (__umulhi(tile, a.nt_magic) + tile) >> a.nt_shift;
}

// CTA pairs: unit u = (block, pair of 128-row tiles); CTA rank r of the pair takes tile
// 2 * pair + r.  No K splits.
__device__ __forceinline__ Unit decode_unit_pair(const GemmArgs& a, uint32_t crank, int64_t u64) {
  const uint32_t u = static_cast<uint32_t>(u64);
  Unit t;
  const uint32_t b = (__umulhi(u, a.nt2_magic) + u) >> a.nt2_shift;
  t.tile = u;
  t.b = static_cast<int>(b);
  t.jt = static_cast<int>(2 * (u - b * static_cast<uint32_t>(a.n_tiles >> 1)) + crank);
  t.split = 0;
  t.nsplit = 1;
  t.ptile = 0;
  t.kb0 = 0;
  t.kb1 = a.n_kb;
  t.gi = 0;
  t.e = __ldg(a.expert_ids + t.b);
  t.ok = t.e >= 0 && t.e < a.E;
  return t;
}

// Fused layer: units [0, units0) are the first GEMM's (gate_up), the rest the second's (down),
// both over the same aligned blocks.  A plain call has one GEMM (a2 is a).
template <bool FUSED, bool PAIR = false>
__device__ __forceinline__ Unit decode_any(const GemmArgs& a, const GemmArgs& a2,
                                           const SplitMap& sm, uint32_t units0, uint32_t crank,
                                           int64_t u64) {
  if (PAIR) return decode_unit_pair(a, crank, u64);
  if (!FUSED) return decode_unit(a, sm, u64);
  const uint32_t u = static_cast<uint32_t>(u64);
  if (u < units0) return decode_unit(a, no_split(), u);
  Unit t = decode_unit(a2, no_split(), u - units0);
  t.gi = 1;
  return t;
}

// The per-GEMM arguments of a unit.
template <bool FUSED>
__device__ __forceinline__ const GemmArgs& args_of(const GemmArgs& a, const GemmArgs& a2,
                                                   const Unit& un) {
  return (FUSED && un.gi) ? a2 : a;
}

__device__ __forceinline__ void named_bar_epi() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// the 64 threads of the activation warps (2 and 3)
__device__ __forceinline__ void named_bar_act() {
  asm volatile("bar.sync 2, 64;" ::: "memory");
}

// OR of `pred` over the 128 epilogue threads (they all take the same branch afterwards, which
// warp-collective tcgen05 loads and the named barrier require).
__device__ __forceinline__ bool epi_any(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return out != 0;
}

// 256-bit global stores (sm_100 and later; the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(float* p, float4 x, float4 y) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(x.x),
               "f"(x.y), "f"(x.z), "f"(x.w), "f"(y.x), "f"(y.y), "f"(y.z), "f"(y.w)
               : "memory");
}
__device__ __forceinline__ void st_global_v8(uint16_t* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Output row of token column j of the unit's block, or -1 when nothing is written there.
__device__ __forceinline__ int64_t out_row(const GemmArgs& a, const Unit& un, int j, int32_t slot) {
  if (a.c_sorted) return static_cast<int64_t>(un.b) * a.block_m + j;  // padding rows get zeros
  return (slot >= 0 && slot < a.total_slots) ? slot : -1;
}

// Writes token columns [c0, c0 + 16) of this warp's 32 tile rows (lanes) to C.  The values go
// through the warp's staging area so that each lane ends up with consecutive output columns of
// one token row and stores them with 16-byte vector stores (lane l: token l / 2, half l % 2).
__device__ __forceinline__ void store_chunk16(const GemmArgs& a, const Unit& un, int q, int lane,
                                              int c0, const int32_t* rows,
                                              const uint32_t (&r)[16], uint8_t* stage) {
  const int tok = lane >> 1, half = lane & 1;
  const int32_t slot = rows[c0 + tok];
  const bool routed = (slot >= 0 && slot < a.total_slots);
  const int64_t row = out_row(a, un, c0 + tok, slot);
  if (a.epilogue == W4A16_EPILOGUE_SILU_MUL) {
    // Lane l < 16 holds gate rows and lane l + 16 the matching up rows.  For each pair of
    // tokens (j, j + 1) one exchange lets lane l compute token j and lane l + 16 token j + 1.
    // SiLU-and-mul takes the FP32 sums as they leave the accumulator (no BF16 gate_up tensor
    // exists between the two GEMMs); h is rounded to BF16 once.
    uint16_t* st = reinterpret_cast<uint16_t*>(stage);  // [16 tokens][16 columns]
    const bool hi = lane >= 16;
#pragma unroll
    for (int jj = 0; jj < 16; jj += 2) {
      const float v0 = __uint_as_float(r[jj]), v1 = __uint_as_float(r[jj + 1]);
      const float recv = __shfl_xor_sync(0xffffffffu, hi ? v0 : v1, 16);
      const float g = hi ? recv : v0;
      const float u = hi ? v1 : recv;
      const float h = __fdividef(g, 1.0f + __expf(-g)) * u;
      st[(jj + (hi ? 1 : 0)) * 16 + (lane & 15)] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
    }
    __syncwarp();
    if (row >= 0) {
      uint4 v = reinterpret_cast<const uint4*>(st)[tok * 2 + half];
      if (!routed) v = make_uint4(0, 0, 0, 0);
      const int col = 64 * un.jt + 16 * q + 8 * half;
      *reinterpret_cast<uint4*>(a.C + row * a.ldc + col) = v;
    }
  } else {
    // [16 tokens][36]: rows padded by 16 bytes so that the 16-byte reads below (lanes 2t and
    // 2t + 1 read token t) fall on distinct banks within each quarter warp
    float* st = reinterpret_cast<float*>(stage);
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) st[jj * 36 + lane] = __uint_as_float(r[jj]);
    __syncwarp();
    if (row >= 0) {
      const int col = tile_row_to_canonical(un.jt, 32 * q + 16 * half, a.N, a.paired != 0);
      const float4* src = reinterpret_cast<const float4*>(st + tok * 36 + 16 * half);
      if (a.merge_w) {
        // top-k merge: this slot's weighted row is added into its token's FP32 row
        if (routed) {
          const float w = __ldg(a.merge_w + slot);
          float* dst = reinterpret_cast<float*>(a.C) + static_cast<int64_t>(slot / a.merge_k) * a.ldc + col;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 v = src[k];
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * k),
                         "f"(w * v.x), "f"(w * v.y), "f"(w * v.z), "f"(w * v.w)
                         : "memory");
          }
        }
      } else if (a.c_f32) {
        float* dst = reinterpret_cast<float*>(a.C) + row * a.ldc + col;
        if (a.c_st256) {  // 32-byte aligned rows: half the store instructions
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            float4 x = src[2 * k], y = src[2 * k + 1];
            if (!routed) x = y = make_float4(0.f, 0.f, 0.f, 0.f);
            st_global_v8(dst + 8 * k, x, y);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            reinterpret_cast<float4*>(dst)[k] = routed ? src[k] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      } else {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 x = src[k];
          auto pk = [&](float lo, float hi2) {
            return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(routed ? lo : 0.f))) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(routed ? hi2 : 0.f))) << 16);
          };
          w[2 * k] = pk(x.x, x.y);
          w[2 * k + 1] = pk(x.z, x.w);
        }
        uint16_t* dst = a.C + row * a.ldc + col;
        if (a.c_st256) {
          st_global_v8(dst, w);
        } else {
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
  }
  __syncwarp();  // the staging area is reused by the next chunk
}

template <bool PAIR>
__device__ __forceinline__ void mma_any(uint32_t d, uint32_t a_tmem, uint64_t bd, uint32_t idesc,
                                        uint32_t acc) {
  if (PAIR) mma_ts_pair(d, a_tmem, bd, idesc, acc); else mma_ts(d, a_tmem, bd, idesc, acc);
}
template <bool PAIR>
__device__ __forceinline__ void commit_any(uint32_t bar) {
  if (PAIR) mma_commit_pair(bar); else mma_commit(bar);
}
// A hand-off arrival from a warp: in a pair kernel lane 0 arrives for the warp on the even
// CTA's barrier (locally or remotely); otherwise every thread arrives locally.
template <bool PAIR>
__device__ __forceinline__ void arrive_handoff(uint32_t bar, bool leader, int lane) {
  if (PAIR) {
    __syncwarp();
    if (lane == 0) {
      if (leader) mbar_arrive(bar); else mbar_arrive_remote(mapa_shared(bar, 0));
    }
  } else {
    mbar_arrive(bar);
  }
}

// TPU: 128-row tiles per unit (tile groups of short-K plain calls; 1 otherwise).
template <int NT, int KS, bool FUSED, bool PAIR = false, int TPU = 1>
__device__ __forceinline__ void gemm_body(const GemmArgs& a, const GemmArgs& a2) {
  using Cfg = GemmCfg<NT, KS, PAIR, TPU>;
  static_assert(TPU == 1 || (!FUSED && !PAIR), "tile groups are for plain calls");
  // PAIR: two-CTA clusters taking the two tiles of a tile pair of one block, with one
  // cta_group::2 MMA over both CTAs.
  constexpr bool CL = PAIR;
  constexpr int S_W = Cfg::kWStages;
  constexpr int S_B = Cfg::kBStages;
  constexpr int S_A = Cfg::kAStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* b_ring = base;                              // S_B x KS x [NT rows x 128 B], swizzled
  uint8_t* w_ring = base + S_B * Cfg::kBBytes;         // S_W x KS x 4608-byte chunks
  uint64_t* bars = reinterpret_cast<uint64_t*>(w_ring + S_W * Cfg::kWBytes);
  uint64_t* wfull = bars;              // weight stage landed (TMA bytes)
  uint64_t* wempty = wfull + S_W;      // weight stage read into registers (4 dequant warps)
  uint64_t* bfull = wempty + S_W;      // activation stage landed
  uint64_t* bempty = bfull + S_B;      // the MMAs reading the activation stage finished
  uint64_t* afull = bempty + S_B;      // dequantised A stage in TMEM written (128 threads)
  uint64_t* aempty = afull + S_A;      // the MMAs reading the A stage finished
  uint64_t* accfull = aempty + S_A;
  uint64_t* accempty = accfull + 2;
  uint64_t* drain = accempty + 2;
  uint32_t* misc = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* tmem_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(misc + 2);
  uint32_t* w_issued = misc + 3;
  uint32_t* b_issued = misc + 4;
  int32_t* epi_rows = reinterpret_cast<int32_t*>(misc + 16);  // sorted_ids of the unit's block
  // per-epilogue-warp staging for vectorised stores (16-byte aligned)
  uint8_t* epi_stage_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(epi_rows + NT) + 15) & ~static_cast<uintptr_t>(15));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // CTA pairs: the even CTA of each two-CTA cluster issues the MMAs; the odd CTA's activation
  // copies complete on the even CTA's barriers (cta_group::2 tensor copies) and its dequant and
  // epilogue warps arrive there remotely
  const uint32_t crank = CL ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const int64_t unit0 = CL ? (blockIdx.x >> 1) : blockIdx.x;
  const int64_t ustride = CL ? (gridDim.x >> 1) : gridDim.x;
  const bool gather = !a.a_sorted;
  // a fused call may mix gathered and TMA-loaded activations (one GEMM each): every stage then
  // completes on 64 arrivals, the TMA path's lane 0 also expecting the tile's bytes
  const bool any_tma = FUSED ? (a.a_sorted || a2.a_sorted) : a.a_sorted;

  if (tid == 0) {
    for (int s = 0; s < S_W; ++s) {
      mbar_init(smem_u32(&wfull[s]), 1);
      mbar_init(smem_u32(&wempty[s]), 4);
    }
    for (int s = 0; s < S_B; ++s) {
      mbar_init(smem_u32(&bfull[s]), PAIR ? 1 : ((FUSED || gather) ? kGatherThreads : 1));
      mbar_init(smem_u32(&bempty[s]), 1);
    }
    for (int s = 0; s < S_A; ++s) {
      mbar_init(smem_u32(&afull[s]), PAIR ? 8 : 128);  // pairs: one arrival per warp of both CTAs
      mbar_init(smem_u32(&aempty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&accfull[s]), 1);
      mbar_init(smem_u32(&accempty[s]), PAIR ? 8 : 128);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *last_flag = 0;
    *w_issued = 0;
    *b_issued = 0;
    fence_mbar_init();
  }
  if (warp == 2 && lane == 0) {
    if (a.a_sorted) tma_prefetch_desc(FUSED ? &a.tmap_a : &a.tmap_a3);
    if (FUSED && a2.a_sorted) tma_prefetch_desc(&a2.tmap_a);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CL) cluster_sync();  // both CTAs' barriers exist before either arrives on the other's
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (!a.routing_ready) pdl_wait();  // sorted_ids / expert_ids / ntp come from the align kernel
  // Dependents may start once every CTA is past this point; they only read routing we have
  // already waited for, and wait on our completion before reading our outputs.
  pdl_launch_dependents();

  int ntp = __ldg(a.ntp);
  if (ntp < 0) ntp = 0;
  if (ntp > a.capacity) ntp = static_cast<int>(a.capacity);
  const int64_t nblocks = ntp / a.block_m;
  // Decode schedule from the routed blocks (every role computes the same map from
  // num_tokens_padded).  When the whole-tile units end in a partial wave of at most half the
  // grid, the tiles of that last wave are cut into K slices (of >= kMinSplitKb K blocks) that
  // fill it: with no full wave (few tiles, long K) every tile is sliced.  A fixed split slices
  // every tile.  Fewer slices when the sliced tiles would overflow the partial-sum scratch.
  const int64_t units1 = nblocks * a.n_tg;
  SplitMap sm = no_split();
  int64_t units_split = units1;
  if (!FUSED && !CL && units1 > 0) {
    int64_t tail = units1;
    int sn = 1;
    if (a.split_auto) {
      const int64_t G = gridDim.x;
      const int64_t R = units1 % G;
      if (R > 0 && 2 * R <= G) {
        int ss = static_cast<int>(min(static_cast<int64_t>(a.split_k), G / R));
        while (ss > 1 && (a.n_kb < ss * kMinSplitKb || R * ss > a.max_split_units)) --ss;
        if (ss > 1) {
          sn = ss;
          tail = units1 - R;
        }
      }
    } else if (a.split_k > 1) {
      int ss = a.split_k;
      while (ss > 1 && units1 * ss > a.max_split_units) --ss;
      if (ss > 1) {
        sn = ss;
        tail = 0;
      }
    }
    if (sn > 1) {
      sm.tail = static_cast<uint32_t>(tail);
      sm.s = static_cast<uint32_t>(sn);
      units_split = tail + (units1 - tail) * sn;
    }
  }
  const int64_t units0 = CL ? nblocks * (a.n_tiles >> 1) : units_split;
  const int64_t n_units = FUSED ? units0 + nblocks * a2.n_tg : units0;
  const uint32_t units0_u = static_cast<uint32_t>(units0);

  if (warp == 0) {
    // ---------------- weight producer: one bulk copy per stage, on a rotating lane ------------
    // One thread's bulk copies are serviced one after another (about 300 ns each on GB300), so
    // successive stages go to different lanes and many copies are in flight at once.
    // Weights never depend on the previous kernel, so they stream before pdl_wait.
    const uint64_t policy = a.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
    uint32_t it = 0;
    for (int64_t u = CL ? unit0 : blockIdx.x; u < n_units; u += CL ? ustride : gridDim.x) {
      const Unit un = decode_any<FUSED, CL>(a, a2, sm, units0_u, crank, u);
      if (!un.ok) continue;
      const GemmArgs& g = args_of<FUSED>(a, a2, un);
      const uint8_t* strip = g.wblob + kHeaderBytes +
                             ((static_cast<int64_t>(un.e) * g.n_tiles + un.jt) * g.n_kb) * kChunkBytes;
      for (int kb = un.kb0; kb < un.kb1; kb += KS, ++it) {
        const int nsub = min(KS, un.kb1 - kb);
        const int s = it % S_W;
        const uint32_t ph = (it / S_W) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&wempty[s]), ph ^ 1, abort_flag, a.dev_err)))
          goto wprod_done;
        if (lane == static_cast<int>(it & 31)) {
          const uint32_t wb = smem_u32(&wfull[s]);
          mbar_arrive_expect_tx(wb, nsub * kChunkBytes);
          bulk_g2s(smem_u32(w_ring + s * Cfg::kWBytes), strip + static_cast<int64_t>(kb) * kChunkBytes,
                   nsub * kChunkBytes, wb, policy);
        }
        __syncwarp();
      }
    }
  wprod_done:
    if (lane == 0) *w_issued = it;
  } else if (warp == 2 || warp == 3) {
    // ---------------- activation producer ----------------
    pdl_wait();  // activations may be the previous kernel's output
    uint32_t it = 0;
    if constexpr (FUSED) {
      // Per unit: gathered rows (cp.async, both warps) or sorted rows (TMA issued by warp 2);
      // every stage completes on the 64 threads' arrivals.  Units of the second GEMM read rows
      // that other CTAs' first-GEMM epilogues write during this launch: thread 0 waits for the
      // block's completion count, then the async proxy is fenced before the tensor loads.
      const int gt = tid - 64;
      const int c = gt & 7;
      constexpr int R = NT / 8;
      for (int64_t u = CL ? unit0 : blockIdx.x; u < n_units; u += CL ? ustride : gridDim.x) {
        const Unit un = decode_any<FUSED, CL>(a, a2, sm, units0_u, crank, u);
        if (!un.ok) continue;
        const GemmArgs& g = args_of<FUSED>(a, a2, un);
        if (g.wait_done) {
          if (gt == 0)
            wait_count_at_least(g.wait_done + un.b, g.wait_count, abort_flag, g.dev_err,
                                g.wait_limit > 0 ? g.wait_limit : kWaitLimitCycles);
          named_bar_act();
          if (*abort_flag) goto fprod_done;
          fence_proxy_async_global();
        }
        if (!g.a_sorted) {
          // per row of this thread: its source (chunk c, K block 0), null for a padding row,
          // and its swizzled destination offset within a sub-block
          const uint16_t* srow[R];
          uint32_t doff[R];
#pragma unroll
          for (int j = 0; j < R; ++j) {
            const int32_t i = __ldg(g.sorted_ids + static_cast<int64_t>(un.b) * g.block_m + (gt >> 3) + 8 * j);
            const int r = (gt >> 3) + 8 * j;
            srow[j] = (i >= 0 && i < g.total_slots)
                          ? g.A + static_cast<int64_t>(i / g.a_row_div) * g.lda + c * 8
                          : nullptr;
            doff[j] = static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
          }
          for (int kb = un.kb0; kb < un.kb1; kb += KS, ++it) {
            const int nsub = min(KS, un.kb1 - kb);
            const int s = it % S_B;
            const uint32_t ph = (it / S_B) & 1;
            if (!mbar_wait(smem_u32(&bempty[s]), ph ^ 1, abort_flag, g.dev_err)) goto fprod_done;
            const uint32_t bdst = smem_u32(b_ring + s * Cfg::kBBytes);
            for (int sb = 0; sb < nsub; ++sb) {
              const uint32_t sdst = bdst + sb * Cfg::kSubB;
              const int koff = (kb + sb) * kBlockK;
#pragma unroll
              for (int j = 0; j < R; ++j)
                if (srow[j]) cp_async_16(sdst + doff[j], srow[j] + koff, 16u);
            }
            cp_async_arrive_noinc(smem_u32(&bfull[s]));
          }
        } else {
          for (int kb = un.kb0; kb < un.kb1; kb += KS, ++it) {
            const int nsub = min(KS, un.kb1 - kb);
            const int s = it % S_B;
            const uint32_t ph = (it / S_B) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bempty[s]), ph ^ 1, abort_flag, g.dev_err)))
              goto fprod_done;
            const uint32_t bb = smem_u32(&bfull[s]);
            if (gt == 0)
              mbar_arrive_expect_tx(bb, nsub * Cfg::kSubB);
            else
              mbar_arrive(bb);
            if (warp == 2) {
              __syncwarp();
              for (int sb = 0; sb < nsub; ++sb)
                if (lane == static_cast<int>(it & 31))
                  tma_load_2d(smem_u32(b_ring + s * Cfg::kBBytes + sb * Cfg::kSubB), &g.tmap_a,
                              (kb + sb) * kBlockK, static_cast<int>(un.b * g.block_m), bb);
              __syncwarp();
            }
          }
        }
      }
    fprod_done:
      cp_async_wait_all();
      if (warp == 2 && lane == 0) *b_issued = it;
    } else if (gather) {
      // rows gathered with 16-byte cp.async into the 128-byte-swizzled K-major layout
      const int g = tid - 64;
      const int c = g & 7;  // 16-byte chunk of a 128-byte row handled by this thread
      constexpr int R = NT / 8;  // rows per thread: (g >> 3) + 8j
      for (int64_t u = CL ? unit0 : blockIdx.x; u < n_units; u += CL ? ustride : gridDim.x) {
        const Unit un = decode_any<FUSED, CL>(a, a2, sm, units0_u, crank, u);
        if (!un.ok) continue;
        // per row of this thread: its source (chunk c of the row, K block 0) and its swizzled
        // destination offset within a sub-block; null source for padding rows
        const uint16_t* srow[R];
        uint32_t doff[R];
#pragma unroll
        for (int j = 0; j < R; ++j) {
          const int32_t i = __ldg(a.sorted_ids + static_cast<int64_t>(un.b) * a.block_m + (g >> 3) + 8 * j);
          const int r = (g >> 3) + 8 * j;
          srow[j] = (i >= 0 && i < a.total_slots)
                        ? a.A + static_cast<int64_t>(i / a.a_row_div) * a.lda + c * 8
                        : nullptr;
          doff[j] = static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
        }
        // a tile group's tiles share the block's activation stages: they are loaded once
        const int kb_end = TPU > 1 ? a.n_kb : un.kb1;
        for (int kb = un.kb0; kb < kb_end; kb += KS, ++it) {
          const int nsub = min(KS, kb_end - kb);
          const int s = it % S_B;
          const uint32_t ph = (it / S_B) & 1;
          if (!mbar_wait(smem_u32(&bempty[s]), ph ^ 1, abort_flag, a.dev_err)) goto bprod_done;
          const uint32_t bdst = smem_u32(b_ring + s * Cfg::kBBytes);
          // Padding rows are not loaded: MMA column j reads only B row j, so whatever a
          // padding row holds lands in a token column that the epilogue discards.
          for (int sb = 0; sb < nsub; ++sb) {
            const uint32_t sdst = bdst + sb * Cfg::kSubB;
            const int koff = (kb + sb) * kBlockK;
#pragma unroll
            for (int j = 0; j < R; ++j)
              if (srow[j]) cp_async_16(sdst + doff[j], srow[j] + koff, 16u);
          }
          cp_async_arrive_noinc(smem_u32(&bfull[s]));
        }
      }
    bprod_done:
      cp_async_wait_all();
    } else if (warp == 2) {
      // rows already in sorted order: one 3-D tensor copy per stage, issued by a lane that
      // rotates over the warp
      for (int64_t u = CL ? unit0 : blockIdx.x; u < n_units; u += CL ? ustride : gridDim.x) {
        const Unit un = decode_any<FUSED, CL>(a, a2, sm, units0_u, crank, u);
        if (!un.ok) continue;
        const int kb_end = TPU > 1 ? a.n_kb : un.kb1;  // tile groups: loaded once
        for (int kb = un.kb0; kb < kb_end; kb += KS, ++it) {
          const int s = it % S_B;
          const uint32_t ph = (it / S_B) & 1;
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bempty[s]), ph ^ 1, abort_flag, a.dev_err)))
            goto tprod_done;
          // pairs: both CTAs' halves complete on the even CTA's barrier, which expects both
          const uint32_t bb = PAIR ? mapa_shared(smem_u32(&bfull[s]), 0) : smem_u32(&bfull[s]);
          // the copy always moves KS blocks of 64 K: in a short last stage the blocks past K are
          // zero-filled (and still counted), those past a K slice's end are loaded and unused
          if (lane == 0 && (!PAIR || leader))
            mbar_arrive_expect_tx(smem_u32(&bfull[s]), (PAIR ? 2 : 1) * KS * Cfg::kSubB);
          __syncwarp();
          if (lane == static_cast<int>(it & 31)) {
            const uint32_t dst = smem_u32(b_ring + s * Cfg::kBBytes);
            const int y = static_cast<int>(un.b * a.block_m + (PAIR ? crank * (NT / 2) : 0));
            if (PAIR) tma_load_3d_pair(dst, &a.tmap_a3, 0, y, kb, bb);
            else tma_load_3d(dst, &a.tmap_a3, 0, y, kb, bb);
          }
          __syncwarp();
        }
      }
    tprod_done:
      if (lane == 0) *b_issued = it;
    }
  } else if (warp == 1) {
    // ---------------- MMA issue: one elected thread runs the whole loop ----------------
    // Measured on GB300: a burst of MMAs issued from a fully unrolled sequence inside one
    // long-lived elected region costs ~9 cycles per N=16 MMA, while re-electing every stage or
    // issuing from a rolled loop costs several hundred cycles per stage.
    constexpr uint32_t idesc = idesc_bf16_f32(PAIR ? 256 : 128, NT);
    const uint64_t b_desc0 = smem_desc_sw128(smem_u32(b_ring));
    if (PAIR && !leader) {
      // odd CTA of a pair: wait for the pair's last MMAs before the TMEM they write is released
      if (elect_one()) mbar_wait_plain(smem_u32(drain), 0);
    } else if (elect_one()) {
      uint32_t it = 0, itb = 0, lu = 0;  // A ring, activation ring, accumulator positions
      constexpr int tpu = TPU;
      for (int64_t u = CL ? unit0 : blockIdx.x; u < n_units; u += CL ? ustride : gridDim.x) {
        const Unit un = decode_any<FUSED, CL>(a, a2, sm, units0_u, crank, u);
        if (!un.ok) continue;
        const bool rows_gathered = FUSED ? !args_of<FUSED>(a, a2, un).a_sorted : gather;
        const int ab = lu & 1;
        const uint32_t pab = (lu >> 1) & 1;
        if (!mbar_wait(smem_u32(&accempty[ab]), pab ^ 1, abort_flag, a.dev_err)) goto mma_done;
        tc_fence_after();
        // a tile group's tiles accumulate side by side: buffer ab holds tpu * NT columns
        const uint32_t d_tmem = tmem_base + ab * (NT * tpu);
        // A stage's release (the commits to its two "empty" barriers) is issued only after the
        // next stage's operands are seen ready, just before that stage's MMAs: measured on GB300
        // a wait issued right after the commits costs ~3% at decode.  The commits still follow
        // the stage's own MMAs, so they track exactly those.  The tiles of a group read the
        // block's activation stages in turn; a stage is released after the last tile's MMAs.
        int prev_sbi = -1, prev_sa = 0;
        bool prev_rel_b = true;
        int bs = 0;  // activation stage of this K stage within the unit (per tile in a group)
        int tg = 0;  // tile of the group
        for (int kb = un.kb0; kb < un.kb1; kb += KS, ++it) {
          const int nsub = min(KS, un.kb1 - kb);
          const uint32_t jb = itb + static_cast<uint32_t>(bs);
          const int sbi = jb % S_B;
          const uint32_t pb = (jb / S_B) & 1;
          const int sa = it % S_A;
          const uint32_t pa = (it / S_A) & 1;
          if (!mbar_wait(smem_u32(&afull[sa]), pa, abort_flag, a.dev_err)) goto mma_done;
          if (tg == 0) {
            if (!mbar_wait(smem_u32(&bfull[sbi]), pb, abort_flag, a.dev_err)) goto mma_done;
            if (rows_gathered) fence_proxy_async_smem();  // cp.async (generic proxy) rows -> tensor core
          }
          tc_fence_after();
          if (prev_sbi >= 0) {
            if (prev_rel_b) commit_any<PAIR>(smem_u32(&bempty[prev_sbi]));
            commit_any<PAIR>(smem_u32(&aempty[prev_sa]));
          }
          const uint64_t b_desc = b_desc0 + static_cast<uint64_t>((sbi * Cfg::kBBytes) >> 4);
          const uint32_t a_tmem = tmem_base + Cfg::kACol0 + sa * (KS * 32);
          const uint32_t acc0 = bs > 0 ? 1u : 0u;
          const uint32_t dt = d_tmem + static_cast<uint32_t>(tg * NT);
          if (nsub == KS) {
#pragma unroll
            for (int sb = 0; sb < KS; ++sb) {
              const uint64_t bd = b_desc + static_cast<uint64_t>((sb * Cfg::kSubB) >> 4);
              const uint32_t at = a_tmem + sb * 32;
              mma_any<PAIR>(dt, at, bd, idesc, sb > 0 ? 1u : acc0);
              mma_any<PAIR>(dt, at + 8, bd + 2, idesc, 1u);
              mma_any<PAIR>(dt, at + 16, bd + 4, idesc, 1u);
              mma_any<PAIR>(dt, at + 24, bd + 6, idesc, 1u);
            }
          } else {  // K tail shorter than a full stage
            for (int sb = 0; sb < nsub; ++sb) {
              const uint64_t bd = b_desc + static_cast<uint64_t>((sb * Cfg::kSubB) >> 4);
              const uint32_t at = a_tmem + sb * 32;
              mma_any<PAIR>(dt, at, bd, idesc, sb > 0 ? 1u : acc0);
              mma_any<PAIR>(dt, at + 8, bd + 2, idesc, 1u);
              mma_any<PAIR>(dt, at + 16, bd + 4, idesc, 1u);
              mma_any<PAIR>(dt, at + 24, bd + 6, idesc, 1u);
            }
          }
          prev_sbi = sbi;
          prev_sa = sa;
          prev_rel_b = tg == tpu - 1;
          ++bs;
          if (tpu > 1 && bs * KS >= a.n_kb) {  // next tile of the group
            bs = 0;
            ++tg;
          }
        }
        if (prev_sbi >= 0) {
          if (prev_rel_b) commit_any<PAIR>(smem_u32(&bempty[prev_sbi]));
          commit_any<PAIR>(smem_u32(&aempty[prev_sa]));
        }
        commit_any<PAIR>(smem_u32(&accfull[ab]));
        itb += static_cast<uint32_t>(tpu > 1 ? a.n_kb / KS : bs);
        ++lu;
      }
    mma_done:
      commit_any<PAIR>(smem_u32(drain));
      mbar_wait_plain(smem_u32(drain), 0);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---------------- epilogue warpgroup ----------------
    pdl_wait();  // outputs may still be read by the previous kernel
    const int q = warp - 4;
    const int t = q * 32 + lane;  // tile row = TMEM lane
    uint8_t* epi_stage = epi_stage_base + q * kEpiStageBytes;
    uint32_t lu = 0;
    // single-kernel layer: zero this CTA's slice of the FP32 token sums, then count it
    bool sums_zeroed = !(FUSED && a2.sync);
    if (FUSED && a2.sync) {
      float4* sums = reinterpret_cast<float4*>(a2.C);
      const int64_t n4 = a2.sum_elems / 4;
      for (int64_t i = static_cast<int64_t>(blockIdx.x) * 128 + t; i < n4;
           i += static_cast<int64_t>(gridDim.x) * 128)
        sums[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      named_bar_epi();
      if (t == 0) red_release_add(a2.sync, 1);
    }
    // Plain calls on 64- and 128-token blocks without the SiLU epilogue (the FP32 down
    // projection, whose epilogue bounds it at prefill), and plain calls whose units are at
    // most two pipeline stages (K <= 512), load the next unit's row ids while draining this
    // one.  Measured on GB300: Qwen3 T=4096 down 116.7 -> 113 us; Kimi-K2 TP8 down (K = 256,
    // 16-token blocks) 70.3 -> 64.2 us at T=32, 137.9 -> 125.6 at T=256, 193.2 -> 178.8 at
    // T=1024 (single flushed calls); the SiLU epilogue and 16-token blocks of longer units
    // ran 0.1-0.7 us slower with it.  (Loading every role's expert ids two units ahead was
    // slower everywhere, e.g. the TP8 down at T=1024 back to 211.6 us.)
    const bool ids_ahead = !FUSED && !CL &&
                           ((NT >= 64 && a.epilogue != W4A16_EPILOGUE_SILU_MUL) || a.n_kb <= 8);
    int64_t ahead_u = -1;
    int32_t ahead_row = 0;
    for (int64_t u = CL ? unit0 : blockIdx.x; u < n_units; u += CL ? ustride : gridDim.x) {
      const Unit un = decode_any<FUSED, CL>(a, a2, sm, units0_u, crank, u);
      if (!un.ok) continue;
      const GemmArgs& g = args_of<FUSED>(a, a2, un);
      named_bar_epi();  // the previous unit's readers of epi_rows / last_flag are done
      if (t < NT)
        epi_rows[t] = ahead_u == u ? ahead_row
                                   : __ldg(a.sorted_ids + static_cast<int64_t>(un.b) * a.block_m + t);
      named_bar_epi();
      const int ab = lu & 1;
      const uint32_t pab = (lu >> 1) & 1;
      const bool ok = mbar_wait(smem_u32(&accfull[ab]), pab, abort_flag, a.dev_err);
      if (epi_any(!ok)) break;
      if (ids_ahead && u + gridDim.x < n_units) {
        ahead_u = u + gridDim.x;
        const uint32_t nb = unit_block(a, sm, ahead_u);
        ahead_row = t < NT ? __ldg(a.sorted_ids + static_cast<int64_t>(nb) * a.block_m + t) : 0;
      }
      if (FUSED && g.sync && !sums_zeroed) {
        // the first merge of this CTA: every CTA's slice of the sums must be zero
        if (t == 0) wait_count_at_least(g.sync, static_cast<int32_t>(gridDim.x), abort_flag, g.dev_err);
        named_bar_epi();
        sums_zeroed = true;
      }
      tc_fence_after();
      // a tile group's accumulators sit side by side: tpu * NT columns, tile c / NT
      constexpr int ncol = NT * TPU;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * ncol;
      if (un.nsplit == 1) {
        // TMEM loads are double-buffered: the next 16 columns are in flight while the current
        // ones are converted and stored.
        auto store_cols = [&](int c, const uint32_t(&r)[16]) {
          Unit ut = un;
          ut.jt = un.jt + c / NT;
          store_chunk16(g, ut, q, lane, c % NT, epi_rows, r, epi_stage);
        };
        uint32_t r0[16], r1[16];
        tmem_ld16(taddr, r0);
#pragma unroll 1
        for (int c0 = 0; c0 < ncol; c0 += 32) {
          tmem_wait_ld16(r0);
          if (c0 + 16 < ncol) tmem_ld16(taddr + c0 + 16, r1);
          if (c0 + 16 >= ncol) {
            tc_fence_before();
            arrive_handoff<PAIR>(smem_u32(&accempty[ab]), leader, lane);
          }
          store_cols(c0, r0);
          if (c0 + 16 < ncol) {
            tmem_wait_ld16(r1);
            if (c0 + 32 < ncol) tmem_ld16(taddr + c0 + 32, r0);
            if (c0 + 32 >= ncol) {
              tc_fence_before();
              arrive_handoff<PAIR>(smem_u32(&accempty[ab]), leader, lane);
            }
            store_cols(c0 + 16, r1);
          }
        }
      } else {
        const int nsplit = un.nsplit;
        float* part = a.part + (static_cast<int64_t>(un.ptile) * nsplit + un.split) * (128 * NT);
#pragma unroll 1
        for (int c0 = 0; c0 < NT; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(taddr + c0, r);
          tmem_wait_ld16(r);
          if (c0 + 16 >= NT) {
            tc_fence_before();
            arrive_handoff<PAIR>(smem_u32(&accempty[ab]), leader, lane);
          }
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) __stcg(part + (c0 + jj) * 128 + t, __uint_as_float(r[jj]));
        }
        __threadfence();
        named_bar_epi();
        if (t == 0) *last_flag = (atomicAdd(a.cnt + un.ptile, 1) == nsplit - 1) ? 1 : 0;
        named_bar_epi();
        if (*last_flag) {
          __threadfence();
          const float* tile_parts = a.part + static_cast<int64_t>(un.ptile) * nsplit * (128 * NT);
#pragma unroll 1
          for (int c0 = 0; c0 < NT; c0 += 16) {
            // splits summed in order; the 16 columns of one split load together
            float v[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) v[jj] = __ldcg(tile_parts + (c0 + jj) * 128 + t);
            for (int s = 1; s < nsplit; ++s) {
              float w[16];
#pragma unroll
              for (int jj = 0; jj < 16; ++jj)
                w[jj] = __ldcg(tile_parts + s * (128 * NT) + (c0 + jj) * 128 + t);
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) v[jj] += w[jj];
            }
            uint32_t r[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) r[jj] = __float_as_uint(v[jj]);
            store_chunk16(g, un, q, lane, c0, epi_rows, r, epi_stage);
          }
          if (t == 0) a.cnt[un.ptile] = 0;  // ready for the next call
        }
      }
      if (FUSED && g.signal_done) {
        // the unit's rows are stored: count the tile done for its block (the barrier orders
        // every epilogue thread's stores before thread 0's release increment)
        named_bar_epi();
        if (t == 0) red_release_add(g.signal_done + un.b, 1);
      }
      ++lu;
    }
    if (FUSED && a2.sync && a2.final_out) {
      // every CTA's merges are done: round this CTA's slice of the sums to BF16
      named_bar_epi();
      if (t == 0) {
        red_release_add(a2.sync + 1, 1);
        wait_count_at_least(a2.sync + 1, static_cast<int32_t>(gridDim.x), abort_flag, a2.dev_err);
      }
      named_bar_epi();
      if (!*abort_flag) {
        const float4* sums = reinterpret_cast<const float4*>(a2.C);
        uint4* out = reinterpret_cast<uint4*>(a2.final_out);
        const int64_t n8 = a2.sum_elems / 8;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * 128 + t; i < n8;
             i += static_cast<int64_t>(gridDim.x) * 128) {
          const float4 x = __ldcg(sums + 2 * i), y = __ldcg(sums + 2 * i + 1);
          auto pk = [](float lo, float hi) {
            return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
                   (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
          };
          out[i] = make_uint4(pk(x.x, x.y), pk(x.z, x.w), pk(y.x, y.y), pk(y.z, y.w));
        }
      }
    }
  } else if (warp >= 8) {
    // ---------------- dequant warpgroups (stages rotate over the groups) ----------------
    const int g = (warp - 8) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + Cfg::kACol0;
    uint32_t it = 0;
    for (int64_t u = CL ? unit0 : blockIdx.x; u < n_units; u += CL ? ustride : gridDim.x) {
      const Unit un = decode_any<FUSED, CL>(a, a2, sm, units0_u, crank, u);
      if (!un.ok) continue;
      // the tile's INT4 conversion (uniform over a tile, read while the weights are in flight;
      // a tile group's modes are read together, one byte per tile)
      const GemmArgs& ga = args_of<FUSED>(a, a2, un);
      constexpr int tpu = TPU;
      uint32_t modes = 0;
      for (int j = 0; j < tpu; ++j)
        modes |= static_cast<uint32_t>(
                     __ldg(ga.tile_mode + static_cast<int64_t>(un.e) * ga.n_tiles + un.jt + j))
                 << (8 * j);
      const bool nvfp4 = ga.nvfp4 != 0;
      for (int kb = un.kb0; kb < un.kb1; kb += KS, ++it) {
        if (it % kDqGroups != static_cast<uint32_t>(g)) continue;
        const int tg = tpu > 1 ? kb / ga.n_kb : 0;  // tile of the group this stage belongs to
        const bool scaled = ((modes >> (8 * tg)) & 0xFFu) == kTileScaled;
        const int nsub = min(KS, un.kb1 - kb);
        const int sw = it % S_W;
        const uint32_t pw = (it / S_W) & 1;
        const int sa = it % S_A;
        const uint32_t pa = (it / S_A) & 1;
        // warp-uniform decisions: tcgen05.st below is a warp-collective instruction
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&wfull[sw]), pw, abort_flag, a.dev_err)))
          goto dq_done;
        if (TPU > 1 && scaled && !nvfp4) {
          // tile groups (one stage per tile): block 0 is converted while the A slot is still
          // busy, the other blocks' codes are read after it frees (the weight stage is released
          // after them).  Measured on GB300: Kimi-K2 TP8 down at T=1024 (32-token blocks,
          // groups of 2) 142.0 -> 131.7 us; without groups it gained nothing and cost up to
          // 2 us at 16-token gate_up calls.
          const uint8_t* wst = w_ring + sw * Cfg::kWBytes;
          uint32_t v0[32];
          dequant_row64_scaled(reinterpret_cast<const uint4*>(wst)[t],
                               reinterpret_cast<const uint4*>(wst + kCodeHalfBytes)[t],
                               reinterpret_cast<const uint32_t*>(wst + kScaleOffset)[t], v0);
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&aempty[sa]), pa ^ 1, abort_flag, a.dev_err)))
            goto dq_done;
          tc_fence_after();
          tmem_st32(lane_base + sa * (KS * 32), v0);
#pragma unroll
          for (int sb = 1; sb < KS; ++sb) {
            if (sb < nsub) {
              const uint8_t* ch = wst + sb * kChunkBytes;
              uint32_t v[32];
              dequant_row64_scaled(reinterpret_cast<const uint4*>(ch)[t],
                                   reinterpret_cast<const uint4*>(ch + kCodeHalfBytes)[t],
                                   reinterpret_cast<const uint32_t*>(ch + kScaleOffset)[t], v);
              tmem_st32(lane_base + sa * (KS * 32) + sb * 32, v);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&wempty[sw]));
          tmem_wait_st();
          tc_fence_before();
          arrive_handoff<PAIR>(smem_u32(&afull[sa]), leader, lane);
          continue;
        }
        uint4 lo[KS], hi[KS];
        uint32_t s2[KS];
#pragma unroll
        for (int sb = 0; sb < KS; ++sb) {
          if (sb < nsub) {
            const uint8_t* ch = w_ring + sw * Cfg::kWBytes + sb * kChunkBytes;
            lo[sb] = reinterpret_cast<const uint4*>(ch)[t];
            hi[sb] = reinterpret_cast<const uint4*>(ch + kCodeHalfBytes)[t];
            s2[sb] = reinterpret_cast<const uint32_t*>(ch + kScaleOffset)[t];
          }
        }
        __syncwarp();  // every lane holds its rows: the weight stage may be refilled
        if (lane == 0) mbar_arrive(smem_u32(&wempty[sw]));
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&aempty[sa]), pa ^ 1, abort_flag, a.dev_err)))
          goto dq_done;
        tc_fence_after();
        if (nvfp4) {
#pragma unroll
          for (int sb = 0; sb < KS; ++sb) {
            if (sb < nsub) {
              uint32_t v[32];
              dequant_row64_nvfp4(lo[sb], hi[sb], s2[sb], v);
              tmem_st32(lane_base + sa * (KS * 32) + sb * 32, v);
            }
          }
        } else if (scaled) {
#pragma unroll
          for (int sb = 0; sb < KS; ++sb) {
            if (sb < nsub) {
              uint32_t v[32];
              dequant_row64_scaled(lo[sb], hi[sb], s2[sb], v);
              tmem_st32(lane_base + sa * (KS * 32) + sb * 32, v);
            }
          }
        } else {
#pragma unroll
          for (int sb = 0; sb < KS; ++sb) {
            if (sb < nsub) {
              uint32_t v[32];
              dequant_row64(lo[sb], hi[sb], s2[sb], v);
              tmem_st32(lane_base + sa * (KS * 32) + sb * 32, v);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        arrive_handoff<PAIR>(smem_u32(&afull[sa]), leader, lane);
      }
    }
  dq_done:;
  }

  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // give in-flight copies a bounded chance to land before the CTA's memory goes away
    const uint32_t nw = *w_issued, nb = *b_issued;
    for (uint32_t j = (nw > static_cast<uint32_t>(S_W) ? nw - S_W : 0); j < nw; ++j)
      mbar_wait_plain(smem_u32(&wfull[j % S_W]), (j / S_W) & 1);
    if (any_tma && (!PAIR || leader))  // a pair's activation loads complete on the even CTA
      for (uint32_t j = (nb > static_cast<uint32_t>(S_B) ? nb - S_B : 0); j < nb; ++j)
        mbar_wait_plain(smem_u32(&bfull[j % S_B]), (j / S_B) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (CL) cluster_sync();  // the peer is done with the pair's TMEM and barriers
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, kTmemCols); else tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int NT, int KS, int TPU>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmArgs a) {
  gemm_body<NT, KS, false, false, TPU>(a, a);
}

// CTA pairs (128-token blocks): launched as two-CTA clusters; one M = 256 MMA covers the two
// CTAs' 128-row weight tiles, each CTA holding half of the block's activation rows.
template <int NT, int KS>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ GemmArgs a) {
  gemm_body<NT, KS, false, true>(a, a);
}

// Fused layer: the gate_up GEMM (a, SiLU-and-mul into sorted rows) and the down GEMM (a2, rows
// of the first by TMA, top-k merge epilogue) walked as one persistent unit sequence.  Down
// units wait per block for the gate_up tiles of that block, which earlier units of this grid
// produce; the launch is cooperative so that every CTA is resident.
template <int NT, int KS>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_layer_kernel(const __grid_constant__ GemmArgs a, const __grid_constant__ GemmArgs a2) {
  gemm_body<NT, KS, true>(a, a2);
}

// ------------------------------------------------------------------------------------------
// Host side: planner, tensor maps and launcher.
// ------------------------------------------------------------------------------------------

// Stage depth: every stage costs barrier round trips and an MMA burst on top of its bytes, so
// blocks up to 64 tokens move four 64-wide K blocks per stage (18432-byte weight copies, 16
// MMAs; measured fastest on GB300 against 2, 3, 5 and 6); 128-token blocks keep two, since
// their activation tiles and accumulators then bound shared memory and TMEM.
template <int NT> struct StageK { static constexpr int value = NT <= 64 ? 4 : 2; };

int stages_for_block_m(int block_m) {
  switch (block_m) {
    case 16: return GemmCfg<16, StageK<16>::value>::kWStages;
    case 32: return GemmCfg<32, StageK<32>::value>::kWStages;
    case 64: return GemmCfg<64, StageK<64>::value>::kWStages;
    case 128: return GemmCfg<128, StageK<128>::value>::kWStages;
    default: return 0;
  }
}

// Expected number of aligned blocks: experts hit at least once (Poisson estimate), each with
// ceil(rows / block_m) blocks.
double expected_blocks(int total_slots, int E, int block_m, double rows_per_expert) {
  if (E <= 0 || total_slots <= 0) return 0.0;
  const double r = rows_per_expert > 0 ? rows_per_expert : static_cast<double>(total_slots) / E;
  const double active = E * (1.0 - std::exp(-r));
  const double per = std::max(1.0, std::ceil(r / block_m));
  return std::min(active * per, static_cast<double>(total_slots));
}

// Split-K: the split itself is chosen on the device from the routed block count (the host
// cannot know it without a read-back).  For decode block sizes the planner allows up to
// kMaxAutoSplit slices of at least kMinSplitKb K blocks and launches one CTA per SM unless its
// estimate of units fills half the grid without slicing.  On the device: where the routed
// units leave SMs idle (one or a few experts with long K, e.g. 32 tiles of K = 7168) every
// tile is sliced until the units fill one wave; where the units end in a partial wave of at
// most half the grid, only that wave's tiles are sliced to fill it (Kimi-K2 EP8 T=16 gate_up,
// 512 units on 152 CTAs: the last 56 tiles in two slices, 62.1 -> 58.0 us).
// Measured on GB300: slicing K = 2048 in two with no full wave (Kimi-K2 EP8 down at T=1, 56
// tiles -> 112 units) is slower (7.5 -> 8.3 us), slicing K = 7168 in four (32 tiles -> 128
// units) much faster (gate_up 16.3 -> 10.5 us); a second wave of half-length units plus the
// partial round trip is slower than one wave of whole ones (Qwen3 T=1 gate_up, 96 units:
// 7.9 -> 11.1 us).
void plan_gemm(int total_slots, int E, int N, int K, int block_m, int rows_per_expert,
               int num_sms, w4a16_plan_t* plan) {
  const int n_tiles = N / kTileRows, n_kb = K / kBlockK;
  const double blocks = expected_blocks(total_slots, E, block_m, rows_per_expert);
  const double units1 = std::max(1.0, std::ceil(blocks)) * n_tiles;
  const int split_max =
      block_m <= kMaxSplitBlockM ? std::max(1, std::min(kMaxAutoSplit, n_kb / kMinSplitKb)) : 1;
  plan->block_m = block_m;
  plan->split_k = split_max;
  plan->est_units = static_cast<int32_t>(std::min(units1, 2.0e9));
  const bool few = 2.0 * units1 < num_sms;
  plan->num_ctas = (split_max > 1 && few) ? num_sms
                                          : std::max(1, std::min(num_sms, plan->est_units));
  plan->stages = stages_for_block_m(block_m);
  plan->cta_pairs = pairs_pay(block_m, n_tiles, n_kb) ? 2 : 1;
}

// cuTensorMapEncodeTiled from the driver (fetched once; no link-time libcuda dependency).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Activations as a 2-D BF16 tensor [rows, K] with row stride lda, 128-byte swizzle; the box is
// 64 columns by box_rows rows (the single-kernel layer's sorted tiles, one copy per 64 K).
cudaError_t make_act_tmap(CUtensorMap* map, const uint16_t* A, int64_t rows, int K, int64_t lda,
                          int box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(lda) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(A), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The same rows as a 3-D tensor [K / 64][rows][64] (x: 64 columns, y: rows, z: K block), box
// 64 x box_rows x box_kb: one copy fills a pipeline stage of box_kb blocks, laid out as box_kb
// consecutive [box_rows][64] tiles (the swizzle follows the shared-memory address, so this is
// the layout of box_kb separate 2-D copies).  Measured on GB300 against one 2-D copy per
// block: Qwen3 T=4096 gate_up 170.7 -> 165.0 us, Kimi-K2 EP8 T=8192 326.3 -> 314.0.
cudaError_t make_act_tmap3(CUtensorMap* map, const uint16_t* A, int64_t rows, int K, int64_t lda,
                           int box_rows, int box_kb) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kBlockK), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(K / kBlockK)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(lda) * 2,
                                 static_cast<cuuint64_t>(kBlockK) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_kb)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(A), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int NT, int TPU>
cudaError_t launch_gemm_tpu(GemmArgs& args, int grid, bool pdl, cudaStream_t stream) {
  constexpr int KS = StageK<NT>::value;
  using Cfg = GemmCfg<NT, KS, false, TPU>;
  static bool configured = false;  // per-process; attribute applies to the current device
  if (!configured) {
    cudaError_t err = cudaFuncSetAttribute(moe_gemm_kernel<NT, KS, TPU>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(Cfg::kSmemBytes));
    if (err != cudaSuccess) return err;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gemm_kernel<NT, KS, TPU>, args);
}

template <int NT>
cudaError_t launch_gemm_t(GemmArgs& args, int grid, bool pdl, cudaStream_t stream) {
  if constexpr (tile_group_max(NT) >= 4)
    if (args.tpu == 4) return launch_gemm_tpu<NT, 4>(args, grid, pdl, stream);
  if constexpr (tile_group_max(NT) >= 2)
    if (args.tpu == 2) return launch_gemm_tpu<NT, 2>(args, grid, pdl, stream);
  if (args.tpu != 1) return cudaErrorInvalidValue;
  return launch_gemm_tpu<NT, 1>(args, grid, pdl, stream);
}

template <int NT>
cudaError_t launch_layer_t(GemmArgs& a, GemmArgs& a2, int grid, cudaStream_t stream) {
  constexpr int KS = StageK<NT>::value;
  using Cfg = GemmCfg<NT, KS>;
  static bool configured = false;
  if (!configured) {
    cudaError_t err = cudaFuncSetAttribute(moe_layer_kernel<NT, KS>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(Cfg::kSmemBytes));
    if (err != cudaSuccess) return err;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;  // down units wait on other CTAs' gate_up units
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, moe_layer_kernel<NT, KS>, a, a2);
}

cudaError_t launch_layer_fused(GemmArgs& a, GemmArgs& a2, int grid, cudaStream_t stream) {
  if (a.block_m != a2.block_m || a.split_k != 1 || a2.split_k != 1) return cudaErrorInvalidValue;
  if (a.capacity <= 0) return cudaSuccess;
  if (a.a_sorted) {
    cudaError_t err = make_act_tmap(&a.tmap_a, a.A, a.capacity, a.K, a.lda, a.block_m);
    if (err != cudaSuccess) return err;
  }
  if (a2.a_sorted) {
    cudaError_t err = make_act_tmap(&a2.tmap_a, a2.A, a2.capacity, a2.K, a2.lda, a2.block_m);
    if (err != cudaSuccess) return err;
  }
  switch (a.block_m) {
    case 16: return launch_layer_t<16>(a, a2, grid, stream);
    case 32: return launch_layer_t<32>(a, a2, grid, stream);
    case 64: return launch_layer_t<64>(a, a2, grid, stream);
    case 128: return launch_layer_t<128>(a, a2, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

static cudaError_t launch_gemm_pair(GemmArgs& args, int grid, bool pdl, cudaStream_t stream) {
  constexpr int NT = 128, KS = StageK<NT>::value;
  using Cfg = GemmCfg<NT, KS, true>;
  auto kernel = moe_gemm_pair_kernel<NT, KS>;
  static bool configured = false;
  if (!configured) {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(Cfg::kSmemBytes));
    if (err != cudaSuccess) return err;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid & ~1);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

cudaError_t launch_gemm(GemmArgs& args, int grid, bool pdl, cudaStream_t stream) {
  if (args.pair) {  // block_m 128, sorted rows, even tile count, no K split (checked by the caller)
    if (args.block_m != 128 || !args.a_sorted || args.split_k != 1 || args.n_tiles % 2 || grid < 2)
      return cudaErrorInvalidValue;
    cudaError_t err = make_act_tmap3(&args.tmap_a3, args.A, args.capacity, args.K, args.lda,
                                     args.block_m / 2, StageK<128>::value);
    if (err != cudaSuccess) return err;
    return launch_gemm_pair(args, grid, pdl, stream);
  }
  const int64_t rows = args.a_sorted
                           ? args.capacity
                           : (static_cast<int64_t>(args.total_slots) + args.a_row_div - 1) /
                                 args.a_row_div;
  if (rows <= 0) return cudaSuccess;  // nothing can be routed
  if (args.a_sorted) {  // sorted rows: one 3-D TMA copy of block_m rows per pipeline stage
    const int stage_kb = args.block_m <= 64 ? StageK<64>::value : StageK<128>::value;
    cudaError_t err = make_act_tmap3(&args.tmap_a3, args.A, rows, args.K, args.lda, args.block_m,
                                     stage_kb);
    if (err != cudaSuccess) return err;
  }
  switch (args.block_m) {
    case 16: return launch_gemm_t<16>(args, grid, pdl, stream);
    case 32: return launch_gemm_t<32>(args, grid, pdl, stream);
    case 64: return launch_gemm_t<64>(args, grid, pdl, stream);
    case 128: return launch_gemm_t<128>(args, grid, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4a16
