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
//   * warp 0 streams 4608-byte packed chunks with 1-D bulk TMA (evict_first for streamed
//     weights); warps 2-3 gather activation rows with cp.async (row = sorted_ids[p] / div);
//     warps 8-15 (two dequant warpgroups, alternating stages) turn codes into BF16 pairs and
//     store them to TMEM with tcgen05.st; warp 1 issues tcgen05.mma from one thread; warps
//     4-7 drain the double-buffered accumulator with tcgen05.ld and write BF16 results;
//   * a persistent grid walks (block, 128-row tile, K split) units found from
//     num_tokens_padded on the device (no host read-back); K splits (decode) write FP32
//     partials and the last CTA to arrive on a per-tile counter sums them in split order,
//     so results are deterministic.
#include <algorithm>
#include <cmath>

#include "gemm.cuh"

namespace w4a16 {

constexpr int kGemmThreads = 512;
constexpr int kTmemCols = 512;
constexpr int kACol0 = 256;  // TMEM columns [256, 512): dequantised A stages, 32 columns each
constexpr int kAStages = 8;
constexpr int kGatherThreads = 64;  // warps 2 and 3
constexpr int kSmemBudget = 200 * 1024;

template <int NT>
struct GemmCfg {
  static constexpr int kBBytes = NT * 128;  // NT rows x 64 BF16
  static constexpr int kStageBytes = kBBytes + kChunkBytes;
  static constexpr int kStagesRaw = (kSmemBudget - 2048) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 32 ? 32 : kStagesRaw;
  static constexpr int kBarBytes = (3 * kStages + 2 * kAStages + 5) * 8;
  static constexpr size_t kSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + kBarBytes + 64;
  static_assert(NT % 16 == 0 && NT >= 16 && NT <= 128, "MMA N must be 16..128 in steps of 16");
  static_assert(2 * NT <= kACol0, "accumulators must fit below the A stages");
};



struct Unit {
  int b, jt, split, kb0, kb1, e;
  int64_t tile;
  bool ok;  // the block names a valid expert
};

__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, int split_k, int64_t u) {
  Unit t;
  t.split = static_cast<int>(u % split_k);
  t.tile = u / split_k;
  t.jt = static_cast<int>(t.tile % a.n_tiles);
  t.b = static_cast<int>(t.tile / a.n_tiles);
  t.kb0 = t.split * a.n_kb / split_k;
  t.kb1 = (t.split + 1) * a.n_kb / split_k;
  t.e = __ldg(a.expert_ids + t.b);
  t.ok = t.e >= 0 && t.e < a.E;
  return t;
}

__device__ __forceinline__ void named_bar_epi() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
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

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// Store one accumulator column (token column j of the block) for tile row t.
__device__ __forceinline__ void store_column(const GemmArgs& a, const Unit& un, int t, int j,
                                             float v) {
  // SiLU-and-mul needs the up value from lane + 16 of the same warp (all lanes shuffle).
  const float up = __shfl_down_sync(0xffffffffu, v, 16);
  const int64_t p = static_cast<int64_t>(un.b) * a.block_m + j;
  int64_t row;
  if (a.c_sorted) {
    row = p;
  } else {
    const int32_t i = __ldg(a.sorted_ids + p);
    if (i >= a.total_slots || i < 0) return;
    row = i;
  }
  if (a.epilogue == W4A16_EPILOGUE_SILU_MUL) {
    const int l = t & 31;
    if (l >= 16) return;
    const float g = bf16_round(v), u = bf16_round(up);
    const float h = g / (1.0f + expf(-g)) * u;
    const int col = 64 * un.jt + 16 * (t >> 5) + l;
    a.C[row * a.ldc + col] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
  } else {
    const int n = tile_row_to_canonical(un.jt, t, a.N, a.paired != 0);
    if (a.c_f32)
      reinterpret_cast<float*>(a.C)[row * a.ldc + n] = v;
    else
      a.C[row * a.ldc + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

template <int NT>
__global__ void __launch_bounds__(kGemmThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmArgs a) {
  using Cfg = GemmCfg<NT>;
  constexpr int S_C = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* b_ring = base;
  uint8_t* c_ring = base + S_C * Cfg::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(c_ring + S_C * kChunkBytes);
  uint64_t* wfull = bars;
  uint64_t* bfull = bars + S_C;
  uint64_t* empty = bars + 2 * S_C;
  uint64_t* afull = bars + 3 * S_C;
  uint64_t* aempty = afull + kAStages;
  uint64_t* accfull = aempty + kAStages;
  uint64_t* accempty = accfull + 2;
  uint64_t* drain = accempty + 2;
  uint32_t* misc = reinterpret_cast<uint32_t*>(drain + 1);
  uint32_t* tmem_slot = misc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(misc + 2);
  uint32_t* issued = misc + 3;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < S_C; ++s) {
      mbar_init(smem_u32(&wfull[s]), 1);
      mbar_init(smem_u32(&bfull[s]), kGatherThreads);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(smem_u32(&afull[s]), 128);
      mbar_init(smem_u32(&aempty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&accfull[s]), 1);
      mbar_init(smem_u32(&accempty[s]), 128);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    *last_flag = 0;
    *issued = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
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
  // Fewer K splits when the routed blocks would overflow the partial-sum scratch.
  int split_k = a.split_k;
  while (split_k > 1 && nblocks * a.n_tiles * split_k > a.max_split_units) --split_k;
  const int64_t n_units = nblocks * a.n_tiles * split_k;

  if (warp == 0) {
    // ---------------- weight stream: one bulk TMA per stage ----------------
    if (lane == 0) {
      const uint64_t policy = a.evict_first ? l2_policy_evict_first() : l2_policy_evict_normal();
      uint32_t it = 0;
      for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit un = decode_unit(a, split_k, u);
        if (!un.ok) continue;
        const uint8_t* src = a.wblob + kHeaderBytes +
                             ((static_cast<int64_t>(un.e) * a.n_tiles + un.jt) * a.n_kb) * kChunkBytes;
        for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
          const int s = it % S_C;
          const uint32_t ph = (it / S_C) & 1;
          if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, abort_flag, a.dev_err)) goto weights_done;
          mbar_arrive_expect_tx(smem_u32(&wfull[s]), kChunkBytes);
          bulk_g2s(smem_u32(c_ring + s * kChunkBytes), src + static_cast<int64_t>(kb) * kChunkBytes,
                   kChunkBytes, smem_u32(&wfull[s]), policy);
        }
      }
    weights_done:
      *issued = it;
    }
  } else if (warp == 2 || warp == 3) {
    // ---------------- activation gather: cp.async rows into swizzled tiles ----------------
    pdl_wait();  // activations may be the previous kernel's output
    const int g = tid - 64;
    uint32_t it = 0;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit un = decode_unit(a, split_k, u);
      if (!un.ok) continue;
      for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
        const int s = it % S_C;
        const uint32_t ph = (it / S_C) & 1;
        if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, abort_flag, a.dev_err)) goto gather_done;
        const uint32_t bdst = smem_u32(b_ring + s * Cfg::kBBytes);
        for (int idx = g; idx < NT * 8; idx += kGatherThreads) {
          const int r = idx >> 3, c = idx & 7;
          const int64_t p = static_cast<int64_t>(un.b) * a.block_m + r;
          int64_t arow;
          bool valid = true;
          if (a.a_sorted) {
            arow = p;
          } else {
            const int32_t i = __ldg(a.sorted_ids + p);
            valid = (i >= 0 && i < a.total_slots);
            arow = valid ? i / a.a_row_div : 0;
          }
          const uint16_t* src = a.A + arow * a.lda + kb * kBlockK + c * 8;
          cp_async_16(bdst + r * 128 + ((c ^ (r & 7)) << 4), valid ? src : a.A, valid ? 16u : 0u);
        }
        cp_async_arrive_noinc(smem_u32(&bfull[s]));
      }
    }
  gather_done:
    cp_async_wait_all();
  } else if (warp == 1) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NT);
      uint32_t it = 0, lu = 0;
      for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit un = decode_unit(a, split_k, u);
        if (!un.ok) continue;
        const int ab = lu & 1;
        const uint32_t pab = (lu >> 1) & 1;
        if (!mbar_wait(smem_u32(&accempty[ab]), pab ^ 1, abort_flag, a.dev_err)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * NT;
        for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
          const int s = it % S_C;
          const uint32_t ph = (it / S_C) & 1;
          const int sa = it % kAStages;
          const uint32_t pa = (it / kAStages) & 1;
          if (!mbar_wait(smem_u32(&bfull[s]), ph, abort_flag, a.dev_err)) goto mma_done;
          if (!mbar_wait(smem_u32(&afull[sa]), pa, abort_flag, a.dev_err)) goto mma_done;
          fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor core reads
          tc_fence_after();
          const uint32_t b_addr = smem_u32(b_ring + s * Cfg::kBBytes);
          const uint32_t a_tmem = tmem_base + kACol0 + sa * 32;
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk) {
            mma_ts(d_tmem, a_tmem + kk * 8, smem_desc_sw128(b_addr + kk * 32), idesc,
                   (kb > un.kb0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&empty[s]));
          mma_commit(smem_u32(&aempty[sa]));
        }
        mma_commit(smem_u32(&accfull[ab]));
        ++lu;
      }
    mma_done:
      mma_commit(smem_u32(drain));
      mbar_wait_plain(smem_u32(drain), 0);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- epilogue warpgroup ----------------
    pdl_wait();  // outputs may still be read by the previous kernel
    const int q = warp - 4;
    const int t = q * 32 + lane;  // tile row = TMEM lane
    uint32_t lu = 0;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit un = decode_unit(a, split_k, u);
      if (!un.ok) continue;
      const int ab = lu & 1;
      const uint32_t pab = (lu >> 1) & 1;
      const bool ok = mbar_wait(smem_u32(&accfull[ab]), pab, abort_flag, a.dev_err);
      if (epi_any(!ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * NT;
      if (split_k == 1) {
#pragma unroll 1
        for (int c0 = 0; c0 < NT; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(taddr + c0, r);
          tmem_wait_ld();
          if (c0 + 16 >= NT) {
            tc_fence_before();
            mbar_arrive(smem_u32(&accempty[ab]));
          }
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) store_column(a, un, t, c0 + jj, __uint_as_float(r[jj]));
        }
      } else {
        float* part = a.part + (un.tile * split_k + un.split) * (128 * NT);
#pragma unroll 1
        for (int c0 = 0; c0 < NT; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(taddr + c0, r);
          tmem_wait_ld();
          if (c0 + 16 >= NT) {
            tc_fence_before();
            mbar_arrive(smem_u32(&accempty[ab]));
          }
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) __stcg(part + (c0 + jj) * 128 + t, __uint_as_float(r[jj]));
        }
        __threadfence();
        named_bar_epi();
        if (t == 0) *last_flag = (atomicAdd(a.cnt + un.tile, 1) == split_k - 1) ? 1 : 0;
        named_bar_epi();
        if (*last_flag) {
          __threadfence();
          const float* tile_parts = a.part + un.tile * split_k * (128 * NT);
#pragma unroll 1
          for (int j = 0; j < NT; ++j) {
            float v = 0.0f;
            for (int s = 0; s < split_k; ++s) v += __ldcg(tile_parts + s * (128 * NT) + j * 128 + t);
            store_column(a, un, t, j, v);
          }
          if (t == 0) a.cnt[un.tile] = 0;  // ready for the next call
        }
        named_bar_epi();
      }
      ++lu;
    }
  } else if (warp >= 8) {
    // ---------------- dequant warpgroups (stages alternate between the two) ----------------
    const int g = (warp - 8) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + kACol0;
    uint32_t it = 0;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x) {
      const Unit un = decode_unit(a, split_k, u);
      if (!un.ok) continue;
      for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
        if ((it & 1) != static_cast<uint32_t>(g)) continue;
        const int s = it % S_C;
        const uint32_t ph = (it / S_C) & 1;
        const int sa = it % kAStages;
        const uint32_t pa = (it / kAStages) & 1;
        // warp-uniform decisions: tcgen05.st below is a warp-collective instruction
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&wfull[s]), ph, abort_flag, a.dev_err)))
          goto dq_done;
        const uint8_t* ch = c_ring + s * kChunkBytes;
        const uint4 lo = reinterpret_cast<const uint4*>(ch)[t];
        const uint4 hi = reinterpret_cast<const uint4*>(ch + kCodeHalfBytes)[t];
        const uint32_t s2 = reinterpret_cast<const uint32_t*>(ch + kScaleOffset)[t];
        uint32_t v[32];
        dequant_row64(lo, hi, s2, v);
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&aempty[sa]), pa ^ 1, abort_flag, a.dev_err)))
          goto dq_done;
        tc_fence_after();
        tmem_st32(lane_base + sa * 32, v);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&afull[sa]));
      }
    }
  dq_done:;
  }

  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // give in-flight weight copies a bounded chance to land before the CTA's memory goes away
    const uint32_t n = *issued;
    for (uint32_t j = (n > static_cast<uint32_t>(S_C) ? n - S_C : 0); j < n; ++j)
      mbar_wait_plain(smem_u32(&wfull[j % S_C]), (j / S_C) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------------
// Host side: planner and launcher.
// ------------------------------------------------------------------------------------------

int stages_for_block_m(int block_m) {
  switch (block_m) {
    case 16: return GemmCfg<16>::kStages;
    case 32: return GemmCfg<32>::kStages;
    case 64: return GemmCfg<64>::kStages;
    case 128: return GemmCfg<128>::kStages;
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

// Split-K choice: minimise the busiest CTA's bytes, ceil(units * S / P) * (W / S + R), where W
// is one tile's packed weight bytes and R the FP32 partial round trip a split adds.
void plan_gemm(int total_slots, int E, int N, int K, int block_m, int rows_per_expert,
               int num_sms, w4a16_plan_t* plan) {
  const int n_tiles = N / kTileRows, n_kb = K / kBlockK;
  const double blocks = expected_blocks(total_slots, E, block_m, rows_per_expert);
  const double units1 = std::max(1.0, std::ceil(blocks)) * n_tiles;
  const double W = static_cast<double>(n_kb) * kChunkBytes;
  const double R = 2.0 * 128 * block_m * 4;
  const int s_max = std::max(1, std::min(16, n_kb / 2));
  int best_s = 1;
  double best = 1e300;
  for (int s = 1; s <= s_max; ++s) {
    const double waves = std::ceil(units1 * s / num_sms);
    const double cost = waves * (W / s + (s > 1 ? R : 0.0));
    if (cost < best * 0.97) {  // prefer fewer splits unless clearly better
      best = cost;
      best_s = s;
    }
  }
  plan->block_m = block_m;
  plan->split_k = best_s;
  plan->est_units = static_cast<int32_t>(std::min(units1 * best_s, 2.0e9));
  plan->num_ctas = std::max(1, std::min(num_sms, plan->est_units));
  plan->stages = stages_for_block_m(block_m);
}

template <int NT>
cudaError_t launch_gemm_t(const GemmArgs& args, int grid, bool pdl, cudaStream_t stream) {
  using Cfg = GemmCfg<NT>;
  static bool configured = false;  // per-process; attribute applies to the current device
  if (!configured) {
    cudaError_t err = cudaFuncSetAttribute(moe_gemm_kernel<NT>,
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
  return cudaLaunchKernelEx(&cfg, moe_gemm_kernel<NT>, args);
}

cudaError_t launch_gemm(const GemmArgs& args, int grid, bool pdl, cudaStream_t stream) {
  switch (args.block_m) {
    case 16: return launch_gemm_t<16>(args, grid, pdl, stream);
    case 32: return launch_gemm_t<32>(args, grid, pdl, stream);
    case 64: return launch_gemm_t<64>(args, grid, pdl, stream);
    case 128: return launch_gemm_t<128>(args, grid, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4a16
