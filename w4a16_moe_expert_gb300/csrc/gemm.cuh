// Arguments of the indexed GEMM kernel, shared by the launcher and the C ABI layer.
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the encoder is fetched from the driver at run time)

#include "common.cuh"

namespace w4a16 {

struct GemmArgs {
  CUtensorMap tmap_a;   // sorted rows, box 64 x block_m (single-kernel layer)
  CUtensorMap tmap_a3;  // sorted rows as [K / 64][rows][64], box 64 x rows x (K blocks a stage)
  const uint16_t* A;
  int64_t lda;
  int a_row_div;
  int a_sorted;
  const uint8_t* wblob;
  int E, N, K, n_tiles, n_kb;
  // Tile groups (short-K plain calls): a unit covers tpu consecutive 128-row tiles of one
  // block, n_tg = n_tiles / tpu units per block (tpu = 1: one tile per unit)
  int tpu, n_tg;
  uint32_t nt_magic, nt_shift;  // division by n_tg: (umulhi(n, magic) + n) >> shift
  int paired;
  int nvfp4;  // the blob holds NVFP4 (E2M1 + E4M3 per 16) weights instead of INT4
  const uint8_t* tile_mode;  // [E * n_tiles] kTilePlain / kTileScaled (INT4 conversion of a tile)
  const int32_t* sorted_ids;
  const int32_t* expert_ids;
  const int32_t* ntp;
  int block_m;
  int total_slots;
  int64_t capacity;
  int epilogue;
  int c_sorted;
  int c_f32;  // C is float (unrounded sums)
  int c_st256;  // C and its rows are 32-byte aligned: the epilogue stores 32 bytes per lane
  const float* merge_w;  // non-null: add merge_w[slot] * value into C row slot / merge_k (FP32)
  int merge_k;
  uint16_t* C;
  int64_t ldc;
  float* part;
  int32_t* cnt;
  int split_k;
  // split_k is an upper bound: the device slices the tiles of a last, partial wave of the
  // routed (block, tile) units into K slices that fill it (every tile when there is no full
  // wave), each slice at least kMinSplitKb K blocks
  int split_auto;
  int64_t max_split_units;  // K splits are reduced on the device until units fit the scratch
  int32_t* dev_err;
  int evict_first;
  int routing_ready;  // routing was complete before the previous kernel started
  // fused layer only: the first GEMM counts finished tiles per block in signal_done; the
  // second waits until wait_done[block] >= wait_count before loading that block's rows
  int32_t* signal_done;
  const int32_t* wait_done;
  int wait_count;
  long long wait_limit;  // cycles before that wait gives up (0: the default, about a second)
  // single-kernel layer, down GEMM only: sync[0] counts CTAs that zeroed their slice of the
  // FP32 token sums C (sum_elems floats), sync[1] CTAs whose units are all done; the last
  // phase rounds the sums into final_out (BF16)
  int32_t* sync;
  int64_t sum_elems;
  uint16_t* final_out;
  // CTA pairs (block_m 128): units are (block, pair of 128-row tiles); divisor n_tiles / 2;
  // one cta_group::2 MMA over both CTAs
  int pair;
  uint32_t nt2_magic, nt2_shift;
};

// Fewest 64-wide K blocks one K slice of an automatically split tile streams (1536 K elements:
// six pipeline stages at decode block sizes).  Measured on GB300: slicing K = 2048 in two
// (Kimi-K2 EP8 down at T=1, 56 tiles -> 112 units) is slower (7.5 -> 8.3 us), slicing
// K = 7168 in four (32 tiles -> 128 units) much faster (gate_up 16.3 -> 10.5 us); slicing the
// last partial wave's tiles into slices of 4 K blocks was no faster at Qwen3 T=8 (K = 2048)
// and slower at T=512 (64.2 -> 72.3 us gate_up).
constexpr int kMinSplitKb = 24;
// Largest block size whose calls the device may split (decode): at prefill the partial sums
// of 128 x block_m tiles cost more than the last wave's imbalance (Qwen3 T=4096 down 117 ->
// 126 us with the last wave sliced).
constexpr int kMaxSplitBlockM = 32;
// Most K slices the planner lets the device choose.
constexpr int kMaxAutoSplit = 8;

// Largest tile group for a block size: its double-buffered accumulators (2 * tpu * block_m
// TMEM columns) stay within the 128 columns reserved for them below 64-token blocks.
constexpr int tile_group_max(int block_m) { return block_m <= 16 ? 4 : (block_m <= 32 ? 2 : 1); }
// K blocks (64 wide) of a unit short enough for tile groups: at most two pipeline stages.
constexpr int kGroupMaxKb = 8;

// CTA pairs by default where a 128-token block's activation rows are long and shared by few
// tiles (N <= 512, K >= 4096): each tile of a block re-reads the block's rows, and a pair reads
// half of them per CTA.  Measured on GB300 (single flushed calls, one CTA per tile against
// pairs): Kimi-K2 TP8 gate_up at T=8192 (4 tiles, K = 7168) 496.3 -> 480.9 us, Zipf routing
// 482.0 -> 459.5; where blocks have 12-56 tiles pairs were 0-5% slower (Qwen3 T=4096 gate_up
// 172.7 -> 176.8, Kimi-K2 EP8 T=16384 gate_up 678.5 -> 697.0, TP8 down 705.2 -> 737.9).
constexpr int kPairMaxTiles = 4;
constexpr int kPairMinKb = 64;
inline bool pairs_pay(int block_m, int n_tiles, int n_kb) {
  return block_m == 128 && n_tiles % 2 == 0 && n_tiles <= kPairMaxTiles && n_kb >= kPairMinKb;
}

// The fused layer call: gate_up (a) then down (a2) in one cooperative persistent launch.
cudaError_t launch_layer_fused(GemmArgs& a, GemmArgs& a2, int grid, cudaStream_t stream);

cudaError_t launch_gemm(GemmArgs& args, int grid, bool pdl, cudaStream_t stream);  // pairs if args.pair

// Multiply-shift constants for dividing 31-bit numerators by d >= 1 (round-up reciprocal).
inline void fast_divisor(uint32_t d, uint32_t* magic, uint32_t* shift) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  const uint64_t m = ((uint64_t(1) << (32 + l)) + d - 1) / d - (uint64_t(1) << 32);
  *magic = static_cast<uint32_t>(m);
  *shift = l;
}
void plan_gemm(int total_slots, int E, int N, int K, int block_m, int rows_per_expert,
               int num_sms, w4a16_plan_t* plan);

}  // namespace w4a16
