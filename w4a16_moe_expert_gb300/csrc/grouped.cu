// Routing for the grouped contracts ("vLLM x Novita AI: Chord, Faster INT4 MoE for Kimi
// K2.x", "Grouped SM90 kernels"): the contiguous prefill layout (rows concatenated by expert,
// each group padded to a 128-row boundary, m_indices per row) and the masked decode layout
// (a fixed row budget max_m per expert, masked_m valid rows).  Each kernel turns its layout
// into the aligned routing (sorted_ids / expert_ids / num_tokens_padded) that the indexed GEMM
// consumes, so both contracts run on the same GEMM kernel.
#include "common.cuh"

namespace w4a16 {

constexpr int kContigBlock = 128;  // the contiguous layout's group padding

// One warp per 128-row block: the block's expert is the id of its first valid row; every row
// with an id is its own sorted position, padding rows get the sentinel m.
__global__ void __launch_bounds__(256)
    contiguous_layout_kernel(const int32_t* __restrict__ m_indices, int m, int E,
                             int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                             int32_t* __restrict__ ntp, int32_t* dev_err) {
  pdl_wait();  // m_indices may come from the previous kernel
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int nblocks = m / kContigBlock;
  if (warp0 == 0 && lane == 0) *ntp = m;
  for (int64_t b = warp0; b < nblocks; b += nwarps) {
    const int64_t r0 = b * kContigBlock;
    int32_t id[kContigBlock / 32];
    int first = -1;  // first valid row of the block (rows r0 + 32 * i + lane)
#pragma unroll
    for (int i = 0; i < kContigBlock / 32; ++i) {
      id[i] = m_indices[r0 + 32 * i + lane];
      const unsigned valid = __ballot_sync(0xffffffffu, id[i] >= 0 && id[i] < E);
      if (first < 0 && valid) first = 32 * i + __ffs(valid) - 1;
    }
    int32_t e = -1;  // first is warp-uniform, so every lane takes the same branch below
#pragma unroll
    for (int i = 0; i < kContigBlock / 32; ++i)
      if (first >= 0 && (first >> 5) == i) e = __shfl_sync(0xffffffffu, id[i], first & 31);
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kContigBlock / 32; ++i) {
      const bool valid = id[i] >= 0 && id[i] < E;
      if (id[i] < -1 || id[i] >= E || (valid && id[i] != e)) bad = true;
      // rows with an id other than the block's are treated as computed with the block's expert
      sorted_ids[r0 + 32 * i + lane] = valid ? static_cast<int32_t>(r0 + 32 * i + lane) : m;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_dev_err(dev_err, W4A16_DEVERR_BAD_EXPERT_ID);
    if (lane == 0) expert_ids[b] = e;
  }
}

// One CTA: valid rows per expert -> blocks of block_m rows per expert in expert order, each row
// pointing at its place g * max_m + r in the [G * max_m, K] activations.
__global__ void __launch_bounds__(1024)
    masked_layout_kernel(const int32_t* __restrict__ masked_m, int G, int max_m, int block_m,
                         int64_t capacity, int32_t* __restrict__ sorted_ids,
                         int32_t* __restrict__ expert_ids, int32_t* __restrict__ ntp,
                         int32_t* dev_err) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;          // [G] valid rows
  int32_t* off = sm + G;      // [G + 1] exclusive prefix of blocks per expert
  __shared__ int32_t warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t sentinel = G * max_m;
  pdl_wait();  // masked_m may come from the previous kernel
  pdl_launch_dependents();

  // blocks per expert, then an exclusive scan over experts (G <= 1024: one per thread)
  int nb = 0;
  if (tid < G) {
    int c = masked_m[tid];
    if (c < 0 || c > max_m) {
      set_dev_err(dev_err, W4A16_DEVERR_CAPACITY);
      c = c < 0 ? 0 : max_m;
    }
    cnt[tid] = c;
    nb = (c + block_m - 1) / block_m;
  }
  int x = nb;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  if (tid < G) off[tid] = x - nb + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (tid == 0) off[G] = warp_sums[31];
  __syncthreads();
  const int nblocks = off[G];
  if (tid == 0) *ntp = nblocks * block_m;

  // owner of block b < nblocks: the last expert whose first block is <= b
  auto owner = [&](int64_t b) {
    int l = 0, h = G - 1;
    while (l < h) {
      const int mid = (l + h + 1) >> 1;
      if (off[mid] <= b) l = mid; else h = mid - 1;
    }
    return l;
  };
  for (int64_t b = tid; b < capacity / block_m; b += blockDim.x)
    expert_ids[b] = b < nblocks ? owner(b) : -1;
  for (int64_t p = tid; p < capacity; p += blockDim.x) {
    const int64_t b = p / block_m;
    int32_t v = sentinel;
    if (b < nblocks) {
      const int g = owner(b);
      const int64_t r = (b - off[g]) * block_m + p % block_m;
      if (r < cnt[g]) v = static_cast<int32_t>(static_cast<int64_t>(g) * max_m + r);
    }
    sorted_ids[p] = v;
  }
}

cudaError_t launch_contiguous_layout(const int32_t* m_indices, int m, int E, int32_t* sorted_ids,
                                     int32_t* expert_ids, int32_t* ntp, int32_t* dev_err,
                                     int num_sms, cudaStream_t stream) {
  const int nblocks = m / kContigBlock;
  int grid = (nblocks + 7) / 8;  // 8 warps per CTA, one block each
  grid = grid < 1 ? 1 : (grid > num_sms * 4 ? num_sms * 4 : grid);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, contiguous_layout_kernel, m_indices, m, E, sorted_ids,
                            expert_ids, ntp, dev_err);
}

cudaError_t launch_masked_layout(const int32_t* masked_m, int G, int max_m, int block_m,
                                 int64_t capacity, int32_t* sorted_ids, int32_t* expert_ids,
                                 int32_t* ntp, int32_t* dev_err, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.dynamicSmemBytes = static_cast<size_t>(2 * G + 1) * sizeof(int32_t);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, masked_layout_kernel, masked_m, G, max_m, block_m, capacity,
                            sorted_ids, expert_ids, ntp, dev_err);
}

}  // namespace w4a16
