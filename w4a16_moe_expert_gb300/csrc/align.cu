// moe_align on the GPU: stable counting sort of the flat slot index by expert.
//
// "vLLM x Novita AI: Chord, Faster INT4 MoE for Kimi K2.x", "Two kernel families" and
// "vLLM integration": the indexed kernels consume sorted_ids / expert_ids /
// num_tokens_padded from an over-allocated align step, read on the device only, so the
// whole path stays CUDA-graph capturable.
//
// One thread-block cluster of up to 8 CTAs x 1024 threads.  The slots are cut into contiguous
// chunks, one per CTA, and each CTA's chunk into contiguous ranges, one per warp, which keeps
// the sort stable without a global sort: every warp counts its range per expert, the CTAs
// exchange their per-expert totals through distributed shared memory, the counts are scanned
// over CTAs, warps and experts, and each warp then places its slots in order (a warp-wide
// match gives each slot its rank among equal ids).
#include <cooperative_groups.h>

#include "common.cuh"

namespace w4a16 {

namespace cg = cooperative_groups;

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kAlignMaxCluster = 8;

__global__ void __launch_bounds__(kAlignThreads, 1)
    moe_align_kernel(const int32_t* __restrict__ topk_ids, int n_slots, int E, int block_m,
                     int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                     int32_t* __restrict__ ntp_out, int64_t capacity, int validate,
                     int32_t* dev_err, int32_t* zero_words, int n_zero_words) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                      // [32][E]: per-warp counts, later per-warp cursors
  int32_t* start = cnt + kAlignWarps * E;  // [E + 1]: padded exclusive prefix
  int32_t* cta_cnt = start + E + 1;        // [E]: this CTA's count per expert (read by peers)
  int32_t* tot = cta_cnt + E;              // [E]: count per expert over all CTAs
  int32_t* pre = tot + E;                  // [E]: count per expert in the chunks before ours
  __shared__ int32_t warp_sums[kAlignWarps];
  __shared__ int bad_id;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int ncta = static_cast<int>(cluster.num_blocks());
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gtid = rank * kAlignThreads + tid, gthreads = ncta * kAlignThreads;
  const int32_t sentinel = n_slots;
  pdl_launch_dependents();  // the next kernel may start its prologue; it waits for our results
  pdl_wait();               // topk_ids may come from the previous kernel in the stream

  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) cnt[i] = 0;
  if (tid == 0) bad_id = 0;
  for (int i = gtid; i < n_zero_words; i += gthreads) zero_words[i] = 0;
  __syncthreads();

  // ---- count per (warp, expert) over this CTA's chunk ----
  const int per_cta = ((n_slots + ncta - 1) / ncta + 1023) & ~1023;
  const int c_lo = min(n_slots, rank * per_cta);
  const int c_hi = min(n_slots, c_lo + per_cta);
  const int per_warp = per_cta / kAlignWarps;  // a multiple of 32
  const int lo = min(c_hi, c_lo + warp * per_warp);
  const int hi = min(c_hi, lo + per_warp);
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    int e = (i < hi) ? topk_ids[i] : -1;
    if (e < -1 || e >= E) {
      if (validate) bad_id = 1;
      e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) cnt[warp * E + e] += __popc(peers);
  }
  __syncthreads();

  // ---- per expert: warp offsets inside the CTA, the CTA's count ----
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = 0;
    for (int w = 0; w < kAlignWarps; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
    cta_cnt[e] = run;
  }
  if (ncta > 1) cluster.sync(); else __syncthreads();  // every CTA's counts are visible

  // ---- per expert: total, count before this chunk, padded size ----
  for (int e = tid; e < E; e += kAlignThreads) {
    int all = cta_cnt[e], before = 0;
    if (ncta > 1) {
      all = 0;
      for (int r = 0; r < ncta; ++r) {
        const int c = *cluster.map_shared_rank(cta_cnt + e, r);
        all += c;
        if (r < rank) before += c;
      }
    }
    tot[e] = all;
    pre[e] = before;
    start[e] = (all + block_m - 1) / block_m * block_m;  // padded size for now
  }
  __syncthreads();

  // ---- exclusive scan of padded sizes over experts (E <= 1024: one element per thread) ----
  {
    const int v = (tid < E) ? start[tid] : 0;
    int x = v;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int s = warp_sums[lane];
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += y;
      }
      warp_sums[lane] = s;  // inclusive over warps
    }
    __syncthreads();
    const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    __syncthreads();
    if (tid < E) start[tid] = excl;
    if (tid == 0) start[E] = warp_sums[kAlignWarps - 1];
  }
  __syncthreads();
  const int ntp = start[E];

  // ---- per-warp cursors become absolute positions ----
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) cnt[i] += start[i % E] + pre[i % E];
  // ---- expert of every block (spread over the cluster) ----
  const int64_t nblocks = capacity / block_m;
  for (int64_t b = gtid; b < nblocks; b += gthreads) {
    const int64_t row = b * block_m;
    int owner = -1;
    if (row < ntp) {  // last expert whose start is <= row (experts with no rows have size 0)
      int l = 0, h = E - 1;
      while (l < h) {
        const int mid = (l + h + 1) >> 1;
        if (start[mid] <= row) l = mid; else h = mid - 1;
      }
      owner = l;
    }
    expert_ids[b] = owner;
  }
  // ---- sentinels: the padding rows of every expert, and everything from num_tokens_padded on ----
  for (int e = gtid; e < E; e += gthreads) {
    const int end = start[e + 1];  // start[E] is num_tokens_padded
    for (int p = start[e] + tot[e]; p < end; ++p)
      if (p < capacity) sorted_ids[p] = sentinel;
  }
  for (int64_t p = static_cast<int64_t>(ntp) + gtid; p < capacity; p += gthreads) sorted_ids[p] = sentinel;
  __syncthreads();

  // ---- stable placement ----
  bool overflow = false;
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    int e = (i < hi) ? topk_ids[i] : -1;
    if (e < -1 || e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int r = __popc(peers & ((1u << lane) - 1u));
      const int pos = cnt[warp * E + e] + r;
      if (pos < capacity) sorted_ids[pos] = i; else overflow = true;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) cnt[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  if (overflow) set_dev_err(dev_err, W4A16_DEVERR_CAPACITY);
  if (rank == 0 && tid == 0) {
    *ntp_out = (ntp <= capacity) ? ntp : static_cast<int32_t>(capacity / block_m * block_m);
    if (ntp > capacity) set_dev_err(dev_err, W4A16_DEVERR_CAPACITY);
  }
  __syncthreads();
  if (tid == 0 && bad_id) set_dev_err(dev_err, W4A16_DEVERR_BAD_EXPERT_ID);
  if (ncta > 1) cluster.sync();  // peers may still be reading this CTA's counts
}

// The same routing for at most 32 slots (decode): warp 0 holds one slot per lane and sorts in
// registers, the other warps clear the counters; after one barrier every thread fills the
// sentinels and the unowned blocks past num_tokens_padded.  A slot's position is the padded
// start of its expert (the sum of the padded counts of the smaller expert ids present) plus
// its rank among the lower lanes holding the same id, so the order is the stable one.
constexpr int kAlignSmallSlots = 32;

__global__ void __launch_bounds__(kAlignThreads, 1)
    moe_align_small_kernel(const int32_t* __restrict__ topk_ids, int n_slots, int E, int block_m,
                           int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                           int32_t* __restrict__ ntp_out, int64_t capacity, int validate,
                           int32_t* dev_err, int32_t* zero_words, int n_zero_words) {
  __shared__ int32_t s_ntp;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t sentinel = n_slots;
  pdl_launch_dependents();  // the next kernel may start its prologue; it waits for our results
  pdl_wait();               // topk_ids may come from the previous kernel in the stream
  if (warp == 0) {
    int e = lane < n_slots ? topk_ids[lane] : -1;
    const bool bad = e < -1 || e >= E;
    if (bad) e = -1;
    if (validate && __any_sync(0xffffffffu, bad) && lane == 0)
      set_dev_err(dev_err, W4A16_DEVERR_BAD_EXPERT_ID);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const bool leader = e >= 0 && lane == __ffs(peers) - 1;
    const int cnt = __popc(peers);
    const int pad = leader ? (cnt + block_m - 1) / block_m * block_m : 0;
    // padded start of this lane's expert, and the total
    int start = 0, ntp = 0;
    for (int j = 0; j < 32; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      const int pj = __shfl_sync(0xffffffffu, pad, j);
      ntp += pj;
      if (ej < e) start += pj;
    }
    if (e >= 0) {
      const int pos = start + __popc(peers & ((1u << lane) - 1u));
      if (pos < capacity) sorted_ids[pos] = lane;
    }
    if (leader) {
      for (int p = start + cnt; p < start + pad; ++p)
        if (p < capacity) sorted_ids[p] = sentinel;
      for (int b = start / block_m; b < (start + pad) / block_m; ++b)
        if (static_cast<int64_t>(b) * block_m < capacity) expert_ids[b] = e;
    }
    if (lane == 0) {
      s_ntp = ntp;
      *ntp_out = (ntp <= capacity) ? ntp : static_cast<int32_t>(capacity / block_m * block_m);
      if (ntp > capacity) set_dev_err(dev_err, W4A16_DEVERR_CAPACITY);
    }
  } else {
    for (int i = tid - 32; i < n_zero_words; i += kAlignThreads - 32) zero_words[i] = 0;
  }
  __syncthreads();
  const int64_t ntp = s_ntp;
  for (int64_t p = ntp + tid; p < capacity; p += kAlignThreads) sorted_ids[p] = sentinel;
  const int64_t nblocks = capacity / block_m;
  for (int64_t b = ntp / block_m + tid; b < nblocks; b += kAlignThreads) expert_ids[b] = -1;
}

// Activation rows in aligned order: out[p, :] = x[sorted_ids[p] / a_row_div, :] for every
// routed position p < num_tokens_padded (padding rows are left as they are).  One warp per
// row, 16-byte vectors; lets the GEMM stream activation tiles with 2-D TMA instead of gathering
// rows itself.
__global__ void __launch_bounds__(256)
    gather_rows_kernel(const uint16_t* __restrict__ x, int64_t ldx, int K, int a_row_div,
                       const int32_t* __restrict__ sorted_ids, const int32_t* __restrict__ ntp_ptr,
                       int total_slots, int64_t capacity, uint16_t* __restrict__ out,
                       int64_t ldo) {
  pdl_wait();  // routing comes from the align kernel
  // The dependent GEMM reads the routing before its own wait, so it may only start once the
  // routing is known to be complete, i.e. after the wait above.
  pdl_launch_dependents();
  int64_t ntp = *ntp_ptr;
  if (ntp < 0) ntp = 0;
  if (ntp > capacity) ntp = capacity;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int vec = K / 8;  // 16-byte vectors per row
  for (int64_t p = warp0; p < ntp; p += nwarps) {
    const int32_t i = __ldg(sorted_ids + p);
    if (i < 0 || i >= total_slots) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(i / a_row_div) * ldx);
    uint4* dst = reinterpret_cast<uint4*>(out + p * ldo);
    for (int v = lane; v < vec; v += 32) dst[v] = __ldg(src + v);
  }
}

cudaError_t launch_gather_rows(const uint16_t* x, int64_t ldx, int K, int a_row_div,
                               const int32_t* sorted_ids, const int32_t* ntp, int total_slots,
                               int64_t capacity, uint16_t* out, int64_t ldo, int num_sms,
                               cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  const int64_t max_rows = capacity < total_slots ? capacity : total_slots;
  int64_t blocks = (max_rows + 7) / 8;  // 8 warps (rows) per block
  const int64_t cap_blocks = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  if (blocks < 1) blocks = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, x, ldx, K, a_row_div, sorted_ids, ntp,
                            total_slots, capacity, out, ldo);
}

size_t align_smem_bytes(int E) {
  return static_cast<size_t>(kAlignWarps * E + 4 * E + 1) * sizeof(int32_t);
}

// Cluster size for n_slots slots: one CTA while each warp's range is at most two passes of 32,
// doubling up to eight CTAs for prefill-sized routings.
static int align_cluster_size(int n_slots) {
  int c = 1;
  while (c < kAlignMaxCluster && n_slots > c * 2 * kAlignThreads) c *= 2;
  return c;
}

cudaError_t launch_moe_align(const int32_t* topk_ids, int n_slots, int E, int block_m,
                             int32_t* sorted_ids, int32_t* expert_ids, int32_t* ntp,
                             int64_t capacity, int validate, int32_t* dev_err,
                             int32_t* zero_words, int n_zero_words, cudaStream_t stream) {
  if (n_slots <= kAlignSmallSlots) {  // decode: one warp sorts in registers
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kAlignThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, moe_align_small_kernel, topk_ids, n_slots, E, block_m,
                              sorted_ids, expert_ids, ntp, capacity, validate, dev_err,
                              zero_words, n_zero_words);
  }
  const size_t smem = align_smem_bytes(E);
  cudaError_t err = cudaFuncSetAttribute(moe_align_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int cluster = align_cluster_size(n_slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(kAlignThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // one CTA launches as a plain grid
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, moe_align_kernel, topk_ids, n_slots, E, block_m, sorted_ids,
                            expert_ids, ntp, capacity, validate, dev_err, zero_words,
                            n_zero_words);
}

}  // namespace w4a16
