// C ABI of the library (declared in include/w4a16_moe.h): argument checks, workspace
// layout, the host planner, the top-k combine kernel and the layer chain.
#include <algorithm>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gemm.cuh"

namespace w4a16 {

// kernels and launchers defined in the other translation units
cudaError_t launch_moe_align(const int32_t* topk_ids, int n_slots, int E, int block_m,
                             int32_t* sorted_ids, int32_t* expert_ids, int32_t* ntp,
                             int64_t capacity, int validate, int32_t* dev_err,
                             int32_t* zero_words, int n_zero_words, cudaStream_t stream);
size_t align_smem_bytes(int E);
cudaError_t launch_gather_rows(const uint16_t* x, int64_t ldx, int K, int a_row_div,
                               const int32_t* sorted_ids, const int32_t* ntp, int total_slots,
                               int64_t capacity, uint16_t* out, int64_t ldo, int num_sms,
                               cudaStream_t stream);
cudaError_t launch_contiguous_layout(const int32_t* m_indices, int m, int E, int32_t* sorted_ids,
                                     int32_t* expert_ids, int32_t* ntp, int32_t* dev_err,
                                     int num_sms, cudaStream_t stream);
cudaError_t launch_masked_layout(const int32_t* masked_m, int G, int max_m, int block_m,
                                 int64_t capacity, int32_t* sorted_ids, int32_t* expert_ids,
                                 int32_t* ntp, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_pack_nvfp4(const uint8_t* codes, const uint8_t* scales, int E, int N, int K,
                              uint32_t flags, void* packed, cudaStream_t stream);
cudaError_t launch_pack(const int32_t* qweight, const uint16_t* scales, int E, int N, int K,
                        uint32_t flags, void* packed, cudaStream_t stream);
cudaError_t launch_debug_dequant(const void* packed, int E, int e, int N, int K, uint32_t flags,
                                 uint16_t* out, cudaStream_t stream);


// ---- error bookkeeping ------------------------------------------------------------------------
static thread_local char g_detail[512] = "";

static w4a16_status_t fail(w4a16_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof g_detail, fmt, ap);
  va_end(ap);
  return st;
}

// Detail text for failures found outside this file.
void set_error_detail(const char* text) { snprintf(g_detail, sizeof g_detail, "%s", text); }

static w4a16_status_t cuda_fail(cudaError_t err, const char* what) {
  cudaGetLastError();  // clear the sticky-free launch error
  return fail(W4A16_CUDA_ERROR, "%s: %s", what, cudaGetErrorString(err));
}

// ---- device facts (cached per device) -----------------------------------------------------------
struct DeviceFacts {
  int checked = 0;
  int ok = 0;
  int num_sms = 0;
};
static DeviceFacts g_dev[64];
static std::mutex g_dev_mu;

static w4a16_status_t device_facts(DeviceFacts* out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(W4A16_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceFacts& f = g_dev[dev];
  if (!f.checked) {
    int major = 0, minor = 0, sms = 0;
    if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(err, "cudaDeviceGetAttribute");
    f.ok = (major == 10 && minor == 3);
    f.num_sms = sms;
    f.checked = 1;
  }
  if (!f.ok) return fail(W4A16_UNSUPPORTED, "this library is built for sm_103a (GB300) only");
  *out = f;
  return W4A16_OK;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static bool valid_block_m(int bm) { return bm == 16 || bm == 32 || bm == 64 || bm == 128; }

// K-split scratch: a fixed 16 MB of FP32 partials, i.e. 32768 / block_m (tile, split) units.
constexpr size_t kPartialBytes = size_t(16) << 20;
static int64_t split_unit_budget(int block_m) { return 32768 / block_m; }

static w4a16_status_t check_packed(const w4a16_packed_weights_t* W) {
  if (!W) return fail(W4A16_INVALID_ARG, "packed weight descriptor is NULL");
  if (W->magic != W4A16_PACK_MAGIC || W->version != W4A16_PACK_VERSION)
    return fail(W4A16_BAD_PACKED_WEIGHT, "packed weight descriptor has a bad magic or version");
  const int group = (W->flags & W4A16_PACK_NVFP4) ? 16 : 32;
  if (W->group != group || W->K % kBlockK || W->N % kTileRows || W->E < 0 || !W->data)
    return fail(W4A16_BAD_PACKED_WEIGHT, "packed weight descriptor has bad sizes");
  if (W->flags & ~(W4A16_PACK_GATE_UP_PAIRED | W4A16_PACK_NVFP4))
    return fail(W4A16_BAD_PACKED_WEIGHT, "packed weight descriptor has unknown flags");
  if (reinterpret_cast<uintptr_t>(W->data) % 256)
    return fail(W4A16_BAD_PACKED_WEIGHT, "packed weight blob must be 256-byte aligned");
  if (W->bytes != w4a16_packed_bytes(W->E, W->N, W->K, W->group, W->flags))
    return fail(W4A16_BAD_PACKED_WEIGHT, "packed weight descriptor has a bad blob size");
  return W4A16_OK;
}

// ---- top-k weighted sum ---------------------------------------------------------------------------
// One thread per 8 output columns of one token; FP32 accumulation over slots in order.
__global__ void __launch_bounds__(256)
    topk_sum_kernel(const float* __restrict__ Y, const int32_t* __restrict__ topk_ids,
                    const float* __restrict__ topk_weights, int T, int top_k, int H,
                    uint16_t* __restrict__ out) {
  pdl_wait();  // Y is the previous kernel's output
  const int vec_per_row = H / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(T) * vec_per_row) return;
  const int64_t t = idx / vec_per_row;
  const int c = static_cast<int>(idx % vec_per_row) * 8;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int s = 0; s < top_k; ++s) {
    const int64_t i = t * top_k + s;
    if (__ldg(topk_ids + i) < 0) continue;
    const float w = __ldg(topk_weights + i);
    const float4 y0 = __ldg(reinterpret_cast<const float4*>(Y + i * H + c));
    const float4 y1 = __ldg(reinterpret_cast<const float4*>(Y + i * H + c + 4));
    acc[0] += w * y0.x;
    acc[1] += w * y0.y;
    acc[2] += w * y0.z;
    acc[3] += w * y0.w;
    acc[4] += w * y1.x;
    acc[5] += w * y1.y;
    acc[6] += w * y1.z;
    acc[7] += w * y1.w;
  }
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q + 1]));
    o[q] = lo | (hi << 16);
  }
  *reinterpret_cast<uint4*>(out + t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
}

static cudaError_t launch_topk_sum(const float* Y, const int32_t* ids, const float* w, int T,
                                   int top_k, int H, uint16_t* out, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(T) * (H / 8);
  if (n == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_sum_kernel, Y, ids, w, T, top_k, H, out);
}

// ---- fused top-k merge helpers: zero the FP32 token sums, then round them to BF16 ------------
__global__ void __launch_bounds__(256) zero_f32_kernel(float* __restrict__ p, int64_t n4) {
  pdl_wait();  // the previous call's last kernel may still read this buffer
  pdl_launch_dependents();
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    reinterpret_cast<float4*>(p)[i] = z;
}

__global__ void __launch_bounds__(256)
    round_bf16_kernel(const float* __restrict__ acc, int64_t n8, uint16_t* __restrict__ out) {
  pdl_wait();  // the sums come from the down GEMM
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    auto pk = [](float lo, float hi) {
      return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
    };
    reinterpret_cast<uint4*>(out)[i] = make_uint4(pk(a.x, a.y), pk(a.z, a.w), pk(b.x, b.y), pk(b.z, b.w));
  }
}

// A grid-stride launch of 256-thread blocks with programmatic dependent launch.
static void pdl_config(int64_t work_items, int num_sms, cudaStream_t stream, cudaLaunchConfig_t* cfg,
                       cudaLaunchAttribute* attr) {
  *cfg = {};
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((work_items + 255) / 256, num_sms * 8));
  cfg->gridDim = dim3(static_cast<unsigned>(blocks));
  cfg->blockDim = dim3(256);
  cfg->stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

static cudaError_t launch_zero_f32(float* p, int64_t n, int num_sms, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(n / 4, num_sms, stream, &cfg, attr);
  return cudaLaunchKernelEx(&cfg, zero_f32_kernel, p, n / 4);
}

static cudaError_t launch_round_bf16(const float* acc, int64_t n, uint16_t* out, int num_sms,
                                     cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(n / 8, num_sms, stream, &cfg, attr);
  return cudaLaunchKernelEx(&cfg, round_bf16_kernel, acc, n / 8, out);
}

// ---- GEMM call shared by the ABI entry and the layer ----------------------------------------------
struct GemmCall {
  const uint16_t* A;
  int64_t lda;
  int a_row_div;
  const w4a16_packed_weights_t* W;
  const w4a16_routing_t* R;
  int epilogue;
  uint32_t row_flags;
  uint16_t* C;
  int64_t ldc;
  void* ws;
  size_t ws_bytes;
  int rows_hint;
  const w4a16_schedule_t* sched;
  int32_t* dev_err;
  int routing_ready;
  const float* merge_w = nullptr;  // fused top-k merge (C = FP32 token sums)
  int merge_k = 0;
  bool one_kernel = false;  // an argument set of the single-kernel layer (one tile per unit)
};

// Checks a GEMM call and fills the kernel arguments and grid; *empty is set when there is
// nothing to compute (no capacity or no experts).
static w4a16_status_t prepare_gemm(const GemmCall& c, const DeviceFacts& dev, GemmArgs* out,
                                   int* out_grid, bool* empty) {
  *empty = false;
  w4a16_status_t st = check_packed(c.W);
  if (st != W4A16_OK) return st;
  const w4a16_routing_t* R = c.R;
  if (!R || !R->sorted_ids || !R->expert_ids || !R->num_tokens_padded)
    return fail(W4A16_INVALID_ARG, "routing tensors must not be NULL");
  if (reinterpret_cast<uintptr_t>(R->sorted_ids) % 16)
    return fail(W4A16_INVALID_ARG, "sorted_ids must be 16-byte aligned");
  if (!valid_block_m(R->block_m))
    return fail(W4A16_UNSUPPORTED, "block_m %d: supported values are 16, 32, 64, 128", R->block_m);
  if (R->capacity < 0 || R->capacity % R->block_m || R->total_slots < 0)
    return fail(W4A16_INVALID_ARG, "capacity must be a non-negative multiple of block_m");
  if (!c.A || !c.C || c.a_row_div <= 0 || c.lda < c.W->K || c.lda % 8 ||
      reinterpret_cast<uintptr_t>(c.A) % 16)
    return fail(W4A16_INVALID_ARG, "A must be 16-byte aligned with lda >= K and lda %% 8 == 0");
  const bool paired = (c.W->flags & W4A16_PACK_GATE_UP_PAIRED) != 0;
  int out_cols = c.W->N;
  if (c.epilogue == W4A16_EPILOGUE_SILU_MUL) {
    if (!paired)
      return fail(W4A16_BAD_PACKED_WEIGHT, "SiLU-and-mul needs a W4A16_PACK_GATE_UP_PAIRED weight");
    out_cols = c.W->N / 2;
  } else if (c.epilogue != W4A16_EPILOGUE_NONE) {
    return fail(W4A16_INVALID_ARG, "unknown epilogue %d", c.epilogue);
  }
  if (c.ldc < out_cols) return fail(W4A16_INVALID_ARG, "ldc smaller than the output width");
  if (reinterpret_cast<uintptr_t>(c.C) % 16 || c.ldc % ((c.row_flags & W4A16_C_FP32) ? 4 : 8))
    return fail(W4A16_INVALID_ARG, "C must be 16-byte aligned with 16-byte aligned rows");
  if ((c.row_flags & W4A16_C_FP32) && c.epilogue != W4A16_EPILOGUE_NONE)
    return fail(W4A16_INVALID_ARG, "FP32 output is available with epilogue NONE only");
  if (R->capacity == 0 || c.W->E == 0) {
    *empty = true;
    return W4A16_OK;
  }

  if ((R->capacity / R->block_m) * static_cast<int64_t>(c.W->N / kTileRows) * 16 >= (int64_t(1) << 31))
    return fail(W4A16_UNSUPPORTED, "routing capacity too large for one call (units must stay below 2^31)");
  w4a16_plan_t plan;
  plan_gemm(R->total_slots, c.W->E, c.W->N, c.W->K, R->block_m, c.rows_hint, dev.num_sms, &plan);
  int split = plan.split_k, grid = plan.num_ctas;
  const int n_kb = c.W->K / kBlockK;
  // an explicit split is taken as given; the planner's is an upper bound for the device
  const bool split_fixed = c.sched && c.sched->split_k > 0;
  if (split_fixed) split = c.sched->split_k;
  if (c.sched && c.sched->num_ctas > 0) grid = c.sched->num_ctas;
  split = std::max(1, std::min(split, std::min(16, n_kb)));
  grid = std::max(1, std::min(grid, dev.num_sms));

  const int64_t budget = split_unit_budget(R->block_m);
  const size_t cnt_bytes = round_up(static_cast<size_t>(budget) * sizeof(int32_t), 256);
  const bool have_scratch = c.ws && c.ws_bytes >= cnt_bytes + kPartialBytes;
  if (split > 1 && !have_scratch) {
    if (split_fixed)
      return fail(W4A16_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes", cnt_bytes + kPartialBytes);
    split = 1;  // no scratch for partial sums: whole-K tiles
  }

  GemmArgs& a = *out;
  std::memset(&a, 0, sizeof a);
  a.A = c.A;
  a.lda = c.lda;
  a.a_row_div = c.a_row_div;
  a.a_sorted = (c.row_flags & W4A16_A_ROWS_SORTED) ? 1 : 0;
  a.wblob = static_cast<const uint8_t*>(c.W->data);
  a.E = c.W->E;
  a.N = c.W->N;
  a.K = c.W->K;
  a.n_tiles = c.W->N / kTileRows;
  a.n_kb = n_kb;
  a.tpu = 1;
  a.n_tg = a.n_tiles;
  fast_divisor(static_cast<uint32_t>(a.n_tg), &a.nt_magic, &a.nt_shift);
  a.paired = paired ? 1 : 0;
  a.nvfp4 = (c.W->flags & W4A16_PACK_NVFP4) ? 1 : 0;
  a.tile_mode = a.wblob + tile_mode_offset(a.E, a.n_tiles, n_kb);
  a.sorted_ids = R->sorted_ids;
  a.expert_ids = R->expert_ids;
  a.ntp = R->num_tokens_padded;
  a.block_m = R->block_m;
  a.total_slots = R->total_slots;
  a.capacity = R->capacity;
  a.epilogue = c.epilogue;
  a.c_sorted = (c.row_flags & W4A16_C_ROWS_SORTED) ? 1 : 0;
  a.c_f32 = (c.row_flags & W4A16_C_FP32) ? 1 : 0;
  a.c_st256 = (reinterpret_cast<uintptr_t>(c.C) % 32 == 0 && c.ldc % (a.c_f32 ? 8 : 16) == 0) ? 1 : 0;
  a.C = c.C;
  a.ldc = c.ldc;
  a.cnt = static_cast<int32_t*>(c.ws);
  a.part = c.ws ? reinterpret_cast<float*>(static_cast<uint8_t*>(c.ws) + cnt_bytes) : nullptr;
  a.split_k = split;
  a.split_auto = (!split_fixed && split > 1) ? 1 : 0;
  a.max_split_units = budget;
  a.dev_err = c.dev_err;
  // weights streamed once per call (few rows per expert) are marked evict-first in L2
  a.evict_first = (c.rows_hint > 0 ? c.rows_hint : R->total_slots / std::max(1, c.W->E)) <= R->block_m;
  a.routing_ready = c.routing_ready;
  a.merge_w = c.merge_w;
  a.merge_k = c.merge_k;
  // CTA pairs (one M = 256 MMA over two CTAs' tiles) for 128-token blocks of sorted rows
  const bool pair_ok = R->block_m == 128 && a.a_sorted && (split == 1 || a.split_auto) &&
                       a.n_tiles % 2 == 0 && grid >= 2 && !c.merge_w;
  const int want_pair = c.sched ? c.sched->cta_pairs : 0;
  if (want_pair < 0 || want_pair > 2)
    return fail(W4A16_INVALID_ARG, "cta_pairs %d: supported values are 0, 1, 2", want_pair);
  if (want_pair == 2 && !pair_ok)
    return fail(W4A16_INVALID_ARG, "CTA pairs need block_m 128, sorted activation rows, an even "
                                   "tile count and no K split");
  const bool pair_pays = pairs_pay(R->block_m, a.n_tiles, n_kb) && !c.one_kernel;
  a.pair = (want_pair == 2 || (want_pair == 0 && pair_ok && pair_pays)) ? 1 : 0;
  if (a.pair) {  // whole-K tiles
    a.split_k = 1;
    a.split_auto = 0;
    grid &= ~1;
    fast_divisor(static_cast<uint32_t>(a.n_tiles / 2), &a.nt2_magic, &a.nt2_shift);
  }
  // Tile groups: where a unit is at most two pipeline stages (K <= 512, the Kimi-K2 TP8 down
  // projection's K = 256), consecutive 128-row tiles of one block share a unit, its
  // activation stages and its per-unit hand-offs.
  const int group_max = tile_group_max(R->block_m);
  const int stage_kb = R->block_m <= 64 ? 4 : 2;
  // (a planner's split of short K yields to the group; a fixed split excludes it)
  const bool group_ok = !a.pair && !c.merge_w && !c.one_kernel &&
                        (a.split_k == 1 || a.split_auto) && n_kb <= kGroupMaxKb &&
                        n_kb % stage_kb == 0;
  const int want_group = c.sched ? c.sched->tile_group : 0;
  if (want_group < 0 || want_group > 4 || want_group == 3)
    return fail(W4A16_INVALID_ARG, "tile_group %d: supported values are 0, 1, 2, 4", want_group);
  int tpu = 1;
  if (want_group > 1) {
    if (!group_ok || want_group > group_max || a.n_tiles % want_group)
      return fail(W4A16_INVALID_ARG, "tile_group %d needs K <= 512 in whole stages, no K split, "
                                     "N / 128 a multiple of it and block_m <= %d",
                  want_group, want_group == 2 ? 32 : 16);
    tpu = want_group;
  } else if (want_group == 0 && group_ok) {
    // the largest group that divides the tiles and still leaves a unit for every CTA (by the
    // planner's estimate of routed blocks): at T=1 parallelism matters more than amortising
    tpu = group_max;
    while (tpu > 1 && (a.n_tiles % tpu || static_cast<int64_t>(plan.est_units) / tpu < grid)) tpu >>= 1;
  }
  if (tpu > 1) {
    a.split_k = 1;
    a.split_auto = 0;
    a.tpu = tpu;
    a.n_tg = a.n_tiles / tpu;
    fast_divisor(static_cast<uint32_t>(a.n_tg), &a.nt_magic, &a.nt_shift);
  }
  *out_grid = grid;
  return W4A16_OK;
}

static w4a16_status_t run_gemm(const GemmCall& c, const DeviceFacts& dev, cudaStream_t stream) {
  GemmArgs a;
  int grid = 0;
  bool empty = false;
  w4a16_status_t st = prepare_gemm(c, dev, &a, &grid, &empty);
  if (st != W4A16_OK || empty) return st;
  cudaError_t err = launch_gemm(a, grid, true, stream);
  if (err != cudaSuccess) return cuda_fail(err, "moe_gemm launch");
  return W4A16_OK;
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

const char* w4a16_status_string(w4a16_status_t s) {
  switch (s) {
    case W4A16_OK: return "ok";
    case W4A16_INVALID_ARG: return "invalid argument";
    case W4A16_UNSUPPORTED: return "unsupported shape, option or device";
    case W4A16_BAD_PACKED_WEIGHT: return "bad packed weight";
    case W4A16_WORKSPACE_TOO_SMALL: return "workspace too small";
    case W4A16_CUDA_ERROR: return "CUDA error";
  }
  return "unknown status";
}

const char* w4a16_last_error_detail(void) { return g_detail; }

int64_t w4a16_align_capacity(int T, int top_k, int E, int block_m) {
  if (T < 0 || top_k <= 0 || E <= 0 || block_m <= 0) return -1;
  const int64_t raw = static_cast<int64_t>(T) * top_k + static_cast<int64_t>(E) * (block_m - 1);
  return (raw + block_m - 1) / block_m * block_m;
}

w4a16_status_t w4a16_moe_align(const int32_t* topk_ids, int T, int top_k, int E, int block_m,
                               int32_t* sorted_ids, int32_t* expert_ids,
                               int32_t* num_tokens_padded, int64_t capacity, int validate,
                               int32_t* dev_err, w4a16_stream_t stream) {
  if (T < 0 || top_k <= 0 || E <= 0 || E > 1024 || block_m <= 0)
    return fail(W4A16_INVALID_ARG, "need T >= 0, top_k > 0, 1 <= E <= 1024, block_m > 0");
  if (static_cast<int64_t>(T) * top_k >= (int64_t(1) << 31))
    return fail(W4A16_INVALID_ARG, "T * top_k must be below 2^31");
  if (capacity % block_m || capacity < w4a16_align_capacity(T, top_k, E, block_m) ||
      capacity >= (int64_t(1) << 31))
    return fail(W4A16_INVALID_ARG, "capacity must be a multiple of block_m, at least "
                "w4a16_align_capacity() and below 2^31");
  if (!sorted_ids || !expert_ids || !num_tokens_padded || (T > 0 && !topk_ids))
    return fail(W4A16_INVALID_ARG, "NULL routing buffer");
  DeviceFacts dev;
  w4a16_status_t st = device_facts(&dev);
  if (st != W4A16_OK) return st;
  cudaError_t err = launch_moe_align(topk_ids, T * top_k, E, block_m, sorted_ids, expert_ids,
                                     num_tokens_padded, capacity, validate, dev_err, nullptr, 0,
                                     stream);
  if (err != cudaSuccess) return cuda_fail(err, "moe_align launch");
  return W4A16_OK;
}

size_t w4a16_packed_bytes(int E, int N, int K, int group, uint32_t flags) {
  const int want = (flags & W4A16_PACK_NVFP4) ? 16 : 32;
  if (E < 0 || N <= 0 || K <= 0 || group != want || K % kBlockK || N % kTileRows) return 0;
  const size_t modes = (static_cast<size_t>(E) * (N / kTileRows) + 15) / 16 * 16;
  return static_cast<size_t>(tile_mode_offset(E, N / kTileRows, K / kBlockK)) + modes;
}

w4a16_status_t w4a16_pack_weights(const int32_t* qweight, const uint16_t* scales, int E, int N,
                                  int K, int group, uint32_t flags, void* packed,
                                  size_t packed_bytes, w4a16_packed_weights_t* desc,
                                  w4a16_stream_t stream) {
  if (group != 32) return fail(W4A16_UNSUPPORTED, "only group size 32 is supported");
  if (E < 0 || N <= 0 || K <= 0 || K % kBlockK || N % kTileRows)
    return fail(W4A16_UNSUPPORTED, "need K %% 64 == 0 and N %% 128 == 0 (got N=%d K=%d)", N, K);
  if (flags & ~W4A16_PACK_GATE_UP_PAIRED) return fail(W4A16_INVALID_ARG, "unknown pack flags");
  if ((flags & W4A16_PACK_GATE_UP_PAIRED) && (N % 2 || (N / 2) % 64))
    return fail(W4A16_UNSUPPORTED, "gate/up pairing needs I = N/2 to be a multiple of 64");
  const size_t need = w4a16_packed_bytes(E, N, K, group, flags);
  if (!packed || !desc || (E > 0 && (!qweight || !scales)))
    return fail(W4A16_INVALID_ARG, "NULL pointer");
  if (packed_bytes < need) return fail(W4A16_INVALID_ARG, "packed buffer needs %zu bytes", need);
  if (reinterpret_cast<uintptr_t>(packed) % 256 || reinterpret_cast<uintptr_t>(qweight) % 16)
    return fail(W4A16_INVALID_ARG, "packed must be 256-byte and qweight 16-byte aligned");
  DeviceFacts dev;
  w4a16_status_t st = device_facts(&dev);
  if (st != W4A16_OK) return st;
  cudaError_t err = launch_pack(qweight, scales, E, N, K, flags, packed, stream);
  if (err != cudaSuccess) return cuda_fail(err, "pack launch");
  desc->magic = W4A16_PACK_MAGIC;
  desc->version = W4A16_PACK_VERSION;
  desc->flags = flags;
  desc->E = E;
  desc->N = N;
  desc->K = K;
  desc->group = group;
  desc->bytes = need;
  desc->data = packed;
  return W4A16_OK;
}

w4a16_status_t w4a16_pack_weights_nvfp4(const uint8_t* codes, const uint8_t* scales, int E, int N,
                                        int K, uint32_t flags, void* packed, size_t packed_bytes,
                                        w4a16_packed_weights_t* desc, w4a16_stream_t stream) {
  if (E < 0 || N <= 0 || K <= 0 || K % kBlockK || N % kTileRows)
    return fail(W4A16_UNSUPPORTED, "need K %% 64 == 0 and N %% 128 == 0 (got N=%d K=%d)", N, K);
  if (flags & ~W4A16_PACK_GATE_UP_PAIRED) return fail(W4A16_INVALID_ARG, "unknown pack flags");
  if ((flags & W4A16_PACK_GATE_UP_PAIRED) && (N % 2 || (N / 2) % 64))
    return fail(W4A16_UNSUPPORTED, "gate/up pairing needs I = N/2 to be a multiple of 64");
  const uint32_t all = flags | W4A16_PACK_NVFP4;
  const size_t need = w4a16_packed_bytes(E, N, K, 16, all);
  if (!packed || !desc || (E > 0 && (!codes || !scales)))
    return fail(W4A16_INVALID_ARG, "NULL pointer");
  if (packed_bytes < need) return fail(W4A16_INVALID_ARG, "packed buffer needs %zu bytes", need);
  if (reinterpret_cast<uintptr_t>(packed) % 256 || reinterpret_cast<uintptr_t>(codes) % 16 ||
      reinterpret_cast<uintptr_t>(scales) % 4)
    return fail(W4A16_INVALID_ARG, "packed must be 256-byte, codes 16-byte and scales 4-byte aligned");
  DeviceFacts dev;
  w4a16_status_t st = device_facts(&dev);
  if (st != W4A16_OK) return st;
  cudaError_t err = launch_pack_nvfp4(codes, scales, E, N, K, all, packed, stream);
  if (err != cudaSuccess) return cuda_fail(err, "pack launch");
  desc->magic = W4A16_PACK_MAGIC;
  desc->version = W4A16_PACK_VERSION;
  desc->flags = all;
  desc->E = E;
  desc->N = N;
  desc->K = K;
  desc->group = 16;
  desc->bytes = need;
  desc->data = packed;
  return W4A16_OK;
}

size_t w4a16_gemm_workspace_size(int total_slots, int E, int N, int K, int block_m) {
  (void)total_slots;
  (void)E;
  (void)N;
  (void)K;
  if (!valid_block_m(block_m)) return 0;
  return round_up(static_cast<size_t>(split_unit_budget(block_m)) * sizeof(int32_t), 256) +
         kPartialBytes;
}

w4a16_status_t w4a16_workspace_clear(void* workspace, size_t workspace_bytes,
                                     w4a16_stream_t stream) {
  if (!workspace && workspace_bytes) return fail(W4A16_INVALID_ARG, "NULL workspace");
  if (!workspace_bytes) return W4A16_OK;
  cudaError_t err = cudaMemsetAsync(workspace, 0, workspace_bytes, stream);
  if (err != cudaSuccess) return cuda_fail(err, "cudaMemsetAsync");
  return W4A16_OK;
}

w4a16_status_t w4a16_moe_gemm(const uint16_t* A, int64_t lda, int a_row_div,
                              const w4a16_packed_weights_t* W, const w4a16_routing_t* routing,
                              int epilogue, uint32_t row_flags, uint16_t* C, int64_t ldc,
                              void* workspace, size_t workspace_bytes,
                              int expected_rows_per_expert, const w4a16_schedule_t* schedule,
                              int32_t* dev_err, w4a16_stream_t stream) {
  DeviceFacts dev;
  w4a16_status_t st = device_facts(&dev);
  if (st != W4A16_OK) return st;
  if (row_flags & ~(W4A16_A_ROWS_SORTED | W4A16_C_ROWS_SORTED | W4A16_C_FP32))
    return fail(W4A16_INVALID_ARG, "unknown row flags");
  GemmCall c{A, lda, a_row_div, W, routing, epilogue, row_flags, C, ldc, workspace,
             workspace_bytes, expected_rows_per_expert, schedule, dev_err, 0};
  return run_gemm(c, dev, stream);
}

// ---- grouped contracts: a layout kernel builds the routing, the indexed GEMM computes ----

struct GroupedLayout {  // routing arrays inside the caller's workspace
  size_t off_expert, off_ntp, total;
};

static GroupedLayout grouped_layout(int64_t capacity, int block_m) {
  GroupedLayout L;
  L.off_expert = round_up(static_cast<size_t>(capacity) * 4, 256);
  L.off_ntp = L.off_expert + round_up(static_cast<size_t>(capacity / block_m) * 4, 256);
  L.total = L.off_ntp + 256;
  return L;
}

size_t w4a16_contiguous_workspace_size(int64_t m) {
  if (m <= 0 || m % 128 || m >= (int64_t(1) << 31)) return 0;
  return grouped_layout(m, 128).total;
}

w4a16_status_t w4a16_contiguous_gemm(const uint16_t* A, int64_t lda, int64_t m,
                                     const int32_t* m_indices, const w4a16_packed_weights_t* W,
                                     int epilogue, uint16_t* C, int64_t ldc, void* workspace,
                                     size_t workspace_bytes, int32_t* dev_err,
                                     w4a16_stream_t stream) {
  w4a16_status_t st = check_packed(W);
  if (st != W4A16_OK) return st;
  if (m < 0 || m % 128 || m >= (int64_t(1) << 31))
    return fail(W4A16_INVALID_ARG, "m must be a multiple of 128 below 2^31");
  if (m == 0) return W4A16_OK;
  if (!m_indices || !workspace || reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(W4A16_INVALID_ARG, "m_indices and a 256-byte aligned workspace are required");
  const GroupedLayout L = grouped_layout(m, 128);
  if (workspace_bytes < L.total)
    return fail(W4A16_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes", L.total);
  DeviceFacts dev;
  st = device_facts(&dev);
  if (st != W4A16_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* sorted_ids = reinterpret_cast<int32_t*>(ws);
  int32_t* expert_ids = reinterpret_cast<int32_t*>(ws + L.off_expert);
  int32_t* ntp = reinterpret_cast<int32_t*>(ws + L.off_ntp);
  cudaError_t err = launch_contiguous_layout(m_indices, static_cast<int>(m), W->E, sorted_ids,
                                             expert_ids, ntp, dev_err, dev.num_sms, stream);
  if (err != cudaSuccess) return cuda_fail(err, "contiguous layout launch");
  const w4a16_routing_t R{sorted_ids, expert_ids, ntp, m, 128, static_cast<int32_t>(m)};
  const w4a16_schedule_t one_split{1, 0};
  GemmCall c{A, lda, 1, W, &R, epilogue, W4A16_A_ROWS_SORTED | W4A16_C_ROWS_SORTED, C, ldc,
             nullptr, 0, 128, &one_split, dev_err, 0};
  return run_gemm(c, dev, stream);
}

// Block size of the masked layout from the expected rows per expert (the indexed planner's
// thresholds).
static int masked_block_m(int expected_m) {
  if (expected_m <= 12) return 16;
  if (expected_m <= 24) return 32;
  if (expected_m <= 48) return 64;
  return 128;
}

static int64_t masked_capacity(int G, int max_m, int block_m) {
  return static_cast<int64_t>(G) * ((max_m + block_m - 1) / block_m) * block_m;
}

size_t w4a16_masked_workspace_size(int G, int max_m, int expected_m) {
  if (G <= 0 || G > 1024 || max_m <= 0 || expected_m <= 0 ||
      static_cast<int64_t>(G) * max_m >= (int64_t(1) << 31))
    return 0;
  const int bm = masked_block_m(expected_m);
  return grouped_layout(masked_capacity(G, max_m, bm), bm).total;
}

w4a16_status_t w4a16_masked_gemm(const uint16_t* A, int64_t lda, int G, int max_m,
                                 const int32_t* masked_m, int expected_m,
                                 const w4a16_packed_weights_t* W, int epilogue, uint16_t* C,
                                 int64_t ldc, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_err, w4a16_stream_t stream) {
  w4a16_status_t st = check_packed(W);
  if (st != W4A16_OK) return st;
  if (G != W->E) return fail(W4A16_INVALID_ARG, "G (%d) must equal the weight's expert count (%d)", G, W->E);
  if (G <= 0 || G > 1024 || max_m <= 0 || expected_m <= 0 ||
      static_cast<int64_t>(G) * max_m >= (int64_t(1) << 31))
    return fail(W4A16_INVALID_ARG, "need 1 <= G <= 1024, max_m > 0, expected_m > 0, G * max_m < 2^31");
  if (!masked_m || !workspace || reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(W4A16_INVALID_ARG, "masked_m and a 256-byte aligned workspace are required");
  const int bm = masked_block_m(expected_m);
  const int64_t cap = masked_capacity(G, max_m, bm);
  const GroupedLayout L = grouped_layout(cap, bm);
  if (workspace_bytes < L.total)
    return fail(W4A16_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes", L.total);
  DeviceFacts dev;
  st = device_facts(&dev);
  if (st != W4A16_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* sorted_ids = reinterpret_cast<int32_t*>(ws);
  int32_t* expert_ids = reinterpret_cast<int32_t*>(ws + L.off_expert);
  int32_t* ntp = reinterpret_cast<int32_t*>(ws + L.off_ntp);
  cudaError_t err = launch_masked_layout(masked_m, G, max_m, bm, cap, sorted_ids, expert_ids, ntp,
                                         dev_err, stream);
  if (err != cudaSuccess) return cuda_fail(err, "masked layout launch");
  const w4a16_routing_t R{sorted_ids, expert_ids, ntp, cap, bm, G * max_m};
  const w4a16_schedule_t one_split{1, 0};
  GemmCall c{A, lda, 1, W, &R, epilogue, 0u, C, ldc, nullptr, 0, expected_m, &one_split, dev_err, 0};
  return run_gemm(c, dev, stream);
}

w4a16_status_t w4a16_gather_rows(const uint16_t* x, int64_t ldx, int K, int a_row_div,
                                 const w4a16_routing_t* routing, uint16_t* out, int64_t ldo,
                                 w4a16_stream_t stream) {
  const w4a16_routing_t* R = routing;
  if (!R || !R->sorted_ids || !R->num_tokens_padded || !x || !out)
    return fail(W4A16_INVALID_ARG, "NULL pointer");
  if (K <= 0 || K % 8 || ldx % 8 || ldo % 8 || ldx < K || ldo < K || a_row_div <= 0 ||
      reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(W4A16_INVALID_ARG, "need K, ldx, ldo multiples of 8 and 16-byte aligned rows");
  if (R->capacity < 0 || R->total_slots < 0) return fail(W4A16_INVALID_ARG, "bad routing sizes");
  DeviceFacts dev;
  w4a16_status_t st = device_facts(&dev);
  if (st != W4A16_OK) return st;
  if (R->capacity == 0 || R->total_slots == 0) return W4A16_OK;
  cudaError_t err = launch_gather_rows(x, ldx, K, a_row_div, R->sorted_ids, R->num_tokens_padded,
                                       R->total_slots, R->capacity, out, ldo, dev.num_sms, stream);
  if (err != cudaSuccess) return cuda_fail(err, "gather_rows launch");
  return W4A16_OK;
}

w4a16_status_t w4a16_topk_sum(const float* Y, const int32_t* topk_ids,
                              const float* topk_weights, int T, int top_k, int H,
                              uint16_t* out, w4a16_stream_t stream) {
  if (T < 0 || top_k <= 0 || H <= 0 || H % 8) return fail(W4A16_INVALID_ARG, "need H %% 8 == 0");
  if (T > 0 && (!Y || !topk_ids || !topk_weights || !out))
    return fail(W4A16_INVALID_ARG, "NULL pointer");
  if (reinterpret_cast<uintptr_t>(Y) % 16 || reinterpret_cast<uintptr_t>(out) % 16)
    return fail(W4A16_INVALID_ARG, "Y and out must be 16-byte aligned");
  DeviceFacts dev;
  w4a16_status_t st = device_facts(&dev);
  if (st != W4A16_OK) return st;
  cudaError_t err = launch_topk_sum(Y, topk_ids, topk_weights, T, top_k, H, out, stream);
  if (err != cudaSuccess) return cuda_fail(err, "topk_sum launch");
  return W4A16_OK;
}

int w4a16_plan_block_m(int T, int top_k, int E, int E_global) {
  if (T <= 0 || top_k <= 0 || E <= 0) return 16;
  const int eg = E_global > 0 ? E_global : E;
  const double rows = static_cast<double>(T) * top_k / eg;  // expected rows per local expert
  if (rows <= 12.0) return 16;
  if (rows <= 24.0) return 32;
  if (rows <= 48.0) return 64;
  return 128;
}

w4a16_status_t w4a16_plan_gemm(int total_slots, int E, int N, int K, int block_m,
                               int expected_rows_per_expert, int num_sms, w4a16_plan_t* plan) {
  if (!plan || total_slots < 0 || E <= 0 || num_sms <= 0)
    return fail(W4A16_INVALID_ARG, "bad planner arguments");
  if (!valid_block_m(block_m) || K % kBlockK || N % kTileRows || K <= 0 || N <= 0)
    return fail(W4A16_UNSUPPORTED, "unsupported shape for the planner");
  plan_gemm(total_slots, E, N, K, block_m, expected_rows_per_expert, num_sms, plan);
  return W4A16_OK;
}

// Layer workspace, in order (each piece 256-byte aligned):
//   sorted_ids [cap] | expert_ids [cap / bm] | ntp [1] | K-split counters | K-split partials |
//   xs (gathered activations, sorted rows) [cap, H] BF16 |
//   h (SiLU output, sorted rows) [cap, I] BF16 | Y (down output, slot rows) [T*top_k, H] FP32
struct LayerLayout {
  int block_m;
  int64_t cap;
  size_t off_sorted, off_expert, off_ntp, off_cnt, off_part, off_xs, off_h, off_y, off_done, total;
};

// Words of the single-kernel layer's counters (per-block gate_up tiles, zeroed sums, finished
// CTAs), a multiple of 4.
static size_t done_words(const LayerLayout& L) {
  return round_up(static_cast<size_t>(L.cap / L.block_m) + 2, 4);
}

static LayerLayout layer_layout(int T, int top_k, int E, int E_global, int H, int I, int block_m) {
  LayerLayout L{};
  L.block_m = block_m > 0 ? block_m : w4a16_plan_block_m(T, top_k, E, E_global);
  L.cap = w4a16_align_capacity(T, top_k, E, L.block_m);
  size_t o = 0;
  L.off_sorted = o;
  o = round_up(o + L.cap * 4, 256);
  L.off_expert = o;
  o = round_up(o + (L.cap / L.block_m) * 4, 256);
  L.off_ntp = o;
  o = round_up(o + 4, 256);
  L.off_cnt = o;
  o = round_up(o + split_unit_budget(L.block_m) * 4, 256);
  L.off_part = o;
  o += kPartialBytes;
  L.off_xs = o;  // gathered activations, used by large blocks only
  o = round_up(o + (L.block_m >= 64 ? static_cast<size_t>(L.cap) * H * 2 : 0), 256);
  L.off_h = o;
  o = round_up(o + static_cast<size_t>(L.cap) * I * 2, 256);
  L.off_y = o;
  o = round_up(o + static_cast<size_t>(T) * top_k * H * 4, 256);
  L.off_done = o;  // single-kernel layer: finished gate_up tiles per block, then 2 phase counts
  o = round_up(o + done_words(L) * 4, 256);
  L.total = o;
  return L;
}

size_t w4a16_layer_workspace_size(int T, int top_k, int E, int E_global, int H, int I,
                                  int block_m) {
  if (T < 0 || top_k <= 0 || E <= 0 || H <= 0 || I <= 0) return 0;
  if (block_m != 0 && !valid_block_m(block_m)) return 0;
  return layer_layout(T, top_k, E, E_global, H, I, block_m).total;
}

w4a16_status_t w4a16_moe_layer(const uint16_t* x, const w4a16_packed_weights_t* w13,
                               const w4a16_packed_weights_t* w2, const int32_t* topk_ids,
                               const float* topk_weights, int T, int top_k, int E_global,
                               int block_m, uint16_t* out, void* workspace,
                               size_t workspace_bytes, int32_t* dev_err, w4a16_stream_t stream) {
  return w4a16_moe_layer_ex(x, w13, w2, topk_ids, topk_weights, T, top_k, E_global, block_m, 0u,
                            out, workspace, workspace_bytes, dev_err, stream);
}

w4a16_status_t w4a16_moe_layer_ex(const uint16_t* x, const w4a16_packed_weights_t* w13,
                                  const w4a16_packed_weights_t* w2, const int32_t* topk_ids,
                                  const float* topk_weights, int T, int top_k, int E_global,
                                  int block_m, uint32_t layer_flags, uint16_t* out,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                  w4a16_stream_t stream) {
  if (layer_flags & ~(W4A16_LAYER_FUSED_TOPK | W4A16_LAYER_FUSED | W4A16_LAYER_DEBUG_WAIT_TIMEOUT))
    return fail(W4A16_INVALID_ARG, "unknown layer flags");
  const bool one_kernel = (layer_flags & W4A16_LAYER_FUSED) != 0;
  if ((layer_flags & W4A16_LAYER_DEBUG_WAIT_TIMEOUT) && !one_kernel)
    return fail(W4A16_INVALID_ARG, "W4A16_LAYER_DEBUG_WAIT_TIMEOUT needs W4A16_LAYER_FUSED");
  const bool fused = one_kernel || (layer_flags & W4A16_LAYER_FUSED_TOPK) != 0;
  w4a16_status_t st = check_packed(w13);
  if (st != W4A16_OK) return st;
  if ((st = check_packed(w2)) != W4A16_OK) return st;
  if (!(w13->flags & W4A16_PACK_GATE_UP_PAIRED))
    return fail(W4A16_BAD_PACKED_WEIGHT, "gate_up weight must be packed with GATE_UP_PAIRED");
  const int E = w13->E, H = w13->K, I = w13->N / 2;
  if (w2->E != E || w2->N != H || w2->K != I)
    return fail(W4A16_BAD_PACKED_WEIGHT, "down weight [%d,%d,%d] does not match gate_up [%d,%d,%d]",
                w2->E, w2->N, w2->K, E, w13->N, H);
  if (T < 0 || top_k <= 0 || E <= 0 || E > 1024 || H % 8)
    return fail(W4A16_INVALID_ARG, "bad layer sizes");
  if (block_m != 0 && !valid_block_m(block_m))
    return fail(W4A16_UNSUPPORTED, "block_m %d: supported values are 16, 32, 64, 128", block_m);
  if (T > 0 && (!x || !topk_ids || !topk_weights || !out))
    return fail(W4A16_INVALID_ARG, "NULL pointer");
  const LayerLayout L = layer_layout(T, top_k, E, E_global, H, I, block_m);
  if (!workspace || workspace_bytes < L.total || reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(W4A16_WORKSPACE_TOO_SMALL, "layer workspace needs %zu bytes, 256-byte aligned",
                L.total);
  DeviceFacts dev;
  if ((st = device_facts(&dev)) != W4A16_OK) return st;
  if (T == 0) return W4A16_OK;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* sorted_ids = reinterpret_cast<int32_t*>(ws + L.off_sorted);
  int32_t* expert_ids = reinterpret_cast<int32_t*>(ws + L.off_expert);
  int32_t* ntp = reinterpret_cast<int32_t*>(ws + L.off_ntp);
  uint16_t* xs = reinterpret_cast<uint16_t*>(ws + L.off_xs);
  uint16_t* h = reinterpret_cast<uint16_t*>(ws + L.off_h);
  float* y = reinterpret_cast<float*>(ws + L.off_y);
  const int n_slots = T * top_k;

  // the align kernel also clears counters for the kernels after it: the K-split counters, or
  // the single-kernel layer's block and phase counts
  int32_t* blk_done = reinterpret_cast<int32_t*>(ws + L.off_done);
  cudaError_t err = launch_moe_align(
      topk_ids, n_slots, E, L.block_m, sorted_ids, expert_ids, ntp, L.cap, 0, dev_err,
      one_kernel ? blk_done : reinterpret_cast<int32_t*>(ws + L.off_cnt),
      static_cast<int>(one_kernel ? done_words(L) : split_unit_budget(L.block_m)), stream);
  if (err != cudaSuccess) return cuda_fail(err, "moe_align launch");
  if (!one_kernel && fused) {  // the down GEMM adds into FP32 token sums held where the per-slot rows would be
    err = launch_zero_f32(y, static_cast<int64_t>(T) * H, dev.num_sms, stream);
    if (err != cudaSuccess) return cuda_fail(err, "zero launch");
  }

  w4a16_routing_t R{sorted_ids, expert_ids, ntp, L.cap, L.block_m, n_slots};
  const int eg = E_global > 0 ? E_global : E;
  const int rows_hint = std::max(1, static_cast<int>(std::lround(static_cast<double>(n_slots) / eg)));
  // Large blocks (prefill) read activation tiles by 2-D TMA from rows gathered into aligned
  // order by a separate kernel (the gate_up GEMM streams its first weights meanwhile); small
  // blocks (decode) gather their few rows inside the GEMM, which saves a launch.
  const bool pre_gather = L.block_m >= 64;
  if (pre_gather) {
    err = launch_gather_rows(x, H, H, top_k, sorted_ids, ntp, n_slots, L.cap, xs, H, dev.num_sms,
                             stream);
    if (err != cudaSuccess) return cuda_fail(err, "gather_rows launch");
  }
  GemmCall g1{pre_gather ? xs : x, H, pre_gather ? 1 : top_k, w13, &R, W4A16_EPILOGUE_SILU_MUL,
              (pre_gather ? W4A16_A_ROWS_SORTED : 0u) | W4A16_C_ROWS_SORTED, h, I,
              ws + L.off_cnt, (L.off_xs - L.off_cnt), rows_hint, nullptr, dev_err,
              pre_gather ? 1 : 0};
  GemmCall g2{h, I, 1, w2, &R, W4A16_EPILOGUE_NONE, W4A16_A_ROWS_SORTED | W4A16_C_FP32,
              reinterpret_cast<uint16_t*>(y), H,
              ws + L.off_cnt, (L.off_xs - L.off_cnt), rows_hint, nullptr, dev_err, 1};
  if (one_kernel) {
    const w4a16_schedule_t one_split{1, 0, 0, 1};
    g1.sched = &one_split;
    g2.sched = &one_split;
    g1.one_kernel = g2.one_kernel = true;
    g2.merge_w = topk_weights;
    g2.merge_k = top_k;
    GemmArgs a1, a2;
    int grid1 = 0, grid2 = 0;
    bool empty1 = false, empty2 = false;
    if ((st = prepare_gemm(g1, dev, &a1, &grid1, &empty1)) != W4A16_OK) return st;
    if ((st = prepare_gemm(g2, dev, &a2, &grid2, &empty2)) != W4A16_OK) return st;
    if (empty1 || empty2) {  // nothing routed: the output is zeros
      err = cudaMemsetAsync(out, 0, static_cast<size_t>(T) * H * sizeof(uint16_t), stream);
      if (err != cudaSuccess) return cuda_fail(err, "output clear");
      return W4A16_OK;
    }
    a1.signal_done = blk_done;
    a2.wait_done = blk_done;
    a2.wait_count = a1.n_tiles;
    if (layer_flags & W4A16_LAYER_DEBUG_WAIT_TIMEOUT) {  // a count nothing reaches, short limit
      a2.wait_count = a1.n_tiles + 1;
      a2.wait_limit = 1ll << 20;
    }
    a2.routing_ready = a1.routing_ready;
    // the kernel zeroes the sums, merges into them and rounds them into out
    a2.sync = blk_done + L.cap / L.block_m;
    a2.sum_elems = static_cast<int64_t>(T) * H;
    a2.final_out = out;
    err = launch_layer_fused(a1, a2, dev.num_sms, stream);
    if (err != cudaSuccess) return cuda_fail(err, "fused layer launch");
    return W4A16_OK;
  }
  if ((st = run_gemm(g1, dev, stream)) != W4A16_OK) return st;
  if (fused) {
    const w4a16_schedule_t one_split{1, 0};  // the merge is the reduction: no K splits
    g2.sched = &one_split;
    g2.merge_w = topk_weights;
    g2.merge_k = top_k;
    if ((st = run_gemm(g2, dev, stream)) != W4A16_OK) return st;
    err = launch_round_bf16(y, static_cast<int64_t>(T) * H, out, dev.num_sms, stream);
    if (err != cudaSuccess) return cuda_fail(err, "round launch");
    return W4A16_OK;
  }
  if ((st = run_gemm(g2, dev, stream)) != W4A16_OK) return st;
  err = launch_topk_sum(y, topk_ids, topk_weights, T, top_k, H, out, stream);
  if (err != cudaSuccess) return cuda_fail(err, "topk_sum launch");
  return W4A16_OK;
}

w4a16_status_t w4a16_debug_dequant(const w4a16_packed_weights_t* W, int expert, uint16_t* out,
                                   w4a16_stream_t stream) {
  w4a16_status_t st = check_packed(W);
  if (st != W4A16_OK) return st;
  if (expert < 0 || expert >= W->E || !out) return fail(W4A16_INVALID_ARG, "bad expert or output");
  DeviceFacts dev;
  if ((st = device_facts(&dev)) != W4A16_OK) return st;
  cudaError_t err = launch_debug_dequant(W->data, W->E, expert, W->N, W->K, W->flags, out, stream);
  if (err != cudaSuccess) return cuda_fail(err, "debug_dequant launch");
  return W4A16_OK;
}

}  // extern "C"
