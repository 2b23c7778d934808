// w4a16_moe_gemm_static_scratch: the indexed GEMM for callers that cannot allocate memory.
//
// Some callers cannot hand the library a workspace: an inference-engine plugin whose enqueue
// hook receives only its input and output buffers, or a serving loop that must not call
// cudaMalloc after start-up (the call can synchronise the device and fragment memory that
// was budgeted up front).  For them the GEMM's K-split scratch (per-tile arrival counters and
// FP32 partial sums) lives in this file-scope device array instead of a caller workspace.
// Every GPU that loads the library holds the array until the process exits.
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace w4a16 {

void set_error_detail(const char* text);  // api.cu

// Counters for the smallest block size (32768 / 16 int32, rounded to 256 bytes) followed by the
// 16 MB of FP32 partials: exactly what w4a16_gemm_workspace_size() asks for at most.
constexpr size_t kStaticScratchBytes = W4A16_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_scratch_mu;
// Device address of g_static_scratch per device ordinal, with the CUDA context it was looked
// up in: a device reset (or a released and re-created primary context) gives the device a new
// context, in which the array has a new address, so the lookup is repeated then.
void* g_scratch_ptr[64] = {};
void* g_scratch_ctx[64] = {};

typedef int (*CtxGetCurrentFn)(void**);  // cuCtxGetCurrent, fetched from the driver at run time

void* current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    tried = true;
  }
  void* ctx = nullptr;
  if (fn && fn(&ctx) != 0) ctx = nullptr;
  return ctx;
}
}  // namespace

// Device address of the array for the current device, looked up on the first call in each
// device's context.  (In host code the array's name is only a host-side stand-in, not a device
// address.)
static cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const void* ctx = current_context();  // NULL before the runtime has set up the device
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_static_scratch);  // sets up the device's context if needed
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context();
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace w4a16

using namespace w4a16;

extern "C" w4a16_status_t w4a16_moe_gemm_static_scratch(
    const uint16_t* A, int64_t lda, int a_row_div, const w4a16_packed_weights_t* W,
    const w4a16_routing_t* routing, int epilogue, uint32_t row_flags, uint16_t* C, int64_t ldc,
    int expected_rows_per_expert, const w4a16_schedule_t* schedule, int32_t* dev_err,
    w4a16_stream_t stream) {
  if (!W || !routing) return w4a16_moe_gemm(A, lda, a_row_div, W, routing, epilogue, row_flags,
                                            C, ldc, nullptr, 0, expected_rows_per_expert,
                                            schedule, dev_err, stream);
  const size_t need = w4a16_gemm_workspace_size(routing->total_slots, W->E, W->N, W->K,
                                                routing->block_m);
  if (need > kStaticScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof msg,
             "this GEMM needs %zu bytes of scratch, more than the %zu-byte static scratch", need,
             kStaticScratchBytes);
    set_error_detail(msg);
    return W4A16_WORKSPACE_TOO_SMALL;
  }
  void* scratch = nullptr;
  cudaError_t err = scratch_address(&scratch);
  if (err != cudaSuccess) {
    cudaGetLastError();
    char msg[160];
    snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch: %s",
             cudaGetErrorString(err));
    set_error_detail(msg);
    return W4A16_CUDA_ERROR;
  }
  // The per-tile arrival counters (the first bytes of the scratch) must start at zero; a
  // finished call leaves them zero, this also covers a call that gave up part way.
  if (need > 0) {
    const size_t counter_bytes = need - (size_t(16) << 20);
    err = cudaMemsetAsync(scratch, 0, counter_bytes, stream);
    if (err != cudaSuccess) {
      cudaGetLastError();
      set_error_detail("clearing the static scratch counters failed");
      return W4A16_CUDA_ERROR;
    }
  }
  return w4a16_moe_gemm(A, lda, a_row_div, W, routing, epilogue, row_flags, C, ldc, scratch,
                        kStaticScratchBytes, expected_rows_per_expert, schedule, dev_err, stream);
}
