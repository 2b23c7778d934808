// Offline weight repack and the debug dequantiser.
//
// "vLLM x Novita AI: Chord, Faster INT4 MoE for Kimi K2.x", "Grouped SM90 kernels": weights
// are repacked once for the kernel that reads them and the prepared weight records its mode.
// Here the target is the GB300 GEMM's stream of 4608-byte chunks, one per (expert, 128-row
// tile, 64-wide K block), read by one bulk copy each:
//   bytes [0, 2048)     row r at 16*r: canonical words 0..3 of the block (K 0..31)
//   bytes [2048, 4096)  row r at 2048 + 16*r: words 4..7 (K 32..63)
//   bytes [4096, 4608)  row r at 4096 + 4*r: the two BF16 scales of the block
// Words are nibble-interleaved (positions 0..3 hold elements 0,2,4,6 and 4..7 hold 1,3,5,7)
// so that one mask yields two neighbouring elements in the two halves of a register.
// After the chunks, one mode byte per (expert, tile): a tile whose scales all lie in (0, 2^-5)
// stores them as s * 2^133 and is converted with one multiply-add per pair (kTileScaled);
// any other tile keeps its scales and the subtract-then-multiply conversion (kTilePlain).
// NVFP4 blobs use the same chunk geometry with the codes in their natural byte order (one
// byte = one E2M1 pair, which the hardware converts as a pair) and four E4M3 scales per row.
#include "common.cuh"

namespace w4a16 {

// Mode byte of each (expert, tile): scaled when every scale of its 128 rows is in (0, 2^-5).
// One thread per tile row; grid (n_tiles, E).
__global__ void __launch_bounds__(kTileRows)
    tile_mode_kernel(const uint16_t* __restrict__ scales, int N, int K, int n_tiles, int n_kb,
                     int paired, uint8_t* __restrict__ out) {
  const int j = blockIdx.x, e = blockIdx.y, r = threadIdx.x;
  const int n = tile_row_to_canonical(j, r, N, paired != 0);
  const uint16_t* s = scales + (static_cast<int64_t>(e) * N + n) * (K / 32);
  bool ok = true;
  for (int g = 0; g < K / 32; ++g) {
    const uint16_t v = __ldg(s + g);
    ok = ok && v >= 1u && v <= kScaledMaxBits;
  }
  ok = __syncthreads_and(ok) != 0;
  if (r == 0)
    out[tile_mode_offset(gridDim.y, n_tiles, n_kb) + static_cast<int64_t>(e) * n_tiles + j] =
        ok ? kTileScaled : kTilePlain;
}

// One thread per tile row; grid (n_kb, n_tiles, E).  Runs after tile_mode_kernel.
__global__ void __launch_bounds__(kTileRows)
    pack_kernel(const int32_t* __restrict__ qweight, const uint16_t* __restrict__ scales, int N,
                int K, int n_tiles, int n_kb, int paired, uint8_t* __restrict__ out) {
  const int kb = blockIdx.x, j = blockIdx.y, e = blockIdx.z, r = threadIdx.x;
  const int n = tile_row_to_canonical(j, r, N, paired != 0);
  const int64_t row = static_cast<int64_t>(e) * N + n;
  const uint32_t* src = reinterpret_cast<const uint32_t*>(qweight) + row * (K / 8) + kb * 8;
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = interleave_nibbles(__ldg(src + i));
  const uint16_t* s = scales + row * (K / 32) + kb * 2;
  uint16_t s0 = __ldg(s), s1 = __ldg(s + 1);
  if (out[tile_mode_offset(gridDim.z, n_tiles, n_kb) + static_cast<int64_t>(e) * n_tiles + j] ==
      kTileScaled) {
    s0 = scale_times_2p133(s0);
    s1 = scale_times_2p133(s1);
  }
  const uint32_t s2 = static_cast<uint32_t>(s0) | (static_cast<uint32_t>(s1) << 16);
  uint8_t* chunk =
      out + kHeaderBytes + ((static_cast<int64_t>(e) * n_tiles + j) * n_kb + kb) * kChunkBytes;
  reinterpret_cast<uint4*>(chunk)[r] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(chunk + kCodeHalfBytes)[r] = make_uint4(w[4], w[5], w[6], w[7]);
  reinterpret_cast<uint32_t*>(chunk + kScaleOffset)[r] = s2;
}

// NVFP4 (one thread per tile row): the row's 32 code bytes of the K block in order (bytes
// 0..15 at 16*r, 16..31 at 2048 + 16*r) and its four E4M3 scale bytes at 4096 + 4*r.
__global__ void __launch_bounds__(kTileRows)
    pack_nvfp4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int N,
                      int K, int n_tiles, int n_kb, int paired, uint8_t* __restrict__ out) {
  const int kb = blockIdx.x, j = blockIdx.y, e = blockIdx.z, r = threadIdx.x;
  const int n = tile_row_to_canonical(j, r, N, paired != 0);
  const int64_t row = static_cast<int64_t>(e) * N + n;
  const uint4* src = reinterpret_cast<const uint4*>(codes + row * (K / 2) + kb * 32);
  const uint32_t s4 = __ldg(reinterpret_cast<const uint32_t*>(scales + row * (K / 16) + kb * 4));
  uint8_t* chunk =
      out + kHeaderBytes + ((static_cast<int64_t>(e) * n_tiles + j) * n_kb + kb) * kChunkBytes;
  reinterpret_cast<uint4*>(chunk)[r] = __ldg(src);
  reinterpret_cast<uint4*>(chunk + kCodeHalfBytes)[r] = __ldg(src + 1);
  reinterpret_cast<uint32_t*>(chunk + kScaleOffset)[r] = s4;
}

__global__ void write_header_kernel(PackedHeader h, uint8_t* out) {
  *reinterpret_cast<PackedHeader*>(out) = h;
}

// Debug: dequantise expert e back to canonical [N, K] with the GEMM's conversion routine.
__global__ void __launch_bounds__(kTileRows)
    debug_dequant_kernel(const uint8_t* __restrict__ packed, int E, int e, int N, int K,
                         int n_tiles, int n_kb, int paired, int nvfp4,
                         uint16_t* __restrict__ out) {
  const int kb = blockIdx.x, j = blockIdx.y, r = threadIdx.x;
  const uint8_t* chunk =
      packed + kHeaderBytes + ((static_cast<int64_t>(e) * n_tiles + j) * n_kb + kb) * kChunkBytes;
  const uint4 lo = reinterpret_cast<const uint4*>(chunk)[r];
  const uint4 hi = reinterpret_cast<const uint4*>(chunk + kCodeHalfBytes)[r];
  const uint32_t s2 = reinterpret_cast<const uint32_t*>(chunk + kScaleOffset)[r];
  const uint8_t mode = packed[tile_mode_offset(E, n_tiles, n_kb) + static_cast<int64_t>(e) * n_tiles + j];
  uint32_t v[32];
  if (nvfp4)
    dequant_row64_nvfp4(lo, hi, s2, v);
  else if (mode == kTileScaled)
    dequant_row64_scaled(lo, hi, s2, v);
  else
    dequant_row64(lo, hi, s2, v);
  const int n = tile_row_to_canonical(j, r, N, paired != 0);
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<int64_t>(n) * K + kb * kBlockK);
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

cudaError_t launch_pack(const int32_t* qweight, const uint16_t* scales, int E, int N, int K,
                        uint32_t flags, void* packed, cudaStream_t stream) {
  const int n_tiles = N / kTileRows, n_kb = K / kBlockK;
  PackedHeader h{};
  h.magic = W4A16_PACK_MAGIC;
  h.version = W4A16_PACK_VERSION;
  h.flags = flags;
  h.E = E;
  h.N = N;
  h.K = K;
  h.group = 32;
  h.n_tiles = n_tiles;
  h.n_kb = n_kb;
  uint8_t* out = static_cast<uint8_t*>(packed);
  write_header_kernel<<<1, 1, 0, stream>>>(h, out);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (E == 0) return cudaSuccess;
  const int paired = (flags & W4A16_PACK_GATE_UP_PAIRED) ? 1 : 0;
  tile_mode_kernel<<<dim3(n_tiles, E), kTileRows, 0, stream>>>(scales, N, K, n_tiles, n_kb,
                                                                 paired, out);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  pack_kernel<<<dim3(n_kb, n_tiles, E), kTileRows, 0, stream>>>(qweight, scales, N, K, n_tiles,
                                                                n_kb, paired, out);
  return cudaGetLastError();
}

cudaError_t launch_pack_nvfp4(const uint8_t* codes, const uint8_t* scales, int E, int N, int K,
                              uint32_t flags, void* packed, cudaStream_t stream) {
  const int n_tiles = N / kTileRows, n_kb = K / kBlockK;
  PackedHeader h{};
  h.magic = W4A16_PACK_MAGIC;
  h.version = W4A16_PACK_VERSION;
  h.flags = flags;
  h.E = E;
  h.N = N;
  h.K = K;
  h.group = 16;
  h.n_tiles = n_tiles;
  h.n_kb = n_kb;
  uint8_t* out = static_cast<uint8_t*>(packed);
  write_header_kernel<<<1, 1, 0, stream>>>(h, out);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (E == 0) return cudaSuccess;
  err = cudaMemsetAsync(out + tile_mode_offset(E, n_tiles, n_kb), kTilePlain,
                        static_cast<size_t>(E) * n_tiles, stream);
  if (err != cudaSuccess) return err;
  pack_nvfp4_kernel<<<dim3(n_kb, n_tiles, E), kTileRows, 0, stream>>>(
      codes, scales, N, K, n_tiles, n_kb, (flags & W4A16_PACK_GATE_UP_PAIRED) ? 1 : 0, out);
  return cudaGetLastError();
}

cudaError_t launch_debug_dequant(const void* packed, int E, int e, int N, int K, uint32_t flags,
                                 uint16_t* out, cudaStream_t stream) {
  const int n_tiles = N / kTileRows, n_kb = K / kBlockK;
  debug_dequant_kernel<<<dim3(n_kb, n_tiles), kTileRows, 0, stream>>>(
      static_cast<const uint8_t*>(packed), E, e, N, K, n_tiles, n_kb,
      (flags & W4A16_PACK_GATE_UP_PAIRED) ? 1 : 0, (flags & W4A16_PACK_NVFP4) ? 1 : 0, out);
  return cudaGetLastError();
}

}  // namespace w4a16
