// Device-side building blocks for the sm_103a kernels: mbarriers, bulk TMA,
// cp.async, tcgen05 (TMEM allocation, MMA, loads/stores), proxy fences and
// programmatic dependent launch.  Hand-written inline PTX; every wait is
// bounded so a broken pipeline reports an error instead of hanging.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "w4a16_moe.h"

namespace w4a16 {

// ---- packed-weight geometry (shared by the packer, the GEMM and debug dequant) -----------
constexpr int kTileRows = 128;             // weight rows per tile = MMA M
constexpr int kBlockK = 64;                // K elements per pipeline stage
constexpr int kCodeHalfBytes = kTileRows * 16;           // 4 words of 128 rows
constexpr int kScaleOffset = 2 * kCodeHalfBytes;         // 4096
constexpr int kChunkBytes = kScaleOffset + kTileRows * 4;  // 4608 bytes per (tile, kb)
constexpr int kHeaderBytes = 256;

// After the chunks, one mode byte per (expert, tile): kTileScaled when every scale of the tile
// lies in (0, 2^-5) and the chunks hold each scale as s * 2^133 (the multiply-add conversion),
// kTilePlain otherwise (scales as given, the subtract-then-multiply conversion).
constexpr uint8_t kTilePlain = 0, kTileScaled = 1;
constexpr uint16_t kScaledMaxBits = 0x3CFF;  // largest BF16 s with s * 2^133 finite (< 2^-5)
__host__ __device__ inline int64_t tile_mode_offset(int E, int n_tiles, int n_kb) {
  return kHeaderBytes + static_cast<int64_t>(E) * n_tiles * n_kb * kChunkBytes;
}

// BF16 bits of s * 2^133 for 0 < s < 2^-5 (bits 0x0001..0x3CFF): exact, since a power-of-two
// factor only moves the exponent (a subnormal s = m * 2^-133 becomes the integer m).
__host__ __device__ inline uint16_t scale_times_2p133(uint16_t s) {
  if (s >= 0x0080u) return static_cast<uint16_t>(s + (133u << 7));
  int p = 6;  // subnormal: value m = s (1..127); normalise its leading bit
  while (!((s >> p) & 1u)) --p;
  return static_cast<uint16_t>(((127u + p) << 7) | ((static_cast<uint32_t>(s) << (7 - p)) & 0x7Fu));
}

// Device header at the start of every packed blob.
struct PackedHeader {
  uint64_t magic;
  uint32_t version;
  uint32_t flags;
  int32_t E, N, K, group;
  int32_t n_tiles, n_kb;
};

// Canonical weight row of tile-row r (0..127) of tile j.  Paired gate/up tiles interleave
// 16-row groups: lanes [32w, 32w+16) of a tile hold gate rows, [32w+16, 32w+32) the up rows
// with the same intermediate index.
__host__ __device__ inline int tile_row_to_canonical(int j, int r, int N, bool paired) {
  if (!paired) return j * kTileRows + r;
  const int I = N / 2;
  const int w = r >> 5, l = r & 31;
  const int col = 64 * j + 16 * w + (l & 15);
  return (l < 16) ? col : I + col;
}

// Nibble position p of a packed word holds element kPerm[p] of the canonical word, so that
// (word >> 4m) & 0x000F000F yields elements (2m, 2m+1) in the two 16-bit halves.
__host__ __device__ inline uint32_t interleave_nibbles(uint32_t w) {
  uint32_t out = 0;
  // positions 0..3 <- elements 0,2,4,6 ; positions 4..7 <- elements 1,3,5,7
  for (int m = 0; m < 4; ++m) {
    out |= ((w >> (8 * m)) & 0xFu) << (4 * m);
    out |= ((w >> (8 * m + 4)) & 0xFu) << (4 * (m + 4));
  }
  return out;
}

// ---- small helpers --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_dev_err(int32_t* dev_err, int bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

// Two BF16 weights from a packed word: bits (m, m+4) -> ((q - 8) * s) rounded once.
// 0x4300 | q is the BF16 value 128 + q exactly; subtracting 136 leaves q - 8 exactly; the
// product with the scale pair is one round-to-nearest-even BF16 multiply.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t shifted_word, uint32_t scale2) {
  uint32_t v;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(v) : "r"(shifted_word), "r"(0x000F000Fu), "r"(0x43004300u));
  uint32_t t, w;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(v), "r"(0x43084308u));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w) : "r"(t), "r"(scale2));
  return w;
}

// Eight dequantised pairs (16 weights, columns 4w..4w+3 for two words) from one packed word:
// writes out[0..3] = pairs (0,1),(2,3),(4,5),(6,7) of the word's 8 elements.
__device__ __forceinline__ void dequant_word(uint32_t word, uint32_t scale2, uint32_t* out) {
  out[0] = dequant_pair(word, scale2);
  out[1] = dequant_pair(word >> 4, scale2);
  out[2] = dequant_pair(word >> 8, scale2);
  out[3] = dequant_pair(word >> 12, scale2);
}

// Scaled tiles: the conversion without the subtraction.  Masked in place, a nibble at bits 0-3
// of a BF16 half is the subnormal q * 2^-133, and at bits 4-7 it is q * 2^-129 (bit patterns
// below 0x100 are linear in value across the subnormal/normal boundary).  With the chunk's
// scale taken as s * 2^133 (and s * 2^129), one fused multiply-add with -8s forms (q - 8) * s
// exactly before its single round-to-nearest-even, so the BF16 result equals the
// subtract-then-scale definition (for s > 0; zero results are +0 as there).
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ void dequant_word_scaled(uint32_t word, uint32_t s133, uint32_t s129,
                                                    uint32_t neg8s, uint32_t* out) {
  out[0] = fma_bf16x2(word & 0x000F000Fu, s133, neg8s);
  out[1] = fma_bf16x2(word & 0x00F000F0u, s129, neg8s);
  const uint32_t w8 = word >> 8;
  out[2] = fma_bf16x2(w8 & 0x000F000Fu, s133, neg8s);
  out[3] = fma_bf16x2(w8 & 0x00F000F0u, s129, neg8s);
}

// Same output as dequant_row64 for a chunk of a scaled tile (scales2x = the two groups'
// s * 2^133).
__device__ __forceinline__ void dequant_row64_scaled(uint4 lo, uint4 hi, uint32_t scales2x,
                                                     uint32_t (&r)[32]) {
  uint32_t s129, neg8s;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(s129) : "r"(scales2x), "r"(0x3D803D80u));  // x 2^-4
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(neg8s) : "r"(s129), "r"(0x80808080u));     // x -2^-126
  const uint32_t a0 = __byte_perm(scales2x, 0, 0x1010), a1 = __byte_perm(scales2x, 0, 0x3232);
  const uint32_t b0 = __byte_perm(s129, 0, 0x1010), b1 = __byte_perm(s129, 0, 0x3232);
  const uint32_t c0 = __byte_perm(neg8s, 0, 0x1010), c1 = __byte_perm(neg8s, 0, 0x3232);
  dequant_word_scaled(lo.x, a0, b0, c0, &r[0]);
  dequant_word_scaled(lo.y, a0, b0, c0, &r[4]);
  dequant_word_scaled(lo.z, a0, b0, c0, &r[8]);
  dequant_word_scaled(lo.w, a0, b0, c0, &r[12]);
  dequant_word_scaled(hi.x, a1, b1, c1, &r[16]);
  dequant_word_scaled(hi.y, a1, b1, c1, &r[20]);
  dequant_word_scaled(hi.z, a1, b1, c1, &r[24]);
  dequant_word_scaled(hi.w, a1, b1, c1, &r[28]);
}

// Dequantise one tile row of a 64-wide K block from a chunk (shared or global memory):
// 32 BF16x2 registers in K order (register c holds elements 2c, 2c+1).
__device__ __forceinline__ void dequant_row64(uint4 lo, uint4 hi, uint32_t scales2x,
                                              uint32_t (&r)[32]) {
  const uint32_t s0 = __byte_perm(scales2x, 0, 0x1010);
  const uint32_t s1 = __byte_perm(scales2x, 0, 0x3232);
  dequant_word(lo.x, s0, &r[0]);
  dequant_word(lo.y, s0, &r[4]);
  dequant_word(lo.z, s0, &r[8]);
  dequant_word(lo.w, s0, &r[12]);
  dequant_word(hi.x, s1, &r[16]);
  dequant_word(hi.y, s1, &r[20]);
  dequant_word(hi.z, s1, &r[24]);
  dequant_word(hi.w, s1, &r[28]);
}

// NVFP4 row of a 64-wide K block: 32 bytes of E2M1 pairs (element 2c in the low nibble of byte
// c; bytes 0..15 in lo, 16..31 in hi) and four E4M3 scales (one per 16 elements, byte i of
// scales4) -> 32 BF16x2 registers in K order.  Every product of an E2M1 value and an E4M3 scale
// is exact in BF16, and so is each step: the E2M1 pair converts to FP16 exactly (the
// e2m1x2 -> f16x2 conversion), the FP16 bits shifted right by 3 (sign kept) are the BF16 bits
// of the same value times 2^-112, and the scale is taken as BF16 times 2^112, so the one
// BF16 multiply yields the exact product.
__device__ __forceinline__ void nvfp4_scales(uint32_t scales4, uint32_t (&sb)[4]) {
  uint32_t f01, f23;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f01) : "h"(static_cast<uint16_t>(scales4 & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f23) : "h"(static_cast<uint16_t>(scales4 >> 16)));
  const uint32_t f[2] = {f01, f23};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint16_t b;
    asm("cvt.rn.bf16.f16 %0, %1;" : "=h"(b) : "h"(static_cast<uint16_t>(f[i >> 1] >> (16 * (i & 1)))));
    const uint32_t pair = static_cast<uint32_t>(b) * 0x00010001u;  // the scale in both halves
    uint32_t scaled;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(scaled) : "r"(pair), "r"(0x77807780u));  // x 2^112
    sb[i] = scaled;
  }
}

// Four E2M1 pairs of one word -> four BF16x2 products with the (2^112-scaled) scale pair sb.
__device__ __forceinline__ void nvfp4_word(uint32_t word, uint32_t sb, uint32_t* out) {
  uint32_t h0, h1, h2, h3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(word));
  const uint32_t h[4] = {h0, h1, h2, h3};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = ((h[i] & 0x7FFF7FFFu) >> 3) | (h[i] & 0x80008000u);  // BF16 of value * 2^-112
    uint32_t w;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(w) : "r"(v), "r"(sb));
    out[i] = w;
  }
}

__device__ __forceinline__ void dequant_row64_nvfp4(uint4 lo, uint4 hi, uint32_t scales4,
                                                    uint32_t (&r)[32]) {
  uint32_t sb[4];
  nvfp4_scales(scales4, sb);
  nvfp4_word(lo.x, sb[0], &r[0]);  // elements 0..7
  nvfp4_word(lo.y, sb[0], &r[4]);  // 8..15
  nvfp4_word(lo.z, sb[1], &r[8]);  // 16..23
  nvfp4_word(lo.w, sb[1], &r[12]);
  nvfp4_word(hi.x, sb[2], &r[16]);  // 32..39
  nvfp4_word(hi.y, sb[2], &r[20]);
  nvfp4_word(hi.z, sb[3], &r[24]);
  nvfp4_word(hi.w, sb[3], &r[28]);
}

// ---- mbarrier ------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread for up to `ns` nanoseconds; it still returns as soon
// as the phase completes, so waiting warps stop taking issue slots from the working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait: ~2^31 cycles (about a second) before giving up.  `abort_flag` (shared) lets
// the other roles of the CTA leave promptly once one of them has given up.
constexpr long long kWaitLimitCycles = 1ll << 31;
constexpr uint32_t kSuspendNs = 20000;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* dev_err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *abort_flag = 1;
      set_dev_err(dev_err, W4A16_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Wait without an abort check (teardown drains).
__device__ __forceinline__ bool mbar_wait_plain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kSuspendNs)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}

// Release increment of a counter in global memory (pairs with wait_count_at_least).
__device__ __forceinline__ void red_release_add(int32_t* p, int32_t v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until a counter in global memory reaches `want` (acquire: what was stored
// before the increments is visible afterwards).  On timeout the CTA's abort flag and the
// caller's error word are set.
__device__ __forceinline__ bool wait_count_at_least(const int32_t* p, int32_t want,
                                                    volatile int* abort_flag, int32_t* dev_err,
                                                    long long limit = kWaitLimitCycles) {
  const long long t0 = clock64();
  while (true) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= want) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      set_dev_err(dev_err, W4A16_DEVERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
    __nanosleep(200);
  }
}

// ---- bulk TMA and cp.async -------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 16-byte async copy with zero fill when src_bytes == 0.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// Arrive on `bar` once all earlier cp.async of this thread have landed (count not raised).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// generic-proxy writes to global memory (seen through an acquire) -> later async-proxy reads
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ---- programmatic dependent launch --------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- tcgen05 -------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16 (BF16 inputs, FP32 accumulate).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ---- CTA pairs (tcgen05 cta_group::2): one MMA spans the TMEM and shared memory of two CTAs
// of a cluster; every tcgen05 allocation, MMA and commit of such a kernel uses cta_group::2.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster, with the default semantics (release at
// CTA scope); the waiting side uses the plain waits above.  The arriving warps have finished
// their tensor-memory stores (tcgen05.wait::st, then tcgen05.fence::before_thread_sync)
// before they arrive.  Measured on GB300: cluster-scope release arrivals and acquire waits made
// the CTA-pair GEMM 1.9x slower than one CTA per tile (Qwen3 T=4096 gate_up 338.6 against
// 174.8 us with these forms, the results bitwise the same).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// M = 256 across the pair: A rows [0, 128) from this CTA's TMEM, [128, 256) from the peer's
// (same address); B rows [0, N/2) from this CTA's shared memory, [N/2, N) from the peer's
// (same offset); D rows split like A.  Issued by the even CTA only.
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at `bar`'s offset in both CTAs of the pair when the pair MMAs
// issued so far complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread (lane l) gets columns [c, c+32) of lane l.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// Wait for this thread's tcgen05.ld operations, with the 16 destination registers as operands so
// the compiler cannot move their uses above the wait.
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte swizzle layout:
// rows of 128 bytes (64 BF16), 8-row groups 1024 bytes apart, tile base 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);       // start address
  d |= static_cast<uint64_t>(1u) << 16;                      // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;              // stride byte offset: 8-row groups
  d |= static_cast<uint64_t>(1u) << 46;                      // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: BF16 A and B (K-major), FP32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                   // D format: F32
         | (1u << 7)                                 // A format: BF16
         | (1u << 10)                                // B format: BF16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

}  // namespace w4a16

namespace w4a16 {

// ---- single-lane election and tensor TMA ----------------------------------------------------
// true in exactly one lane of a converged warp
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// 2-D tiled tensor load: box at (x = column, y = row) of the tensor map into shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// A 3-D tile [z][y][x] (sorted activation rows viewed as [K / 64][rows][64]): one copy loads a
// whole pipeline stage of 64-wide K blocks, each block's rows after the previous block's.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// CTA pairs: the same copy into this CTA's shared memory, its completion signalled on an
// mbarrier of either CTA of the pair (`bar` is a shared::cluster address, e.g. the even CTA's).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, int x, int y,
                                                 int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

}  // namespace w4a16
