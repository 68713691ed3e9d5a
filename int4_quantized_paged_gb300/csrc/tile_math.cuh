// Fragment-level helpers shared by the decode and prefill attention kernels:
// exact conversions of cache codes to f16, packing, mma.sync wrappers, the
// 128B-swizzle address map of TMA tiles, TMA tile copies.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "kvq_internal.h"

namespace kvq {

// 2^x, flushing results below 2^-126 to zero: every use is a softmax weight
// or a rescale factor relative to a running maximum, where such a value is
// negligible beside the weight 1 of the maximum itself.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tma_tile_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// One box of a 3-D tensor map at coordinates (x, y, z) into shared memory.
__device__ __forceinline__ void tma_tile_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// As tma_tile_2d, with an L2 eviction-priority policy (createpolicy) for
// data read once.
__device__ __forceinline__ void tma_tile_2d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 policy for copies: evict first (data streamed once, larger than L2) or
// normal priority (data that may still be in L2 at its next use).
__device__ __forceinline__ uint64_t l2_copy_policy(bool evict_first) {
  uint64_t pol;
  if (evict_first)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Four E4M3 codes (one word) -> two f16x2: bytes 0,1 -> lo; bytes 2,3 -> hi.
// The conversion is exact.
__device__ __forceinline__ void e4m3x4_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %2; cvt.rn.f16x2.e4m3x2 %0, a; cvt.rn.f16x2.e4m3x2 %1, b; }"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// The two's-complement nibbles at bits 4P..4P+3 and 16+4P..19+4P of x (P = 0
// or 1) -> f16x2 of 16^P times their signed values, exactly.  Flipping bit 3
// of a nibble makes it offset binary m = n + 8; placed in the mantissa under
// the exponent of 1024 it reads 1024 + 16^P m, and subtracting 1024 + 8 16^P
// leaves 16^P n.  The flip, the mask and the exponent bits are one
// three-input logic operation.
template <int P>
__device__ __forceinline__ uint32_t nib2_f16x2(uint32_t x) {
  constexpr uint32_t M = 0x000F000Fu << (4 * P);
  constexpr uint32_t C = (0x00080008u << (4 * P)) | 0x64006400u;
  constexpr uint32_t S = P == 0 ? 0x64086408u : 0x64806480u;   // f16 1032 / 1152
  const uint32_t h = (x & M) ^ C;
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(S));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float f16_lo(uint32_t h2) {
  float f;
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %1; cvt.f32.f16 %0, a; }" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t h2) {
  float f;
  asm("{ .reg .b16 a, b; mov.b32 {a, b}, %1; cvt.f32.f16 %0, b; }" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float bf16_lo(uint32_t h2) { return __uint_as_float(h2 << 16); }

// y rounded to E4M3 (nearest even, saturating to +-448), as a float: the
// value of the code the cache write would store for y.
__device__ __forceinline__ float e4m3_round(float y) {
  unsigned short c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(0.f), "f"(y));
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return f16_lo(h2);
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

template <bool BF>
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// ------------------------------------------------------------------ layout
template <int MODE>
constexpr int row_bytes(int D) {
  return MODE == BF16 ? 2 * D : (MODE == INT4_PER_TOKEN_HEAD ? D / 2 : D);
}

// Shared-memory byte offset of logical byte `o` of a tile written by a TMA
// copy with 128-byte rows and 128B swizzle (buffer 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(uint32_t o) {
  return o ^ (((o >> 7) & 7u) << 4);
}

// 2^e for e in [-126, 127] (exact, from the exponent bits); 0 below.
__device__ __forceinline__ float pow2i(int e) {
  return e < -126 ? 0.f : __uint_as_float((uint32_t)(e + 127) << 23);
}

// Unbiased exponent of a positive normal float.
__device__ __forceinline__ int f32_exp(float x) {
  return (int)((__float_as_uint(x) >> 23) & 0xFF) - 127;
}

}  // namespace kvq
