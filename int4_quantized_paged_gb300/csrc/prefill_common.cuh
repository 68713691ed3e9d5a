// Pieces shared by the two prefill kernels: the launch arguments and the
// exact conversion of 16 raw cache bytes into f16 (bf16 for BF16 layers).
#pragma once

#include <stdint.h>

#include "kvq_internal.h"
#include "tile_math.cuh"

namespace kvq {

struct PrefillArgs {
  DecodeArgs d;                  // caches, scales, block table, context_lens, q, out
  const int* query_start;        // [B + 1]
  int qtiles;                    // query tiles per (sequence, KV head) in the grid
};

// 16 raw code bytes -> their f16 (bf16 for BF16) values: 8 (BF16), 16 (FP8)
// or 32 (INT4) elements, as 1, 2 or 4 16-byte chunks.  Exact.
template <int MODE>
__device__ __forceinline__ void convert16(uint4 w, uint4 (&o)[4]) {
  if constexpr (MODE == BF16) {
    o[0] = w;
  } else if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t x = ws[q];
      // low nibble of byte j = element 2j: e = {b0.lo, b1.lo}, h = 16 {b0.hi, b1.hi}
      const uint32_t e0 = nib2_f16x2<0>(__byte_perm(x, 0u, 0x7170));
      const uint32_t h0 = nib2_f16x2<1>(__byte_perm(x, 0u, 0x7170));
      const uint32_t e1 = nib2_f16x2<0>(__byte_perm(x, 0u, 0x7372));
      const uint32_t h1 = nib2_f16x2<1>(__byte_perm(x, 0u, 0x7372));
      uint32_t hs0, hs1;
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hs0) : "r"(h0), "r"(0x2C002C00u));   // x 1/16
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hs1) : "r"(h1), "r"(0x2C002C00u));
      o[q].x = __byte_perm(e0, hs0, 0x5410);
      o[q].y = __byte_perm(e0, hs0, 0x7632);
      o[q].z = __byte_perm(e1, hs1, 0x5410);
      o[q].w = __byte_perm(e1, hs1, 0x7632);
    }
  } else {
    e4m3x4_f16(w.x, o[0].x, o[0].y);
    e4m3x4_f16(w.y, o[0].z, o[0].w);
    e4m3x4_f16(w.z, o[1].x, o[1].y);
    e4m3x4_f16(w.w, o[1].z, o[1].w);
  }
}

}  // namespace kvq
