// Paged GQA decode attention over the quantized cache, with split-K over the
// context and a log-sum-exp merge.
//
// What it computes: for each sequence b and query head hq, the softmax over
// retained positions p in [lo, L) of softmax_scale * <q, K_hat[p]> weights
// V_hat[p]; K_hat = code * K scale, V_hat = code * V scale.  The K scale is
// applied to the dot product of q with the raw codes and the V scale to the
// softmax weight, so codes are never rescaled element by element.
// Scale layouts: "Per-tensor vs per-head FP8 KV cache scales"; windows and
// BF16 (skipped) layers: "FP8 KV cache layer skipping vs per-head scales",
// sections "FP8 KV cache layer skipping vs per-head scales" and "Layer
// skipping follows retained-token footprint".
//
// Decomposition: one CTA of 4 warps per (sequence, KV head, split).  The
// split's positions are cut into 32-position tiles; warp w takes tiles w,
// w+4, ...  In a tile, lane i owns position tile*32+i for the QK products of
// all G query heads of the group (q lives in shared memory, pre-multiplied by
// softmax_scale*log2(e)), the online softmax runs in log2 units, and the PV
// update spreads the tile's V rows over the lanes, 8 elements per lane.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int WARPS = 4;
constexpr int TILE = 32;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two E4M3 codes (low byte first) -> two floats; the conversion is exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  uint32_t h2;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(two));
  const unsigned short lo = (unsigned short)(h2 & 0xFFFFu), hi = (unsigned short)(h2 >> 16);
  float2 r;
  asm("cvt.f32.f16 %0, %1;" : "=f"(r.x) : "h"(lo));
  asm("cvt.f32.f16 %0, %1;" : "=f"(r.y) : "h"(hi));
  return r;
}

// 8 row elements starting at element 8*c of a cached row, as floats (codes,
// not yet scaled).
template <int MODE, int D>
__device__ __forceinline__ void load8(const uint8_t* row, int c, float v[8]) {
  if constexpr (MODE == BF16) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + 16 * c);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(ws[i] << 16);
      v[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
    }
  } else if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + 4 * c);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = (float)(((int)(w << (28 - 4 * i))) >> 28);
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(row + 8 * c);
    float2 a = e4m3x2_to_float2(w.x & 0xFFFFu), b = e4m3x2_to_float2(w.x >> 16);
    float2 d = e4m3x2_to_float2(w.y & 0xFFFFu), e = e4m3x2_to_float2(w.y >> 16);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    v[4] = d.x; v[5] = d.y; v[6] = e.x; v[7] = e.y;
  }
}

template <int MODE>
constexpr int row_bytes(int D) {
  return MODE == BF16 ? 2 * D : (MODE == INT4_PER_TOKEN_HEAD ? D / 2 : D);
}

template <int MODE, int D, int G>
__global__ void __launch_bounds__(WARPS * 32) decode_kernel(DecodeArgs a) {
  constexpr int RB = row_bytes<MODE>(D);
  constexpr int LPR = D / 8;            // lanes per row in the PV phase
  constexpr int RPI = 32 / LPR;         // rows per pass in the PV phase
  constexpr bool DYN = (MODE == FP8_PER_TOKEN_HEAD || MODE == INT4_PER_TOKEN_HEAD);

  __shared__ __align__(16) float q_s[G][D];
  __shared__ float p_s[WARPS][TILE][G];
  __shared__ long long row_s[WARPS][TILE];      // cell index of each tile row, -1 = none
  __shared__ float m_s[WARPS][G], l_s[WARPS][G];
  __shared__ __align__(16) float o_s[WARPS][G][D];

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int j = i / D, d = i - j * D;
    const uint16_t qb = a.q[((long long)b * a.Hq + g * G + j) * D + d];
    q_s[j][d] = __uint_as_float((uint32_t)qb << 16) * a.qk_scale;
  }
  __syncthreads();

  int L = a.context_lens[b];
  if (L < 0) {
    if (threadIdx.x == 0 && split == 0 && g == 0) atomicOr(a.err, ERR_BAD_INDEX);
    L = 0;
  }
  const int lo = (a.window > 0 && L > a.window) ? L - a.window : 0;
  const int t0 = lo / TILE, t1 = (L + TILE - 1) / TILE;
  const int n_tiles = t1 - t0;
  const int tps = (n_tiles + a.splits - 1) / a.splits;
  const int my_t0 = t0 + split * tps;
  const int my_t1 = min(t1, my_t0 + tps);

  float ks_static = 1.f, vs_static = 1.f;
  if constexpr (MODE == FP8_PER_TENSOR) { ks_static = a.k_scale[0]; vs_static = a.v_scale[0]; }
  if constexpr (MODE == FP8_PER_HEAD) { ks_static = a.k_scale[g]; vs_static = a.v_scale[g]; }

  float m[G], l[G], o[G][8];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[j][e] = 0.f;
  }

  const int pr = lane / LPR, pc = lane % LPR;   // PV-phase row group and column chunk
  const int* bt = a.block_table + (long long)b * a.max_blocks;

  for (int tile = my_t0 + warp; tile < my_t1; tile += WARPS) {
    // ---- QK: lane owns one position
    const int pos = tile * TILE + lane;
    long long cell = -1;
    if (pos >= lo && pos < L) {
      const int blk = bt[pos / a.bs];
      if (blk >= 0 && blk < a.num_blocks) {
        cell = ((long long)blk * a.Hkv + g) * a.bs + (pos % a.bs);
      } else {
        atomicOr(a.err, ERR_BAD_INDEX);
      }
    }
    float s[G];
#pragma unroll
    for (int j = 0; j < G; ++j) s[j] = 0.f;
    float vsc = 0.f;
    if (cell >= 0) {
      const uint8_t* krow = a.k_cache + cell * RB;
#pragma unroll 4
      for (int c = 0; c < D / 8; ++c) {
        float kv[8];
        load8<MODE, D>(krow, c, kv);
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float4 qa = *reinterpret_cast<const float4*>(&q_s[j][8 * c]);
          const float4 qb = *reinterpret_cast<const float4*>(&q_s[j][8 * c + 4]);
          s[j] += qa.x * kv[0] + qa.y * kv[1] + qa.z * kv[2] + qa.w * kv[3] +
                  qb.x * kv[4] + qb.y * kv[5] + qb.z * kv[6] + qb.w * kv[7];
        }
      }
      const float ksc = DYN ? a.k_cs[cell] : ks_static;
      vsc = DYN ? a.v_cs[cell] : vs_static;
#pragma unroll
      for (int j = 0; j < G; ++j) s[j] *= ksc;
    } else {
#pragma unroll
      for (int j = 0; j < G; ++j) s[j] = -INFINITY;
    }
    // ---- online softmax (log2 units)
    float alpha[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float mt = s[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float mn = fmaxf(m[j], mt);
      if (mn == -INFINITY) {
        alpha[j] = 1.f;
        p_s[warp][lane][j] = 0.f;
      } else {
        alpha[j] = ex2(m[j] - mn);           // m = -inf -> 0
        const float p = (cell >= 0) ? ex2(s[j] - mn) : 0.f;
        l[j] = l[j] * alpha[j] + p;          // per-lane partial sum
        p_s[warp][lane][j] = p * vsc;
      }
      m[j] = mn;
    }
    row_s[warp][lane] = cell;
    __syncwarp();
    // ---- PV: lane group pr walks rows pr, pr+RPI, ...; column chunk pc
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[j][e] *= alpha[j];
    for (int r = pr; r < TILE; r += RPI) {
      const long long vc = row_s[warp][r];
      if (vc < 0) continue;
      float vv[8];
      load8<MODE, D>(a.v_cache + vc * RB, pc, vv);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float p = p_s[warp][r][j];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[j][e] += p * vv[e];
      }
    }
    __syncwarp();
  }

  // ---- reduce inside the warp: l over lanes, o over the RPI row groups
#pragma unroll
  for (int j = 0; j < G; ++j) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l[j] += __shfl_xor_sync(0xffffffffu, l[j], off);
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[j][e] += __shfl_xor_sync(0xffffffffu, o[j][e], off);
  }
  if (lane < LPR) {
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) o_s[warp][j][8 * pc + e] = o[j][e];
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < G; ++j) { m_s[warp][j] = m[j]; l_s[warp][j] = l[j]; }
  }
  __syncthreads();

  // ---- combine the warps, then write the output or the split's partial
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int j = i / D, d = i - j * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, m_s[w][j]);
    float acc = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < WARPS; ++w) {
        const float f = ex2(m_s[w][j] - M);
        acc += f * o_s[w][j][d];
        den += f * l_s[w][j];
      }
    }
    const long long head = (long long)b * a.Hq + g * G + j;
    if (a.splits == 1) {
      a.out[head * D + d] = den > 0.f ? acc / den : 0.f;
    } else {
      const long long part = (((long long)b * a.Hkv + g) * a.splits + split) * G + j;
      a.ws_o[part * D + d] = acc;
      if (d == 0) { a.ws_ml[2 * part] = M; a.ws_ml[2 * part + 1] = den; }
    }
  }
}

// Log-sum-exp merge of the splits: one CTA of D threads per (sequence, KV head).
template <int D, int G>
__global__ void __launch_bounds__(D) merge_kernel(DecodeArgs a) {
  const int g = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const long long base = ((long long)b * a.Hkv + g) * a.splits;
  for (int j = 0; j < G; ++j) {
    float M = -INFINITY;
    for (int s = 0; s < a.splits; ++s) M = fmaxf(M, a.ws_ml[2 * ((base + s) * G + j)]);
    float acc = 0.f, den = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < a.splits; ++s) {
        const long long part = (base + s) * G + j;
        const float f = ex2(a.ws_ml[2 * part] - M);
        acc += f * a.ws_o[part * D + d];
        den += f * a.ws_ml[2 * part + 1];
      }
    }
    a.out[((long long)b * a.Hq + g * G + j) * D + d] = den > 0.f ? acc / den : 0.f;
  }
}

template <int MODE, int D, int G>
cudaError_t launch3(const DecodeArgs& a, cudaStream_t st) {
  dim3 grid(a.splits, a.Hkv, a.B);
  decode_kernel<MODE, D, G><<<grid, WARPS * 32, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  merge_kernel<D, G><<<dim3(a.Hkv, a.B), D, 0, st>>>(a);
  return cudaGetLastError();
}

template <int MODE, int D>
cudaError_t launch2(int G, const DecodeArgs& a, cudaStream_t st) {
  switch (G) {
    case 1: return launch3<MODE, D, 1>(a, st);
    case 2: return launch3<MODE, D, 2>(a, st);
    case 4: return launch3<MODE, D, 4>(a, st);
    case 8: return launch3<MODE, D, 8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int MODE>
cudaError_t launch1(int D, int G, const DecodeArgs& a, cudaStream_t st) {
  switch (D) {
    case 64: return launch2<MODE, 64>(G, a, st);
    case 128: return launch2<MODE, 128>(G, a, st);
    case 256: return launch2<MODE, 256>(G, a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool decode_supported(int mode, int D, int G) {
  return mode >= BF16 && mode <= INT4_PER_TOKEN_HEAD && (D == 64 || D == 128 || D == 256) &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_decode(int mode, int D, int G, const DecodeArgs& a, cudaStream_t st) {
  if (a.B == 0) return cudaSuccess;
  switch (mode) {
    case BF16: return launch1<BF16>(D, G, a, st);
    case FP8_PER_TENSOR: return launch1<FP8_PER_TENSOR>(D, G, a, st);
    case FP8_PER_HEAD: return launch1<FP8_PER_HEAD>(D, G, a, st);
    case FP8_PER_TOKEN_HEAD: return launch1<FP8_PER_TOKEN_HEAD>(D, G, a, st);
    case INT4_PER_TOKEN_HEAD: return launch1<INT4_PER_TOKEN_HEAD>(D, G, a, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
