// Fused quantize-and-scatter cache write, static per-head calibration and the
// stand-alone E4M3 encoder.
//
// Scale layouts: "Per-tensor vs per-head FP8 KV cache scales" (sections
// "Per-tensor vs per-head FP8 KV cache scales" and "Dynamic per-token-head
// scales add 3.125 percent"); packed INT4: "Per-token-head KV cache scale
// overhead", section "INT4 makes the metadata fraction larger".
//
// The write is a pure HBM stream: per token and KV head it reads 2*2D bytes
// of bf16 K/V and writes 2*D*elem code bytes plus 8 scale bytes.  Two kernels
// share the arithmetic: write_staged_kernel for large writes (token rows
// streamed into a shared-memory ring by bulk copies; one group of D/16 lanes
// per head vector) and write_kernel for small writes and BF16 layers (one
// group of D/8 lanes per vector, 16-byte loads straight into registers).  In
// both the amax is a shuffle reduction inside the group.
#include <cuda_runtime.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "kvq_internal.h"

namespace kvq {

__device__ unsigned g_error_word;

unsigned* error_word() {
  static unsigned* ptr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptr[dev] = static_cast<unsigned*>(p);
  }
  return ptr[dev];
}

namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448
// (hardware cvt with .satfinite).  `lo` lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Max over the LPV lanes of one vector group.  Groups of one warp may take
// different paths (a skipped slot, the end of the grid-stride loop), so the
// shuffle names only the group's own lanes.
template <int LPV>
__device__ __forceinline__ float group_max(float v) {
  const unsigned lane = threadIdx.x & 31u;
  const unsigned mask = (LPV == 32) ? 0xffffffffu
                                    : (((1u << LPV) - 1u) << (lane & ~(unsigned)(LPV - 1)));
#pragma unroll
  for (int o = LPV / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(mask, v, o));
  return v;
}

// Unpacks 8 bf16 (one 16-byte word group) to fp32.
__device__ __forceinline__ void unpack8(float* x, const uint4 raw) {
  x[0] = bf16_lo(raw.x); x[1] = bf16_hi(raw.x);
  x[2] = bf16_lo(raw.y); x[3] = bf16_hi(raw.y);
  x[4] = bf16_lo(raw.z); x[5] = bf16_hi(raw.z);
  x[6] = bf16_lo(raw.w); x[7] = bf16_hi(raw.w);
}

// Dynamic scale from the vector's amax: s = RN32(amax / qmax), 1.0 for a zero
// vector.  Computed by the reciprocal correction below (exact for every bf16
// amax >= 2^-100); IEEE division under that.
template <int MODE>
__device__ __forceinline__ float dynamic_scale(float m) {
  constexpr float qmax = (MODE == INT4_PER_TOKEN_HEAD) ? 7.0f : 448.0f;
  constexpr float rq = 1.0f / qmax;                         // RN(1/qmax)
  if (m >= 0x1p-100f) {
    const float q0 = __fmul_rn(m, rq);
    return __fmaf_rn(__fmaf_rn(-q0, qmax, m), rq, q0);
  }
  return (m == 0.f) ? 1.0f : __fdiv_rn(m, qmax);
}

// y = RN32(x / s).  One correctly rounded reciprocal per vector, then per
// element q0 = RN(x r) and the FMA correction q1 = RN(q0 + RN(x - q0 s) r),
// which is the correctly rounded quotient while the remainder x - q0 s is
// exact (Markstein's theorem: r within half an ulp of 1/s, q0 within an ulp).
// That holds away from fp32 underflow; below the guard the kernel divides.
// Verified equal to IEEE division over every dynamic scale (every bf16 amax,
// /448 and /7, every bf16 |x| <= amax) where the result decides a code, and
// over random static scales.  With a static scale the quotient can be huge;
// past 1e30 it saturates either way, so the correction is skipped there.
// With a dynamic scale |x/s| <= qmax (1 + 2^-23), so no guard is needed.
template <int MODE, int N>
__device__ __forceinline__ void divide_rn(float* y, const float* x, float s) {
  constexpr bool DYN = (MODE == FP8_PER_TOKEN_HEAD || MODE == INT4_PER_TOKEN_HEAD);
  constexpr float kLo = DYN ? 0x1p-100f : 0x1p-60f;
  if (s >= kLo && s <= 0x1p100f) {
    const float r = __frcp_rn(s);
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float q0 = __fmul_rn(x[i], r);
      const float q1 = __fmaf_rn(__fmaf_rn(-q0, s, x[i]), r, q0);
      y[i] = (DYN || fabsf(q0) < 1e30f) ? q1 : q0;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) y[i] = __fdiv_rn(x[i], s);
  }
}

// Codes of N quotients: E4M3 bytes (N/4 words) or packed INT4 nibbles, even
// element in the low nibble (N/8 words).
//
// INT4: for |y| < 2^22, RN(y + 1.5 * 2^23) = 1.5 * 2^23 + RNE(y) exactly (the
// sum's ulp is 1, ties go to the even significand, i.e. to even RNE(y)), and
// the bit pattern of that float is the pattern of 1.5 * 2^23 (low bits 0)
// plus RNE(y), so its low four bits are RNE(y) as a two's-complement nibble.
// The per-token-head scale keeps |y| <= 7 (1 + 2^-23) (s = RN(amax / 7),
// |x| <= amax, and the scale's rounding error is far below 1/14 down to the
// smallest bf16 amax), so RNE(y) already lies in [-7, 7] and needs no clamp.
template <int MODE, int N>
__device__ __forceinline__ void encode(uint32_t* w, const float* y) {
  if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
    constexpr float kRound = 12582912.0f;                     // 1.5 * 2^23
#pragma unroll
    for (int k = 0; k < N / 8; ++k) {
      uint32_t b[4];                                          // byte j in the low 8 bits
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = __float_as_uint(__fadd_rn(y[8 * k + 2 * j], kRound));
        const uint32_t hi = __float_as_uint(__fadd_rn(y[8 * k + 2 * j + 1], kRound));
        b[j] = (lo & 0x0Fu) | ((hi << 4) & 0xF0u);
      }
      w[k] = __byte_perm(__byte_perm(b[0], b[1], 0x0040u), __byte_perm(b[2], b[3], 0x0040u),
                         0x5410u);
    }
  } else {
#pragma unroll
    for (int k = 0; k < N / 4; ++k)
      w[k] = e4m3x2(y[4 * k], y[4 * k + 1]) | (e4m3x2(y[4 * k + 2], y[4 * k + 3]) << 16);
  }
}

// Quantize and store one vector's 8-element slice held by this lane.
template <int MODE, int D>
__device__ __forceinline__ void quantize_store(const WriteArgs& a, const uint4 raw, int is_v, int h,
                                               long long cell, int sub) {
  constexpr int LPV = D / 8;
  uint8_t* cache = is_v ? a.v_cache : a.k_cache;
  if constexpr (MODE == BF16) {
    reinterpret_cast<uint4*>(cache + cell * (2 * D))[sub] = raw;
  } else {
    float x[8];
    unpack8(x, raw);
    float s;
    if constexpr (MODE == FP8_PER_TENSOR) {
      s = __ldg(is_v ? a.v_scale : a.k_scale);
    } else if constexpr (MODE == FP8_PER_HEAD) {
      s = __ldg((is_v ? a.v_scale : a.k_scale) + h);
    } else {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
      s = dynamic_scale<MODE>(group_max<LPV>(m));
      if (sub == 0) (is_v ? a.v_cs : a.k_cs)[cell] = s;
    }
    float y[8];
    divide_rn<MODE, 8>(y, x, s);
    uint32_t w[2];
    encode<MODE, 8>(w, y);
    if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
      reinterpret_cast<uint32_t*>(cache + cell * (D / 2))[sub] = w[0];
    } else {
      reinterpret_cast<uint2*>(cache + cell * D)[sub] = make_uint2(w[0], w[1]);
    }
  }
}

// One group of LPV = D/8 lanes per (token, head, K|V) vector; each group
// handles UNROLL grid-strided vectors per pass, issuing all their loads
// before any arithmetic so several 16-byte loads per lane are in flight.
template <int MODE, int D>
__global__ void __launch_bounds__(256) write_kernel(WriteArgs a) {
  constexpr int LPV = D / 8;
  constexpr int UNROLL = 4;
  const long long lane_id = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int sub = threadIdx.x % LPV;
  const long long per_tensor = a.T * a.Hkv;
  const long long n_vec = 2 * per_tensor;
  const long long stride_vec = ((long long)gridDim.x * blockDim.x) / LPV;
  // vector index -> (tensor, token, head) in 32-bit arithmetic (the host
  // refuses writes of 2^31 vectors or more)
  const unsigned per_t = (unsigned)per_tensor, hkv = (unsigned)a.Hkv;
  for (long long base = lane_id / LPV; base < n_vec; base += UNROLL * stride_vec) {
    uint4 raw[UNROLL];
    long long slot[UNROLL];
    int hh[UNROLL], vv[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const long long vec = base + u * stride_vec;
      slot[u] = -1;
      if (vec < n_vec) {
        const unsigned v32 = (unsigned)vec;
        const int is_v = v32 >= per_t;
        const unsigned th = is_v ? v32 - per_t : v32;
        const unsigned t = th / hkv;
        const int h = (int)(th - t * hkv);
        hh[u] = h;
        vv[u] = is_v;
        const uint16_t* src = (is_v ? a.v_new : a.k_new) + (long long)t * a.token_stride + (long long)h * D;
        raw[u] = __ldg(reinterpret_cast<const uint4*>(src) + sub);
        slot[u] = __ldg(a.slots + t);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const long long vec = base + u * stride_vec;
      if (vec >= n_vec) break;                                // whole group agrees
      const int is_v = vv[u], h = hh[u];
      if (slot[u] < 0) continue;                              // whole group agrees
      if (slot[u] >= a.num_blocks * a.bs) {
        if (sub == 0 && !is_v && h == 0) atomicOr(a.err, ERR_BAD_INDEX);
        continue;
      }
      const long long blk = slot[u] >> a.bs_shift;
      const int off = (int)(slot[u] & (a.bs - 1));
      const long long cell = (blk * a.Hkv + h) * a.bs + off;
      quantize_store<MODE, D>(a, raw[u], is_v, h, cell, sub);
    }
  }
}

// Staged write for large token counts.  Each CTA takes chunks of TT tokens
// (chunk c, c + grid, ...).  A producer warp streams the chunks' K and V rows
// (one bulk copy per token row) and slot indices through a WNS-stage
// shared-memory ring; eight consumer warps quantize from it, one group of
// D/16 lanes per head vector, 16 elements per lane, and release each stage on
// its "empty" barrier, so no warp waits for another except through the ring.
// Bytes in flight do not depend on registers.  The arithmetic is that of
// write_kernel.
constexpr int WNS = 3;            // ring stages
constexpr int WCONSUMERS = 256;   // consumer threads (8 warps)
constexpr int WTHREADS = WCONSUMERS + 32;
constexpr int WMAXTT = 32;        // tokens per chunk at most

struct StagedLayout {
  unsigned row;                   // bytes of one token's K (or V) row: Hkv * D * 2
  int tt;                         // tokens per chunk
  unsigned stage;                 // 2 * tt * row
  unsigned smem;                  // ring + slot table + full and empty barriers
};

__host__ __device__ inline StagedLayout staged_layout(int Hkv, int D) {
  StagedLayout l;
  l.row = (unsigned)Hkv * D * 2;
  int tt = (int)(8192u / l.row);    // about 16 KB of K and V rows per stage
  l.tt = tt < 1 ? 1 : (tt > WMAXTT ? WMAXTT : tt);
  l.stage = 2u * l.tt * l.row;
  l.smem = WNS * l.stage + WNS * WMAXTT * 8 + 2 * WNS * 8;
  return l;
}

template <int MODE, int D>
__global__ void __launch_bounds__(WTHREADS, 4) write_staged_kernel(const WriteArgs a) {
  constexpr int LPV = D / 16;                 // lanes per vector
  constexpr int GROUPS = WCONSUMERS / LPV;
  constexpr int RB = (MODE == BF16) ? 2 * D : (MODE == INT4_PER_TOKEN_HEAD ? D / 2 : D);
  extern __shared__ __align__(128) uint8_t smem[];
  const StagedLayout ly = staged_layout(a.Hkv, D);
  const int TT = ly.tt;
  long long* slot_s = reinterpret_cast<long long*>(smem + WNS * ly.stage);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + WNS * ly.stage + WNS * WMAXTT * 8);
  uint64_t* empty = full + WNS;
  const int tid = threadIdx.x, lane = tid & 31;
  const long long nchunks = (a.T + TT - 1) / TT;
  if ((long long)blockIdx.x >= nchunks) return;     // whole CTA: before any barrier
  if (tid == 0) {
    for (int s = 0; s < WNS; ++s) {
      mbar_init(&full[s], 2);                       // copies' arrive + slots' arrive
      mbar_init(&empty[s], WCONSUMERS / 32);        // one arrive per consumer warp
    }
    mbar_init_fence();
  }
  __syncthreads();                                  // the only CTA-wide barrier

  if (tid >= WCONSUMERS) {
    // ---------------- producer warp
    int st = 0;
    long long k = 0;                                // chunks of this CTA so far
    for (long long c = blockIdx.x; c < nchunks; c += gridDim.x, ++k) {
      // the k-th chunk reuses stage k % WNS after the consumers released
      // chunk k - WNS there: phase k / WNS - 1 of its empty barrier
      if (k >= WNS && !mbar_wait(&empty[st], (uint32_t)(k / WNS - 1) & 1u)) {
        if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
        return;
      }
      const long long t0 = c * TT;
      const int nt = (int)min((long long)TT, a.T - t0);
      uint8_t* dst = smem + st * ly.stage;
      if (lane == 0) {
        fence_proxy_async();
        mbar_expect_tx(&full[st], 2u * nt * ly.row);
        for (int i = 0; i < nt; ++i) {
          const long long src = (t0 + i) * a.token_stride;
          bulk_copy(dst + i * ly.row, a.k_new + src, ly.row, &full[st]);
          bulk_copy(dst + (TT + i) * ly.row, a.v_new + src, ly.row, &full[st]);
        }
      }
      // the chunk's slots, loaded while its rows are in flight; the arrive
      // after the warp barrier publishes them with the stage
      if (lane < nt) slot_s[st * WMAXTT + lane] = __ldg(a.slots + t0 + lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
      if (++st == WNS) st = 0;
    }
    return;
  }

  // ---------------- consumer warps
  const int grp = tid / LPV, sub = tid % LPV;
  const long long cells = a.num_blocks * a.bs;      // < 2^31 (checked on the host)
  const unsigned hkv = (unsigned)a.Hkv;
  // r / Hkv as a multiply-high: exact for r < 2^32 / Hkv, and r < 64 Hkv here
  const unsigned long long magic = ((1ull << 32) + hkv - 1) / hkv;
  int st = 0;
  uint32_t par = 0;
  for (long long c = blockIdx.x; c < nchunks; c += gridDim.x) {
    const long long t0 = c * TT;
    const int nt = (int)min((long long)TT, a.T - t0);
    if (!mbar_wait(&full[st], par)) {
      if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
      return;
    }
    const uint8_t* rows = smem + st * ly.stage;
    const int nvec = nt * a.Hkv;                     // vectors per tensor in the chunk
    for (int v = grp; v < 2 * nvec; v += GROUPS) {
      const int is_v = v >= nvec;
      const int r = is_v ? v - nvec : v;
      const unsigned i = (unsigned)(((unsigned long long)(unsigned)r * magic) >> 32);
      const unsigned h = (unsigned)r - i * hkv;
      const long long slot = slot_s[st * WMAXTT + i];
      if (slot < 0) continue;                        // whole group agrees
      if (slot >= cells) {
        if (sub == 0 && !is_v && h == 0) atomicOr(a.err, ERR_BAD_INDEX);
        continue;
      }
      const unsigned sl = (unsigned)slot;
      const unsigned cell = (((sl >> a.bs_shift) * hkv + h) << a.bs_shift) | (sl & (a.bs - 1));
      const uint8_t* src = rows + (is_v ? TT + i : i) * ly.row + h * (2 * D) + sub * 32;
      const uint4 r0 = *reinterpret_cast<const uint4*>(src);
      const uint4 r1 = *reinterpret_cast<const uint4*>(src + 16);
      uint8_t* dst = (is_v ? a.v_cache : a.k_cache) + (size_t)cell * RB;
      if constexpr (MODE == BF16) {
        reinterpret_cast<uint4*>(dst)[2 * sub] = r0;
        reinterpret_cast<uint4*>(dst)[2 * sub + 1] = r1;
      } else {
        float x[16];
        unpack8(x, r0);
        unpack8(x + 8, r1);
        float s;
        if constexpr (MODE == FP8_PER_TENSOR) {
          s = __ldg(is_v ? a.v_scale : a.k_scale);
        } else if constexpr (MODE == FP8_PER_HEAD) {
          s = __ldg((is_v ? a.v_scale : a.k_scale) + h);
        } else {
          float m = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(x[e]));
          s = dynamic_scale<MODE>(group_max<LPV>(m));
          if (sub == 0) (is_v ? a.v_cs : a.k_cs)[cell] = s;
        }
        float y[16];
        divide_rn<MODE, 16>(y, x, s);
        uint32_t w[4];
        encode<MODE, 16>(w, y);
        if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
          reinterpret_cast<uint2*>(dst)[sub] = make_uint2(w[0], w[1]);
        } else {
          reinterpret_cast<uint4*>(dst)[sub] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    __syncwarp();                                    // this warp is done with stage st
    if (lane == 0) mbar_arrive(&empty[st]);
    if (++st == WNS) { st = 0; par ^= 1u; }
  }
}

// Resident staged-write CTAs per SM for this layout (0: not launchable).
template <int MODE, int D>
int staged_ctas_per_sm(unsigned smem) {
  static int max_set[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  auto kern = write_staged_kernel<MODE, D>;
  if (!max_set[dev]) {
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
            cudaSuccess)
      return 0;
    max_set[dev] = optin;
  }
  if ((int)smem > max_set[dev]) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, WTHREADS, smem) != cudaSuccess)
    return 0;
  return n;
}

template <int MODE, int D>
cudaError_t launch_write_d(const WriteArgs& a, cudaStream_t st) {
  // staged path once there is at least one chunk per SM (a BF16 layer is a
  // plain copy, which the direct kernel streams faster)
  const StagedLayout ly = staged_layout(a.Hkv, D);
  const long long nchunks = (a.T + ly.tt - 1) / ly.tt;
  if (MODE != BF16 && nchunks >= sm_count()) {
    const int per_sm = staged_ctas_per_sm<MODE, D>(ly.smem);
    if (per_sm > 0) {
      long long grid = (long long)sm_count() * per_sm;
      if (grid > nchunks) grid = nchunks;
      write_staged_kernel<MODE, D><<<(unsigned)grid, WTHREADS, ly.smem, st>>>(a);
      return cudaGetLastError();
    }
  }
  const long long lanes_needed = 2 * a.T * a.Hkv * (D / 8);
  const int threads = 256;
  long long blocks = (lanes_needed + threads - 1) / threads;
  const long long cap = (long long)sm_count() * 8 * 4;      // resident blocks x 4; grid-stride beyond
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  write_kernel<MODE, D><<<(unsigned)blocks, threads, 0, st>>>(a);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(int D, const WriteArgs& a, cudaStream_t st) {
  switch (D) {
    case 64: return launch_write_d<MODE, 64>(a, st);
    case 128: return launch_write_d<MODE, 128>(a, st);
    case 256: return launch_write_d<MODE, 256>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------- calibration
// amax per KV head over a [T][Hkv][D] bf16 sample.  Positive floats order like
// their bit patterns, so an integer atomicMax on the bits is a float max.
__global__ void calib_zero(unsigned* amax_bits, int Hkv) {
  int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < Hkv) amax_bits[h] = 0u;
}

// Grid: x over token chunks, y = KV head.  One atomic per block.
__global__ void calib_amax(const uint16_t* x, long long T, int Hkv, int D, unsigned* amax_bits) {
  const int h = blockIdx.y;
  const long long n = T * D;                 // elements of head h
  float m = 0.f;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / D, d = i - t * D;
    m = fmaxf(m, fabsf(__uint_as_float((uint32_t)x[(t * Hkv + h) * D + d] << 16)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wmax[32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, wmax[w]);
    atomicMax(amax_bits + h, __float_as_uint(r));
  }
}

__global__ void calib_finish(unsigned* amax_bits, int Hkv, float qmax) {
  int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < Hkv) {
    const float m = __uint_as_float(amax_bits[h]);
    reinterpret_cast<float*>(amax_bits)[h] = (m == 0.f) ? 1.0f : __fdiv_rn(m, qmax);
  }
}

// The bounded wait of the decode and cache-write kernels, made to run out:
// the barrier expects bytes that no copy delivers (none is issued, so nothing
// is in flight when the wait gives up), and the warp flags TIMEOUT exactly as
// those kernels do.
__global__ void wait_check_kernel(unsigned* err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  const int lane = threadIdx.x & 31;
  if (lane == 0) mbar_init(&bar, 1);
  mbar_init_fence();
  __syncwarp();
  if (lane == 0) mbar_expect_tx(&bar, 16);
  __syncwarp();
  if (!mbar_wait(&bar, 0, limit) && lane == 0) atomicOr(err, ERR_TIMEOUT);
}

__global__ void e4m3_encode_kernel(const float* in, uint8_t* out, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    out[i] = (uint8_t)(e4m3x2(in[i], 0.f) & 0xFFu);
}

}  // namespace

cudaError_t launch_cache_write(int mode, int D, const WriteArgs& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  switch (mode) {
    case BF16: return launch_mode<BF16>(D, a, st);
    case FP8_PER_TENSOR: return launch_mode<FP8_PER_TENSOR>(D, a, st);
    case FP8_PER_HEAD: return launch_mode<FP8_PER_HEAD>(D, a, st);
    case FP8_PER_TOKEN_HEAD: return launch_mode<FP8_PER_TOKEN_HEAD>(D, a, st);
    case INT4_PER_TOKEN_HEAD: return launch_mode<INT4_PER_TOKEN_HEAD>(D, a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_calibrate(const uint16_t* x, long long T, int Hkv, int D, float qmax,
                             float* out, cudaStream_t st) {
  unsigned* bits = reinterpret_cast<unsigned*>(out);
  const int tb = 256;
  calib_zero<<<(Hkv + tb - 1) / tb, tb, 0, st>>>(bits, Hkv);
  const long long n = T * D;
  if (n > 0) {
    long long blocks = (n + tb - 1) / tb;
    if (blocks > 64) blocks = 64;
    calib_amax<<<dim3((unsigned)blocks, (unsigned)Hkv), tb, 0, st>>>(x, T, Hkv, D, bits);
  }
  calib_finish<<<(Hkv + tb - 1) / tb, tb, 0, st>>>(bits, Hkv, qmax);
  return cudaGetLastError();
}

cudaError_t launch_wait_check(long long limit_cycles, cudaStream_t st) {
  unsigned* err = error_word();
  if (!err) return cudaErrorInvalidValue;
  wait_check_kernel<<<1, 32, 0, st>>>(err, limit_cycles);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, long long n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int tb = 256;
  long long blocks = (n + tb - 1) / tb;
  const long long cap = (long long)sm_count() * 16;
  if (blocks > cap) blocks = cap;
  e4m3_encode_kernel<<<(unsigned)blocks, tb, 0, st>>>(in, out, n);
  return cudaGetLastError();
}

}  // namespace kvq
