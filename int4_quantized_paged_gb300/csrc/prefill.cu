// Prefill (chunked multi-query) attention over the quantized paged cache.
//
// What it computes: sequence b appends n_b tokens at positions
// [L_b - n_b, L_b) (their K/V already written by the cache write); each new
// token's query at position p attends causally to the retained positions
// [lo(p), p], lo(p) = max(0, p + 1 - W) for a window W, else 0, with the same
// scores, scales and softmax as decode.  This is the prefill stage whose
// time to first token the pages record ("FP8 KV cache layer skipping vs
// per-head scales", section "Run a four-way ablation"; "Per-tensor vs per-head
// FP8 KV cache scales", section "Use a three-stage decision").
//
// Work decomposition (one CTA per query tile, no split of the keys):
//  * A CTA owns ROWS = 128 query rows of one (sequence, KV head): QP = 128/G
//    consecutive new positions times the G query heads of that KV head, so a
//    key/value tile is fetched and dequantized once for all of them.  CTAs
//    with the latest (longest) query tiles start first.
//  * Keys stream in tiles of 64 positions (four 16-position page tiles, one
//    2-D TMA box each for K and V, plus 64-byte bulk copies of the dynamic
//    scales) through NSR raw stages.  After each tile lands, all threads
//    convert it once into f16 (bf16 for BF16 layers) shared-memory tiles K16
//    and V16 (exact: E4M3 and INT4 codes are f16 values); positions outside
//    the CTA's key range become zeros, so no stale byte reaches a product.
//  * Eight warps, each 16 rows, in FlashAttention-2 layout on mma.m16n8k16:
//    S = Q K^T with Q and K fragments from ldmatrix, the online softmax on
//    the accumulators (log2 units, causal and window masks per row), and
//    O += P' V with the S accumulators reused as the A fragments and V
//    fragments from ldmatrix.trans.  P' = p x v_scale x 2^k as in decode
//    (k a power-of-two range factor per warp), split into f16 hi + lo (three
//    bf16 terms for BF16 layers) so the weights keep fp32-class accuracy.
//  * q is prescaled per row by a power of two so its bf16 values are exact
//    in f16; the factor returns on the score.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "kvq_internal.h"
#include "tile_math.cuh"

namespace kvq {
namespace {

constexpr int PWARPS = 8;                  // warps per CTA
constexpr int ROWS = 16 * PWARPS;          // query rows per CTA
constexpr int KT = 64;                     // key positions per tile
constexpr int SUB = KT / 16;               // 16-position page tiles per key tile
constexpr int PKP = 13;                    // P' = p v_scale 2^(PKP - vexp) < 2^14

__device__ __forceinline__ void ldsm_x4(uint32_t r[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

template <int MODE, int D>
struct PCfg {
  static constexpr int RB = row_bytes<MODE>(D);
  static constexpr int TB = 16 * RB;                       // one page tile (16 positions)
  static constexpr int TBP = (TB + 1023) / 1024 * 1024;
  static constexpr bool DYN = (MODE == FP8_PER_TOKEN_HEAD || MODE == INT4_PER_TOKEN_HEAD);
  static constexpr bool BF = (MODE == BF16);
  static constexpr int RAW = 2 * SUB * TBP;                 // K and V page tiles of a key tile
  static constexpr int SCB = DYN ? 2 * SUB * 64 : 0;        // their K and V scales
  static constexpr int LD = D + 8;                          // f16 row pitch (elements)
  static constexpr int KV16 = KT * LD * 2;                  // bytes of K16 (and of V16)
  static constexpr int Q16 = ROWS * LD * 2;
  static constexpr int FIXED = 2 * KV16 + Q16 + 2 * KT * 4 + ROWS * 8 + 64;
  // raw stages: two where they fit beside the rest in 227 KB, else one
  static constexpr int NSR = (2 * (RAW + SCB) + FIXED + 2048 <= 232448) ? 2 : 1;
  static constexpr int RAWS = (RAW + SCB + 1023) / 1024 * 1024;   // stage pitch
  static constexpr int SMEM = NSR * RAWS + FIXED + 1024;           // + alignment slack
  static constexpr int NPART = BF ? 3 : 2;                  // terms of the P' split
};

struct PrefillArgs {
  DecodeArgs d;                  // caches, scales, block table, context_lens, q, out
  const int* query_start;        // [B + 1]
  int qtiles;                    // query tiles per (sequence, KV head) in the grid
};

template <int MODE, int D, int G>
__global__ void __launch_bounds__(PWARPS * 32, 1)
    prefill_kernel(const PrefillArgs pa, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap) {
  using C = PCfg<MODE, D>;
  using ET = uint16_t;
  const DecodeArgs& a = pa.d;
  constexpr int QP = ROWS / G;                 // positions per query tile
  constexpr int LD = C::LD;
  constexpr int NSR = C::NSR;
  constexpr int NT = D / 8;                    // O n-tiles (8 d values each)

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* raw = smem;                                       // NSR stages
  ET* k16 = reinterpret_cast<ET*>(smem + NSR * C::RAWS);
  ET* v16 = k16 + KT * LD;
  ET* q16 = v16 + KT * LD;
  float* ksm = reinterpret_cast<float*>(q16 + ROWS * LD);    // [KT] K scale (0: no key)
  float* vsm = ksm + KT;                                     // [KT] V scale
  float* rowf = vsm + KT;                                    // [ROWS] score factor per row
  int* rowp = reinterpret_cast<int*>(rowf + ROWS);           // [ROWS] position (-1: no row)
  uint64_t* bars = reinterpret_cast<uint64_t*>(rowp + ROWS); // [NSR]
  __shared__ int s_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lg = lane >> 2, lt = lane & 3;

  // ---- this CTA's (sequence, KV head, query tile); latest tiles first
  const int per_tile = a.B * a.Hkv;
  const int qt = pa.qtiles - 1 - (int)(blockIdx.x / per_tile);
  const int rem = (int)(blockIdx.x % per_tile);
  const int b = rem / a.Hkv, g = rem - b * a.Hkv;
  const int q0 = pa.query_start[b];
  const int n_b = pa.query_start[b + 1] - q0;
  int L = a.context_lens[b];
  if (qt * QP >= n_b || n_b <= 0) return;                   // whole CTA: before any barrier
  // the chunk cannot start before 0, and its last position must lie inside
  // the positions the sequence's block-table row covers
  if (L < n_b || (long long)L > ((long long)a.max_blocks << a.bs_shift)) {
    if (tid == 0) atomicOr(a.err, ERR_BAD_INDEX);
    return;
  }
  const int first = L - n_b + qt * QP;                      // position of query index 0
  const int nq = min(QP, n_b - qt * QP);                    // valid query positions here
  const int pmax = first + nq - 1;
  const int kmin = (a.window > 0) ? max(0, first + 1 - a.window) : 0;
  const int t0 = kmin / KT, t1 = pmax / KT;                 // key tiles, inclusive

  if (tid == 0) {
    for (int s = 0; s < NSR; ++s) mbar_init(&bars[s], 1);
    mbar_init_fence();
    s_flag = 0;
  }

  // ---- queries: row r = h * QP + i -> token q0 + qt*QP + i, head g*G + h.
  // Warp w stages rows w, w + 8, ...: one row per pass, D/32 elements a lane.
  float ks_static = 1.f;
  if constexpr (MODE == FP8_PER_TENSOR) ks_static = a.k_scale[0];
  if constexpr (MODE == FP8_PER_HEAD) ks_static = a.k_scale[g];
  for (int r = warp; r < ROWS; r += PWARPS) {
    const int h = r / QP, i = r - h * QP;
    const bool valid = i < nq;
    constexpr int EL = D / 32;
    float x[EL];
    float amax = 0.f;
    if (valid) {
      const uint16_t* src = a.q + ((long long)(q0 + qt * QP + i) * a.Hq + g * G + h) * D;
#pragma unroll
      for (int e = 0; e < EL; ++e) {
        x[e] = __uint_as_float((uint32_t)src[lane + 32 * e] << 16);
        amax = fmaxf(amax, fabsf(x[e]));
      }
    } else {
#pragma unroll
      for (int e = 0; e < EL; ++e) x[e] = 0.f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int qexp = 0;
    if (!C::BF && amax > 0.f) qexp = max(((int)(__float_as_uint(amax) >> 23) & 0xFF) - 127, -100);
    const float qmul = C::BF ? 1.f : pow2i(14 - qexp);
#pragma unroll
    for (int e = 0; e < EL; ++e) {
      const float v = x[e] * qmul;
      q16[r * LD + lane + 32 * e] =
          C::BF ? (uint16_t)(pack_bf16x2(v, 0.f) & 0xFFFFu) : (uint16_t)(pack_f16x2(v, 0.f) & 0xFFFFu);
    }
    if (lane == 0) {
      rowf[r] = a.qk_scale * ks_static * (C::BF ? 1.f : pow2i(qexp - 14));
      rowp[r] = valid ? first + i : -1;
    }
  }
  __syncthreads();

  // ---- copies of key tile t into raw stage st: warp 0, lane s < SUB takes
  // page tile s.  Page tiles wholly outside [kmin, pmax] are not fetched.
  auto issue = [&](int t, int st) {
    const int pos = t * KT + 16 * lane;
    int blk = -1;
    bool want = false;
    if (lane < SUB) {
      want = pos + 16 > kmin && pos <= pmax;
      if (want) {
        blk = __ldg(a.block_table + (long long)b * a.max_blocks + (pos >> a.bs_shift));
        if (blk < 0 || blk >= a.num_blocks) {
          atomicOr(a.err, ERR_BAD_INDEX);
          want = false;
        }
      }
    }
    const unsigned fetch = __ballot_sync(0xffffffffu, want);
    uint8_t* base = raw + st * C::RAWS;
    if (lane == 0)
      mbar_expect_tx(&bars[st], (uint32_t)__popc(fetch) * (2 * C::TB + (C::DYN ? 128 : 0)));
    __syncwarp();
    if (want) {
      const unsigned cell = ((unsigned)blk * (unsigned)a.Hkv + (unsigned)g) * (unsigned)a.bs +
                            (unsigned)(pos & (a.bs - 1));
      const int rowc = (int)(((unsigned long long)cell * C::RB) >> 7);
      tma_tile_2d(base + lane * C::TBP, &kmap, 0, rowc, &bars[st]);
      tma_tile_2d(base + (SUB + lane) * C::TBP, &vmap, 0, rowc, &bars[st]);
      if constexpr (C::DYN) {
        float* sc = reinterpret_cast<float*>(base + C::RAW);
        bulk_copy(sc + 16 * lane, a.k_cs + cell, 64, &bars[st]);
        bulk_copy(sc + 16 * (SUB + lane), a.v_cs + cell, 64, &bars[st]);
      }
    }
    return fetch;
  };
  unsigned fetched[2] = {0u, 0u};                  // page tiles fetched per stage (warp 0)
  if (warp == 0)
    for (int s = 0; s < NSR && t0 + s <= t1; ++s) fetched[s] = issue(t0 + s, s);

  // ---- per-warp state: rows rA = 16 warp + lg and rB = rA + 8
  const int rA = 16 * warp + lg, rB = rA + 8;
  const int pA = rowp[rA], pB = rowp[rB];
  const int loA = (a.window > 0) ? max(0, pA + 1 - a.window) : 0;
  const int loB = (a.window > 0) ? max(0, pB + 1 - a.window) : 0;
  const float fA = rowf[rA], fB = rowf[rB];
  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  int vexp = -1000;
  float fv = 0.f;                                  // 2^(PKP - vexp)
  float vs_static = 1.f;
  if constexpr (MODE == FP8_PER_TENSOR) vs_static = a.v_scale[0];
  if constexpr (MODE == FP8_PER_HEAD) vs_static = a.v_scale[g];

  for (int t = t0; t <= t1; ++t) {
    const int st = (t - t0) % NSR;
    const uint32_t par = (uint32_t)(((t - t0) / NSR) & 1);
    const bool ok = mbar_wait(&bars[st], par);
    if (__syncthreads_or(!ok)) {
      // a copy never completed: flag it, let the other stage's copies land
      // (bounded), and stop
      if (tid == 0) {
        atomicOr(a.err, ERR_TIMEOUT);
        if (NSR == 2 && t + 1 <= t1)
          (void)mbar_wait(&bars[st ^ 1], (uint32_t)(((t + 1 - t0) / NSR) & 1));
      }
      return;
    }
    // which page tiles of this key tile hold data (warp 0 knows; share it)
    if (tid == 0) s_flag = (int)fetched[st];
    __syncthreads();
    const unsigned have = (unsigned)s_flag;
    const uint8_t* base = raw + st * C::RAWS;
    // ---- convert the tile into K16 / V16 (zeros where nothing was fetched or
    // the position lies outside [kmin, pmax]); scales into ksm / vsm
    {
      constexpr int CH = C::RB / 16;               // 16-byte chunks per position row
      for (int c = tid; c < 2 * KT * CH; c += PWARPS * 32) {
        const int isv = c >= KT * CH;
        const int cc = isv ? c - KT * CH : c;
        const int key = cc / CH, ch = cc - key * CH;
        const int sub = key >> 4, kr = key & 15;
        const int pos = t * KT + key;
        const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (live)
          w = *reinterpret_cast<const uint4*>(base + (isv ? SUB + sub : sub) * C::TBP +
                                             swz((uint32_t)(kr * C::RB + ch * 16)));
        ET* dst = (isv ? v16 : k16) + key * LD;
        if constexpr (MODE == BF16) {
          *reinterpret_cast<uint4*>(dst + ch * 8) = w;
        } else if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
          // 32 nibbles -> 32 f16 (exact): low nibble of byte j = element 2j
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t x = ws[q];
            const uint32_t e0 = nib2_f16x2<0>(__byte_perm(x, 0u, 0x7170));   // bytes 0,1 low
            const uint32_t h0 = nib2_f16x2<1>(__byte_perm(x, 0u, 0x7170));   // bytes 0,1 high x16
            const uint32_t e1 = nib2_f16x2<0>(__byte_perm(x, 0u, 0x7372));
            const uint32_t h1 = nib2_f16x2<1>(__byte_perm(x, 0u, 0x7372));
            // e0 = {b0.lo, b1.lo}, h0 = 16 {b0.hi, b1.hi}: order b0.lo b0.hi b1.lo b1.hi
            uint32_t hs0, hs1;
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hs0) : "r"(h0), "r"(0x2C002C00u));   // x 1/16
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hs1) : "r"(h1), "r"(0x2C002C00u));
            uint4 o;
            o.x = __byte_perm(e0, hs0, 0x5410);
            o.y = __byte_perm(e0, hs0, 0x7632);
            o.z = __byte_perm(e1, hs1, 0x5410);
            o.w = __byte_perm(e1, hs1, 0x7632);
            *reinterpret_cast<uint4*>(dst + ch * 32 + 8 * q) = o;
          }
        } else {
          uint4 o0, o1;
          e4m3x4_f16(w.x, o0.x, o0.y);
          e4m3x4_f16(w.y, o0.z, o0.w);
          e4m3x4_f16(w.z, o1.x, o1.y);
          e4m3x4_f16(w.w, o1.z, o1.w);
          *reinterpret_cast<uint4*>(dst + ch * 16) = o0;
          *reinterpret_cast<uint4*>(dst + ch * 16 + 8) = o1;
        }
      }
      if (tid < 2 * KT) {
        const int isv = tid >= KT;
        const int key = isv ? tid - KT : tid;
        const int sub = key >> 4;
        const int pos = t * KT + key;
        const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
        float sc = live ? 1.f : 0.f;
        if constexpr (C::DYN)
          if (live) sc = reinterpret_cast<const float*>(base + C::RAW)[16 * (isv ? SUB + sub : sub) + (key & 15)];
        (isv ? vsm : ksm)[key] = sc;
      }
    }
    __syncthreads();
    // the raw stage is free: fetch key tile t + NSR into it
    if (warp == 0 && t + NSR <= t1) {
      fence_proxy_async();
      fetched[st] = issue(t + NSR, st);
    }

    // ---- S = Q K^T for this warp's 16 rows and the 64 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
    {
      const int m = lane >> 3;                     // ldmatrix: this lane's matrix
      const ET* qrow = q16 + (16 * warp + (m & 1) * 8 + (lane & 7)) * LD + (m >> 1) * 8;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t af[4];
        ldsm_x4(af, qrow + 16 * kk);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t bf[4];
          ldsm_x4(bf, k16 + (16 * np + (m >> 1) * 8 + (lane & 7)) * LD + 16 * kk + (m & 1) * 8);
          mma16816<C::BF>(s[2 * np], af, bf[0], bf[1]);
          mma16816<C::BF>(s[2 * np + 1], af, bf[2], bf[3]);
        }
      }
    }

    // ---- scores (log2 units) with the causal / window masks of each row
    float mtA = -INFINITY, mtB = -INFINITY;
    int et = -1000;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int key = 8 * j + 2 * lt + c;
        const int pos = t * KT + key;
        const float kscale = ksm[key];
        // a key whose page was not fetched (bad block id) has scale 0: masked
        const bool okA = pA >= 0 && pos >= loA && pos <= pA && kscale != 0.f;
        const bool okB = pB >= 0 && pos >= loB && pos <= pB && kscale != 0.f;
        s[j][c] = okA ? s[j][c] * kscale * fA : -INFINITY;
        s[j][2 + c] = okB ? s[j][2 + c] * kscale * fB : -INFINITY;
        mtA = fmaxf(mtA, s[j][c]);
        mtB = fmaxf(mtB, s[j][2 + c]);
        if constexpr (C::DYN)
          if (kscale != 0.f) et = max(et, f32_exp(vsm[key]));
      }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      mtA = fmaxf(mtA, __shfl_xor_sync(0xffffffffu, mtA, o));
      mtB = fmaxf(mtB, __shfl_xor_sync(0xffffffffu, mtB, o));
    }
    const float mnA = fmaxf(mA, mtA), mnB = fmaxf(mB, mtB);
    float alA = (mnA == -INFINITY) ? 1.f : ex2(mA - mnA);
    float alB = (mnB == -INFINITY) ? 1.f : ex2(mB - mnB);
    mA = mnA;
    mB = mnB;
    lA *= alA;
    lB *= alB;
    if constexpr (C::DYN) {
      // warp-uniform V-scale exponent: every key of the tile is in each quad
      et = __reduce_max_sync(0xffffffffu, et);
      const int vnew = max(vexp, max(et, -100));
      if (vnew != vexp) {
        const float vfix = pow2i(vexp - vnew);     // 0 on the first data (O is 0)
        alA *= vfix;
        alB *= vfix;
        vexp = vnew;
        fv = pow2i(PKP - vexp);
      }
    }
    if (__any_sync(0xffffffffu, alA != 1.f || alB != 1.f)) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        acc[n][0] *= alA;
        acc[n][1] *= alA;
        acc[n][2] *= alB;
        acc[n][3] *= alB;
      }
    }
    // weights p, row sums, and P' = p x (v_scale 2^(PKP - vexp) | 2^14 | 1)
    const float muA = (mA == -INFINITY) ? 0.f : mA, muB = (mB == -INFINITY) ? 0.f : mB;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int key = 8 * j + 2 * lt + c;
        const float pa_ = ex2(s[j][c] - muA), pb_ = ex2(s[j][2 + c] - muB);
        lA += pa_;
        lB += pb_;
        float vf;
        if constexpr (C::DYN) vf = vsm[key] * fv;
        else if constexpr (C::BF) vf = 1.f;
        else vf = 16384.f;
        s[j][c] = pa_ * vf;
        s[j][2 + c] = pb_ * vf;
      }

    // ---- O += P' V: the S accumulators of keys 16kk.. are the A fragments
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ap[C::NPART][4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int j = 2 * kk + (h >> 1);
        const int e = (h & 1) * 2;                 // h: 0 (row A, j0) 1 (row B, j0) 2 (A, j1) 3 (B, j1)
        const float x0 = s[j][e], x1 = s[j][e + 1];
        if constexpr (C::BF) {
          const uint32_t h0 = pack_bf16x2(x0, x1);
          const float r0 = x0 - bf16_lo(h0), r1 = x1 - bf16_lo(h0 >> 16);
          const uint32_t m0 = pack_bf16x2(r0, r1);
          ap[0][h] = h0;
          ap[1][h] = m0;
          ap[2][h] = pack_bf16x2(r0 - bf16_lo(m0), r1 - bf16_lo(m0 >> 16));
        } else {
          const uint32_t h0 = pack_f16x2(x0, x1);
          ap[0][h] = h0;
          ap[1][h] = pack_f16x2(x0 - f16_lo(h0), x1 - f16_lo(h0 >> 16));
        }
      }
      // fragment order: a0 (row g, keys 0-7), a1 (row g+8), a2 (row g, keys 8-15), a3
      const int m = lane >> 3;
      const ET* vrow = v16 + (16 * kk + (m & 1) * 8 + (lane & 7)) * LD + (m >> 1) * 8;
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        uint32_t bf[4];
        ldsm_x4_t(bf, vrow + 16 * dn);
#pragma unroll
        for (int k = 0; k < C::NPART; ++k) {
          mma16816<C::BF>(acc[2 * dn], ap[k], bf[0], bf[1]);
          mma16816<C::BF>(acc[2 * dn + 1], ap[k], bf[2], bf[3]);
        }
      }
    }
    __syncthreads();                               // K16 / V16 are rewritten next
  }

  // ---- epilogue: out = O x unscale / l per row
#pragma unroll
  for (int o = 1; o < 4; o <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, o);
    lB += __shfl_xor_sync(0xffffffffu, lB, o);
  }
  float unscale;
  if constexpr (C::BF) unscale = 1.f;
  else if constexpr (C::DYN) unscale = pow2i(vexp - PKP);
  else unscale = vs_static * (1.f / 16384.f);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int r = half ? rB : rA;
    const int p = half ? pB : pA;
    if (p < 0) continue;
    const float l = half ? lB : lA;
    const float f = l > 0.f ? unscale / l : 0.f;
    const int h = r / QP, i = r - h * QP;
    float* dst = a.out + ((long long)(q0 + qt * QP + i) * a.Hq + g * G + h) * D;
#pragma unroll
    for (int n = 0; n < NT; ++n)
      *reinterpret_cast<float2*>(dst + 8 * n + 2 * lt) =
          make_float2(acc[n][2 * half] * f, acc[n][2 * half + 1] * f);
  }
}

template <int MODE, int D, int G>
cudaError_t plaunch3(const PrefillArgs& pa, cudaStream_t st) {
  using C = PCfg<MODE, D>;
  const DecodeArgs& a = pa.d;
  const long long total = a.num_blocks * a.Hkv * a.bs * (long long)C::RB;
  CUtensorMap km, vm;
  if (total > 0) {
    if (!make_tile_map(&km, a.k_cache, total, C::TB) || !make_tile_map(&vm, a.v_cache, total, C::TB))
      return cudaErrorInvalidValue;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = prefill_kernel<MODE, D, G>;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long grid = (long long)pa.qtiles * a.B * a.Hkv;
  if (grid <= 0) return cudaSuccess;
  kern<<<(unsigned)grid, PWARPS * 32, C::SMEM, st>>>(pa, km, vm);
  return cudaGetLastError();
}

template <int MODE, int D>
cudaError_t plaunch2(int G, const PrefillArgs& pa, cudaStream_t st) {
  switch (G) {
    case 1: return plaunch3<MODE, D, 1>(pa, st);
    case 2: return plaunch3<MODE, D, 2>(pa, st);
    case 4: return plaunch3<MODE, D, 4>(pa, st);
    case 8: return plaunch3<MODE, D, 8>(pa, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int MODE>
cudaError_t plaunch1(int D, int G, const PrefillArgs& pa, cudaStream_t st) {
  switch (D) {
    case 64: return plaunch2<MODE, 64>(G, pa, st);
    case 128: return plaunch2<MODE, 128>(G, pa, st);
    case 256: return plaunch2<MODE, 256>(G, pa, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int prefill_rows_per_cta() { return ROWS; }

cudaError_t launch_prefill(int mode, int D, int G, const DecodeArgs& a, const int* query_start,
                           int max_query_len, cudaStream_t st) {
  if (a.B == 0 || max_query_len <= 0) return cudaSuccess;
  PrefillArgs pa;
  pa.d = a;
  pa.query_start = query_start;
  const int qp = ROWS / G;
  pa.qtiles = (max_query_len + qp - 1) / qp;
  switch (mode) {
    case BF16: return plaunch1<BF16>(D, G, pa, st);
    case FP8_PER_TENSOR: return plaunch1<FP8_PER_TENSOR>(D, G, pa, st);
    case FP8_PER_HEAD: return plaunch1<FP8_PER_HEAD>(D, G, pa, st);
    case FP8_PER_TOKEN_HEAD: return plaunch1<FP8_PER_TOKEN_HEAD>(D, G, pa, st);
    case INT4_PER_TOKEN_HEAD: return plaunch1<INT4_PER_TOKEN_HEAD>(D, G, pa, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
