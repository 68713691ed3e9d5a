// Prefill (chunked multi-query) attention over a quantized paged cache (FP8 or
// INT4 codes at head_dim 64, 128 or 256; BF16 layers at 64 and 128),
// warp-specialised on the fifth-generation tensor cores.  It computes what the single-role prefill kernel computes
// (causal attention of each new token's query over the retained positions,
// the scales folded into score and weight: "Per-tensor vs per-head FP8 KV
// cache scales", section "Use a three-stage decision"; "FP8 KV cache layer
// skipping vs per-head scales", section "Run a four-way ablation") with the
// work of one key tile spread over warps with their own roles, so that the
// tensor cores, the code conversion and the softmax run at the same time.
//
// A CTA owns two query tiles of M = 128 rows each (128/G consecutive new
// positions times the G query heads of one KV head; tile 1 follows tile 0),
// and streams the keys of both in tiles of 64 positions.  At head_dim 256 a
// CTA owns one query tile (its O takes 256 tensor-memory columns) and keeps
// Q in tensor memory, the A operand of S; the roles below then have one
// softmax warpgroup and the other warps move down by four.  Roles (14 warps):
//  * warp 12, producer: 2-D TMA copies of the key tile's K and V page tiles
//    (and 64-byte bulk copies of their dynamic scales) into a ring of raw
//    stages; lane s takes page tile s.
//  * warps 8-11, converters: raw codes -> f16 in the tensor cores' layout,
//    K as 64 rows of D (K-major, 128-byte swizzle) and V transposed (D rows
//    of 64 keys, by a byte transpose in registers); K and V scales (zero for a
//    key outside the CTA's range or on a page that was not fetched) and the
//    tile's largest V-scale exponent.  Three operand buffers.  BF16 layers:
//    K stays bf16 (S is a bf16 MMA; at head_dim 128 the producer copies it
//    straight into its operand buffer), and the converters give each V row
//    the power-of-two V scale that maps its largest exponent to 2^14,
//    converting it to f16 exactly; the rest then runs as for dynamic scales.
//  * warp 13, MMA issuer (one thread): S_j = Q_j K^T (M 128, N 64) into
//    tensor memory for each query tile j, and O_j += P'_j V with P'_j read
//    from tensor memory, every term of its f16 hi + lo split.  Each query
//    tile has two S/P' buffers (key tile t uses buffer t & 1; P' replaces S
//    there).  Order per key tile t: PV_0(t), PV_1(t), then S_0(t+2) and
//    S_1(t+2) once the PV that last read each buffer has completed, so a
//    softmax warpgroup finds the scores of its next tile ready and the
//    tensor cores work on one query tile while the other's softmax runs.
//  * warps 0-3 and 4-7, softmax of query tile 0 and 1: one thread per row
//    (its tensor-memory lane) loads the row's 64 scores, applies the K scale
//    and masks, keeps a lazily moved reference max (moved only when a tile's
//    max exceeds it by more than 8 in log2 units), rescales the row of O in tensor memory
//    when it moves, and stores P' = p x v_scale x 2^k (f16 hi + lo) over the
//    scores it has read.
// Tensor memory: two S/P' buffers per query tile (64 columns each), O_0, O_1
// (D each).
// Every wait is bounded; a wait that runs out flags TIMEOUT and sets a
// shared abort flag that ends every role's loop, the work already issued is
// waited for (bounded again), and tensor memory is freed before the CTA exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "kvq_internal.h"
#include "prefill_common.cuh"
#include "tcgen05.cuh"
#include "tile_math.cuh"

namespace kvq {
namespace {

constexpr int WS_CONV = 4;                          // converter warps
constexpr int WROWS = 128;                          // rows per query tile (the MMA's M)

// A 16-byte shared-memory load that stays after the tensor-memory stores
// issued before it (both are volatile asm): the softmax reads a chunk's V
// scales just before it uses them, instead of the compiler hoisting all
// sixteen loads of a tile to its start, where their 64 registers pushed the
// thread past its 128-register share and spilled.
__device__ __forceinline__ float4 lds_v4_ordered(const float4* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"((uint32_t)__cvta_generic_to_shared(p)));
  return v;
}

// Warp roles: NQ query tiles per CTA (two at head_dim 64 and 128; one at 256,
// whose O needs 256 tensor-memory columns), a softmax warpgroup per query
// tile, then the converters, the producer and the MMA issuer.
template <int D>
struct WRoles {
  static constexpr int NQ = (D == 256) ? 1 : 2;
  static constexpr int SOFT = 4 * NQ;                // softmax warps
  static constexpr int PROD = SOFT + WS_CONV;        // producer warp
  static constexpr int MMA = PROD + 1;               // MMA-issuing warp
  static constexpr int THREADS = (MMA + 1) * 32;     // 448 or 320
};
constexpr int WKT = 64;                             // keys per tile
constexpr int WKP = 6;                              // P' = p v_scale 2^(WKP - vexp) < 2^15 (p <= 2^8)
constexpr float WLAZY = 8.f;                        // the reference max moves when exceeded by this
// static FP8 scales: P' = p x 2^6 (< 2^14)
constexpr int CONV_BAR = 1;                         // named barrier of the converter warps

template <int MODE, int D>
struct WCfg {
  static constexpr int RB = row_bytes<MODE>(D);
  static constexpr int TB = 16 * RB;                       // one page tile (16 positions)
  static constexpr int TBP = (TB + 1023) / 1024 * 1024;
  // scales copied from the cache with the codes (dynamic FP8, INT4)
  static constexpr bool FETCH = (MODE == FP8_PER_TOKEN_HEAD || MODE == INT4_PER_TOKEN_HEAD);
  // BF16 layers: K stays bf16 (S is a bf16 MMA against bf16 queries); each V
  // row is scaled by the power of two that maps its largest exponent to 2^14
  // and converted to f16 exactly, and its V scale is that power's inverse
  static constexpr bool BFK = (MODE == BF16);
  // per-key V scales in the scale buffer, followed by the softmax's range factor
  static constexpr bool DYN = FETCH || BFK;
  static constexpr int SUB = WKT / 16;                      // page tiles per key tile
  // BF16 at head_dim 128: K is copied straight into its operand buffer, which
  // halves the raw stage so that three raw stages and three operand buffers
  // fit (two and two otherwise).  At 64 both already fit three and four, and
  // the producer keeps its four-stage lookahead by staging K like V.
  static constexpr bool KDIRECT = BFK && D == 128;
  // a raw stage: the K and V page tiles of a key tile (V only with KDIRECT),
  // then their scales
  static constexpr int RAW = (KDIRECT ? 1 : 2) * SUB * TBP;
  static constexpr int VOFF = KDIRECT ? 0 : SUB * TBP;      // V page tiles in a raw stage
  static constexpr int SCB = FETCH ? 2 * SUB * 64 : 0;
  static constexpr int RAWS = (RAW + SCB + 1023) / 1024 * 1024;
  static constexpr int NQ = WRoles<D>::NQ;
  static constexpr int QB = WROWS * D * 2;                  // one query tile: D/64 blocks of 128 x 128 B
  // queries in shared memory (two query tiles); with one query tile (D 256)
  // they live in tensor memory instead, the A operand of S
  static constexpr int QSM = (NQ == 2) ? 2 * QB : 0;
  static constexpr int KB = WKT * D * 2;                    // one K buffer: D/64 blocks of 64 x 128 B
  static constexpr int VTB = D * WKT * 2;                   // one V^T buffer: D rows of 128 B
  // one scale buffer: K scales, V scales, then ints: V-scale exponent of
  // each 32-key half, whether every page tile was fetched
  static constexpr int SCS = 2 * WKT * 4 + 16;
  static constexpr int ROWB = 2 * 2 * WROWS * 4;            // row factor and position per row
  static constexpr int BARB = 32 * 8;                       // barriers
  static constexpr int LIMIT = 232448 - 1024;               // per-CTA shared memory, minus slack
  // operand buffers (K, V^T, scales): three when they fit beside two raw stages
  static constexpr int fixed_of(int nb) { return QSM + nb * (KB + VTB + SCS) + ROWB + BARB + 64; }
  static constexpr int NB = (fixed_of(3) + 2 * RAWS <= LIMIT) ? 3 : 2;
  static constexpr int FIXED = fixed_of(NB);
  static constexpr int NR = (FIXED + 4 * RAWS <= LIMIT) ? 4 : ((FIXED + 3 * RAWS <= LIMIT) ? 3 : 2);
  static constexpr int SMEM = NR * RAWS + FIXED + 1024;
  // Tensor-memory columns.  S/P' buffer b of query tile j: S (fp32, 64
  // columns), then P' (f16 hi in the first 32 columns, lo in the next 32) in
  // its place.  Two query tiles: S/P' at 64 (2 j + b), O_j at 256 + D j.  One
  // query tile (D 256): O at 0, S/P' at 256 + 64 b, Q (f16, D / 2 columns) at
  // 384.
  __host__ __device__ static constexpr int scol(int j, int b) { return NQ == 2 ? 64 * (2 * j + b) : 256 + 64 * b; }
  __host__ __device__ static constexpr int ocol(int j) { return NQ == 2 ? 256 + D * j : 0; }
  static constexpr int QCOL = 384;
  static constexpr int TCOLS = 512;
  static_assert(NQ == 2 ? 256 + 2 * D <= TCOLS : QCOL + D / 2 <= TCOLS, "tensor memory");
  static_assert(SMEM <= 232448, "shared memory");
};

template <int MODE, int D, int G>
__global__ void __launch_bounds__(WRoles<D>::THREADS, 1)
    prefill_ws_kernel(const PrefillArgs pa, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  using C = WCfg<MODE, D>;
  using RL = WRoles<D>;
  constexpr int NQ = RL::NQ;
  const DecodeArgs& a = pa.d;
  constexpr int SUB = C::SUB;
  constexpr int NR = C::NR;
  constexpr int NB = C::NB;
  constexpr int QP = WROWS / G;                // positions per query tile
  constexpr int CPR = C::RB / 16;              // 16-byte raw chunks per position row
  constexpr int EPC = (MODE == INT4_PER_TOKEN_HEAD) ? 32 : (MODE == BF16 ? 8 : 16);   // elements per raw chunk

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* raw = smem;                                       // NR stages
  uint8_t* q16 = raw + NR * C::RAWS;                         // 2 query tiles (none for NQ 1)
  uint8_t* k16 = q16 + C::QSM;                               // NB K buffers
  uint8_t* vt16 = k16 + NB * C::KB;                          // NB V^T buffers
  uint8_t* scb = vt16 + NB * C::VTB;                         // NB scale buffers
  float* rowf = reinterpret_cast<float*>(scb + NB * C::SCS); // [2][128] score factor per row
  int* rowp = reinterpret_cast<int*>(rowf + 2 * WROWS);      // [2][128] position (-1: no row)
  uint64_t* bars = reinterpret_cast<uint64_t*>(rowp + 2 * WROWS);
  uint64_t* raw_full = bars;                                 // [NR] producer -> converters
  uint64_t* raw_empty = raw_full + NR;                       // [NR] converters -> producer
  uint64_t* kv_full = raw_empty + NR;                        // [NB] converters -> MMA
  uint64_t* kv_empty = kv_full + NB;                         // [NB] MMA (commit) -> converters
  uint64_t* s_full = kv_empty + NB;                          // [2][2] MMA (commit) -> softmax j, per S buffer
  // P' of query tile j in S/P' buffer b: [2][2], 128 arrivals each.  One
  // barrier per buffer: a softmax warpgroup may finish key tile t + 1 before
  // the MMA issuer waits for its tile t, and a barrier per query tile would
  // then complete two phases ahead of its waiter.
  uint64_t* p_full = s_full + 4;
  uint64_t* pv_done = p_full + 4;                            // [2] MMA (commit) -> softmax j
  uint64_t* o_fin = pv_done + 2;                             // MMA (commit) -> softmax, at the end
  int* s_have = reinterpret_cast<int*>(bars + 32);           // [NR] fetched page tiles per stage
  volatile int* s_abort = s_have + 4;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_have + 5);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- this CTA's (sequence, KV head, pair of query tiles); latest first
  const int per_tile = a.B * a.Hkv;
  const int ct = pa.qtiles - 1 - (int)(blockIdx.x / per_tile);
  const int rem = (int)(blockIdx.x % per_tile);
  const int b = rem / a.Hkv, g = rem - b * a.Hkv;
  const int q0 = pa.query_start[b];
  const int n_b = pa.query_start[b + 1] - q0;
  const int L = a.context_lens[b];
  if (ct * NQ * QP >= n_b || n_b <= 0) return;              // whole CTA: before any barrier
  if (L < n_b || (long long)L > ((long long)a.max_blocks << a.bs_shift)) {
    if (tid == 0) atomicOr(a.err, ERR_BAD_INDEX);
    return;
  }
  const int qbase = ct * NQ * QP;                           // query index of tile 0, row 0
  const int first = L - n_b + qbase;                        // its position
  const int nq = min(NQ * QP, n_b - qbase);                 // valid query positions here
  const int pmax = first + nq - 1;
  const int kmin = (a.window > 0) ? max(0, first + 1 - a.window) : 0;
  const int t0 = kmin / WKT, t1 = pmax / WKT;               // key tiles, inclusive
  const int ntl = t1 - t0 + 1;

  if (tid == 0) {
    for (int s = 0; s < NR; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 1);
    }
    for (int s = 0; s < NB; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4 * 32);
    }
    for (int s = 0; s < 2; ++s) mbar_init(&pv_done[s], 1);
    mbar_init(o_fin, 1);
    mbar_init_fence();
    *s_abort = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_tmem)),
                 "r"(C::TCOLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // ---- queries: row R = 128 j + h * QP + i of query tile j -> query index
  // qbase + j * QP + i, head g*G + h, prescaled by a power of two so the bf16
  // values are exact in f16 (BF16 layers: the bf16 values as they are).
  float ks_static = 1.f;
  if constexpr (MODE == FP8_PER_TENSOR) ks_static = a.k_scale[0];
  if constexpr (MODE == FP8_PER_HEAD) ks_static = a.k_scale[g];
  if constexpr (NQ == 2) {
    // into shared memory (K-major, 128-byte swizzle); lane l holds elements
    // l + 32e of the row
    for (int R = warp; R < NQ * WROWS; R += RL::THREADS / 32) {
      const int j = R / WROWS, r = R - j * WROWS;
      const int h = r / QP, i = r - h * QP;
      const int qi = j * QP + i;                             // query index within the CTA
      const bool valid = qi < nq;
      constexpr int EL = D / 32;
      float x[EL];
      float amax = 0.f;
      if (valid) {
        const uint16_t* src = a.q + ((long long)(q0 + qbase + qi) * a.Hq + g * G + h) * D;
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
      if (amax > 0.f) qexp = max(((int)(__float_as_uint(amax) >> 23) & 0xFF) - 127, -100);
      if constexpr (C::BFK) qexp = 14;
      const float qmul = pow2i(14 - qexp);
      uint8_t* qt = q16 + j * C::QB;
#pragma unroll
      for (int e = 0; e < EL; ++e) {
        const int d = lane + 32 * e;
        const uint16_t h16 = C::BFK ? (uint16_t)(__float_as_uint(x[e]) >> 16)
                                    : (uint16_t)(pack_f16x2(x[e] * qmul, 0.f) & 0xFFFFu);
        *reinterpret_cast<uint16_t*>(qt + (d >> 6) * (WROWS * 128) + swc(r, (d & 63) >> 3) + (d & 7) * 2) = h16;
      }
      if (lane == 0) {
        rowf[R] = a.qk_scale * ks_static * pow2i(qexp - 14);
        rowp[R] = valid ? first + qi : -1;
      }
    }
  } else {
    // into tensor memory, the A operand of S: the softmax warps' thread r
    // owns row r (its lane) and stores its D / 2 f16 pairs as columns
    if (warp < RL::SOFT) {
      const int r = warp * 32 + lane;
      const int h = r / QP, i = r - h * QP;
      const bool valid = i < nq;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + ((long long)(q0 + qbase + (valid ? i : 0)) * a.Hq + g * G + h) * D);
      float amax = 0.f;
      if (valid) {
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = src[c];
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w4[e] << 16)),
                                     fabsf(__uint_as_float(w4[e] & 0xFFFF0000u))));
        }
      }
      int qexp = 0;
      if (amax > 0.f) qexp = max(((int)(__float_as_uint(amax) >> 23) & 0xFF) - 127, -100);
      const float qmul = pow2i(14 - qexp);
      const uint32_t trq = tmem + ((uint32_t)(warp * 32) << 16) + C::QCOL;
#pragma unroll 1
      for (int c0 = 0; c0 < D / 2; c0 += 32) {     // 32 columns = 64 elements at a time
        uint32_t wq[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = valid ? src[(c0 * 2) / 8 + c] : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            wq[4 * c + e] = pack_f16x2(__uint_as_float(w4[e] << 16) * qmul,
                                       __uint_as_float(w4[e] & 0xFFFF0000u) * qmul);
        }
        uint32_t lo16[16], hi16[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) { lo16[e] = wq[e]; hi16[e] = wq[16 + e]; }
        tmem_st16_nowait(trq + c0, lo16);
        tmem_st16_nowait(trq + c0 + 16, hi16);
      }
      tmem_wait_st();
      rowf[r] = a.qk_scale * ks_static * pow2i(qexp - 14);
      rowp[r] = valid ? first + i : -1;
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ================================================================ roles
  if (warp == RL::PROD) {
    // ---- producer: key tile t into raw stage (t - t0) % NR; lane s < SUB
    // copies page tile s.  Page tiles wholly outside [kmin, pmax] are not
    // fetched.
    int last[NR];                                  // tile index last issued into each stage
#pragma unroll
    for (int s = 0; s < NR; ++s) last[s] = -1;
    for (int i = 0; i < ntl; ++i) {
      const int st = i % NR;
      if (i >= NR) {
        const bool ok = mbar_wait(&raw_empty[st], (uint32_t)((i / NR - 1) & 1));
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) { *s_abort = 1; atomicOr(a.err, ERR_TIMEOUT); }
          break;
        }
      }
      if constexpr (C::KDIRECT) {
        // K lands in operand buffer i % NB: wait until the MMAs of its last
        // tile are done with it
        if (i >= NB) {
          const bool ok = mbar_wait(&kv_empty[i % NB], (uint32_t)((i / NB - 1) & 1));
          if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) { *s_abort = 1; atomicOr(a.err, ERR_TIMEOUT); }
            break;
          }
        }
      }
      if (__any_sync(0xffffffffu, *s_abort)) break;
      const int t = t0 + i;
      const int pos = t * WKT + 16 * lane;
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
      fence_proxy_async();
      if (lane == 0) {
        s_have[st] = (int)fetch;
        mbar_expect_tx(&raw_full[st], (uint32_t)__popc(fetch) * (2 * C::TB + (C::FETCH ? 128 : 0)));
      }
      __syncwarp();
      if (want) {
        const unsigned cell = ((unsigned)blk * (unsigned)a.Hkv + (unsigned)g) * (unsigned)a.bs +
                              (unsigned)(pos & (a.bs - 1));
        const int rowc = (int)(((unsigned long long)cell * C::RB) >> 7);
        if constexpr (C::KDIRECT) {
          // bf16 K needs no conversion: each 64-d block of the page tile's 16
          // rows goes to its rows of the K operand (K-major, 128-byte swizzle)
#pragma unroll
          for (int h = 0; h < D / 64; ++h)
            tma_tile_3d(k16 + (i % NB) * C::KB + h * (WKT * 128) + lane * (16 * 128), &kmap, 0, h,
                        (int)cell, &raw_full[st]);
        } else {
          tma_tile_2d(base + lane * C::TBP, &kmap, 0, rowc, &raw_full[st]);
        }
        tma_tile_2d(base + C::VOFF + lane * C::TBP, &vmap, 0, rowc, &raw_full[st]);
        if constexpr (C::FETCH) {
          float* sc = reinterpret_cast<float*>(base + C::RAW);
          bulk_copy(sc + 16 * lane, a.k_cs + cell, 64, &raw_full[st]);
          bulk_copy(sc + 16 * (SUB + lane), a.v_cs + cell, 64, &raw_full[st]);
        }
      }
      last[st] = i;
    }
    // every copy issued has landed before the CTA exits (bounded waits)
    if (lane == 0)
#pragma unroll
      for (int s = 0; s < NR; ++s)
        if (last[s] >= 0) (void)mbar_wait(&raw_full[s], (uint32_t)((last[s] / NR) & 1));
  } else if (warp >= RL::SOFT && warp < RL::PROD) {
    // ---- converters (128 threads)
    const int ct_ = tid - RL::SOFT * 32;
    for (int i = 0; i < ntl; ++i) {
      const int st = i % NR, buf = i % NB;
      const int t = t0 + i;
      bool ok = mbar_wait(&raw_full[st], (uint32_t)((i / NR) & 1));
      if (i >= NB) ok = mbar_wait(&kv_empty[buf], (uint32_t)((i / NB - 1) & 1)) && ok;
      if (!ok) { *s_abort = 1; atomicOr(a.err, ERR_TIMEOUT); }
      // every converter thread takes the same decision (a barrier reduction)
      if (named_sync_or(CONV_BAR, WS_CONV * 32, !ok || *s_abort)) break;
      const unsigned have = (unsigned)s_have[st];
      const uint8_t* base = raw + st * C::RAWS;
      uint8_t* kb = k16 + buf * C::KB;
      // K into kb; zeros where nothing was fetched or the position lies
      // outside [kmin, pmax].  Each thread takes NIT chunks; all loads first,
      // then conversions.  (KDIRECT: the producer copied K there; rows of
      // keys not fetched or outside [kmin, pmax] hold whatever was there, and
      // the softmax masks their scores by their K scale 0.)
      constexpr int NIT = WKT * CPR / (WS_CONV * 32);
      static_assert(NIT * WS_CONV * 32 == WKT * CPR, "chunks per converter thread");
      if constexpr (!C::KDIRECT) {
        uint4 wk[NIT];
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
          const int cc = ct_ + it * WS_CONV * 32;
          const int key = cc / CPR, ch = cc % CPR;
          const int sub = key >> 4, kr = key & 15;
          const int pos = t * WKT + key;
          const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
          const uint32_t off = swz((uint32_t)(kr * C::RB + ch * 16));
          wk[it] = live ? *reinterpret_cast<const uint4*>(base + sub * C::TBP + off)
                        : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
          const int cc = ct_ + it * WS_CONV * 32;
          const int key = cc / CPR, ch = cc % CPR;
          const int d0 = ch * EPC;
          uint4 ok_[4];
          convert16<MODE>(wk[it], ok_);
#pragma unroll
          for (int qq = 0; qq < EPC / 8; ++qq) {
            const int d = d0 + 8 * qq;
            *reinterpret_cast<uint4*>(kb + (d >> 6) * (WKT * 128) + swc(key, (d & 63) >> 3)) = ok_[qq];
          }
        }
      }
      uint8_t* vb = vt16 + buf * C::VTB;
      if constexpr (MODE == BF16) {
        // V of a BF16 layer.  First the largest exponent e of each key row
        // (two threads per key, half a row each): the key's V scale is
        // 2^(e - 14), and the row times 2^(14 - e) has its largest value in
        // [2^14, 2^15), so every bf16 value down to 2^-28 of it converts to
        // f16 exactly.
        float* vsm = reinterpret_cast<float*>(scb + buf * C::SCS) + WKT;
        {
          const int key = ct_ >> 1, hh = ct_ & 1;
          const int sub = key >> 4, kr = key & 15;
          const int pos = t * WKT + key;
          const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
          uint32_t em = 0;                          // exponent fields (<< 7) of both halves of a word
          if (live) {
#pragma unroll
            for (int c = 0; c < CPR / 2; ++c) {
              const uint4 w = *reinterpret_cast<const uint4*>(
                  base + C::VOFF + sub * C::TBP + swz((uint32_t)(kr * C::RB + (hh * (CPR / 2) + c) * 16)));
              em = __vmaxu2(em, w.x & 0x7F807F80u);
              em = __vmaxu2(em, w.y & 0x7F807F80u);
              em = __vmaxu2(em, w.z & 0x7F807F80u);
              em = __vmaxu2(em, w.w & 0x7F807F80u);
            }
          }
          em = max(em & 0xFFFFu, em >> 16) >> 7;    // biased exponent, 0 for zeros
          em = max(em, __shfl_xor_sync(0xffffffffu, em, 1));
          const int e = em ? max((int)em - 127, -100) : 0;
          if (hh == 0) vsm[key] = live ? pow2i(e - 14) : 0.f;
        }
        named_sync(CONV_BAR, WS_CONV * 32);         // every key's V scale is in place
        // V^T: a task is 8 keys x one d pair (one word per key).  Each key's
        // two values are scaled by the inverse of its V scale (a power of two:
        // exact) and packed, keys 2q and 2q + 1 per word, into the rows of
        // d = 2 dp (low halves) and 2 dp + 1 (high halves).  Consecutive
        // lanes take consecutive d pairs of the same keys (one 128-byte row
        // per load), and lanes with bit 2 set store their odd row first, so
        // that each 8-lane phase of a store meets every bank once.
        constexpr int DP = D / 2;
        constexpr int NTB = 8 * DP / (WS_CONV * 32);
        static_assert(NTB * WS_CONV * 32 == 8 * DP, "V^T tasks per converter thread");
#pragma unroll
        for (int it = 0; it < NTB; ++it) {
          const int task = ct_ + it * WS_CONV * 32;
          const int dp = task % DP, kg = task / DP;
          const float4 s0 = *reinterpret_cast<const float4*>(vsm + 8 * kg);
          const float4 s1 = *reinterpret_cast<const float4*>(vsm + 8 * kg + 4);
          const float sk[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
          uint32_t x[8];
          float inv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int key = 8 * kg + k;
            const int sub = key >> 4, kr = key & 15;
            const int pos = t * WKT + key;
            const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
            x[k] = live ? *reinterpret_cast<const uint32_t*>(base + C::VOFF + sub * C::TBP +
                                                            swz((uint32_t)(kr * C::RB + 4 * dp)))
                        : 0u;
            // 2^(14 - e) from 2^(e - 14); 2^127 for a key with no data (its values are 0)
            inv[k] = __uint_as_float((254u - (__float_as_uint(sk[k]) >> 23)) << 23);
          }
          uint32_t ev[4], od[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            ev[q] = pack_f16x2(__uint_as_float(x[2 * q] << 16) * inv[2 * q],
                               __uint_as_float(x[2 * q + 1] << 16) * inv[2 * q + 1]);
            od[q] = pack_f16x2(__uint_as_float(x[2 * q] & 0xFFFF0000u) * inv[2 * q],
                               __uint_as_float(x[2 * q + 1] & 0xFFFF0000u) * inv[2 * q + 1]);
          }
          const uint4 E = make_uint4(ev[0], ev[1], ev[2], ev[3]);
          const uint4 O = make_uint4(od[0], od[1], od[2], od[3]);
          const bool swp = (lane >> 2) & 1;
          *reinterpret_cast<uint4*>(vb + swc(2 * dp + (swp ? 1 : 0), kg)) = swp ? O : E;
          *reinterpret_cast<uint4*>(vb + swc(2 * dp + (swp ? 0 : 1), kg)) = swp ? E : O;
        }
      }
      if constexpr (MODE != INT4_PER_TOKEN_HEAD && MODE != BF16) {
        // V^T straight from the raw FP8 codes: a task is 8 keys x 4 d.  Its
        // 8 words (one per key: codes of d..d+3) are transposed in registers
        // into 4 rows of 8 codes each, converted, and stored as one 16-byte
        // chunk per d row.  Lane-to-task map: consecutive lanes take
        // consecutive d groups, and the key group turns with the lane pair and
        // the warp, so the 4-byte loads and the 16-byte stores of a warp meet
        // no bank twice.
        constexpr int DG = D / 4;                   // d groups of 4
        constexpr int NT = 8 * DG / (WS_CONV * 32); // tasks per thread (4 at D 256, 2 at 128, 1 at 64)
        static_assert(NT * WS_CONV * 32 == 8 * DG, "V^T tasks per converter thread");
        const int cw = warp - RL::SOFT;              // converter warp 0..3
#pragma unroll
        for (int it = 0; it < NT; ++it) {
          int dg, kg;
          if constexpr (DG > 32) {                  // D 256: two sweeps of 32 d groups
            dg = lane + 32 * (it & 1);
            kg = (((lane >> 1) + cw) & 3) + 4 * (it >> 1);
          } else {
            dg = lane % DG;
            kg = (((dg >> 1) + cw) & 3) + 4 * (it + lane / DG);
          }
          uint32_t x[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int key = 8 * kg + k;
            const int sub = key >> 4, kr = key & 15;
            const int pos = t * WKT + key;
            const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
            x[k] = live ? *reinterpret_cast<const uint32_t*>(base + (SUB + sub) * C::TBP +
                                                            swz((uint32_t)(kr * C::RB + 4 * dg)))
                        : 0u;
          }
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t* y = x + 4 * half;
            const uint32_t t0 = __byte_perm(y[0], y[1], 0x5140), t1 = __byte_perm(y[0], y[1], 0x7362);
            const uint32_t t2 = __byte_perm(y[2], y[3], 0x5140), t3 = __byte_perm(y[2], y[3], 0x7362);
            uint32_t* o = half ? hi : lo;
            o[0] = __byte_perm(t0, t2, 0x5410);     // byte dd of keys 0..3 (or 4..7)
            o[1] = __byte_perm(t0, t2, 0x7632);
            o[2] = __byte_perm(t1, t3, 0x5410);
            o[3] = __byte_perm(t1, t3, 0x7632);
          }
#pragma unroll
          for (int dd = 0; dd < 4; ++dd) {
            uint4 v;
            e4m3x4_f16(lo[dd], v.x, v.y);
            e4m3x4_f16(hi[dd], v.z, v.w);
            *reinterpret_cast<uint4*>(vb + swc(4 * dg + dd, kg)) = v;
          }
        }
      }
      if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
        // V^T straight from the raw INT4 codes: a task is 8 keys x 4 bytes
        // (8 d).  The 8 words are transposed as for FP8; byte bb of 4 keys
        // then gives the f16 values of d = 2bb (low nibbles) and 2bb + 1 (high
        // nibbles, read 16x and scaled back exactly).
        constexpr int BG = D / 8;                   // 4-byte groups of a key row
        constexpr int NTI = (8 * BG > WS_CONV * 32) ? 8 * BG / (WS_CONV * 32) : 1;
        const int cw = warp - RL::SOFT;
#pragma unroll
        for (int it = 0; it < NTI; ++it) {
        int bg, kg;
        if constexpr (BG >= 32) {                   // D 256: 256 tasks, two per thread
          bg = lane;
          kg = (((lane >> 1) + cw) & 3) + 4 * it;
        } else if constexpr (BG >= 16) {            // 128 tasks, one per thread
          bg = lane % BG;
          kg = (((bg >> 1) + cw) & 3) + 4 * (lane / BG);
        } else {                                    // 64 tasks: the first 64 threads
          bg = ct_ % BG;
          kg = ct_ / BG;
        }
        if (kg < 8) {
          uint32_t x[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int key = 8 * kg + k;
            const int sub = key >> 4, kr = key & 15;
            const int pos = t * WKT + key;
            const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
            x[k] = live ? *reinterpret_cast<const uint32_t*>(base + (SUB + sub) * C::TBP +
                                                            swz((uint32_t)(kr * C::RB + 4 * bg)))
                        : 0u;
          }
          uint32_t lo[4], hi[4];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t* y = x + 4 * half;
            const uint32_t t0 = __byte_perm(y[0], y[1], 0x5140), t1 = __byte_perm(y[0], y[1], 0x7362);
            const uint32_t t2 = __byte_perm(y[2], y[3], 0x5140), t3 = __byte_perm(y[2], y[3], 0x7362);
            uint32_t* o = half ? hi : lo;
            o[0] = __byte_perm(t0, t2, 0x5410);
            o[1] = __byte_perm(t0, t2, 0x7632);
            o[2] = __byte_perm(t1, t3, 0x5410);
            o[3] = __byte_perm(t1, t3, 0x7632);
          }
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            uint32_t ev[4], od[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              // keys 2q, 2q + 1: bytes (q & 1) * 2 and +1 of lo or hi
              const uint32_t wq = (q < 2) ? lo[bb] : hi[bb];
              const uint32_t pr = __byte_perm(wq, 0u, (q & 1) ? 0x7372 : 0x7170);
              ev[q] = nib2_f16x2<0>(pr);
              const uint32_t h16 = nib2_f16x2<1>(pr);
              asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(od[q]) : "r"(h16), "r"(0x2C002C00u));   // x 1/16
            }
            const int d = 8 * bg + 2 * bb;
            *reinterpret_cast<uint4*>(vb + swc(d, kg)) = make_uint4(ev[0], ev[1], ev[2], ev[3]);
            *reinterpret_cast<uint4*>(vb + swc(d + 1, kg)) = make_uint4(od[0], od[1], od[2], od[3]);
          }
        }
        }
      }
      {
        // scales: threads 0..63 K, 64..127 V (scale 0: no key)
        float* ksm = reinterpret_cast<float*>(scb + buf * C::SCS);
        float* vsm = ksm + WKT;
        int* tinfo = reinterpret_cast<int*>(vsm + WKT);
        const int isv = ct_ >= WKT;
        const int key = isv ? ct_ - WKT : ct_;
        const int sub = key >> 4;
        const int pos = t * WKT + key;
        const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
        float sc = live ? 1.f : 0.f;
        if constexpr (C::FETCH)
          if (live) sc = reinterpret_cast<const float*>(base + C::RAW)[16 * (isv ? SUB + sub : sub) + (key & 15)];
        if constexpr (C::BFK) {
          if (isv) sc = vsm[key];                   // the BF16 V scale found above
          else ksm[key] = sc;
        } else {
          (isv ? vsm : ksm)[key] = sc;
        }
        if constexpr (C::DYN) {
          if (isv) {
            const int e = __reduce_max_sync(0xffffffffu, live ? f32_exp(sc) : -1000);
            if (lane == 0) tinfo[(ct_ - WKT) >> 5] = e;
          }
        }
        if (ct_ == 0) tinfo[2] = (have == (1u << SUB) - 1u) ? 1 : 0;
      }
      fence_proxy_async();
      named_sync(CONV_BAR, WS_CONV * 32);
      if (ct_ == 0) {
        mbar_arrive(&raw_empty[st]);                // the raw stage has been read
        mbar_arrive(&kv_full[buf]);
      }
    }
  } else if (warp == RL::MMA) {
    // ---- MMA issuer: one elected lane issues and commits (elect.sync picks
    // the same lane each time: the warp is converged); the warp waits together
    constexpr uint32_t IDS = mma_idesc<C::BFK>(WROWS, WKT);   // bf16 Q and K for BF16 layers
    constexpr uint32_t IDO = mma_idesc<false>(WROWS, D);
    auto wait = [&](uint64_t* bar, uint32_t par) -> bool {
      const bool w = __all_sync(0xffffffffu, mbar_wait(bar, par));
      if (!w && lane == 0) { *s_abort = 1; atomicOr(a.err, ERR_TIMEOUT); }
      return w && !__any_sync(0xffffffffu, *s_abort);
    };
    // Descriptors of the operand buffers' starts; an operand at byte offset
    // o is the start's descriptor plus o / 16 (the 14-bit address field
    // cannot carry: shared memory ends below 2^18 bytes)
    const uint64_t dq = sw128_desc(q16), dk = sw128_desc(k16), dv = sw128_desc(vt16);
    // S_j = Q_j K^T from K buffer kbuf into S buffer sb of query tile j (Q
    // from shared memory with two query tiles, from tensor memory with one)
    auto issue_s = [&](int j, int kbuf, int sb) {
      const uint64_t qa = dq + (uint64_t)(j * (C::QB >> 4));
      const uint64_t kb = dk + (uint64_t)(kbuf * (C::KB >> 4));
      const uint32_t td = tmem + C::scol(j, sb);
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int s2 = 0; s2 < D / 16; ++s2) {
          const uint64_t db = kb + (uint64_t)((((s2 >> 2) * (WKT * 128)) + (s2 & 3) * 32) >> 4);
          if constexpr (NQ == 2)
            umma(td, qa + (uint64_t)((((s2 >> 2) * (WROWS * 128)) + (s2 & 3) * 32) >> 4), db, IDS,
                 s2 > 0);
          else
            umma_tmem_a(td, tmem + C::QCOL + 8 * s2, db, IDS, s2 > 0);
        }
        umma_commit(&s_full[2 * j + sb]);
      }
      __syncwarp();
    };
    // O_j += P'_j V, both terms of the split, P' from S/P' buffer sb, V^T
    // from buffer vbuf
    auto issue_pv = [&](int j, int vbuf, int sb, bool acc) {
      const uint64_t vb = dv + (uint64_t)(vbuf * (C::VTB >> 4));
      const uint32_t td = tmem + C::ocol(j);
      const uint32_t ta = tmem + C::scol(j, sb);
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int kk = 0; kk < WKT / 16; ++kk)
            umma_tmem_a(td, ta + 32 * h + 8 * kk, vb + (uint64_t)(kk * 2), IDO, acc || h > 0 || kk > 0);
      }
      __syncwarp();
    };
    // S of key tile t goes into S/P' buffer t & 1 of each query tile, two
    // tiles ahead of the softmax that reads it: S_j(t+2) is issued once
    // PV_j(t), the last reader of that buffer's P', has completed, so the
    // softmax of a query tile finds its next scores ready when it finishes
    if (wait(&kv_full[0], 0u)) {
#pragma unroll
      for (int j = 0; j < NQ; ++j) issue_s(j, 0, 0);
      bool go = true;
      if (ntl > 1) {
        go = wait(&kv_full[1 % NB], (uint32_t)((1 / NB) & 1));
        if (go)
#pragma unroll
          for (int j = 0; j < NQ; ++j) issue_s(j, 1 % NB, 1);
      }
      for (int i = 0; go && i < ntl; ++i) {
        const int buf = i % NB, sb = i & 1;
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          if (!wait(&p_full[2 * j + sb], (uint32_t)((i >> 1) & 1))) { go = false; break; }
          issue_pv(j, buf, sb, i > 0);
          if (elect_one()) umma_commit(&pv_done[j]);
          __syncwarp();
        }
        if (!go) break;
        // every PV of this key tile has read its operands: buffer free
        if (elect_one()) umma_commit(&kv_empty[buf]);
        __syncwarp();
        if (i + 2 < ntl) {
          const int nb2 = (i + 2) % NB;
          if (!wait(&kv_full[nb2], (uint32_t)(((i + 2) / NB) & 1))) break;
#pragma unroll
          for (int j = 0; j < NQ; ++j) {
            if (!wait(&pv_done[j], (uint32_t)(i & 1))) { go = false; break; }
            issue_s(j, nb2, sb);
          }
          if (!go) break;
        }
      }
    }
    // everything issued completes before the epilogue and the exit
    if (elect_one()) umma_commit(o_fin);
    __syncwarp();
    (void)mbar_wait(o_fin, 0u);
  } else {
    // ---- softmax of query tile j: one thread per row (its tensor-memory lane)
    const int j = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int R = j * WROWS + r;
    const int pA = rowp[R];
    const int loA = (a.window > 0) ? max(0, pA + 1 - a.window) : 0;
    const float fA = rowf[R];
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tO = trow + C::ocol(j);
    // positions of this query tile's first and last rows: a key tile inside
    // [last row's window start, first row] is visible to every row
    const int firstj = first + j * QP;
    const int pmaxj = min(firstj + QP - 1, pmax);
    // mU: the row's reference max (log2 units) the weights are taken against;
    // it moves only when a tile exceeds it by more than WLAZY, so O is
    // rescaled rarely and the weights stay below 2^WLAZY
    float mU = -INFINITY, l = 0.f;
    int vexp = -1000;
    float vs_static = 1.f;
    if constexpr (MODE == FP8_PER_TENSOR) vs_static = a.v_scale[0];
    if constexpr (MODE == FP8_PER_HEAD) vs_static = a.v_scale[g];
    bool ok = true;
    for (int i = 0; i < ntl; ++i) {
      const int buf = i % NB, t = t0 + i;
      // S of this tile in S/P' buffer i & 1 (its P' replaces it there)
      const int sb = i & 1;
      const uint32_t tS = trow + C::scol(j, sb), tP = tS;
      const bool w = __all_sync(0xffffffffu, mbar_wait(&s_full[2 * j + sb], (uint32_t)((i >> 1) & 1)));
      if (!w && lane == 0) { *s_abort = 1; atomicOr(a.err, ERR_TIMEOUT); }
      if (!w || __any_sync(0xffffffffu, *s_abort)) { ok = false; break; }
      tc_fence_after();
      uint32_t s0[32], s1[32];
      tmem_ld32_nowait(tS, s0);
      tmem_ld32_nowait(tS + 32, s1);
      tmem_wait_ld();
      const float* ksm = reinterpret_cast<const float*>(scb + buf * C::SCS);
      const float* vsm = ksm + WKT;
      const int* tinfo = reinterpret_cast<const int*>(vsm + WKT);
      const bool fast = tinfo[2] != 0 && t * WKT + WKT - 1 <= firstj &&
                        (a.window <= 0 || t * WKT >= pmaxj + 1 - a.window);
      // scores times the K scale (or -inf where masked); four running maxima.
      // The test for a wholly visible tile is taken once, outside the
      // unrolled loops, so neither loop branches per key.
      const float4* ks4 = reinterpret_cast<const float4*>(ksm);
      float sv[WKT];
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (fast) {
#pragma unroll
        for (int k4 = 0; k4 < WKT / 4; ++k4) {
          const float4 kq = ks4[k4];
          const float ksv[4] = {kq.x, kq.y, kq.z, kq.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = 4 * k4 + e;
            const float x = __uint_as_float(k < 32 ? s0[k] : s1[k - 32]) * ksv[e];
            sv[k] = x;
            m4[e] = fmaxf(m4[e], x);
          }
        }
      } else {
        // keys of this row: [loA, pA] relative to the tile; a key outside the
        // CTA's range or on a page not fetched has scale 0
        const int klo = loA - t * WKT, khi = pA < 0 ? -1 : pA - t * WKT;
#pragma unroll
        for (int k4 = 0; k4 < WKT / 4; ++k4) {
          const float4 kq = ks4[k4];
          const float ksv[4] = {kq.x, kq.y, kq.z, kq.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = 4 * k4 + e;
            const bool okk = k >= klo && k <= khi && ksv[e] != 0.f;
            const float x = okk ? __uint_as_float(k < 32 ? s0[k] : s1[k - 32]) * ksv[e] : -INFINITY;
            sv[k] = x;
            m4[e] = fmaxf(m4[e], x);
          }
        }
      }
      const float mrow = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * fA;
      float al = 1.f;
      if (mrow > mU + WLAZY || (mU == -INFINITY && mrow > -INFINITY)) {
        al = (mU == -INFINITY) ? 0.f : ex2(mU - mrow);
        mU = mrow;
      }
      if constexpr (C::DYN) {
        const int et = max(tinfo[0], tinfo[1]);     // the same for every row (same keys)
        const int vnew = max(vexp, max(et, -100));
        if (vnew != vexp) {
          al *= pow2i(vexp - vnew);                 // 0 on the first data (O is 0)
          vexp = vnew;
        }
      }
      // l and O both carry the range factor 2^(WKP - vexp) (64 for static
      // scales), so both follow the max and the V-scale exponent
      l *= al;
      // O holds data from the first PV on; it is rescaled (rarely) once the
      // previous PV has updated it.  P' needs no wait: its buffer held this
      // tile's S, and the PV that last read P' there completed before that S
      // was issued.
      if (i > 0 && __any_sync(0xffffffffu, al != 1.f)) {
        const bool w2 = __all_sync(0xffffffffu, mbar_wait(&pv_done[j], (uint32_t)((i - 1) & 1)));
        if (!w2 && lane == 0) { *s_abort = 1; atomicOr(a.err, ERR_TIMEOUT); }
        if (!w2 || __any_sync(0xffffffffu, *s_abort)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float v[32];
          tmem_ld32(tO + c0, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] *= al;
          tmem_st32(tO + c0, v);
        }
      }
      // p x 2^k = 2^(score - (mU - k)): the power-of-two range factor k
      // (WKP - vexp, or 6 for static scales) enters the exponent, exactly
      const float mu = ((mU == -INFINITY) ? 0.f : mU) - (C::DYN ? (float)(WKP - vexp) : 6.f);
      const float4* vs4 = reinterpret_cast<const float4*>(vsm);
      float lp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int k = 16 * c + 4 * q4;
          float x[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            x[e] = ex2(fmaf(sv[k + e], fA, -mu));
            lp[e] += x[e];
          }
          if constexpr (C::DYN) {
            const float4 vq = lds_v4_ordered(vs4 + (k >> 2));
            x[0] *= vq.x; x[1] *= vq.y; x[2] *= vq.z; x[3] *= vq.w;
          }
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint32_t h = pack_f16x2(x[2 * h2], x[2 * h2 + 1]);
            hw[2 * q4 + h2] = h;
            lw[2 * q4 + h2] = pack_f16x2(x[2 * h2] - f16_lo(h), x[2 * h2 + 1] - f16_hi(h));
          }
        }
        tmem_st8_nowait(tP + 8 * c, hw);
        tmem_st8_nowait(tP + 32 + 8 * c, lw);
      }
      l += (lp[0] + lp[1]) + (lp[2] + lp[3]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[2 * j + sb]);
    }
    // ---- epilogue: out = O x unscale / l (rows without a query store nothing)
    const bool fin = __all_sync(0xffffffffu, mbar_wait(o_fin, 0u));
    if (ok && fin && !__any_sync(0xffffffffu, *s_abort)) {
      tc_fence_after();
      // O / l: the range factor cancels; static scales multiply by v_scale
      const float f = l > 0.f ? (C::DYN ? 1.f : vs_static) / l : 0.f;
      const int h = r / QP, ii = r - h * QP;
      float* dst = a.out + ((long long)(q0 + qbase + j * QP + ii) * a.Hq + g * G + h) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        tmem_ld32(tO + c0, v);
        if (pA >= 0) {
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4)
            *reinterpret_cast<float4*>(dst + c0 + 4 * i4) =
                make_float4(v[4 * i4] * f, v[4 * i4 + 1] * f, v[4 * i4 + 2] * f, v[4 * i4 + 3] * f);
        }
      }
    }
  }

  // ---- tensor memory is freed once every role is done with it
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::TCOLS));
  }
}

using WsEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

WsEncodeFn ws_encode_fn() {
  static WsEncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<WsEncodeFn>(p);
  }
  return fn;
}

// A BF16 layer's K buffer as a 3-D uint8 tensor [cell][64-d block][128 bytes]:
// one box is one 64-d block of 16 consecutive cells, which lands as 16 rows
// of the K operand (128-byte swizzle).
bool make_kblock_map(CUtensorMap* m, const void* base, long long total_bytes, int row_bytes) {
  WsEncodeFn fn = ws_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)(row_bytes / 128), (cuuint64_t)(total_bytes / row_bytes)};
  cuuint64_t strides[2] = {128, (cuuint64_t)row_bytes};
  cuuint32_t box[3] = {128, 1, 16};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int D, int G>
cudaError_t wslaunch3(const PrefillArgs& pa0, int max_query_len, cudaStream_t st) {
  using C = WCfg<MODE, D>;
  const DecodeArgs& a = pa0.d;
  const long long total = a.num_blocks * a.Hkv * a.bs * (long long)C::RB;
  CUtensorMap km, vm;
  if (total > 0) {
    const bool kok = C::KDIRECT ? make_kblock_map(&km, a.k_cache, total, C::RB)
                                : make_tile_map(&km, a.k_cache, total, C::TB);
    if (!kok || !make_tile_map(&vm, a.v_cache, total, C::TB)) return cudaErrorInvalidValue;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = prefill_ws_kernel<MODE, D, G>;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  PrefillArgs pa = pa0;
  const int qp2 = WRoles<D>::NQ * (WROWS / G);      // query positions per CTA
  pa.qtiles = (max_query_len + qp2 - 1) / qp2;
  const long long grid = (long long)pa.qtiles * a.B * a.Hkv;
  if (grid <= 0) return cudaSuccess;
  kern<<<(unsigned)grid, WRoles<D>::THREADS, C::SMEM, st>>>(pa, km, vm);
  return cudaGetLastError();
}

template <int MODE, int D>
cudaError_t wslaunch2(int G, const PrefillArgs& pa, int mq, cudaStream_t st) {
  switch (G) {
    case 1: return wslaunch3<MODE, D, 1>(pa, mq, st);
    case 2: return wslaunch3<MODE, D, 2>(pa, mq, st);
    case 4: return wslaunch3<MODE, D, 4>(pa, mq, st);
    case 8: return wslaunch3<MODE, D, 8>(pa, mq, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int MODE>
cudaError_t wslaunch1(int D, int G, const PrefillArgs& pa, int mq, cudaStream_t st) {
  switch (D) {
    case 64: return wslaunch2<MODE, 64>(G, pa, mq, st);
    case 128: return wslaunch2<MODE, 128>(G, pa, mq, st);
    case 256: return wslaunch2<MODE, 256>(G, pa, mq, st);
    default: return cudaErrorInvalidValue;
  }
}

// BF16 layers at head_dim 64 and 128 (a BF16 raw stage at 256 does not fit
// beside the operand buffers)
cudaError_t wslaunch1_bf16(int D, int G, const PrefillArgs& pa, int mq, cudaStream_t st) {
  switch (D) {
    case 64: return wslaunch2<BF16, 64>(G, pa, mq, st);
    case 128: return wslaunch2<BF16, 128>(G, pa, mq, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool prefill_ws_supports(int mode, int D) {
  if (mode == BF16) return D == 64 || D == 128;
  return D == 64 || D == 128 || D == 256;
}

cudaError_t launch_prefill_ws(int mode, int D, int G, const DecodeArgs& a, const int* query_start,
                              int max_query_len, cudaStream_t st) {
  if (a.B == 0 || max_query_len <= 0) return cudaSuccess;
  PrefillArgs pa;
  pa.d = a;
  pa.query_start = query_start;
  pa.qtiles = 0;
  switch (mode) {
    case FP8_PER_TENSOR: return wslaunch1<FP8_PER_TENSOR>(D, G, pa, max_query_len, st);
    case FP8_PER_HEAD: return wslaunch1<FP8_PER_HEAD>(D, G, pa, max_query_len, st);
    case FP8_PER_TOKEN_HEAD: return wslaunch1<FP8_PER_TOKEN_HEAD>(D, G, pa, max_query_len, st);
    case INT4_PER_TOKEN_HEAD: return wslaunch1<INT4_PER_TOKEN_HEAD>(D, G, pa, max_query_len, st);
    case BF16: return wslaunch1_bf16(D, G, pa, max_query_len, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
