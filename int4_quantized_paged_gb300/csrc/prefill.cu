// Prefill (chunked multi-query) attention over the quantized paged cache on
// the fifth-generation tensor cores (tcgen05, accumulators in tensor memory),
// single-role: every warp takes each phase in turn.  It serves BF16 layers
// at head_dim 256, whose bf16 pages do not fit the warp-specialised kernel's
// raw stages beside its operand buffers; every other layer goes to that
// kernel (launch_prefill below dispatches).
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
//  * A CTA owns M = 128 query rows of one (sequence, KV head): 128/G
//    consecutive new positions times the G query heads of that KV head, so a
//    key/value tile is fetched and dequantized once for all of them.  CTAs
//    with the latest (longest) query tiles start first.
//  * Keys stream in tiles of KT positions (64; 32 for BF16 at D = 256, whose
//    pages are largest): KT/16 page tiles by 2-D TMA for K and V plus 64-byte
//    bulk copies of the dynamic scales, through NSR raw stages.  All threads
//    convert a landed tile once into f16 (bf16 for BF16 layers; exact) in the
//    tensor cores' shared-memory layout: K as KT rows of D (K-major, 128-byte
//    swizzle) and V transposed, D rows of KT keys, through a row-major
//    staging copy.  Positions outside the CTA's key range become zeros.
//  * S = Q K^T: one thread issues D/16 tcgen05.mma (M 128, N KT, K 16) from
//    shared-memory descriptors into KT tensor-memory columns, and commits them
//    to a shared-memory barrier.
//  * Softmax: every warp takes 32 query rows (its tensor-memory lanes) and one
//    half of the tile's keys; a thread loads its row's KT/2 scores
//    (tcgen05.ld), applies the K scale and, on tiles not wholly visible to
//    every row, the causal / window masks, and the two halves exchange their
//    maxima through shared memory.  The row's reference max moves only when
//    a tile exceeds it by more than 2^8 (log2 units 8), so the output
//    accumulator in tensor memory is rescaled rarely (each half rescales its
//    half of the columns); the weights stay below 2^8 and meet V as
//    P' = p x v_scale x 2^k (k keeps P' below 2^15), split into f16 hi + lo
//    (three bf16 terms for BF16 layers) and written to shared memory, K-major.
//  * O += P' V: one thread issues the split's terms (M 128, N D, K 16 each)
//    into D tensor-memory columns and commits.  The next tile's conversion
//    waits for that commit before it overwrites the operands.
//  * Epilogue: each thread reads its half of its row of O (tcgen05.ld),
//    divides by the row sum (both halves' sums) and stores fp32.  Tensor memory is allocated and freed
//    by warp 0; every wait is bounded, and a wait that runs out flags TIMEOUT,
//    lets the work already issued finish (bounded again) and frees tensor
//    memory before the CTA exits.
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

constexpr int TWARPS = 8;                  // warps per CTA
constexpr int TROWS = 128;                 // query rows per CTA (the MMA's M)
constexpr int TKP = 6;                     // P' = p v_scale 2^(TKP - vexp) < 2^15 (p <= 2^8)
constexpr float TLAZY = 8.f;               // the row's reference max moves when exceeded by this
constexpr float TSTATIC = 64.f;            // P' = p x 64 for static FP8 scales (< 2^14)

// ------------------------------------------------------------ configuration
template <int MODE, int D>
struct TCfg {
  static constexpr int RB = row_bytes<MODE>(D);
  static constexpr int TB = 16 * RB;                       // one page tile (16 positions)
  static constexpr int TBP = (TB + 1023) / 1024 * 1024;
  static constexpr bool DYN = (MODE == FP8_PER_TOKEN_HEAD || MODE == INT4_PER_TOKEN_HEAD);
  static constexpr bool BF = (MODE == BF16);
  static constexpr int KT = (BF && D == 256) ? 32 : 64;    // keys per tile
  static constexpr int SUB = KT / 16;                       // page tiles per key tile
  static constexpr int NPART = BF ? 3 : 2;                  // terms of the P' split
  static constexpr int RAW = 2 * SUB * TBP;                 // K and V page tiles of a key tile
  static constexpr int SCB = DYN ? 2 * SUB * 64 : 0;        // their K and V scales
  static constexpr int RAWS = (RAW + SCB + 1023) / 1024 * 1024;
  static constexpr int QB = TROWS * D * 2;                  // Q: D/64 blocks of 128 x 128 B
  static constexpr int KB = KT * D * 2;                     // K: D/64 blocks of KT x 128 B
  static constexpr int VTB = D * 128;                       // V^T: D rows of 128 B (KT keys)
  static constexpr int PB = TROWS * 128;                    // one P' term: 128 rows of 128 B
  static constexpr int LDV = (D + 8) * 2;                   // row pitch (bytes) of the V staging copy
  // the P' terms' region, which also holds the V staging copy during conversion
  static constexpr int PREG = (NPART * PB > KT * LDV) ? NPART * PB : KT * LDV;
  // the operands of one key tile: K, V^T and the P' region
  static constexpr int BUF = (KB + VTB + PREG + 1023) / 1024 * 1024;
  // K and V scales and the tile's V-scale exponents
  static constexpr int SCB1 = 2 * KT * 4 + 16;
  // row data, per-half row maxima / sums, barriers, flags
  static constexpr int SMALLC = TROWS * 8 + 2 * TROWS * 4 + 128;
  static constexpr int LIMIT = 232448 - 1024;               // per-CTA shared memory, minus slack
  static constexpr int FIXED = QB + BUF + SCB1 + SMALLC;
  static constexpr int NSR = (2 * RAWS + FIXED <= LIMIT) ? 2 : 1;
  static constexpr int SMEM = NSR * RAWS + FIXED + 1024;
  static constexpr int OCOL = KT;                           // S: [0, KT), O: [KT, KT + D)
  static constexpr int TCOLS = (OCOL + D <= 128) ? 128 : ((OCOL + D <= 256) ? 256 : 512);
};

template <int MODE, int D, int G>
__global__ void __launch_bounds__(TWARPS * 32, 1)
    prefill_tc_kernel(const PrefillArgs pa, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  using C = TCfg<MODE, D>;
  using ET = uint16_t;
  const DecodeArgs& a = pa.d;
  constexpr int KT = C::KT;
  constexpr int SUB = C::SUB;
  constexpr int NSR = C::NSR;
  constexpr int QP = TROWS / G;                // positions per query tile
  constexpr int CPR = C::RB / 16;              // 16-byte raw chunks per position row
  constexpr int EPC = (MODE == BF16) ? 8 : (MODE == INT4_PER_TOKEN_HEAD ? 32 : 16);  // elements per raw chunk

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* raw = smem;                                       // NSR stages
  uint8_t* q16 = smem + NSR * C::RAWS;                       // Q, K-major swizzled
  uint8_t* k16 = q16 + C::QB;                                // K, K-major swizzled
  uint8_t* vt16 = k16 + C::KB;                               // V^T, K-major swizzled
  uint8_t* p16 = vt16 + C::VTB;                              // P' terms; also the V staging copy
  float* ksm = reinterpret_cast<float*>(k16 + C::BUF);      // [KT] K scale (0: no key)
  float* vsm = ksm + KT;                                     // [KT] V scale
  int* etile = reinterpret_cast<int*>(vsm + KT);             // [4] tile V-scale exponents
  float* rowf = reinterpret_cast<float*>(etile + 4);         // [TROWS] score factor per row
  int* rowp = reinterpret_cast<int*>(rowf + TROWS);          // [TROWS] position (-1: no row)
  float* mx = reinterpret_cast<float*>(rowp + TROWS);       // [2][TROWS] per-half row max / sum
  uint64_t* bars = reinterpret_cast<uint64_t*>(mx + 2 * TROWS);  // [NSR] raw, then S, then O
  uint64_t* bar_s = bars + NSR;
  uint64_t* bar_o = bar_s + 1;
  int& s_flag = *reinterpret_cast<int*>(bar_o + 1);
  uint32_t& s_tmem = *(reinterpret_cast<uint32_t*>(bar_o + 1) + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- this CTA's (sequence, KV head, query tile); latest tiles first
  const int per_tile = a.B * a.Hkv;
  const int qt = pa.qtiles - 1 - (int)(blockIdx.x / per_tile);
  const int rem = (int)(blockIdx.x % per_tile);
  const int b = rem / a.Hkv, g = rem - b * a.Hkv;
  const int q0 = pa.query_start[b];
  const int n_b = pa.query_start[b + 1] - q0;
  const int L = a.context_lens[b];
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
    for (int s = 0; s < NSR + 2; ++s) mbar_init(&bars[s], 1);
    mbar_init_fence();
    s_flag = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&s_tmem)),
                 "r"(C::TCOLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  // ---- queries: row r = h * QP + i -> token q0 + qt*QP + i, head g*G + h,
  // prescaled by a power of two so the bf16 values are exact in f16.  Warp w
  // stages rows w, w + 8, ...; lane l holds elements l + 32e.
  float ks_static = 1.f;
  if constexpr (MODE == FP8_PER_TENSOR) ks_static = a.k_scale[0];
  if constexpr (MODE == FP8_PER_HEAD) ks_static = a.k_scale[g];
  for (int r = warp; r < TROWS; r += TWARPS) {
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
      const int d = lane + 32 * e;
      const float v = x[e] * qmul;
      const ET h16 = C::BF ? (ET)(pack_bf16x2(v, 0.f) & 0xFFFFu) : (ET)(pack_f16x2(v, 0.f) & 0xFFFFu);
      *reinterpret_cast<ET*>(q16 + (d >> 6) * (TROWS * 128) + swc(r, (d & 63) >> 3) + (d & 7) * 2) = h16;
    }
    if (lane == 0) {
      rowf[r] = a.qk_scale * ks_static * (C::BF ? 1.f : pow2i(qexp - 14));
      rowp[r] = valid ? first + i : -1;
    }
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

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
  int pend[2] = {-1, -1};                          // tile issued into each stage, not yet landed
  if (warp == 0)
    for (int s = 0; s < NSR && t0 + s <= t1; ++s) {
      fetched[s] = issue(t0 + s, s);
      pend[s] = t0 + s;
    }

  // ---- softmax state.  Every warp scores half of each key tile for 32 rows:
  // warp w takes rows (w & 3) * 32 + lane (its tensor-memory lanes) and keys
  // [half * KH, half * KH + KH) with half = w >> 2.
  constexpr int KH = KT / 2;
  const int r = (warp & 3) * 32 + lane;
  const int half = warp >> 2;
  const int pA = rowp[r];
  const int loA = (a.window > 0) ? max(0, pA + 1 - a.window) : 0;
  const float fA = rowf[r];
  const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  // mU: the row's reference max (log2 units) the weights are taken against;
  // it moves only when a tile's max exceeds it by more than TLAZY, so the
  // output accumulator is rescaled rarely and the weights stay below 2^TLAZY
  float mU = -INFINITY, lH = 0.f;                  // lH: this half's running sum
  int vexp = -1000;
  float fv = 0.f;                                  // 2^(TKP - vexp)
  float vs_static = 1.f;
  if constexpr (MODE == FP8_PER_TENSOR) vs_static = a.v_scale[0];
  if constexpr (MODE == FP8_PER_HEAD) vs_static = a.v_scale[g];
  constexpr uint32_t IDS = mma_idesc<C::BF>(TROWS, KT);
  constexpr uint32_t IDO = mma_idesc<C::BF>(TROWS, D);

  bool failed = false;
  int issued_s = 0, issued_o = 0;                  // S and PV commits issued (barrier phases)
  unsigned have = 0u;                              // fetched pages of the current key tile

  // Waits for key tile tt's pages and for the last PV (the previous reader of
  // K, V^T and P'), converts the tile and issues S = Q K^T.
  auto convert_and_score = [&](int tt) -> bool {
    const int st = (tt - t0) % NSR;
    const uint32_t par = (uint32_t)(((tt - t0) / NSR) & 1);
    bool ok = mbar_wait(&bars[st], par);
    if (issued_o > 0) ok = mbar_wait(bar_o, (uint32_t)((issued_o - 1) & 1)) && ok;
    if (__syncthreads_or(!ok)) return false;
    pend[st] = -1;
    tc_fence_after();
    // which page tiles of this key tile hold data (warp 0 knows; share it)
    if (tid == 0) s_flag = (int)fetched[st];
    __syncthreads();
    have = (unsigned)s_flag;
    const uint8_t* base = raw + st * C::RAWS;
    uint8_t* kb = k16;
    uint8_t* pb = p16;
    // K into kb, V into the row-major staging copy in pb (zeros where
    // nothing was fetched or the position lies outside [kmin, pmax]).  Each
    // thread takes NIT chunks of K and as many of V; all loads first, then
    // the conversions, with no branch per chunk.
    // (INT4 at D 64 has fewer chunks than threads: the rest idle, whole warps)
    constexpr int NIT = (KT * CPR + TWARPS * 32 - 1) / (TWARPS * 32);
    {
      uint4 wk[NIT], wv[NIT];
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        const int cc = tid + it * TWARPS * 32;
        const int key = cc / CPR, ch = cc % CPR;
        const int sub = key >> 4, kr = key & 15;
        const int pos = tt * KT + key;
        const bool live = cc < KT * CPR && ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
        const uint32_t off = swz((uint32_t)(kr * C::RB + ch * 16));
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        wk[it] = live ? *reinterpret_cast<const uint4*>(base + sub * C::TBP + off) : z;
        wv[it] = live ? *reinterpret_cast<const uint4*>(base + (SUB + sub) * C::TBP + off) : z;
      }
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        const int cc = tid + it * TWARPS * 32;
        if (cc >= KT * CPR) break;
        const int key = cc / CPR, ch = cc % CPR;
        uint4 ok_[4], ov[4];
        convert16<MODE>(wk[it], ok_);
        convert16<MODE>(wv[it], ov);
        const int d0 = ch * EPC;
#pragma unroll
        for (int q = 0; q < EPC / 8; ++q) {
          const int d = d0 + 8 * q;
          *reinterpret_cast<uint4*>(kb + (d >> 6) * (KT * 128) + swc(key, (d & 63) >> 3)) = ok_[q];
          *reinterpret_cast<uint4*>(pb + key * C::LDV + d * 2) = ov[q];
        }
      }
    }
    if (tid < 2 * KT) {
      const int isv = tid >= KT;
      const int key = isv ? tid - KT : tid;
      const int sub = key >> 4;
      const int pos = tt * KT + key;
      const bool live = ((have >> sub) & 1u) && pos >= kmin && pos <= pmax;
      float sc = live ? 1.f : 0.f;
      if constexpr (C::DYN)
        if (live) sc = reinterpret_cast<const float*>(base + C::RAW)[16 * (isv ? SUB + sub : sub) + (key & 15)];
      (isv ? vsm : ksm)[key] = sc;
      if constexpr (C::DYN) {
        // the largest V-scale exponent of the tile's live keys (whole warps)
        if (isv) {
          const int e = __reduce_max_sync(0xffffffffu, live ? f32_exp(sc) : -1000);
          if (lane == 0) etile[(tid - KT) >> 5] = e;
        }
      }
    }
    __syncthreads();
    // the raw stage is free: fetch key tile tt + NSR into it
    if (warp == 0 && tt + NSR <= t1) {
      fence_proxy_async();
      fetched[st] = issue(tt + NSR, st);
      pend[st] = tt + NSR;
    }
    // V^T: rows d, chunks of 8 keys, from the staging copy
    uint8_t* vb = vt16;
    constexpr int NVT = (KT / 8) * (D / 2) / (TWARPS * 32);
    static_assert(NVT * TWARPS * 32 == (KT / 8) * (D / 2), "V^T tasks per thread");
#pragma unroll
    for (int it = 0; it < NVT; ++it) {
      const int u = tid + it * TWARPS * 32;
      const int dp = u % (D / 2), kg = u / (D / 2);
      uint32_t wv[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        wv[k] = *reinterpret_cast<const uint32_t*>(pb + (8 * kg + k) * C::LDV + dp * 4);
      uint4 e, f;
      e.x = __byte_perm(wv[0], wv[1], 0x5410);
      e.y = __byte_perm(wv[2], wv[3], 0x5410);
      e.z = __byte_perm(wv[4], wv[5], 0x5410);
      e.w = __byte_perm(wv[6], wv[7], 0x5410);
      f.x = __byte_perm(wv[0], wv[1], 0x7632);
      f.y = __byte_perm(wv[2], wv[3], 0x7632);
      f.z = __byte_perm(wv[4], wv[5], 0x7632);
      f.w = __byte_perm(wv[6], wv[7], 0x7632);
      *reinterpret_cast<uint4*>(vb + swc(2 * dp, kg)) = e;
      *reinterpret_cast<uint4*>(vb + swc(2 * dp + 1, kg)) = f;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && elect_one()) {               // lane 0 of the converged warp 0
      tc_fence_after();
#pragma unroll
      for (int s2 = 0; s2 < D / 16; ++s2) {
        const uint64_t da = sw128_desc(q16 + (s2 >> 2) * (TROWS * 128) + (s2 & 3) * 32);
        const uint64_t db = sw128_desc(kb + (s2 >> 2) * (KT * 128) + (s2 & 3) * 32);
        umma(tmem, da, db, IDS, s2 > 0);
      }
      umma_commit(bar_s);
    }
    ++issued_s;
    return true;
  };

  if (!convert_and_score(t0)) failed = true;
  for (int t = t0; t <= t1 && !failed; ++t) {
    // ---- softmax: this warp's half of the row's scores; rescale O; write P'
    // key tile fully visible to every query row of the CTA: no mask needed
    const bool fast = have == (1u << SUB) - 1u && t * KT + KT - 1 <= first &&
                      (a.window <= 0 || t * KT >= pmax + 1 - a.window);
    const float* kss = ksm;
    const float* vss = vsm;
    float sv[KH];
    // S of this tile, and the last PV (O is rescaled below); warp-uniform, so
    // the warp-wide tensor-memory loads stay converged
    bool sok = mbar_wait(bar_s, (uint32_t)((issued_s - 1) & 1));
    if (issued_o > 0) sok = mbar_wait(bar_o, (uint32_t)((issued_o - 1) & 1)) && sok;
    sok = __all_sync(0xffffffffu, sok);
    if (sok) {
      tc_fence_after();
      if constexpr (KH == 32) {
        tmem_ld32(trow + half * KH, sv);
      } else {
        tmem_ld16(trow + half * KH, sv);
      }
      // the test for a wholly visible tile is taken once, outside the
      // unrolled loops, so neither loop branches per key
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (fast) {
#pragma unroll
        for (int j = 0; j < KH; ++j) {
          sv[j] *= kss[half * KH + j];
          m4[j & 3] = fmaxf(m4[j & 3], sv[j]);
        }
      } else {
        // keys of this row relative to the tile; a key whose page was not
        // fetched (bad block id) has scale 0: masked
        const int klo = loA - t * KT, khi = pA < 0 ? -1 : pA - t * KT;
#pragma unroll
        for (int j = 0; j < KH; ++j) {
          const int key = half * KH + j;
          const float ks = kss[key];
          const bool okj = key >= klo && key <= khi && ks != 0.f;
          sv[j] = okj ? sv[j] * ks : -INFINITY;
          m4[j & 3] = fmaxf(m4[j & 3], sv[j]);
        }
      }
      const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      mx[half * TROWS + r] = mt;
    }
    if (__syncthreads_or(!sok)) {
      failed = true;
      break;
    }
    {
      // the row's tile max (both halves), in log2 units
      const float mrow = fmaxf(mx[r], mx[TROWS + r]) * fA;
      float al = 1.f;
      if (mrow > mU + TLAZY || (mU == -INFINITY && mrow > -INFINITY)) {
        al = (mU == -INFINITY) ? 0.f : ex2(mU - mrow);
        mU = mrow;
      }
      // the sum of weights follows the max only; O (whose weights carry the
      // V-scale factor 2^(TKP - vexp)) also follows the V-scale exponent
      lH *= al;
      if constexpr (C::DYN) {
        // the V-scale exponent is the same for every row (same keys)
        int et = etile[0];
        if constexpr (KT > 32) et = max(et, etile[1]);
        const int vnew = max(vexp, max(et, -100));
        if (vnew != vexp) {
          al *= pow2i(vexp - vnew);               // 0 on the first data (O is 0)
          vexp = vnew;
          fv = pow2i(TKP - vexp);
        }
      }
      // O holds no data before the first tile's PV; each half rescales its
      // half of the row's columns
      if (issued_o > 0 && __any_sync(0xffffffffu, al != 1.f)) {
#pragma unroll 1
        for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
          float v[32];
          tmem_ld32(trow + C::OCOL + c0, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= al;
          tmem_st32(trow + C::OCOL + c0, v);
        }
      }
      const float mu = (mU == -INFINITY) ? 0.f : mU;
      uint8_t* pb = p16;
#pragma unroll
      for (int c8 = 0; c8 < KH / 8; ++c8) {
        uint32_t hp[C::NPART][4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          float x[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = 8 * c8 + 2 * e2 + h;
            const float p = ex2(fmaf(sv[j], fA, -mu));
            lH += p;
            float vf;
            if constexpr (C::DYN) vf = vss[half * KH + j] * fv;
            else if constexpr (C::BF) vf = 1.f;
            else vf = TSTATIC;
            x[h] = p * vf;
          }
          if constexpr (C::BF) {
            const uint32_t h0 = pack_bf16x2(x[0], x[1]);
            const float r0 = x[0] - bf16_lo(h0), r1 = x[1] - bf16_lo(h0 >> 16);
            const uint32_t m0 = pack_bf16x2(r0, r1);
            hp[0][e2] = h0;
            hp[1][e2] = m0;
            hp[2 % C::NPART][e2] = pack_bf16x2(r0 - bf16_lo(m0), r1 - bf16_lo(m0 >> 16));
          } else {
            const uint32_t h0 = pack_f16x2(x[0], x[1]);
            hp[0][e2] = h0;
            hp[1][e2] = pack_f16x2(x[0] - f16_lo(h0), x[1] - f16_hi(h0));
          }
        }
#pragma unroll
        for (int k = 0; k < C::NPART; ++k)
          *reinterpret_cast<uint4*>(pb + k * C::PB + swc(r, half * (KH / 8) + c8)) =
              make_uint4(hp[k][0], hp[k][1], hp[k][2], hp[k][3]);
      }
      fence_proxy_async();
      tc_fence_before();
    }
    __syncthreads();
    // ---- O += P' V^T, every term of the split
    if (warp == 0 && elect_one()) {
      tc_fence_after();
      const uint8_t* pb = p16;
      const uint8_t* vb = vt16;
#pragma unroll
      for (int k = 0; k < C::NPART; ++k)
#pragma unroll
        for (int s2 = 0; s2 < KT / 16; ++s2) {
          const uint64_t da = sw128_desc(pb + k * C::PB + s2 * 32);
          const uint64_t db = sw128_desc(vb + s2 * 32);
          umma(tmem + C::OCOL, da, db, IDO, issued_o > 0 || k > 0 || s2 > 0);
        }
      umma_commit(bar_o);
    }
    ++issued_o;
    // the next tile is converted once this PV has read the operands
    if (t + 1 <= t1 && !convert_and_score(t + 1)) {
      failed = true;
      break;
    }
  }

  // ---- the last PV completes; on a failure, also the last S and every raw
  // tile still in flight (each wait bounded), so nothing is pending when
  // tensor memory is freed and the CTA exits
  bool fin = true;
  if (issued_o > 0) fin = mbar_wait(bar_o, (uint32_t)((issued_o - 1) & 1));
  failed = __syncthreads_or(failed || !fin);
  if (failed) {
    if (tid == 0) {
      atomicOr(a.err, ERR_TIMEOUT);
      if (issued_s > 0) (void)mbar_wait(bar_s, (uint32_t)((issued_s - 1) & 1));
    }
    if (warp == 0 && lane == 0)
      for (int s2 = 0; s2 < NSR; ++s2)
        if (pend[s2] >= 0) (void)mbar_wait(&bars[s2], (uint32_t)(((pend[s2] - t0) / NSR) & 1));
  } else {
    // ---- epilogue: out = O x unscale / l per row; each half stores its half
    // of the row's columns (the loads are warp-wide; rows without a query
    // store nothing)
    mx[half * TROWS + r] = lH;
    __syncthreads();
    const float l = mx[r] + mx[TROWS + r];
    tc_fence_after();
    float unscale;
    if constexpr (C::BF) unscale = 1.f;
    else if constexpr (C::DYN) unscale = pow2i(vexp - TKP);
    else unscale = vs_static * (1.f / TSTATIC);
    const float f = l > 0.f ? unscale / l : 0.f;
    const int h = r / QP, i = r - h * QP;
    float* dst = a.out + ((long long)(q0 + qt * QP + i) * a.Hq + g * G + h) * D;
#pragma unroll 1
    for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
      float v[32];
      tmem_ld32(trow + C::OCOL + c0, v);
      if (pA >= 0) {
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4)
          *reinterpret_cast<float4*>(dst + c0 + 4 * i4) =
              make_float4(v[4 * i4] * f, v[4 * i4 + 1] * f, v[4 * i4 + 2] * f, v[4 * i4 + 3] * f);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::TCOLS));
  }
}

template <int MODE, int D, int G>
cudaError_t tclaunch3(const PrefillArgs& pa, cudaStream_t st) {
  using C = TCfg<MODE, D>;
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
  auto kern = prefill_tc_kernel<MODE, D, G>;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long grid = (long long)pa.qtiles * a.B * a.Hkv;
  if (grid <= 0) return cudaSuccess;
  kern<<<(unsigned)grid, TWARPS * 32, C::SMEM, st>>>(pa, km, vm);
  return cudaGetLastError();
}

template <int MODE, int D>
cudaError_t tclaunch2(int G, const PrefillArgs& pa, cudaStream_t st) {
  switch (G) {
    case 1: return tclaunch3<MODE, D, 1>(pa, st);
    case 2: return tclaunch3<MODE, D, 2>(pa, st);
    case 4: return tclaunch3<MODE, D, 4>(pa, st);
    case 8: return tclaunch3<MODE, D, 8>(pa, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int MODE>
cudaError_t tclaunch1(int D, int G, const PrefillArgs& pa, cudaStream_t st) {
  switch (D) {
    case 64: return tclaunch2<MODE, 64>(G, pa, st);
    case 128: return tclaunch2<MODE, 128>(G, pa, st);
    case 256: return tclaunch2<MODE, 256>(G, pa, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int prefill_rows_per_cta() { return TROWS; }

cudaError_t launch_prefill(int mode, int D, int G, const DecodeArgs& a, const int* query_start,
                           int max_query_len, cudaStream_t st) {
  if (a.B == 0 || max_query_len <= 0) return cudaSuccess;
  if (prefill_ws_supports(mode, D))
    return launch_prefill_ws(mode, D, G, a, query_start, max_query_len, st);
  PrefillArgs pa;
  pa.d = a;
  pa.query_start = query_start;
  const int qp = TROWS / G;
  pa.qtiles = (max_query_len + qp - 1) / qp;
  switch (mode) {
    case BF16: return tclaunch1<BF16>(D, G, pa, st);
    case FP8_PER_TENSOR: return tclaunch1<FP8_PER_TENSOR>(D, G, pa, st);
    case FP8_PER_HEAD: return tclaunch1<FP8_PER_HEAD>(D, G, pa, st);
    case FP8_PER_TOKEN_HEAD: return tclaunch1<FP8_PER_TOKEN_HEAD>(D, G, pa, st);
    case INT4_PER_TOKEN_HEAD: return tclaunch1<INT4_PER_TOKEN_HEAD>(D, G, pa, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
