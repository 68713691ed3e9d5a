// Paged GQA decode attention over the quantized cache.
//
// What it computes: for each sequence b and query head hq, the softmax over
// retained positions p in [lo, L) of softmax_scale * <q, K_hat[p]> weights
// V_hat[p]; K_hat = code * K scale, V_hat = code * V scale.  The K scale
// multiplies the dot product of q with the raw codes and the V scale the
// softmax weight, so codes are never rescaled element by element.  Scale
// layouts: "Per-tensor vs per-head FP8 KV cache scales"; packed INT4:
// "Per-token-head KV cache scale overhead", section "INT4 makes the metadata
// fraction larger"; windows and BF16 (skipped) layers: "FP8 KV cache layer
// skipping vs per-head scales", sections "FP8 KV cache layer skipping vs
// per-head scales" and "Layer skipping follows retained-token footprint".
//
// Work decomposition (split-K over the context, balanced over warps):
//  * A sequence's retained positions are cut into 16-position tiles (a tile
//    never straddles a page: block_size is a multiple of 16).  All tiles of
//    all (sequence, KV head) items, in that order, form one list of T tiles.
//    Worker warp w takes tiles [w T / W, (w+1) T / W): every warp gets the
//    same number of tiles whatever the context lengths, and a warp's share
//    runs across item boundaries.  For each item segment it covers, a warp
//    either writes the final output (it covered the whole item) or a partial
//    (running max m, sum l, unnormalised O) that a merge kernel combines by
//    log-sum-exp; the merge is a programmatic dependent launch, so its launch
//    overlaps this grid's tail.  Warps never wait on one another.
//  * Each warp streams its tiles through an NS-stage ring in shared memory
//    with TMA: a 2-D tensor copy each for the K and V code tile (128-byte
//    rows, 128B swizzle so the fragment loads below hit no bank conflicts)
//    and, for dynamic scales, a 64-byte bulk copy each of the tile's K and V
//    scales, completing on the stage's mbarrier.  The copies of the next
//    NS-1 tiles (of this or the next item) are in flight while one tile is
//    computed.  Pages of a layer larger than L2 are copied evict-first.
//    Every wait is bounded: a wait that runs out sets the TIMEOUT bit of the
//    device error word, drains the warp's copies and stops.
//  * QK on tensor cores: S^T[16 positions x 8 columns] = K_tile . Q^T with
//    mma.m16n8k16, fp32 accumulate.  E4M3 and INT4 codes convert exactly to
//    f16; q (bf16) times a power of two converts exactly to f16 (an FP8
//    query's E4M3 values are f16 values).  Columns are the G query heads of
//    the KV head, repeated once per term of the weight split when they fit
//    in the 8 columns, so a QK column is already the PV column it feeds.
//  * Online softmax in log2 units on the fragments, against a reference max
//    that moves (reduced over the warp, O and l rescaled) only on tiles where
//    some lane holds a score above it by more than 8 (a weight factor of
//    2^8), so the weights p stay below 2^8.  The weights that meet V are P' = p * v_scale * 2^k, with k a
//    power-of-two range factor that keeps P' below 2^14, so both f16 terms of
//    its split stay normal numbers.
//  * PV on tensor cores with d as the M dimension: O^T[d x cols] += V^T P'.
//    P' is split into two f16 terms (hi + lo, about 22 bits; three bf16
//    terms for BF16 layers) so the weighted sum keeps fp32-class accuracy;
//    for G*terms <= 8 all terms share one 8-column tile.  The P' fragment
//    comes from the S^T fragment by movmatrix (in-register 8x8 transpose).
//  * Outputs are fp32, or their round-to-nearest-even bf16 for the bf16
//    variant.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "async_copy.cuh"
#include "kvq_internal.h"
#include "tile_math.cuh"

namespace kvq {
namespace {

constexpr int WARPS = 4;         // worker warps per CTA (independent)
// Tuning knob (build-time): the QK accumulator chains (2 shortens the MMA
// dependency chain).
#ifndef KVQ_QK2
#define KVQ_QK2 1
#endif
constexpr int TILE = 16;         // positions per tile
// The reference max m_run a column's weights are taken against moves only
// when a tile's score exceeds it by more than LAZY (log2 units), so most
// tiles rescale nothing and the weights p stay below 2^LAZY.
constexpr float LAZY = 8.f;
constexpr int KP = 5;            // P' = p v_scale 2^(KP - vexp) < 2^14 (dynamic scales)
constexpr float PSTATIC = 64.f;  // P' = p x 64 < 2^14 (static FP8 scales)

template <int N>
__device__ __forceinline__ void lds(uint32_t (&r)[N], const uint8_t* base, uint32_t o) {
  static_assert(N == 1 || N == 2 || N == 4, "");
  const uint8_t* p = base + swz(o);
  if constexpr (N == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
  } else if constexpr (N == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    r[0] = v.x; r[1] = v.y;
  } else {
    r[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}

// d index of QK k-slot j (0: 2t, 1: 2t+1, 2: 2t+8, 3: 2t+9) at k-step s for
// lane column t: the order the QK A-fragment loader produces.
template <int MODE, int D>
__device__ __forceinline__ int qk_d(int t, int s, int j) {
  if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
    const int base = t * (D / 4) + 8 * (s >> 1) + 2 * (s & 1);
    const int off[4] = {0, 4, 1, 5};
    return base + off[j];
  } else {
    return t * (D / 4) + 4 * s + j;
  }
}

// Term k of the split of a weight x into f16 (hi, lo) or bf16 (hi, mid, lo)
// parts whose sum reproduces x to about 22 (f16) or 24 (bf16) bits.
template <bool BF>
__device__ __forceinline__ float split_term(float x, int k) {
  if constexpr (BF) {
    const float h = bf16_lo(pack_bf16x2(x, 0.f));
    const float r = x - h;
    const float m = bf16_lo(pack_bf16x2(r, 0.f));
    return k == 0 ? h : (k == 1 ? m : r - m);
  } else {
    const float h = f16_lo(pack_f16x2(x, 0.f));
    return k == 0 ? h : x - h;
  }
}

// SEG bytes of a token row segment from a swizzled tile into 32-bit words;
// zeros when the token is masked (its bytes may be anything).
template <int SEG>
__device__ __forceinline__ void load_seg(uint32_t* w, const uint8_t* tile, uint32_t off, bool ok) {
  if constexpr (SEG >= 16) {
#pragma unroll
    for (int h = 0; h < SEG / 16; ++h) {
      uint32_t r[4];
      lds<4>(r, tile, off + 16 * h);
#pragma unroll
      for (int e = 0; e < 4; ++e) w[4 * h + e] = ok ? r[e] : 0u;
    }
  } else if constexpr (SEG == 8) {
    uint32_t r[2];
    lds<2>(r, tile, off);
    w[0] = ok ? r[0] : 0u;
    w[1] = ok ? r[1] : 0u;
  } else {
    uint32_t r[1];
    lds<1>(r, tile, off);
    w[0] = ok ? r[0] : 0u;
  }
}

// QK of one 16-position sub-tile: sacc (rows lg, lg+8; columns 2lt, 2lt+1)
// += K_tile . Q^T.  The lane reads its D/4-element segment of rows lg, lg+8.
template <int MODE, int D>
__device__ __forceinline__ void qk_tile(float sacc_out[4], const uint8_t* kt, int lg, int lt,
                                        const uint32_t (*qf)[2]) {
  constexpr int RB = row_bytes<MODE>(D);
  constexpr int KSTEPS = D / 16;
  constexpr int NCH = KVQ_QK2 ? 2 : 1;     // independent accumulator chains
  const int r0 = lg, r1 = lg + 8;
  float sacc2[NCH][4];
#pragma unroll
  for (int c = 0; c < NCH; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) sacc2[c][e] = 0.f;
  if constexpr (MODE == BF16) {
#pragma unroll
    for (int s4 = 0; s4 < KSTEPS; s4 += 2) {
      uint32_t w0[4], w1[4];
      lds<4>(w0, kt, r0 * RB + lt * (D / 2) + 8 * s4);
      lds<4>(w1, kt, r1 * RB + lt * (D / 2) + 8 * s4);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t af[4] = {w0[2 * u], w1[2 * u], w0[2 * u + 1], w1[2 * u + 1]};
        mma16816<true>(sacc2[u % NCH], af, qf[s4 + u][0], qf[s4 + u][1]);
      }
    }
  } else if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
    constexpr int SEGB = D / 8;          // bytes of the lane segment; a word = two k-steps
    constexpr int NW = SEGB / 4;
    uint32_t w0[NW], w1[NW];
    load_seg<SEGB>(w0, kt, r0 * RB + lt * SEGB, true);
    load_seg<SEGB>(w1, kt, r1 * RB + lt * SEGB, true);
#pragma unroll
    for (int s = 0; s < KSTEPS; ++s) {
      // k-slots 0, 1: nibbles 2(s&1) and 4 + 2(s&1) of the word; k-slots 2, 3:
      // the next ones, read 16x (q carries the 1/16 for them)
      const uint32_t x0 = (s & 1) ? (w0[s >> 1] >> 8) : w0[s >> 1];
      const uint32_t x1 = (s & 1) ? (w1[s >> 1] >> 8) : w1[s >> 1];
      const uint32_t af[4] = {nib2_f16x2<0>(x0), nib2_f16x2<0>(x1), nib2_f16x2<1>(x0),
                              nib2_f16x2<1>(x1)};
      mma16816<false>(sacc2[s % NCH], af, qf[s][0], qf[s][1]);
    }
  } else {
#pragma unroll
    for (int s4 = 0; s4 < KSTEPS; s4 += 4) {
      uint32_t w0[4], w1[4];
      lds<4>(w0, kt, r0 * RB + lt * (D / 4) + 4 * s4);
      lds<4>(w1, kt, r1 * RB + lt * (D / 4) + 4 * s4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t af[4];
        e4m3x4_f16(w0[u], af[0], af[2]);
        e4m3x4_f16(w1[u], af[1], af[3]);
        mma16816<false>(sacc2[u % NCH], af, qf[s4 + u][0], qf[s4 + u][1]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float v = sacc2[0][e];
    if constexpr (NCH == 2) v += sacc2[NCH - 1][e];
    sacc_out[e] += v;
  }
}

// PV of one 16-position sub-tile: acc[n][i] (rows d, columns) += V^T . P'.
// The lane reads its d-segment of positions 2lt, 2lt+1, 2lt+8, 2lt+9; with
// WHOLE false, positions outside [lo, L) are zeroed (their bytes may be
// anything).
template <int MODE, int D, int NT, bool WHOLE>
__device__ __forceinline__ void pv_tile(float (*acc)[D / 16][4], const uint8_t* vt, int lg,
                                        int lt, const uint32_t (*pb)[2], int pos0, int lo, int L) {
  constexpr int RB = row_bytes<MODE>(D);
  constexpr int SEG = (MODE == BF16) ? D / 4 : (MODE == INT4_PER_TOKEN_HEAD ? D / 16 : D / 8);
  constexpr int SW = SEG / 4;
  constexpr bool BF = (MODE == BF16);
  const int ta = 2 * lt, tb = 2 * lt + 1, tc = 2 * lt + 8, td = 2 * lt + 9;
  bool va = true, vb = true, vc = true, vd = true;
  if constexpr (!WHOLE) {
    va = pos0 + ta >= lo && pos0 + ta < L;
    vb = pos0 + tb >= lo && pos0 + tb < L;
    vc = pos0 + tc >= lo && pos0 + tc < L;
    vd = pos0 + td >= lo && pos0 + td < L;
  }
  // With 64-byte rows two positions share a 128-byte swizzle row, and if
  // every lane read its even position first, half of the banks would serve
  // each load twice.  Lanes with bit 1 of lg set read the odd position of
  // each pair first (wa <-> wb, wc <-> wd) and select its bytes back with a
  // swapped byte permutation, so each load touches all 32 banks once.
  const bool sw = (RB == 64) && ((lg >> 1) & 1);
  uint32_t wa[SW], wb[SW], wc[SW], wd[SW];
  const int seg0 = lg * SEG;
  load_seg<SEG>(wa, vt, (sw ? tb : ta) * RB + seg0, sw ? vb : va);
  load_seg<SEG>(wb, vt, (sw ? ta : tb) * RB + seg0, sw ? va : vb);
  load_seg<SEG>(wc, vt, (sw ? td : tc) * RB + seg0, sw ? vd : vc);
  load_seg<SEG>(wd, vt, (sw ? tc : td) * RB + seg0, sw ? vc : vd);
#pragma unroll
  for (int i = 0; i < D / 16; ++i) {
    uint32_t af[4];
    if constexpr (MODE == BF16) {
      // elements 2i and 2i+1 of each position's segment = word i
      af[0] = __byte_perm(wa[i], wb[i], 0x5410);
      af[1] = __byte_perm(wa[i], wb[i], 0x7632);
      af[2] = __byte_perm(wc[i], wd[i], 0x5410);
      af[3] = __byte_perm(wc[i], wd[i], 0x7632);
    } else if constexpr (MODE == INT4_PER_TOKEN_HEAD) {
      // byte i of the segment: low nibble = d 2i, high nibble = d 2i+1; the
      // high nibbles (rows lg + 8: odd d) are read 16x and scaled back in
      // the epilogue
      const int wi = i >> 2, k = i & 3;
      const uint32_t sel = sw ? (uint32_t)((4 + k) | ((4 + k) << 4) | (k << 8) | (k << 12))
                              : (uint32_t)(k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12));
      const uint32_t x = __byte_perm(wa[wi], wb[wi], sel);
      const uint32_t y = __byte_perm(wc[wi], wd[wi], sel);
      af[0] = nib2_f16x2<0>(x);
      af[1] = nib2_f16x2<1>(x);
      af[2] = nib2_f16x2<0>(y);
      af[3] = nib2_f16x2<1>(y);
    } else {
      // bytes 2i, 2i+1 of each position's segment
      const int wi = i >> 1;
      const uint32_t sel = (i & 1) ? (sw ? 0x3726u : 0x7362u) : (sw ? 0x1504u : 0x5140u);
      e4m3x4_f16(__byte_perm(wa[wi], wb[wi], sel), af[0], af[1]);
      e4m3x4_f16(__byte_perm(wc[wi], wd[wi], sel), af[2], af[3]);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) mma16816<BF>(acc[n][i], af, pb[n][0], pb[n][1]);
  }
}

// ------------------------------------------------------------------ kernel
template <int MODE, int D>
struct Cfg {
  static constexpr int RB = row_bytes<MODE>(D);
  static constexpr int TB = TILE * RB;                       // tile bytes
  static constexpr int TBP = (TB + 1023) / 1024 * 1024;      // padded to 1024
  static constexpr bool DYN = (MODE == FP8_PER_TOKEN_HEAD || MODE == INT4_PER_TOKEN_HEAD);
  static constexpr bool BF = (MODE == BF16);
  static constexpr int STAGE = 2 * TBP;                      // K + V code tiles
  static constexpr int SCALES = DYN ? 128 : 0;               // K + V scales per stage
  static constexpr int KSTEPS = D / 16;
  static constexpr int MTILES = D / 16;
};

// Resident CTAs per SM the register budget is sized for: four (16 warps,
// <= 128 registers) where the accumulators fit without spilling, three
// (<= 168) for the eight-column split of GQA-8 at D = 128, else two.
template <int MODE, int D, int G>
struct MinCtas {
  static constexpr int value =
      (D == 256 || (MODE == BF16 && G >= 4)) ? 2 : ((G == 8 && D >= 128) ? 3 : 4);
};

// Shared memory: the warps' rings first (1024-aligned stages for the
// swizzled copies), then per warp its scale slots, q staging and barriers.
template <int MODE, int D, int G>
struct Layout {
  using C = Cfg<MODE, D>;
  static constexpr int q = G * D * 2;
  static constexpr int aux_of(int ns) { return (ns * C::SCALES + q + ns * 8 + 127) / 128 * 128; }
  static constexpr int warp_bytes(int ns) { return ns * C::STAGE + aux_of(ns); }
  // Ring depth: two stages (one tile in flight per warp while one is
  // computed keeps ~64 KB in flight per SM, enough for the copy bandwidth;
  // deeper rings measured slower), three for the 4 KB tiles of quantized
  // D = 256 layers; fewer if MinCtas CTAs would not share the SM's 228 KB
  // (1 KB per CTA is reserved by the system, 1 KB of each CTA's is alignment
  // slack).
  static constexpr int budget = 233472 / MinCtas<MODE, D, G>::value - 2048;
  static constexpr int fit(int ns) {
    return (ns > 2 && WARPS * warp_bytes(ns) > budget) ? fit(ns - 1) : ns;
  }
#ifdef KVQ_NS
  static constexpr int NS = KVQ_NS < 2 ? 2 : KVQ_NS;
#else
  static constexpr int NS = fit((D == 256 && MODE != BF16) ? 3 : 2);
#endif
  static constexpr int ring = NS * C::STAGE;
  static constexpr int scales = NS * C::SCALES;
  static constexpr int aux = aux_of(NS);
  static constexpr int total = WARPS * (ring + aux) + 1024;   // + alignment slack
};

// Position of one warp's cursor in the tile list.
struct Cursor {
  int b, g, k;      // sequence, KV head, tile within the item
  int n, t0;        // tiles of the item, first tile index (position / 16)
};

// Positions of sequence b that are read: its context length, at least 0 and
// at most the positions its block-table row covers (a longer context is an
// index error: check_len flags it, and only the covered positions are read).
__device__ __forceinline__ int ctx_len(const DecodeArgs& a, int b) {
  const int L = a.context_lens[b];
  const long long cap = (long long)a.max_blocks << a.bs_shift;
  return L < 0 ? 0 : ((long long)L > cap ? (int)cap : L);
}

__device__ __forceinline__ void check_len(const DecodeArgs& a, int b) {
  const int L = a.context_lens[b];
  if (L < 0 || (long long)L > ((long long)a.max_blocks << a.bs_shift))
    atomicOr(a.err, ERR_BAD_INDEX);
}

__device__ __forceinline__ int seq_tiles(const DecodeArgs& a, int b, int* t0) {
  const int L = ctx_len(a, b);
  const int lo = (a.window > 0 && L > a.window) ? L - a.window : 0;
  *t0 = lo / TILE;
  return L > 0 ? (L + TILE - 1) / TILE - lo / TILE : 0;
}

// Total tiles T (all lanes get it) and, if `find` >= 0, the cursor at tile
// `find`.  Sequences are scanned 32 at a time with a warp prefix sum.
__device__ long long scan_tiles(const DecodeArgs& a, long long find, Cursor* cur, int lane) {
  long long base = 0;             // tiles before the current chunk of sequences
  bool found = false;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    const int b = b0 + lane;
    int t0 = 0, n = 0;
    if (b < a.B) {
      check_len(a, b);
      n = seq_tiles(a, b, &t0);
    }
    long long incl = (long long)n * a.Hkv;       // inclusive prefix within the chunk
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const long long excl = incl - (long long)n * a.Hkv;
    if (!found && find >= 0) {
      const bool here = b < a.B && n > 0 && find >= base + excl && find < base + incl;
      const unsigned m = __ballot_sync(0xffffffffu, here);
      if (m) {
        const int src = __ffs(m) - 1;
        const long long off = __shfl_sync(0xffffffffu, find - base - excl, src);
        const int nn = __shfl_sync(0xffffffffu, n, src);
        cur->b = b0 + src;
        cur->n = nn;
        cur->t0 = __shfl_sync(0xffffffffu, t0, src);
        cur->g = (int)(off / nn);
        cur->k = (int)(off % nn);
        found = true;
      }
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return base;
}

// Total tiles T, this warp's share [my0, my1) and the cursor at my0.  For
// B <= 128 one round of context-length loads (four sequences per lane) serves
// both; larger batches scan twice.  Returns the share's tile count.
__device__ int locate(const DecodeArgs& a, int wid, Cursor* cur, int lane) {
  long long T, my0, my1;
  if (a.B > 128) {
    T = scan_tiles(a, -1, cur, lane);
    my0 = (long long)wid * T / a.workers;
    my1 = (long long)(wid + 1) * T / a.workers;
    if (my1 <= my0) return 0;
    scan_tiles(a, my0, cur, lane);
    return (int)(my1 - my0);
  }
  int n[4], t0[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = 32 * i + lane;
    n[i] = t0[i] = 0;
    if (b < a.B) {
      check_len(a, b);
      n[i] = seq_tiles(a, b, &t0[i]);
    }
  }
  long long incl[4], base[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) incl[i] = (long long)n[i] * a.Hkv;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const long long v = __shfl_up_sync(0xffffffffu, incl[i], o);
      if (lane >= o) incl[i] += v;
    }
  }
  base[0] = 0;
#pragma unroll
  for (int i = 1; i < 4; ++i) base[i] = base[i - 1] + __shfl_sync(0xffffffffu, incl[i - 1], 31);
  T = base[3] + __shfl_sync(0xffffffffu, incl[3], 31);
  my0 = (long long)wid * T / a.workers;
  my1 = (long long)(wid + 1) * T / a.workers;
  if (my1 <= my0) return 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long excl = incl[i] - (long long)n[i] * a.Hkv;
    const bool here = n[i] > 0 && my0 >= base[i] + excl && my0 < base[i] + incl[i];
    const unsigned m = __ballot_sync(0xffffffffu, here);
    if (m) {
      const int src = __ffs(m) - 1;
      const long long off = __shfl_sync(0xffffffffu, my0 - base[i] - excl, src);
      const int nn = __shfl_sync(0xffffffffu, n[i], src);
      cur->b = 32 * i + src;
      cur->n = nn;
      cur->t0 = __shfl_sync(0xffffffffu, t0[i], src);
      cur->g = (int)(off / nn);
      cur->k = (int)(off % nn);
      break;
    }
  }
  return (int)(my1 - my0);
}

// Worker 0: item tile offsets P_i (i = b*Hkv + g; P_{B*Hkv} = T) for the
// merge, and zeros for the output of every sequence with no retained position.
template <int G, int D>
__device__ void publish_items(const DecodeArgs& a, int lane) {
  long long base = 0;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    const int b = b0 + lane;
    int t0 = 0, n = 0;
    if (b < a.B) n = seq_tiles(a, b, &t0);
    long long incl = (long long)n * a.Hkv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (b < a.B) {
      const long long first = base + incl - (long long)n * a.Hkv;
      if (a.item_tiles)
        for (int g = 0; g < a.Hkv; ++g) a.item_tiles[(long long)b * a.Hkv + g] = first + (long long)g * n;
      if (n == 0) {
        if (a.out_bf16) {
          uint4* o = reinterpret_cast<uint4*>(a.out_bf16 + (long long)b * a.Hq * D);
          for (int i = 0; i < a.Hq * D / 8; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
        } else {
          float4* o = reinterpret_cast<float4*>(a.out + (long long)b * a.Hq * D);
          for (int i = 0; i < a.Hq * D / 4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0 && a.item_tiles) a.item_tiles[(long long)a.B * a.Hkv] = base;
}

__device__ __forceinline__ void advance(const DecodeArgs& a, Cursor& c) {
  if (++c.k < c.n) return;
  c.k = 0;
  if (++c.g < a.Hkv) return;
  c.g = 0;
  do {
    if (++c.b >= a.B) { c.n = 0; return; }
    c.n = seq_tiles(a, c.b, &c.t0);
  } while (c.n == 0);
}

template <int MODE, int D, int G>
__global__ void __launch_bounds__(WARPS * 32, MinCtas<MODE, D, G>::value)
    decode_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
  using C = Cfg<MODE, D>;
  using LY = Layout<MODE, D, G>;
  constexpr int NS = LY::NS;
  constexpr int NPART = C::BF ? 3 : 2;                       // terms of the P' split
  constexpr bool PACKED = G * NPART <= 8;                    // all terms in one PV tile
  constexpr int NT = PACKED ? 1 : NPART;                     // PV column tiles
  // QK columns that carry scores.  PACKED: column c holds head c % G, and its
  // weight feeds term c / G of the split, so the QK and PV columns coincide.
  constexpr int NCOL = PACKED ? G * NPART : G;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lg = lane >> 2, lt = lane & 3;       // fragment row group / column pair
  const int wid = blockIdx.x * WARPS + warp;
  // the merge kernel may be scheduled now; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (wid >= a.workers) return;                  // no CTA-wide barrier anywhere below

  uint8_t* wcodes = smem + warp * LY::ring;
  uint8_t* waux = smem + WARPS * LY::ring + warp * LY::aux;
  float* wscales = reinterpret_cast<float*>(waux);
  uint16_t* qst = reinterpret_cast<uint16_t*>(waux + LY::scales);
  uint64_t* wbars = reinterpret_cast<uint64_t*>(waux + LY::scales + LY::q);

  // ---- this warp's share of the tile list
  Cursor cc;
  cc.b = cc.g = cc.k = cc.n = cc.t0 = 0;
  const int ntiles = locate(a, wid, &cc, lane);
  if (wid == 0) publish_items<G, D>(a, lane);
  if (ntiles <= 0) return;
  Cursor cp = cc;                                 // producer cursor, NS tiles ahead

  if (lane < NS) mbar_init(&wbars[lane], 1);
  mbar_init_fence();
  __syncwarp();

  const uint64_t l2_policy = l2_copy_policy(a.stream_once != 0);
  unsigned valid_mask = 0;        // bit s: stage s holds a fetched tile
  int pst = 0;                    // stage the next issued tile goes to
  // Block id of the producer cursor's tile, loaded one issue ahead so that its
  // latency is spent on the previous tile's compute.
  auto block_of = [&](const Cursor& p) -> int {
    if (p.n == 0) return -1;      // past the end of the list
    const int pos0 = (p.t0 + p.k) * TILE;
    return __ldg(a.block_table + (long long)p.b * a.max_blocks + (pos0 >> a.bs_shift));
  };
  // Copies of the next tile (cursor p, block id blk) into stage pst.  Cell
  // indices fit in 32 bits (the host refuses caches of 2^31 cells or more).
  auto issue = [&](const Cursor& p, const int blk) {
    const int st = pst;
    pst = (pst + 1 == NS) ? 0 : pst + 1;
    const int pos0 = (p.t0 + p.k) * TILE;
    if (blk >= 0 && blk < a.num_blocks) {
      // every lane holds the same block id and cursor: any one lane issues
      if (elect_one()) {
        const unsigned cell = ((unsigned)blk * (unsigned)a.Hkv + (unsigned)p.g) * (unsigned)a.bs +
                              (unsigned)(pos0 & (a.bs - 1));
        const int row = (int)(((unsigned long long)cell * C::RB) >> 7);
        uint64_t* bar = &wbars[st];
        mbar_expect_tx(bar, 2 * C::TB + C::SCALES);
        uint8_t* kd = wcodes + st * C::STAGE;
        // a layer whose pages cannot stay in L2 streams them evict-first
        tma_tile_2d_hint(kd, &kmap, 0, row, bar, l2_policy);
        tma_tile_2d_hint(kd + C::TBP, &vmap, 0, row, bar, l2_policy);
        if constexpr (C::DYN) {
          bulk_copy(wscales + st * 32, a.k_cs + cell, 64, bar);
          bulk_copy(wscales + st * 32 + 16, a.v_cs + cell, 64, bar);
        }
      }
      valid_mask |= 1u << st;
    } else {
      // nothing is fetched, but the stage's phase must still complete so
      // that the parity of its later uses stays in step
      if (lane == 0) {
        atomicOr(a.err, ERR_BAD_INDEX);
        mbar_arrive(&wbars[st]);
      }
      valid_mask &= ~(1u << st);
    }
  };
  {
    // block ids of the first NS tiles in one round of loads while they lie in
    // the starting item (lane j: tile j)
    int blk0 = -1;
    if (lane < NS && cc.k + lane < cc.n)
      blk0 = __ldg(a.block_table + (long long)cc.b * a.max_blocks +
                   (((cc.t0 + cc.k + lane) * TILE) >> a.bs_shift));
    for (int j = 0; j < NS && j < ntiles; ++j) {
      const int bj = __shfl_sync(0xffffffffu, blk0, j);
      const bool same = cp.b == cc.b && cp.g == cc.g && cp.k == cc.k + j;
      issue(cp, same ? bj : block_of(cp));
      advance(a, cp);
    }
  }
  int blk_next = block_of(cp);

  float ks_static = 1.f, vs_static = 1.f;
  if constexpr (MODE == FP8_PER_TENSOR) { ks_static = a.k_scale[0]; vs_static = a.v_scale[0]; }
  // (per-head scales are read per segment below)

  // ---- per-segment state
  uint32_t qf[C::KSTEPS][2];
  float s_fac = 0.f;
  float m_run[2], l_run[2];
  float m_ref[2] = {0.f, 0.f};    // m_run, or 0 while it is -inf (every score so far -inf)
  float acc[NT][C::MTILES][4];
  int vexp = -1000;               // running max exponent of the V scales (dynamic)
  float fv = 0.f;                 // 2^(KP - vexp)
  float vcap = 0.f;               // 2^(vexp + 1): a V scale at or above it raises vexp
  float qc[2] = {1.f, 1.f};       // per-column query scale (FP8 query, per-head scales)
  float sq[2] = {0.f, 0.f};       // score factor of each column: s_fac x qc
  int seg_b = -1, seg_g = -1, seg_k0 = 0, seg_klast = 0, seg_n = 0;

  // Writes the segment's result: final output if it covered the whole item,
  // else a partial at slot (item + worker) for the merge.
  auto finalize = [&]() {
    float vsg = vs_static;
    if constexpr (MODE == FP8_PER_HEAD) vsg = a.v_scale[seg_g];
    // reduce l over the row groups (m is already uniform across them)
    float l_tot[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v = l_run[c];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      l_tot[c] = v;
    }
    // fold the split terms onto the lanes that own head columns
    float o[C::MTILES][4];
#pragma unroll
    for (int i = 0; i < C::MTILES; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = 0.f;
#pragma unroll
        for (int n = 0; n < NT; ++n) v += acc[n][i][e];
        if constexpr (PACKED && G >= 2) {
#pragma unroll
          for (int k = 1; k < NPART; ++k) v += __shfl_down_sync(0xffffffffu, v, k * (G / 2));
        }
        o[i][e] = v;
      }
    if constexpr (PACKED && G == 1) {
      // head 0: columns 0 and 1 in lane column 0, column 2 (bf16) in lane column 1
#pragma unroll
      for (int i = 0; i < C::MTILES; ++i) {
        const float x0 = (C::BF) ? __shfl_down_sync(0xffffffffu, o[i][0], 1) : 0.f;
        const float x2 = (C::BF) ? __shfl_down_sync(0xffffffffu, o[i][2], 1) : 0.f;
        o[i][0] += o[i][1] + x0;
        o[i][2] += o[i][3] + x2;
      }
    }
    float unscale;
    if constexpr (C::BF) unscale = 1.f;
    else if constexpr (C::DYN) unscale = pow2i(vexp - KP);
    else unscale = vsg * (1.f / PSTATIC);
    const int nh = (G == 1) ? 1 : 2;              // heads owned by this lane column
    const bool owner = (G == 1) ? (lt == 0) : (2 * lt < G);
    const bool full = (seg_k0 == 0 && seg_klast == seg_n - 1);
    const int item = seg_b * a.Hkv + seg_g;
    if (owner) {
#pragma unroll
      for (int e1 = 0; e1 < 2; ++e1) {
        if (e1 >= nh) break;
        const int h = (G == 1) ? 0 : 2 * lt + e1;
        const float l = l_tot[e1];
        const float f = full ? (l > 0.f ? unscale / l : 0.f) : unscale;
        const long long orow = ((long long)seg_b * a.Hq + seg_g * G + h) * D;
        float* dst = full ? a.out + orow : a.ws_o + (((long long)(item + wid) * G + h) * D);
        // INT4: the odd-d rows were accumulated 16x (see pv_tile)
        const float f_odd = (MODE == INT4_PER_TOKEN_HEAD) ? f * 0.0625f : f;
        if (full && a.out_bf16) {
#pragma unroll
          for (int i = 0; i < C::MTILES; ++i) {
            const int d = lg * (D / 8) + 2 * i;
            *reinterpret_cast<uint32_t*>(a.out_bf16 + orow + d) =
                pack_bf16x2(o[i][e1] * f, o[i][2 + e1] * f_odd);
          }
        } else {
#pragma unroll
          for (int i = 0; i < C::MTILES; ++i) {
            const int d = lg * (D / 8) + 2 * i;
            *reinterpret_cast<float2*>(dst + d) = make_float2(o[i][e1] * f, o[i][2 + e1] * f_odd);
          }
        }
        if (!full && lg == 0) {
          float* ml = a.ws_ml + 2 * ((long long)(item + wid) * G + h);
          ml[0] = m_run[e1];
          ml[1] = l;
        }
      }
    }
  };

  int fail_at = -1;
  int L = 0, lo = 0;              // the current item's context length and window start
  int j = 0;
  int cst = 0;                    // stage of tile j
  uint32_t cpar = 0;              // phase parity of stage cst for tile j
  while (j < ntiles) {
    // ---------------- segment boundary: finish the previous item, start the next
    if (cc.b != seg_b || cc.g != seg_g) {
      if (seg_b >= 0) finalize();
      seg_b = cc.b;
      seg_g = cc.g;
      seg_k0 = cc.k;
      seg_n = cc.n;
      L = ctx_len(a, seg_b);
      lo = (a.window > 0 && L > a.window) ? L - a.window : 0;
      __syncwarp();
      // q of this item -> staging -> power-of-two prescale -> f16 B fragments
      const uint4* qsrc =
          reinterpret_cast<const uint4*>(a.q + ((long long)seg_b * a.Hq + seg_g * G) * D);
      float amax = 0.f;
      for (int i = lane; i < G * D / 8; i += 32) {
        const uint4 v = qsrc[i];
        reinterpret_cast<uint4*>(qst)[i] = v;
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w4[e] << 16)),
                                   fabsf(__uint_as_float(w4[e] & 0xFFFF0000u))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      __syncwarp();
      int qexp = 0;                   // q is scaled by 2^(14 - qexp) for f16
      if (!C::BF && amax > 0.f && !a.q_scale)
        qexp = max(((int)(__float_as_uint(amax) >> 23) & 0xFF) - 127, -100);
      const float qmul = (C::BF || a.q_scale) ? 1.f : pow2i(14 - qexp);
      float ks = ks_static;
      if constexpr (MODE == FP8_PER_HEAD) ks = a.k_scale[seg_g];
      s_fac = a.qk_scale * ks * ((C::BF || a.q_scale) ? 1.f : pow2i(qexp - 14));
      // FP8 query: every element becomes the E4M3 value of RN32(q / q_scale)
      // (exact in f16 and bf16) and q_scale multiplies the score: a single
      // scale folds into s_fac, per-head scales into the column factors qc
      float qs_col = 1.f;             // scale of this lane's staged column (lg)
      if (a.q_scale) {
        const bool per_head = a.q_scale_count > 1;
        if (!per_head) s_fac *= a.q_scale[0];
        qs_col = a.q_scale[per_head ? seg_g * G + (lg % G) : 0];
#pragma unroll
        for (int e = 0; e < 2; ++e) qc[e] = per_head ? a.q_scale[seg_g * G + ((2 * lt + e) % G)] : 1.f;
      }
#pragma unroll
      for (int s = 0; s < C::KSTEPS; ++s) {
        float v[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float x = (lg < NCOL)
                        ? __uint_as_float((uint32_t)qst[(lg % G) * D + qk_d<MODE, D>(lt, s, jj)] << 16)
                        : 0.f;
          if (a.q_scale) x = e4m3_round(__fdiv_rn(x, qs_col));
          v[jj] = x * ((MODE == INT4_PER_TOKEN_HEAD && jj >= 2) ? qmul * 0.0625f : qmul);
        }
        if constexpr (C::BF) {
          qf[s][0] = pack_bf16x2(v[0], v[1]);
          qf[s][1] = pack_bf16x2(v[2], v[3]);
        } else {
          qf[s][0] = pack_f16x2(v[0], v[1]);
          qf[s][1] = pack_f16x2(v[2], v[3]);
        }
      }
      sq[0] = s_fac * qc[0];
      sq[1] = s_fac * qc[1];
      m_run[0] = m_run[1] = -INFINITY;
      m_ref[0] = m_ref[1] = 0.f;
      l_run[0] = l_run[1] = 0.f;
      vexp = -1000;
      fv = 0.f;
      vcap = 0.f;
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < C::MTILES; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[n][i][e] = 0.f;
    }

    // ---------------- this iteration: tile j
    const int pos0 = (cc.t0 + cc.k) * TILE;
    const bool ok = (valid_mask >> cst) & 1u;
    const uint8_t* kt = wcodes + cst * C::STAGE;
    const float* ksc = wscales + cst * 32;
    if (ok && !mbar_wait(&wbars[cst], cpar)) {
      fail_at = j;
      break;
    }
    // whole: every position of the tile is retained, so nothing is masked
    const bool whole = ok && pos0 >= lo && pos0 + TILE <= L;

    // ---------------- QK: rows lg, lg+8
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) qk_tile<MODE, D>(sacc, kt, lg, lt, qf);

    // ---------------- scores (log2 units); masked entries are -inf
    // score factor of each accumulator element: the row's K scale (dynamic)
    // times the column factor, formed apart from the QK result so it stays
    // off its dependency chain
    float kq[4] = {sq[0], sq[1], sq[0], sq[1]};
    float vs0 = 1.f, vs1 = 1.f;           // V scales of rows lg, lg + 8 (dynamic)
    bool vraise = false;                  // a retained row's V scale reaches 2^(vexp + 1)
    if constexpr (C::DYN) {
      if (ok) {
        const float k0 = ksc[lg], k1 = ksc[lg + 8];
        kq[0] = k0 * sq[0]; kq[1] = k0 * sq[1]; kq[2] = k1 * sq[0]; kq[3] = k1 * sq[1];
        vs0 = ksc[16 + lg];
        vs1 = ksc[16 + lg + 8];
        // rows outside [lo, L) may hold anything: only retained rows count
        const int p0 = pos0 + lg, p1 = p0 + 8;
        vraise = ((whole || (p0 >= lo && p0 < L)) && vs0 >= vcap) ||
                 ((whole || (p1 >= lo && p1 < L)) && vs1 >= vcap);
      }
    }
    float s_raw[4];
    if (whole && NCOL == 8) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s_raw[e] = sacc[e] * kq[e];
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pos = pos0 + lg + ((e & 2) ? 8 : 0);
        const bool v = ok && (whole || (pos >= lo && pos < L)) && (2 * lt + (e & 1)) < NCOL;
        s_raw[e] = v ? sacc[e] * kq[e] : -INFINITY;
      }
    }

    // ---------------- online softmax.  The reference max m_run (per column,
    // warp-uniform) moves only when some lane holds a score above it by more
    // than LAZY, and the V-scale exponent vexp only when a retained V scale
    // reaches 2^(vexp + 1); only then are they reduced over the warp and O
    // and l rescaled, so most tiles take no shuffle here.
    const float lmax[2] = {fmaxf(s_raw[0], s_raw[2]), fmaxf(s_raw[1], s_raw[3])};
    const bool raise = lmax[0] > m_run[0] + LAZY || lmax[1] > m_run[1] + LAZY || vraise;
    if (__any_sync(0xffffffffu, raise)) {
      float al[2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float mt = lmax[c];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
        const float mn = fmaxf(m_run[c], mt);
        al[c] = (mn == -INFINITY) ? 1.f : ex2(m_run[c] - mn);   // 0 while m_run is -inf
        l_run[c] *= al[c];
        m_run[c] = mn;
        m_ref[c] = (mn == -INFINITY) ? 0.f : mn;
      }
      if constexpr (C::DYN) {
        int et = -1000;                 // largest V-scale exponent of the retained rows
        if (ok) {
          const int p0 = pos0 + lg, p1 = p0 + 8;
          if (whole || (p0 >= lo && p0 < L)) et = f32_exp(vs0);
          if (whole || (p1 >= lo && p1 < L)) et = max(et, f32_exp(vs1));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) et = max(et, __shfl_xor_sync(0xffffffffu, et, o));
        const int vnew = max(vexp, max(et, -100));
        if (vnew != vexp) {
          const float vfix = pow2i(vexp - vnew);     // 0 on the first tile (O is 0)
          al[0] *= vfix;
          al[1] *= vfix;
          vexp = vnew;
          fv = pow2i(KP - vexp);
          vcap = pow2i(vexp + 1);
        }
      }
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < C::MTILES; ++i) {
          acc[n][i][0] *= al[0];
          acc[n][i][1] *= al[1];
          acc[n][i][2] *= al[0];
          acc[n][i][3] *= al[1];
        }
    }
    float pw[4];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      pw[c] = ex2(s_raw[c] - m_ref[c]);
      pw[c + 2] = ex2(s_raw[c + 2] - m_ref[c]);
      l_run[c] += pw[c] + pw[c + 2];
    }
    // weights that meet V: P' = p v_scale 2^(KP - vexp) (dynamic), p 64 (FP8)
    if constexpr (C::DYN) {
      const float f0 = vs0 * fv, f1 = vs1 * fv;
      pw[0] *= f0; pw[1] *= f0; pw[2] *= f1; pw[3] *= f1;
    } else if constexpr (!C::BF) {
#pragma unroll
      for (int e = 0; e < 4; ++e) pw[e] *= PSTATIC;
    }

    // ---------------- PV
    if (ok) {
      const float* pr = pw;
      uint32_t pb[NT][2];
      if constexpr (C::BF) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          float x[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 2 * lt + (e & 1);
            const int k = PACKED ? c / G : n;
            const bool live = PACKED ? (k < NPART) : (c < G);
            x[e] = live ? split_term<true>(pr[e], k) : 0.f;
          }
          pb[n][0] = movmatrix_t(pack_bf16x2(x[0], x[1]));   // positions 0..7
          pb[n][1] = movmatrix_t(pack_bf16x2(x[2], x[3]));   // positions 8..15
        }
      } else {
        // f16 hi + lo: the hi pairs are packed once, the lo pairs are the
        // remainders of their unpacked values
        const uint32_t h01 = pack_f16x2(pr[0], pr[1]), h23 = pack_f16x2(pr[2], pr[3]);
        const uint32_t l01 = pack_f16x2(pr[0] - f16_lo(h01), pr[1] - f16_hi(h01));
        const uint32_t l23 = pack_f16x2(pr[2] - f16_lo(h23), pr[3] - f16_hi(h23));
        if constexpr (PACKED) {
          // column c carries term c / G of head c % G: lanes whose two
          // columns are hi columns take the hi pair, the next G columns the
          // lo pair, dead columns zero (G = 1: column 0 hi, column 1 lo)
          uint32_t p01, p23;
          if constexpr (G == 1) {
            p01 = lt == 0 ? __byte_perm(h01, l01, 0x7610) : 0u;
            p23 = lt == 0 ? __byte_perm(h23, l23, 0x7610) : 0u;
          } else {
            const int k = (2 * lt) / G;
            p01 = k == 0 ? h01 : (k == 1 ? l01 : 0u);
            p23 = k == 0 ? h23 : (k == 1 ? l23 : 0u);
          }
          pb[0][0] = movmatrix_t(p01);
          pb[0][1] = movmatrix_t(p23);
        } else {
          // one column tile per term; columns past G are zero
          const bool live = 2 * lt < G;
          pb[0][0] = movmatrix_t(live ? h01 : 0u);
          pb[0][1] = movmatrix_t(live ? h23 : 0u);
          pb[NT - 1][0] = movmatrix_t(live ? l01 : 0u);
          pb[NT - 1][1] = movmatrix_t(live ? l23 : 0u);
        }
      }
      const uint8_t* vt = kt + C::TBP;
      if (whole) {
        pv_tile<MODE, D, NT, true>(acc, vt, lg, lt, pb, 0, 0, 0);
      } else {
        pv_tile<MODE, D, NT, false>(acc, vt, lg, lt, pb, pos0, lo, L);
      }
    }

    // ---------------- advance; refill the consumed stage
    seg_klast = cc.k;
    advance(a, cc);
    __syncwarp();
    if (j + NS < ntiles) {
      fence_proxy_async();
      issue(cp, blk_next);
      advance(a, cp);
      blk_next = block_of(cp);
    }
    ++j;
    if (++cst == NS) { cst = 0; cpar ^= 1u; }
  }

  if (fail_at >= 0) {
    // a wait ran out: flag it, then drain the copies this warp still has in
    // flight (tiles fail_at .. fail_at+NS-1), each wait bounded again
    if (lane == 0) atomicOr(a.err, ERR_TIMEOUT);
    for (int jj = fail_at, st = cst, par = (int)cpar; jj < ntiles && jj < fail_at + NS; ++jj) {
      if ((valid_mask >> st) & 1u) (void)mbar_wait(&wbars[st], (uint32_t)par);
      if (++st == NS) { st = 0; par ^= 1; }
    }
    return;
  }
  finalize();
}

// Log-sum-exp merge: one CTA per (sequence, KV head) item, one warp per query
// head of the group.  Items covered by one worker (or by none) were written by
// the decode kernel; the others combine the partials of their workers.  The
// partial rows of the first PRE workers are loaded together with the (m, l)
// pairs, so an item split over at most PRE workers costs two dependent rounds
// of loads after the item offsets.
template <int D, int G>
__global__ void __launch_bounds__(32 * G) merge_kernel(const DecodeArgs a) {
  // launched as a programmatic dependent of the decode kernel: wait until that
  // grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int PRE = 8;
  constexpr int DL = D / 32;                            // elements per lane
  const int item = blockIdx.x;
  const int j = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long P = a.item_tiles[item], n = a.item_tiles[item + 1] - P;
  const long long T = a.item_tiles[(long long)a.B * a.Hkv];
  if (n <= 0) return;
  const long long W = a.workers;
  const long long w0 = ((P + 1) * W - 1) / T;           // worker owning tile P
  const long long w1 = ((P + n) * W - 1) / T;           // worker owning tile P + n - 1
  if (w0 == w1) return;
  const int b = item / a.Hkv, g = item - b * a.Hkv;
  // a worker whose share is empty (more workers than tiles) wrote nothing, and
  // its slot may hold anything: such workers get weight 0 and are selected out
  auto live_w = [&](long long w) { return w <= w1 && (w * T) / W != ((w + 1) * T) / W; };
  auto row = [&](long long w) { return a.ws_o + ((item + w) * G + j) * D; };
  float pre[PRE][DL];
#pragma unroll
  for (int u = 0; u < PRE; ++u) {
    const long long w = (w0 + u <= w1) ? w0 + u : w0;
#pragma unroll
    for (int k = 0; k < DL; ++k) pre[u][k] = row(w)[lane + 32 * k];
  }
  float acc[DL];
#pragma unroll
  for (int k = 0; k < DL; ++k) acc[k] = 0.f;
  float M = -INFINITY, lsum = 0.f;
  // chunks of 32 workers: lane w-c0 holds that worker's (m, l)
  for (long long c0 = w0; c0 <= w1; c0 += 32) {
    const long long w = c0 + lane;
    float m = -INFINITY, l = 0.f;
    const bool live = live_w(w);
    const long long part = (item + w) * G + j;
    if (live) {
      m = a.ws_ml[2 * part];
      l = a.ws_ml[2 * part + 1];
    }
    float cm = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
    const float Mn = fmaxf(M, cm);
    const float rescale = (M == -INFINITY) ? 0.f : ex2(M - Mn);
    const float f = live ? ex2(m - Mn) : 0.f;
    float ls = f * l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    lsum = lsum * rescale + ls;
#pragma unroll
    for (int k = 0; k < DL; ++k) acc[k] *= rescale;
    const int cnt = (int)min(32LL, w1 - c0 + 1);
    int i0 = 0;
    if (c0 == w0) {
      // the prefetched rows
#pragma unroll
      for (int u = 0; u < PRE; ++u) {
        const float fu = (u < cnt) ? __shfl_sync(0xffffffffu, f, u) : 0.f;
#pragma unroll
        for (int k = 0; k < DL; ++k) acc[k] = fu != 0.f ? fmaf(fu, pre[u][k], acc[k]) : acc[k];
      }
      i0 = PRE;
    }
    for (; i0 < cnt; i0 += 4) {
      // four partials' loads in flight at once; missing ones read slot c0
      float v[4][DL], fi[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        fi[u] = __shfl_sync(0xffffffffu, f, (i0 + u) & 31);
        const long long ii = (i0 + u < cnt) ? i0 + u : 0;
        if (i0 + u >= cnt) fi[u] = 0.f;
#pragma unroll
        for (int k = 0; k < DL; ++k) v[u][k] = row(c0 + ii)[lane + 32 * k];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int k = 0; k < DL; ++k) acc[k] = fi[u] != 0.f ? fmaf(fi[u], v[u][k], acc[k]) : acc[k];
    }
    M = Mn;
  }
  const long long orow = ((long long)b * a.Hq + g * G + j) * D;
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  if (a.out_bf16) {
#pragma unroll
    for (int k = 0; k < DL; ++k)
      a.out_bf16[orow + lane + 32 * k] = (uint16_t)(pack_bf16x2(acc[k] * inv, 0.f) & 0xFFFFu);
  } else {
#pragma unroll
    for (int k = 0; k < DL; ++k) a.out[orow + lane + 32 * k] = acc[k] * inv;
  }
}

// ------------------------------------------------------------------ host
// Sets the kernel's dynamic shared-memory limit once per device; returns its
// resident CTAs per SM (0 on failure).
template <int MODE, int D, int G>
int prepare(int* smem_out) {
  using LY = Layout<MODE, D, G>;
  const int smem = LY::total;
  if (smem_out) *smem_out = smem;
  static int per_sm[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!per_sm[dev]) {
    auto kern = decode_kernel<MODE, D, G>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, WARPS * 32, smem) !=
            cudaSuccess || n <= 0)
      return 0;
    per_sm[dev] = n;
  }
  return per_sm[dev];
}

template <int MODE, int D, int G>
cudaError_t launch3(const DecodeArgs& a, cudaStream_t st) {
  using C = Cfg<MODE, D>;
  const long long total = a.num_blocks * a.Hkv * a.bs * (long long)C::RB;
  CUtensorMap km, vm;
  if (total > 0) {
    if (!make_tile_map(&km, a.k_cache, total, C::TB) || !make_tile_map(&vm, a.v_cache, total, C::TB))
      return cudaErrorInvalidValue;
  }
  int smem = 0;
  if (prepare<MODE, D, G>(&smem) <= 0) return cudaErrorInvalidConfiguration;
  const int ctas = (a.workers + WARPS - 1) / WARPS;
  decode_kernel<MODE, D, G><<<ctas, WARPS * 32, smem, st>>>(a, km, vm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.workers <= 1) return e;
  // programmatic dependent launch: the merge grid's launch overlaps the
  // decode grid's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * a.Hkv));
  cfg.blockDim = dim3(32 * G);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel<D, G>, a);
}

template <int MODE, int D, int G>
constexpr bool built() {
  return !(D == 256 && (G == 8 || (MODE == BF16 && G == 4)));
}

template <int MODE, int D>
int per_sm2(int G) {
  switch (G) {
    case 1: return prepare<MODE, D, 1>(nullptr);
    case 2: return prepare<MODE, D, 2>(nullptr);
    case 4:
      if constexpr (built<MODE, D, 4>()) return prepare<MODE, D, 4>(nullptr);
      else return 0;
    case 8:
      if constexpr (built<MODE, D, 8>()) return prepare<MODE, D, 8>(nullptr);
      else return 0;
    default: return 0;
  }
}

template <int MODE>
int per_sm1(int D, int G) {
  switch (D) {
    case 64: return per_sm2<MODE, 64>(G);
    case 128: return per_sm2<MODE, 128>(G);
    case 256: return per_sm2<MODE, 256>(G);
    default: return 0;
  }
}

template <int MODE, int D>
cudaError_t launch2(int G, const DecodeArgs& a, cudaStream_t st) {
  switch (G) {
    case 1: return launch3<MODE, D, 1>(a, st);
    case 2: return launch3<MODE, D, 2>(a, st);
    case 4:
      if constexpr (built<MODE, D, 4>()) return launch3<MODE, D, 4>(a, st);
      else return cudaErrorInvalidValue;
    case 8:
      if constexpr (built<MODE, D, 8>()) return launch3<MODE, D, 8>(a, st);
      else return cudaErrorInvalidValue;
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

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  }
  return fn;
}

// The layer's code buffer as a 2-D uint8 tensor of 128-byte rows; one box is
// a 16-position tile of one (block, KV head) page.
bool make_tile_map(CUtensorMap* m, const void* base, long long total_bytes, int tile_bytes) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)(total_bytes / 128)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, (cuuint32_t)(tile_bytes / 128)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int decode_ctas_per_sm(int mode, int D, int G) {
  switch (mode) {
    case BF16: return per_sm1<BF16>(D, G);
    case FP8_PER_TENSOR: return per_sm1<FP8_PER_TENSOR>(D, G);
    case FP8_PER_HEAD: return per_sm1<FP8_PER_HEAD>(D, G);
    case FP8_PER_TOKEN_HEAD: return per_sm1<FP8_PER_TOKEN_HEAD>(D, G);
    case INT4_PER_TOKEN_HEAD: return per_sm1<INT4_PER_TOKEN_HEAD>(D, G);
    default: return 0;
  }
}

int decode_warps_per_cta() { return WARPS; }

bool decode_supported(int mode, int D, int G) {
  if (!(mode >= BF16 && mode <= INT4_PER_TOKEN_HEAD)) return false;
  if (!(D == 64 || D == 128 || D == 256)) return false;
  if (!(G == 1 || G == 2 || G == 4 || G == 8)) return false;
  // the PV accumulators (D/16 tiles x 4 x column tiles) must fit in registers
  if (D == 256 && (G == 8 || (mode == BF16 && G == 4))) return false;
  return true;
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
