// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

enum Mode { BF16 = 0, FP8_PER_TENSOR = 1, FP8_PER_HEAD = 2, FP8_PER_TOKEN_HEAD = 3,
            INT4_PER_TOKEN_HEAD = 4 };

// Device error word bits.
enum : unsigned { ERR_BAD_INDEX = 1u, ERR_TIMEOUT = 2u };

struct WriteArgs {
  const uint16_t* k_new;       // bf16 bits
  const uint16_t* v_new;
  long long token_stride;      // elements between tokens
  const long long* slots;
  long long T;
  int Hkv;
  int bs;
  int bs_shift;                // log2(bs)
  long long num_blocks;
  const float* k_scale;        // static modes
  const float* v_scale;
  uint8_t* k_cache;
  uint8_t* v_cache;
  float* k_cs;                 // dynamic modes
  float* v_cs;
  unsigned* err;
};

struct DecodeArgs {
  const uint16_t* q;           // bf16 [B][Hq][D]
  const float* q_scale;        // FP8 query: [1] or [Hq] scales (nullptr: bf16 query)
  int q_scale_count;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;        // static modes: [1] or [Hkv]
  const float* v_scale;
  const float* k_cs;           // dynamic modes: [num_blocks][Hkv][bs]
  const float* v_cs;
  const int* block_table;      // [B][max_blocks]
  const int* context_lens;     // [B]
  float* out;                  // [B][Hq][D] fp32, or
  uint16_t* out_bf16;          // [B][Hq][D] bf16 (RN of the fp32 result) when non-null
  float* ws_o;                 // [B*Hkv + workers][G][D] unnormalised partial outputs
  float* ws_ml;                // [B*Hkv + workers][G][2] running max (log2 units) and sum
  long long* item_tiles;       // [B*Hkv + 1] first tile of each item in the tile list; T last
  unsigned* err;
  int B, Hq, Hkv, bs, bs_shift, max_blocks, window, workers;
  int stream_once;             // pages larger than L2: copy them evict-first
  long long num_blocks;
  float qk_scale;              // softmax_scale * log2(e)
};

// Launchers (return cudaGetLastError() of the launch).
cudaError_t launch_cache_write(int mode, int D, const WriteArgs& a, cudaStream_t st);
cudaError_t launch_calibrate(const uint16_t* x, long long T, int Hkv, int D, float qmax,
                             float* out, cudaStream_t st);
cudaError_t launch_e4m3_encode(const float* in, uint8_t* out, long long n, cudaStream_t st);
// One warp whose bounded barrier wait runs out after limit_cycles (sets TIMEOUT).
cudaError_t launch_wait_check(long long limit_cycles, cudaStream_t st);
// Returns cudaErrorInvalidValue for an unsupported (mode, D, G) combination.
cudaError_t launch_decode(int mode, int D, int G, const DecodeArgs& a, cudaStream_t st);
bool decode_supported(int mode, int D, int G);
// Prefill: one CTA per (query tile, sequence, KV head); DecodeArgs supplies the
// caches, scales, block table, context lengths, q and out (no workspace).
cudaError_t launch_prefill(int mode, int D, int G, const DecodeArgs& a, const int* query_start,
                           int max_query_len, cudaStream_t st);
// Warp-specialised prefill for quantized layers of head_dim 64 or 128.
bool prefill_ws_supports(int mode, int D);
cudaError_t launch_prefill_ws(int mode, int D, int G, const DecodeArgs& a, const int* query_start,
                              int max_query_len, cudaStream_t st);
int prefill_rows_per_cta();
// Resident decode CTAs per SM on the current device (0 if unknown: no device).
int decode_ctas_per_sm(int mode, int D, int G);
int decode_warps_per_cta();

// 2-D TMA map of a layer's code buffer viewed as [total_bytes / 128] rows of
// 128 bytes, box of tile_bytes / 128 rows, 128B swizzle (false on failure).
bool make_tile_map(CUtensorMap* m, const void* base, long long total_bytes, int tile_bytes);

// Device error word of the current device.
unsigned* error_word();

int sm_count();

}  // namespace kvq
