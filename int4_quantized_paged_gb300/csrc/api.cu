// C ABI of libkvq: argument validation, capacity accounting, split-K planning
// and dispatch to the kernels.  Everything here runs on the host.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>
#include <vector>

#include "kvq.h"
#include "kvq_internal.h"

struct kvq_ctx {
  kvq_config cfg;
  std::vector<int> mode;
  std::vector<int> window;
  float softmax_scale;
};

namespace kvq {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace kvq

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool is_dynamic(int mode) {
  return mode == KVQ_FP8_PER_TOKEN_HEAD || mode == KVQ_INT4_PER_TOKEN_HEAD;
}

double elem_bytes(int mode) {
  return mode == KVQ_BF16 ? 2.0 : (mode == KVQ_INT4_PER_TOKEN_HEAD ? 0.5 : 1.0);
}

long long row_bytes(int mode, int D) {
  return mode == KVQ_BF16 ? 2LL * D : (mode == KVQ_INT4_PER_TOKEN_HEAD ? D / 2 : D);
}

kvq_status check_layer(const kvq_ctx* ctx, int layer) {
  if (!ctx) return KVQ_ERR_INVALID_ARG;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

kvq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

// Worker warps for a decode call: enough to fill every SM at the kernel's
// occupancy, but no more than one per 4 tiles (64 positions) of work, so a
// worker always streams several tiles.
int auto_workers(long long batch, int Hkv, int positions, int per_sm) {
  const long long tiles = batch * Hkv * (((long long)positions + 15) / 16 + 1);
  const long long full = (long long)kvq::sm_count() * (per_sm > 0 ? per_sm : 2) *
                         kvq::decode_warps_per_cta();
  long long w = tiles / 4;
  if (w > full) w = full;
  if (w < 1) w = 1;
  return (int)w;
}

}  // namespace

extern "C" {

kvq_status kvq_create(const kvq_config* cfg, kvq_ctx** out) {
  if (!cfg || !out) return KVQ_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->num_layers <= 0 || cfg->num_q_heads <= 0 || cfg->num_kv_heads <= 0 ||
      cfg->head_dim <= 0 || cfg->block_size <= 0 || cfg->num_blocks < 0 || !cfg->layer_mode)
    return KVQ_ERR_INVALID_ARG;
  if (cfg->num_q_heads % cfg->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  const int G = cfg->num_q_heads / cfg->num_kv_heads;
  if (cfg->head_dim != 64 && cfg->head_dim != 128 && cfg->head_dim != 256)
    return KVQ_ERR_UNSUPPORTED;
  const int bs = cfg->block_size;
  if (bs != 16 && bs != 32 && bs != 64 && bs != 128) return KVQ_ERR_UNSUPPORTED;
  if (!(cfg->softmax_scale >= 0.f) || isinf(cfg->softmax_scale)) return KVQ_ERR_INVALID_ARG;
  // cache cells (block, KV head, slot) are indexed in 32 bits on the device
  if (cfg->num_blocks * (long long)cfg->num_kv_heads * bs >= (1LL << 31)) return KVQ_ERR_UNSUPPORTED;
  for (int l = 0; l < cfg->num_layers; ++l) {
    const int m = cfg->layer_mode[l];
    if (m < KVQ_BF16 || m > KVQ_INT4_PER_TOKEN_HEAD) return KVQ_ERR_INVALID_ARG;
    if (!kvq::decode_supported(m, cfg->head_dim, G)) return KVQ_ERR_UNSUPPORTED;
    // TMA addresses the code buffer in 128-byte rows with a signed 32-bit
    // coordinate
    if (cfg->num_blocks * (long long)cfg->num_kv_heads * bs * row_bytes(m, cfg->head_dim) / 128 >=
        (1LL << 31))
      return KVQ_ERR_UNSUPPORTED;
    if (cfg->layer_window && cfg->layer_window[l] < 0) return KVQ_ERR_INVALID_ARG;
  }
  kvq_ctx* c = new (std::nothrow) kvq_ctx;
  if (!c) return KVQ_ERR_INVALID_ARG;
  c->cfg = *cfg;
  try {  // no exception may cross the C ABI
    c->mode.assign(cfg->layer_mode, cfg->layer_mode + cfg->num_layers);
    if (cfg->layer_window)
      c->window.assign(cfg->layer_window, cfg->layer_window + cfg->num_layers);
    else
      c->window.assign(cfg->num_layers, 0);
  } catch (...) {
    delete c;
    return KVQ_ERR_INVALID_ARG;
  }
  c->cfg.layer_mode = c->mode.data();
  c->cfg.layer_window = c->window.data();
  c->softmax_scale =
      cfg->softmax_scale > 0.f ? cfg->softmax_scale : 1.0f / sqrtf((float)cfg->head_dim);
  *out = c;
  return KVQ_OK;
}

void kvq_destroy(kvq_ctx* ctx) { delete ctx; }

kvq_status kvq_layer_buffer_sizes(const kvq_ctx* ctx, int layer, size_t* code_bytes,
                                  size_t* scale_bytes) {
  kvq_status st = check_layer(ctx, layer);
  if (st != KVQ_OK) return st;
  const kvq_config& c = ctx->cfg;
  const int mode = ctx->mode[layer];
  const long long cells = c.num_blocks * c.num_kv_heads * (long long)c.block_size;
  if (code_bytes) *code_bytes = (size_t)(cells * row_bytes(mode, c.head_dim));
  if (scale_bytes) *scale_bytes = is_dynamic(mode) ? (size_t)cells * sizeof(float) : 0;
  return KVQ_OK;
}

kvq_status kvq_cache_bytes(const kvq_ctx* ctx, long long context_tokens, kvq_capacity* out) {
  if (!ctx || !out || context_tokens < 0) return KVQ_ERR_INVALID_ARG;
  const kvq_config& c = ctx->cfg;
  const double H = c.num_kv_heads, D = c.head_dim;
  kvq_capacity r;
  memset(&r, 0, sizeof(r));
  for (int l = 0; l < c.num_layers; ++l) {
    const int mode = ctx->mode[l];
    const double payload = 2.0 * H * D * elem_bytes(mode);         // K and V codes
    const double scales = is_dynamic(mode) ? 2.0 * H * 4.0 : 0.0;   // one K + one V fp32
    const int W = ctx->window[l];
    const long long kept = (W > 0 && W < context_tokens) ? W : context_tokens;
    r.payload_bytes_per_token += payload;
    r.scale_bytes_per_token += scales;
    r.retained_positions += kept;
    r.cache_bytes += (payload + scales) * (double)kept;
    r.bf16_cache_bytes += 2.0 * H * D * 2.0 * (double)kept;
    if (mode == KVQ_FP8_PER_TENSOR) r.static_scale_bytes += 2 * 4;
    if (mode == KVQ_FP8_PER_HEAD) r.static_scale_bytes += 2LL * 4 * c.num_kv_heads;
  }
  r.bytes_per_token = r.payload_bytes_per_token + r.scale_bytes_per_token;
  r.block_bytes = r.bytes_per_token * c.block_size;
  r.cache_bytes += (double)r.static_scale_bytes;
  *out = r;
  return KVQ_OK;
}

kvq_status kvq_cache_write(const kvq_ctx* ctx, int layer, const void* k_new, const void* v_new,
                           long long kv_token_stride, const long long* slot_mapping,
                           long long num_tokens, const float* k_scale, const float* v_scale,
                           void* k_cache, void* v_cache, float* k_cache_scale,
                           float* v_cache_scale, void* stream) {
  kvq_status st = check_layer(ctx, layer);
  if (st != KVQ_OK) return st;
  if (num_tokens < 0) return KVQ_ERR_INVALID_ARG;
  if (num_tokens == 0) return KVQ_OK;
  if (num_tokens * 2LL * ctx->cfg.num_kv_heads >= (1LL << 31)) return KVQ_ERR_INVALID_ARG;
  const kvq_config& c = ctx->cfg;
  const int mode = ctx->mode[layer];
  const long long HD = (long long)c.num_kv_heads * c.head_dim;
  const long long stride = kv_token_stride == 0 ? HD : kv_token_stride;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return KVQ_ERR_INVALID_ARG;
  if (stride < HD) return KVQ_ERR_INVALID_ARG;
  if (stride % 8 != 0 || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return KVQ_ERR_ALIGNMENT;
  if ((mode == KVQ_FP8_PER_TENSOR || mode == KVQ_FP8_PER_HEAD) && (!k_scale || !v_scale))
    return KVQ_ERR_INVALID_ARG;
  if (is_dynamic(mode)) {
    if (!k_cache_scale || !v_cache_scale) return KVQ_ERR_INVALID_ARG;
    if (!aligned4(k_cache_scale) || !aligned4(v_cache_scale)) return KVQ_ERR_ALIGNMENT;
  }
  unsigned* err = kvq::error_word();
  if (!err) return KVQ_ERR_CUDA;
  kvq::WriteArgs a;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.token_stride = stride;
  a.slots = slot_mapping;
  a.T = num_tokens;
  a.Hkv = c.num_kv_heads;
  a.bs = c.block_size;
  a.bs_shift = __builtin_ctz((unsigned)c.block_size);
  a.num_blocks = c.num_blocks;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.k_cache = static_cast<uint8_t*>(k_cache);
  a.v_cache = static_cast<uint8_t*>(v_cache);
  a.k_cs = k_cache_scale;
  a.v_cs = v_cache_scale;
  a.err = err;
  return cuda_status(
      kvq::launch_cache_write(mode, c.head_dim, a, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_calibrate_per_head(const kvq_ctx* ctx, const void* x, long long num_tokens,
                                  float qmax, float* scale_out, void* stream) {
  if (!ctx || !x || !scale_out || num_tokens < 0 || !(qmax > 0.f)) return KVQ_ERR_INVALID_ARG;
  if (!aligned4(scale_out)) return KVQ_ERR_ALIGNMENT;
  const kvq_config& c = ctx->cfg;
  return cuda_status(kvq::launch_calibrate(static_cast<const uint16_t*>(x), num_tokens,
                                           c.num_kv_heads, c.head_dim, qmax, scale_out,
                                           static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_plan(const kvq_ctx* ctx, int layer, int batch, int max_context,
                           int* num_workers, size_t* workspace_bytes) {
  kvq_status st = check_layer(ctx, layer);
  if (st != KVQ_OK) return st;
  if (!num_workers || batch < 0 || max_context < 0) return KVQ_ERR_INVALID_ARG;
  const kvq_config& c = ctx->cfg;
  const int W = ctx->window[layer];
  const int positions = (W > 0 && W < max_context) ? W + 15 : max_context;
  const int G = c.num_q_heads / c.num_kv_heads;
  int w = *num_workers > 0
              ? *num_workers
              : auto_workers(batch, c.num_kv_heads, positions,
                             kvq::decode_ctas_per_sm(ctx->mode[layer], c.head_dim, G));
  *num_workers = w;
  if (workspace_bytes) {
    // one partial slot per (sequence, KV head) item plus one per worker, and
    // the items' offsets in the tile list
    const size_t items = (size_t)batch * c.num_kv_heads;
    const size_t slots = items + (size_t)w;
    *workspace_bytes = w <= 1 ? 0
                              : slots * G * (c.head_dim + 2) * sizeof(float) +
                                    (items + 1) * sizeof(long long);
  }
  return KVQ_OK;
}

size_t kvq_decode_workspace_size(const kvq_ctx* ctx, int layer, int batch, int max_context) {
  int workers = 0;
  size_t bytes = 0;
  if (kvq_decode_plan(ctx, layer, batch, max_context, &workers, &bytes) != KVQ_OK) return 0;
  return bytes;
}

}  // extern "C"

namespace {

// Shared by the fp32- and bf16-output entry points: exactly one of out and
// out_bf16 is non-null.
kvq_status decode_impl(const kvq_ctx* ctx, int layer, const void* q, const float* q_scale,
                       int q_scale_count, const void* k_cache,
                       const void* v_cache, const float* k_scale, const float* v_scale,
                       const float* k_cache_scale, const float* v_cache_scale,
                       const int* block_table, int max_blocks_per_seq, const int* context_lens,
                       int batch, int max_context, float* out, uint16_t* out_bf16,
                       int num_workers, void* workspace, size_t workspace_bytes, void* stream) {
  kvq_status st = check_layer(ctx, layer);
  if (st != KVQ_OK) return st;
  if (batch < 0 || max_context < 0 || num_workers < 0 || max_blocks_per_seq < 0)
    return KVQ_ERR_INVALID_ARG;
  if (batch == 0) return KVQ_OK;
  const kvq_config& c = ctx->cfg;
  // the block-table rows must cover the longest context
  if ((long long)max_context > (long long)max_blocks_per_seq * c.block_size)
    return KVQ_ERR_INVALID_ARG;
  const int mode = ctx->mode[layer];
  void* out_any = out ? static_cast<void*>(out) : static_cast<void*>(out_bf16);
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out_any)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out_any) ||
      !aligned4(block_table) || !aligned4(context_lens))
    return KVQ_ERR_ALIGNMENT;
  if ((mode == KVQ_FP8_PER_TENSOR || mode == KVQ_FP8_PER_HEAD) && (!k_scale || !v_scale))
    return KVQ_ERR_INVALID_ARG;
  if (is_dynamic(mode)) {
    if (!k_cache_scale || !v_cache_scale) return KVQ_ERR_INVALID_ARG;
    if (!aligned4(k_cache_scale) || !aligned4(v_cache_scale)) return KVQ_ERR_ALIGNMENT;
  }
  if (q_scale) {
    if (q_scale_count != 1 && q_scale_count != c.num_q_heads) return KVQ_ERR_INVALID_ARG;
    if (!aligned4(q_scale)) return KVQ_ERR_ALIGNMENT;
  }
  int workers = num_workers;
  size_t need = 0;
  st = kvq_decode_plan(ctx, layer, batch, max_context, &workers, &need);
  if (st != KVQ_OK) return st;
  if (workers > 1 && (!workspace || workspace_bytes < need)) return KVQ_ERR_WORKSPACE;
  if (workers > 1 && !aligned16(workspace)) return KVQ_ERR_ALIGNMENT;
  if ((long long)workers > 4LL * 65535 * 64) return KVQ_ERR_INVALID_ARG;
  unsigned* err = kvq::error_word();
  if (!err) return KVQ_ERR_CUDA;
  const int G = c.num_q_heads / c.num_kv_heads;
  kvq::DecodeArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.q_scale = q_scale;
  a.q_scale_count = q_scale ? q_scale_count : 0;
  a.k_cache = static_cast<const uint8_t*>(k_cache);
  a.v_cache = static_cast<const uint8_t*>(v_cache);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.k_cs = k_cache_scale;
  a.v_cs = v_cache_scale;
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.out = out;
  a.out_bf16 = out_bf16;
  float* ws = static_cast<float*>(workspace);
  const size_t n_part = ((size_t)batch * c.num_kv_heads + (size_t)workers) * G;
  a.ws_o = workers > 1 ? ws : nullptr;
  a.ws_ml = workers > 1 ? ws + n_part * c.head_dim : nullptr;
  a.item_tiles = workers > 1 ? reinterpret_cast<long long*>(ws + n_part * (c.head_dim + 2))
                             : nullptr;
  a.err = err;
  a.B = batch;
  a.Hq = c.num_q_heads;
  a.Hkv = c.num_kv_heads;
  a.bs = c.block_size;
  a.bs_shift = __builtin_ctz((unsigned)c.block_size);
  a.max_blocks = max_blocks_per_seq;
  a.window = ctx->window[layer];
  a.workers = workers;
  a.num_blocks = c.num_blocks;
  a.qk_scale = ctx->softmax_scale * 1.4426950408889634f;
  {
    // upper bound of the cache bytes this call reads; beyond ~half the L2 the
    // pages cannot survive to the next step, so they are streamed evict-first
    const long long win = ctx->window[layer];
    const long long pos = (win > 0 && win < max_context) ? win : max_context;
    const double bytes = (double)batch * c.num_kv_heads * (double)pos *
                         (2.0 * (double)row_bytes(mode, c.head_dim) + (is_dynamic(mode) ? 8 : 0));
    a.stream_once = bytes > 64.0 * 1024 * 1024;
  }
  return cuda_status(
      kvq::launch_decode(mode, c.head_dim, G, a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

kvq_status kvq_decode_attention(const kvq_ctx* ctx, int layer, const void* q,
                                const void* k_cache, const void* v_cache, const float* k_scale,
                                const float* v_scale, const float* k_cache_scale,
                                const float* v_cache_scale, const int* block_table,
                                int max_blocks_per_seq, const int* context_lens, int batch,
                                int max_context, float* out, int num_workers, void* workspace,
                                size_t workspace_bytes, void* stream) {
  return decode_impl(ctx, layer, q, nullptr, 0, k_cache, v_cache, k_scale, v_scale,
                     k_cache_scale, v_cache_scale, block_table, max_blocks_per_seq, context_lens,
                     batch, max_context, out, nullptr, num_workers, workspace, workspace_bytes,
                     stream);
}

kvq_status kvq_decode_attention_fp8_query(const kvq_ctx* ctx, int layer, const void* q,
                                          const float* q_scale, int q_scale_count,
                                          const void* k_cache, const void* v_cache,
                                          const float* k_scale, const float* v_scale,
                                          const float* k_cache_scale,
                                          const float* v_cache_scale, const int* block_table,
                                          int max_blocks_per_seq, const int* context_lens,
                                          int batch, int max_context, float* out,
                                          int num_workers, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (!q_scale) return KVQ_ERR_INVALID_ARG;
  return decode_impl(ctx, layer, q, q_scale, q_scale_count, k_cache, v_cache, k_scale, v_scale,
                     k_cache_scale, v_cache_scale, block_table, max_blocks_per_seq, context_lens,
                     batch, max_context, out, nullptr, num_workers, workspace, workspace_bytes,
                     stream);
}

kvq_status kvq_decode_attention_bf16(const kvq_ctx* ctx, int layer, const void* q,
                                     const void* k_cache, const void* v_cache,
                                     const float* k_scale, const float* v_scale,
                                     const float* k_cache_scale, const float* v_cache_scale,
                                     const int* block_table, int max_blocks_per_seq,
                                     const int* context_lens, int batch, int max_context,
                                     void* out, int num_workers, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return decode_impl(ctx, layer, q, nullptr, 0, k_cache, v_cache, k_scale, v_scale,
                     k_cache_scale, v_cache_scale, block_table, max_blocks_per_seq, context_lens,
                     batch, max_context, nullptr, static_cast<uint16_t*>(out), num_workers,
                     workspace, workspace_bytes, stream);
}

kvq_status kvq_prefill_attention(const kvq_ctx* ctx, int layer, const void* q,
                                 const void* k_cache, const void* v_cache, const float* k_scale,
                                 const float* v_scale, const float* k_cache_scale,
                                 const float* v_cache_scale, const int* block_table,
                                 int max_blocks_per_seq, const int* query_start,
                                 const int* context_lens, int batch, int max_query_len,
                                 float* out, void* stream) {
  kvq_status st = check_layer(ctx, layer);
  if (st != KVQ_OK) return st;
  if (batch < 0 || max_query_len < 0 || max_blocks_per_seq < 0) return KVQ_ERR_INVALID_ARG;
  if (batch == 0 || max_query_len == 0) return KVQ_OK;
  const kvq_config& c = ctx->cfg;
  const int mode = ctx->mode[layer];
  if (!q || !k_cache || !v_cache || !block_table || !query_start || !context_lens || !out)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned4(block_table) || !aligned4(query_start) || !aligned4(context_lens))
    return KVQ_ERR_ALIGNMENT;
  if ((mode == KVQ_FP8_PER_TENSOR || mode == KVQ_FP8_PER_HEAD) && (!k_scale || !v_scale))
    return KVQ_ERR_INVALID_ARG;
  if (is_dynamic(mode)) {
    if (!k_cache_scale || !v_cache_scale) return KVQ_ERR_INVALID_ARG;
    if (!aligned4(k_cache_scale) || !aligned4(v_cache_scale)) return KVQ_ERR_ALIGNMENT;
  }
  const int G = c.num_q_heads / c.num_kv_heads;
  const long long qtiles = ((long long)max_query_len * G + kvq::prefill_rows_per_cta() - 1) /
                           kvq::prefill_rows_per_cta();
  if (qtiles * batch * c.num_kv_heads >= (1LL << 31)) return KVQ_ERR_INVALID_ARG;
  unsigned* err = kvq::error_word();
  if (!err) return KVQ_ERR_CUDA;
  kvq::DecodeArgs a = {};
  a.q = static_cast<const uint16_t*>(q);
  a.k_cache = static_cast<const uint8_t*>(k_cache);
  a.v_cache = static_cast<const uint8_t*>(v_cache);
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.k_cs = k_cache_scale;
  a.v_cs = v_cache_scale;
  a.block_table = block_table;
  a.context_lens = context_lens;
  a.out = out;
  a.err = err;
  a.B = batch;
  a.Hq = c.num_q_heads;
  a.Hkv = c.num_kv_heads;
  a.bs = c.block_size;
  a.bs_shift = __builtin_ctz((unsigned)c.block_size);
  a.max_blocks = max_blocks_per_seq;
  a.window = ctx->window[layer];
  a.workers = 1;
  a.num_blocks = c.num_blocks;
  a.qk_scale = ctx->softmax_scale * 1.4426950408889634f;
  return cuda_status(kvq::launch_prefill(mode, c.head_dim, G, a, query_start, max_query_len,
                                         static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_e4m3_encode(const float* in, unsigned char* out, long long n, void* stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return KVQ_ERR_INVALID_ARG;
  return cuda_status(kvq::launch_e4m3_encode(in, out, n, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_check_bounded_wait(long long limit_cycles, void* stream) {
  if (limit_cycles <= 0 || limit_cycles > (1LL << 31)) return KVQ_ERR_INVALID_ARG;
  return cuda_status(kvq::launch_wait_check(limit_cycles, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_get_device_error(void* stream) {
  unsigned* err = kvq::error_word();
  if (!err) return KVQ_ERR_CUDA;
  unsigned v = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return KVQ_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVQ_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpyAsync(err, &zero, sizeof(zero), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return KVQ_ERR_CUDA;
  }
  if (v & kvq::ERR_TIMEOUT) return KVQ_ERR_TIMEOUT;
  if (v & kvq::ERR_BAD_INDEX) return KVQ_ERR_BAD_INDEX;
  return KVQ_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- fixed scratch
// Scratch for kvq_decode_attention_fixed_scratch: a file-scope device array,
// present on every GPU that loads the library until the process exits.  Host
// code cannot use the name as an address; the address is looked up once per
// device with cudaGetSymbolAddress while that device is current.
static __device__ __align__(256) unsigned char kvq_fixed_scratch[KVQ_FIXED_SCRATCH_BYTES];

namespace {
std::mutex g_fixed_scratch_mu;
void* g_fixed_scratch_ptr[64] = {nullptr};
}  // namespace

extern "C" {

kvq_status kvq_decode_attention_fixed_scratch(const kvq_ctx* ctx, int layer, const void* q,
                                              const void* k_cache, const void* v_cache,
                                              const float* k_scale, const float* v_scale,
                                              const float* k_cache_scale,
                                              const float* v_cache_scale, const int* block_table,
                                              int max_blocks_per_seq, const int* context_lens,
                                              int batch, int max_context, float* out,
                                              int num_workers, void* stream) {
  kvq_status st = check_layer(ctx, layer);
  if (st != KVQ_OK) return st;
  if (batch < 0 || max_context < 0 || num_workers < 0) return KVQ_ERR_INVALID_ARG;
  // Size check first.  An explicit worker count whose partials do not fit is
  // refused; the automatic plan is cut to the most workers that fit (one
  // worker needs no scratch at all).
  int workers = num_workers;
  size_t need = 0;
  st = kvq_decode_plan(ctx, layer, batch, max_context, &workers, &need);
  if (st != KVQ_OK) return st;
  if (need > (size_t)KVQ_FIXED_SCRATCH_BYTES) {
    if (num_workers > 0) return KVQ_ERR_WORKSPACE;
    const kvq_config& c = ctx->cfg;
    const long long items = (long long)batch * c.num_kv_heads;
    const long long G = c.num_q_heads / c.num_kv_heads;
    const long long per_slot = G * (c.head_dim + 2) * (long long)sizeof(float);
    const long long room = (long long)KVQ_FIXED_SCRATCH_BYTES - (items + 1) * (long long)sizeof(long long);
    long long fit = room > 0 ? room / per_slot - items : 0;
    if (fit > workers) fit = workers;
    workers = fit >= 2 ? (int)fit : 1;
    st = kvq_decode_plan(ctx, layer, batch, max_context, &workers, &need);
    if (st != KVQ_OK) return st;
    if (need > (size_t)KVQ_FIXED_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVQ_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_fixed_scratch_mu);
    if (!g_fixed_scratch_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, kvq_fixed_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
      g_fixed_scratch_ptr[dev] = p;
    }
    scratch = g_fixed_scratch_ptr[dev];
  }
  // Nothing in the scratch needs to start at zero: every partial and offset
  // the merge reads is written by the decode kernel of the same call.
  return kvq_decode_attention(ctx, layer, q, k_cache, v_cache, k_scale, v_scale, k_cache_scale,
                              v_cache_scale, block_table, max_blocks_per_seq, context_lens, batch,
                              max_context, out, workers, scratch,
                              (size_t)KVQ_FIXED_SCRATCH_BYTES, stream);
}

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case KVQ_ERR_WORKSPACE: return "decode workspace missing or too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_BAD_INDEX: return "slot or block id outside the cache";
    case KVQ_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
