/*
 * kvq.h -- C ABI of libkvq, a quantized paged KV cache for one GB300 GPU.
 *
 * Two hot operations, both hand-written CUDA for sm_103a:
 *
 *   kvq_cache_write       new bf16 K/V vectors -> scale -> FP8 E4M3 / packed
 *                         INT4 / BF16 codes -> scatter into paged blocks.
 *   kvq_decode_attention  paged GQA decode over that cache, K scale folded
 *                         into the QK product, V scale into the PV sum.
 *
 * Around them: the work plan of the decode (kvq_decode_plan), its variants
 * (bf16 output, FP8 query, no caller workspace), prefill attention over the
 * same cache (kvq_prefill_attention), static per-head calibration, the
 * capacity accounting of the pages and the device codec on its own.
 *
 * The operations and their scale layouts follow three pages:
 *   [P1] "Per-tensor vs per-head FP8 KV cache scales"
 *   [P2] "Per-token-head KV cache scale overhead"
 *   [P3] "FP8 KV cache layer skipping vs per-head scales"
 *
 * Conventions for every call:
 *  - Pointers named *_cache, q, out, k_new, v_new, slot_mapping, block_table,
 *    context_lens, workspace and the scale arrays are DEVICE pointers owned by
 *    the caller; the library never allocates, frees or retains them.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Device work is enqueued asynchronously on it; a call returns
 *    once the work is enqueued.
 *  - Argument errors are detected on the host before anything is launched and
 *    reported as a kvq_status; nothing is launched in that case.  Index errors
 *    found on the device (a slot or block id outside the cache, a negative
 *    context length) skip the bad access and set a device error word that
 *    kvq_get_device_error() reads.  No call falls back to another path.
 *  - kvq_ctx is host-only configuration; it may be shared between threads
 *    for the read-only calls below.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size or layer index */
  KVQ_ERR_UNSUPPORTED = 2,  /* head_dim, block_size, mode or GQA ratio not built */
  KVQ_ERR_ALIGNMENT = 3,    /* a pointer or stride breaks the 16-byte rule */
  KVQ_ERR_WORKSPACE = 4,    /* workspace missing or smaller than kvq_decode_plan says */
  KVQ_ERR_CUDA = 5,         /* a CUDA launch or query failed */
  KVQ_ERR_BAD_INDEX = 6,    /* device saw a slot / block id outside the cache */
  KVQ_ERR_TIMEOUT = 7       /* a bounded device wait gave up */
} kvq_status;

/* Cache dtype and scale layout of one layer ([P1] "Per-tensor vs per-head FP8
 * KV cache scales"; [P2] "INT4 makes the metadata fraction larger"; [P3] "FP8
 * KV cache layer skipping vs per-head scales"). */
typedef enum kvq_mode {
  KVQ_BF16 = 0,                /* skipped layer: native bf16, no scales */
  KVQ_FP8_PER_TENSOR = 1,      /* E4M3, one K and one V scale per layer */
  KVQ_FP8_PER_HEAD = 2,        /* E4M3, static scale per KV head */
  KVQ_FP8_PER_TOKEN_HEAD = 3,  /* E4M3, scale = amax/448 per token and head */
  KVQ_INT4_PER_TOKEN_HEAD = 4  /* packed symmetric INT4, scale = amax/7 */
} kvq_mode;

/* Model/cache description, the pages' statement of the problem: layers, Hq
 * query heads and Hkv KV heads ([P3] "Per-head scales have fixed overhead"),
 * head size and block size ([P2] "Per-token-head KV cache scale overhead",
 * "Convert bytes into block capacity"), the scale layout of each layer ([P1]
 * "Per-tensor vs per-head FP8 KV cache scales"), and the window and skipped
 * (KVQ_BF16) layers ([P3] "FP8 KV cache layer skipping vs per-head scales",
 * "Layer skipping follows retained-token footprint"). */
typedef struct kvq_config {
  int num_layers;
  int num_q_heads;          /* Hq; a multiple of num_kv_heads, Hq/Hkv <= 16 */
  int num_kv_heads;         /* Hkv */
  int head_dim;             /* D: 64, 128 or 256 */
  int block_size;           /* tokens per block: 16, 32, 64 or 128 */
  long long num_blocks;     /* blocks in each layer's cache */
  const int* layer_mode;    /* host [num_layers] of kvq_mode; copied by kvq_create */
  const int* layer_window;  /* host [num_layers]; 0 = full attention, W > 0 keeps
                               the last W positions; NULL = all full */
  float softmax_scale;      /* 0 => 1/sqrt(head_dim) */
} kvq_config;

typedef struct kvq_ctx kvq_ctx;

/* Validates and copies *cfg into a new context (the description above;
 * [P1] and [P3] as cited there).  Host only; no CUDA call.  Returns
 * KVQ_ERR_INVALID_ARG for a null pointer, a non-positive count, Hq not a
 * multiple of Hkv, a mode outside kvq_mode or a negative window, and
 * KVQ_ERR_UNSUPPORTED for a head size, block size or GQA ratio that is not
 * built or a cache too large for 32-bit cell indices.  *out is NULL on
 * error; the caller releases a context with kvq_destroy. */
kvq_status kvq_create(const kvq_config* cfg, kvq_ctx** out);
void kvq_destroy(kvq_ctx* ctx);

/* Bytes of one layer's K code buffer and K scale buffer (V is the same).
 * Codes: [num_blocks][Hkv][block_size][row] with row = 2D (BF16), D (FP8) or
 * D/2 (INT4) bytes ([P2] "The FP8 scale tax is 4 divided by head size": one
 * byte per FP8 element; "INT4 makes the metadata fraction larger": half a
 * byte per INT4 element).  Scales (dynamic modes only, else 0): [num_blocks]
 * [Hkv][block_size] fp32, one K and one V scale per token and KV head
 * (same section; the pages' padding of each scale is not stored).  Each
 * (block, head) page of codes and of scales is contiguous; a block of
 * block_size tokens holds block_size x the per-token bytes ([P2] "Convert
 * bytes into block capacity").  Host only; KVQ_ERR_INVALID_ARG for a bad
 * context or layer.  The caller allocates the buffers. */
kvq_status kvq_layer_buffer_sizes(const kvq_ctx* ctx, int layer, size_t* code_bytes,
                                  size_t* scale_bytes);

/* Capacity accounting for one sequence of `context_tokens` positions.
 * Payload 2 x Hkv x D x bytes/elem per layer and retained token, dynamic
 * scales 2 x Hkv x 4 bytes ([P2] "Per-token-head KV cache scale overhead"),
 * static scales 8 bytes per per-tensor layer and 8 x Hkv per per-head layer
 * ([P1] "Static per-head metadata is almost free"), window layers retain
 * min(context, W) positions ([P3] "Layer skipping follows retained-token
 * footprint"), block bytes = per-token bytes x block size ([P2] "Convert
 * bytes into block capacity").  Bytes are before allocator rounding. */
typedef struct kvq_capacity {
  double payload_bytes_per_token;   /* all layers, codes only */
  double scale_bytes_per_token;     /* all layers, dynamic scales only */
  double bytes_per_token;           /* payload + scales */
  double block_bytes;               /* bytes_per_token x block_size */
  long long retained_positions;     /* sum over layers of retained positions */
  long long static_scale_bytes;     /* per-tensor and per-head scale arrays */
  double cache_bytes;               /* retained codes + scales + static scales */
  double bf16_cache_bytes;          /* the same retention with every layer BF16 */
} kvq_capacity;
kvq_status kvq_cache_bytes(const kvq_ctx* ctx, long long context_tokens, kvq_capacity* out);

/* Fused quantize-and-scatter of num_tokens new K/V vectors into `layer`.
 *
 * k_new, v_new: bf16 [num_tokens][Hkv][D], token t starting at element
 *   t * kv_token_stride (0 => Hkv*D); 16-byte aligned, stride a multiple of 8.
 * slot_mapping: int64 [num_tokens]; token t goes to block slot/block_size,
 *   offset slot%block_size; slot < 0 skips the token (padding).
 * k_scale, v_scale: fp32, [1] for KVQ_FP8_PER_TENSOR, [Hkv] for
 *   KVQ_FP8_PER_HEAD, ignored (may be NULL) otherwise.
 * k_cache, v_cache: the layer's code buffers (16-byte aligned).
 * k_cache_scale, v_cache_scale: the layer's scale buffers for the dynamic
 *   modes, ignored (may be NULL) otherwise.
 * Per element: y = x / s rounded to fp32, then E4M3 round-to-nearest-even
 * with saturation to +-448, or INT4 q = clamp(rint(y), -7, 7) packed two per
 * byte (even element in the low nibble).  Dynamic scales: s = amax/448 (FP8)
 * or amax/7 (INT4) in fp32, s = 1 when amax = 0 ([P1] "Dynamic per-token-head
 * scales add 3.125 percent"; [P2] "INT4 makes the metadata fraction larger").
 * A slot past the cache skips the token and sets KVQ_ERR_BAD_INDEX on the
 * device word. */
kvq_status kvq_cache_write(const kvq_ctx* ctx, int layer, const void* k_new, const void* v_new,
                           long long kv_token_stride, const long long* slot_mapping,
                           long long num_tokens, const float* k_scale, const float* v_scale,
                           void* k_cache, void* v_cache, float* k_cache_scale,
                           float* v_cache_scale, void* stream);

/* Static per-head calibration: scale_out[h] = amax over a bf16 sample
 * x [num_tokens][Hkv][D] of head h, divided by qmax (448 for E4M3) in fp32;
 * 1.0 for an all-zero head ([P1] "Calibration changes which scale layout
 * exists": an online maximum stands in for warm-up calibration).
 * scale_out: device fp32 [Hkv], overwritten. */
kvq_status kvq_calibrate_per_head(const kvq_ctx* ctx, const void* x, long long num_tokens,
                                  float qmax, float* scale_out, void* stream);

/* Work plan for a decode call.  The retained positions of all (sequence, KV
 * head) items are cut into 16-position tiles and divided evenly among
 * `num_workers` worker warps (split-K over the context, balanced whatever the
 * context lengths); an item shared by several workers is merged by
 * log-sum-exp.  The pages fix no decode schedule; split-K with a
 * log-sum-exp merge is this library's way of spreading the retained
 * positions of few, long sequences ([P3] "Performance can favor the larger
 * cache": latency grows with every context token) over every SM.  On input *num_workers > 0 requests a count, 0 asks for the
 * plan's choice (fill every SM, from the batch, KV heads, the longest
 * context and the device); on output it holds the count and
 * *workspace_bytes what a call with that count needs (0 for one worker). */
kvq_status kvq_decode_plan(const kvq_ctx* ctx, int layer, int batch, int max_context,
                           int* num_workers, size_t* workspace_bytes);

/* Workspace bytes of a decode call with num_workers = 0 (the plan's choice):
 * kvq_decode_plan's *workspace_bytes for that count.  0 when one worker
 * suffices, and also when an argument is invalid (kvq_decode_plan reports
 * which). */
size_t kvq_decode_workspace_size(const kvq_ctx* ctx, int layer, int batch, int max_context);

/* Paged decode attention, one query token per sequence.
 *
 * Scales are folded, never applied element by element: the K scale (per
 * tensor, per KV head or per token and KV head, [P1] "Per-tensor vs per-head
 * FP8 KV cache scales", "Range sharing explains the accuracy trade")
 * multiplies the dot product of q with the raw codes, and the V scale the
 * softmax weight that meets the raw V codes.  Window layers read only their
 * last W positions, and KVQ_BF16 layers their native bf16 values ([P3] "FP8
 * KV cache layer skipping vs per-head scales", "Layer skipping follows
 * retained-token footprint").  Packed INT4 layers as [P2] "INT4 makes the
 * metadata fraction larger".
 *
 * q: bf16 [batch][Hq][D], 16-byte aligned.  Query head hq reads KV head
 *   hq / (Hq/Hkv).
 * block_table: int32 [batch][max_blocks_per_seq]; entries for positions that
 *   are not read may hold anything (e.g. -1).  Row b must cover context_lens[b]
 *   positions (context_lens[b] <= max_blocks_per_seq x block_size): a longer
 *   context is an index error -- only the covered positions are read and
 *   KVQ_ERR_BAD_INDEX is set on the device word.  Only positions [lo, L) are
 *   read, so a window layer may reuse its freed blocks as a ring: with
 *   R = ceil(W / block_size) + 1 physical blocks per sequence, logical block j
 *   may map to ring slot j mod R (the block a new position overwrites holds
 *   only positions outside the window).
 * context_lens: int32 [batch]; L counts the current token, whose K/V were
 *   written first.  The query attends to positions [lo, L), lo = max(0, L-W)
 *   for a window W, else 0.  L = 0 gives a zero output row.
 * out: fp32 [batch][Hq][D] = sum_p softmax(softmax_scale <q, K_hat[p]>) V_hat[p]
 *   with K_hat = code x K scale, V_hat = code x V scale.
 * max_context: an upper bound of context_lens, used only by the plan; more
 *   than max_blocks_per_seq x block_size returns KVQ_ERR_INVALID_ARG.
 * num_workers: worker warps (see kvq_decode_plan); 0 = the plan's choice.
 *   With more than one worker, partials go to `workspace` (16-byte aligned,
 *   kvq_decode_plan gives its size); its contents need no initialisation.
 * Scale pointers as for kvq_cache_write. */
kvq_status kvq_decode_attention(const kvq_ctx* ctx, int layer, const void* q,
                                const void* k_cache, const void* v_cache, const float* k_scale,
                                const float* v_scale, const float* k_cache_scale,
                                const float* v_cache_scale, const int* block_table,
                                int max_blocks_per_seq, const int* context_lens, int batch,
                                int max_context, float* out, int num_workers, void* workspace,
                                size_t workspace_bytes, void* stream);

/* kvq_decode_attention with an FP8 query.  Each query element x becomes the
 * E4M3 code of RN32(x / q_scale) (round to nearest even, saturating to
 * +-448, as kvq_cache_write encodes), and the scores use its value times
 * q_scale: out = sum_p softmax(softmax_scale <q_hat, K_hat[p]>) V_hat[p] with
 * q_hat = E4M3(q / q_scale) x q_scale.  This is the per-tensor FP8 path with
 * one scale each for Q, K and V, and the per-attention-head path with one Q
 * scale per query head ([P3] "FP8 KV cache layer skipping vs per-head
 * scales", opening section).
 * q_scale: device fp32, q_scale_count = 1 (one scale) or Hq (one per query
 *   head), each finite and > 0.  Other arguments, errors and workspace as for
 *   kvq_decode_attention; the output is fp32. */
kvq_status kvq_decode_attention_fp8_query(const kvq_ctx* ctx, int layer, const void* q,
                                          const float* q_scale, int q_scale_count,
                                          const void* k_cache, const void* v_cache,
                                          const float* k_scale, const float* v_scale,
                                          const float* k_cache_scale,
                                          const float* v_cache_scale, const int* block_table,
                                          int max_blocks_per_seq, const int* context_lens,
                                          int batch, int max_context, float* out,
                                          int num_workers, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* kvq_decode_attention with a bf16 output: out is bf16 [batch][Hq][D]
 * (16-byte aligned), each element the round-to-nearest-even bf16 of the fp32
 * value kvq_decode_attention returns for the same arguments and num_workers.
 * The pages leave the attention output's dtype open; this variant returns
 * the model's native bf16 (the dtype [P3] "FP8 KV cache layer skipping vs
 * per-head scales" keeps for unquantized layers) and halves the output
 * traffic.  The arithmetic up to the final rounding is
 * kvq_decode_attention's.  Arguments, errors and workspace as for
 * kvq_decode_attention. */
kvq_status kvq_decode_attention_bf16(const kvq_ctx* ctx, int layer, const void* q,
                                     const void* k_cache, const void* v_cache,
                                     const float* k_scale, const float* v_scale,
                                     const float* k_cache_scale, const float* v_cache_scale,
                                     const int* block_table, int max_blocks_per_seq,
                                     const int* context_lens, int batch, int max_context,
                                     void* out, int num_workers, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Prefill (chunked multi-query) attention over the quantized paged cache:
 * the new tokens of each sequence attend causally to the cache, as at the
 * prefill stage whose time to first token the pages record ([P3] "FP8 KV
 * cache layer skipping vs per-head scales", section "Run a four-way
 * ablation").
 *
 * Sequence b has n_b = query_start[b+1] - query_start[b] new tokens at
 * positions [L_b - n_b, L_b), L_b = context_lens[b] >= n_b; their K/V were
 * written first (kvq_cache_write).  Query row query_start[b] + i of q (bf16
 * [T][Hq][D], T = query_start[batch], 16-byte aligned) sits at position
 * p = L_b - n_b + i and attends to positions [lo(p), p], lo(p) =
 * max(0, p + 1 - W) for a window W, else 0; out (fp32 [T][Hq][D]) is the
 * softmax(softmax_scale <q, K_hat>) weighted sum of V_hat over them, exactly
 * what kvq_decode_attention returns for that query with context p + 1.
 * query_start: int32 [batch + 1], query_start[0] = 0, non-decreasing.
 * max_query_len: an upper bound of every n_b (sizes the grid; rows past n_b
 *   do no work).
 * Scale pointers and block table as for kvq_decode_attention.  No workspace;
 * n_b > L_b, or L_b beyond the positions the sequence's block-table row
 * covers (max_blocks_per_seq x block_size), sets the BAD_INDEX bit of the
 * device error word and skips that sequence; a block id outside
 * [0, num_blocks) sets the same bit, nothing is read for that page, and its
 * positions are left out of the softmax (the output stays finite). */
kvq_status kvq_prefill_attention(const kvq_ctx* ctx, int layer, const void* q,
                                 const void* k_cache, const void* v_cache, const float* k_scale,
                                 const float* v_scale, const float* k_cache_scale,
                                 const float* v_cache_scale, const int* block_table,
                                 int max_blocks_per_seq, const int* query_start,
                                 const int* context_lens, int batch, int max_query_len,
                                 float* out, void* stream);

/* Decode attention that allocates nothing and needs no workspace from the
 * caller.  The pages have no counterpart to this call; it exists for callers
 * that cannot provide device scratch: code running where no device allocator
 * may be used (a serving loop that forbids allocations after start-up, a
 * plugin inside a host process that owns every device buffer) or bindings
 * that cannot manage device memory at all.
 *
 * Arguments and results are those of kvq_decode_attention without
 * `workspace`/`workspace_bytes`.  The split-K partials live instead in one
 * static device array of KVQ_FIXED_SCRATCH_BYTES (16 MiB) per GPU, held by
 * every GPU that loads the library until the process exits.  With
 * num_workers = 0 the plan's worker count is cut to the most workers whose
 * partials fit (at worst one worker, which needs no scratch).  An explicit
 * num_workers whose plan (kvq_decode_plan for the same batch, max_context
 * and num_workers) needs more than the array returns KVQ_ERR_WORKSPACE and
 * launches nothing; pass a smaller num_workers to fit.
 *
 * The first call on a device looks the array's address up on that device
 * (make that device current first; make the first call before any stream
 * capture).  Every call on a device shares the one array: calls whose GPU
 * work overlaps (different streams, concurrent host threads) race on it and
 * must be serialised by the caller.  The array keeps the last call's
 * contents; no call reads anything it did not write itself. */
#define KVQ_FIXED_SCRATCH_BYTES (16u * 1024u * 1024u)
kvq_status kvq_decode_attention_fixed_scratch(const kvq_ctx* ctx, int layer, const void* q,
                                              const void* k_cache, const void* v_cache,
                                              const float* k_scale, const float* v_scale,
                                              const float* k_cache_scale,
                                              const float* v_cache_scale, const int* block_table,
                                              int max_blocks_per_seq, const int* context_lens,
                                              int batch, int max_context, float* out,
                                              int num_workers, void* stream);

/* The device codec on its own: out[i] = E4M3 code of in[i] (RNE, saturating
 * to +-448), exactly as kvq_cache_write encodes y.  in: device fp32 [n],
 * out: device uint8 [n]. */
kvq_status kvq_e4m3_encode(const float* in, unsigned char* out, long long n, void* stream);

/* Synchronizes `stream`, returns the device error word of the current device
 * as a status (KVQ_OK, KVQ_ERR_BAD_INDEX or KVQ_ERR_TIMEOUT) and clears it. */
kvq_status kvq_get_device_error(void* stream);

/* Check of the timeout path (no counterpart on the pages).  Every wait of the
 * decode, prefill and staged cache-write kernels on a shared-memory barrier
 * is bounded (about 2 s); a wait that runs out sets the TIMEOUT bit of the
 * device error word and the kernel stops instead of hanging the GPU.  This
 * call enqueues one warp that waits in the same way on a barrier that expects
 * bytes no copy ever delivers (no copy is issued, so nothing is in flight
 * when it gives up), with a limit of `limit_cycles` SM clock cycles
 * (0 < limit_cycles <= 2^31; 2,000,000 is about 1 ms).  Afterwards
 * kvq_get_device_error() returns KVQ_ERR_TIMEOUT and the context stays
 * usable.  Returns KVQ_ERR_INVALID_ARG for a limit outside the range. */
kvq_status kvq_check_bounded_wait(long long limit_cycles, void* stream);

const char* kvq_status_string(kvq_status s);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H_ */
