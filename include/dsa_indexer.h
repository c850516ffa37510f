/*
 * dsa_indexer.h -- C ABI of the DSA lightning-indexer step on one GB300 GPU
 * (library: libdsa_indexer.so, kernels for sm_103a).
 *
 * The step, per F ("full") layer of a DeepSeek Sparse Attention model:
 *   1. write each new token's 128-d indexer key into the paged FP8 cache;
 *   2. score every query token against its request's cached keys;
 *   3. keep the top `index_topk` keys per query in a shared int32 buffer;
 * and, over a layer stack, 4. the IndexCache F/S schedule: S ("shared")
 * layers run no indexer and read what the last F layer wrote in this pass.
 *
 * Sources, by page title and section:
 *   [IC]  "vLLM IndexCache 实战指南" -- §二 How It Works (shared
 *         topk_indices_buffer, -1 clear before scatter, S layers read the
 *         buffer written earlier in the same forward pass), §三 配置参数参考
 *         (index_topk_freq, index_topk_pattern, index_skip_topk_offset and
 *         the skip rule), §四 方式二 (layers beyond the pattern are F).
 *   [KV]  "GLM-5.3 推理全链路(十二): 主 KV 与索引器缓存的分页预算、前缀命中与驱逐"
 *         -- byte-accounting table (132 B per token per layer), SGLang
 *         _buffer_shape (8448-byte page rows), IndexKeyCache.move comment
 *         (all key bytes of a page, then all scale bytes), the
 *         topk_indices_buffer passage, the write-path section
 *         (store_quantized), and "64 token 页的由来" (64-token pages).
 *   [HBM] "HBM 索引架构设计" -- §2.3 (slot = block_table[req, pos/bs]*bs + pos%bs);
 *         §5.1-5.3 (compressed caches: one entry per compress_ratio tokens,
 *         slot only for a token with (pos+1) % ratio == 0, -1 otherwise).
 *   [DSA] DeepSeek-V3.2 report (arXiv:2512.02556, in [KV]'s references):
 *         score(t,s) = sum_h w[t,h] * ReLU(q[t,h] . k[s]).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers unless stated; the caller owns
 *     every buffer (caches, outputs, workspace).  Nothing here allocates,
 *     frees or synchronises: each call only enqueues kernels on `stream`
 *     (a cudaStream_t; NULL = legacy default stream) and returns.
 *   - head_dim is 128 and the page is 64 tokens; both are fixed.
 *   - Page layout (one uint8 row of DSA_PAGE_BYTES per physical page): the
 *     E4M3 key of in-page offset o at bytes [o*128, o*128+128), its FP32
 *     scale at byte DSA_PAGE_SCALE_OFFSET + 4*o.
 *   - Batch metadata (int32, device): query_start_loc [R+1] with
 *     query_start_loc[0] = 0 and query_start_loc[R] = T (request r owns query
 *     rows [qsl[r], qsl[r+1])); seq_lens [R] = context length of request r
 *     AFTER this step (its new tokens are the last q_len[r] positions);
 *     block_table [R, max_blocks] row-major, physical page of each 64-token
 *     block of the request.
 *   - Quantisation: one FP32 scale per 128-element block, s = amax/448 in
 *     FP32 (s = 1 for an all-zero block), codes = E4M3(x / s) rounded to
 *     nearest-even with saturation to +-448.  Inputs must be finite.
 *   - Returned top-k indices are logical token positions inside the request
 *     (0 .. ctx-1), in no particular order; row t holds min(ctx(t), index_topk)
 *     valid indices followed by -1, ctx(t) = pos(t)+1 (causal, self included).
 *   - Compressed cache (the *_compressed entry points, compress_ratio N >= 1;
 *     N = 1 is the plain cache): entry c of a request holds the key of its
 *     token at position (c+1)*N - 1, the token that completes the entry; the
 *     block table maps 64-entry pages (entry c in block c/64, offset c%64),
 *     so a request needs ceil((seq_len/N) / 64) blocks.  Row t sees the
 *     entries c < ctx(t) = (pos(t)+1)/N (integer division: those whose
 *     completing token is at or before it) and its indices are entry numbers.
 *     Rows that see no entry are all -1.
 *   - Return value: DSA_OK or a negative DSA_ERR_*; the message of the last
 *     failing call on this thread is dsa_last_error().  Faults in device-side
 *     metadata (e.g. a block id outside [0, num_pages)) do not trap: the
 *     affected keys/tokens are skipped and a DSA_STATUS_* bit is OR-ed into
 *     *dev_status (int32, device, may be NULL) for the caller to read later.
 */
#ifndef DSA_INDEXER_H_
#define DSA_INDEXER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* same type as cudaStream_t */

#define DSA_HEAD_DIM 128
#define DSA_PAGE_TOKENS 64
#define DSA_TOKEN_BYTES 132               /* [KV] byte-accounting table */
#define DSA_PAGE_BYTES 8448               /* [KV] 64 * (128 + 128/128*4) */
#define DSA_PAGE_SCALE_OFFSET 8192        /* [KV] keys first, then scales */
#define DSA_MAX_TOPK 2048

/* return codes */
#define DSA_OK 0
#define DSA_ERR_INVALID_ARG (-1)
#define DSA_ERR_UNSUPPORTED (-2)
#define DSA_ERR_WORKSPACE_TOO_SMALL (-3)
#define DSA_ERR_CUDA (-4)
#define DSA_ERR_TIMEOUT (-5)

/* bits OR-ed into *dev_status by the kernels */
#define DSA_STATUS_BAD_PAGE 0x1      /* block_table entry outside [0, num_pages) */
#define DSA_STATUS_BAD_METADATA 0x2  /* q_len < 0, seq_len < q_len, seq_len > 64*max_blocks */
#define DSA_STATUS_TIMEOUT 0x4       /* a bounded on-chip wait gave up; results invalid */

/* Version of this ABI (major*100 + minor). */
int dsa_abi_version(void);

/* Thread-local message describing the last non-zero return on this thread. */
const char* dsa_last_error(void);

/*
 * Steps 1 ([HBM] §2.3 and [KV] write path): quantise the FP32 key of every
 * new token and store it in the paged cache.
 *   k              [T, 128] FP32, row t = key of query row t.
 *   k_cache        [num_pages, 8448] uint8, this layer's page pool (written).
 *   slot_mapping   [T] int64 or NULL; receives page*64 + pos%64 per token.
 * Tokens whose page is invalid are not written (slot -1, DSA_STATUS_BAD_PAGE).
 * Errors: INVALID_ARG (null required pointer, T < 0, R < 1, max_blocks < 1,
 * num_pages < 1); CUDA (launch failure).
 */
int dsa_indexer_write_k(const float* k, int T, const int32_t* query_start_loc,
                        const int32_t* seq_lens, int R, const int32_t* block_table,
                        int max_blocks, uint8_t* k_cache, int64_t num_pages,
                        int64_t* slot_mapping, int32_t* dev_status, dsa_stream_t stream);

/*
 * Step 1 with BF16 inputs, and the upstream query quantisation fused into the
 * same launch (the cache write of the page "GLM-5.3 推理全链路(十二)" takes the
 * key already quantised; here one kernel quantises both the new keys and the
 * layer's query rows with the rule of the cache write).  The pages print no
 * BF16 interface; BF16 widens to FP32 exactly, so the results equal
 * dsa_indexer_write_k / dsa_quantize_fp8_blocks on the widened values.
 *   k          [T, 128] BF16 (16-byte aligned) new-token keys.
 *   q          [T, H, 128] BF16 query rows, or NULL (keys only).
 *   q_fp8      [T, H, 128] E4M3 out, q_scale [T, H] FP32 out (when q != NULL).
 * Other arguments and errors as dsa_indexer_write_k; H must be >= 1 with q.
 */
int dsa_indexer_write_k_bf16(const void* k, int T, const int32_t* query_start_loc,
                             const int32_t* seq_lens, int R, const int32_t* block_table,
                             int max_blocks, uint8_t* k_cache, int64_t num_pages,
                             const void* q, int H, uint8_t* q_fp8, float* q_scale,
                             int64_t* slot_mapping, int32_t* dev_status, dsa_stream_t stream);

/*
 * Step 1 for a compressed cache ([HBM] §5.2): like dsa_indexer_write_k, but
 * only a token with (pos+1) % compress_ratio == 0 is stored, as entry
 * pos / compress_ratio (see the conventions above); the other tokens write
 * nothing and get slot -1.  k holds one row per new token (the rows of tokens
 * that complete no entry are read but not stored).
 *   slot_mapping  [T] int64 or NULL: page*64 + entry%64, or -1.
 * Errors: as dsa_indexer_write_k, plus INVALID_ARG for compress_ratio < 1.
 */
int dsa_indexer_write_k_compressed(const float* k, int T, const int32_t* query_start_loc,
                                   const int32_t* seq_lens, int R, const int32_t* block_table,
                                   int max_blocks, uint8_t* k_cache, int64_t num_pages,
                                   int compress_ratio, int64_t* slot_mapping,
                                   int32_t* dev_status, dsa_stream_t stream);

/*
 * Per-block FP8 quantiser used for keys, exposed for queries: x [n_blocks, 128]
 * FP32 -> codes [n_blocks, 128] E4M3 bytes + scales [n_blocks] FP32, same rule
 * as the cache write ([KV] byte-accounting table: 128 FP8 bytes + one FP32
 * scale per 128-element block).  Used to produce q_fp8 / q_scale.
 */
int dsa_quantize_fp8_blocks(const float* x, int64_t n_blocks, uint8_t* codes, float* scales,
                            dsa_stream_t stream);

/*
 * Bytes of device workspace that dsa_indexer_score_topk / dsa_layer_stack_run
 * need for a batch of T query rows with H heads and this index_topk.  Returns
 * 0 for invalid arguments.  Pure host function.
 *   max_ctx  0, or a bound on the keys any query row sees (its request's
 *            seq_len; seq_len / compress_ratio for a compressed cache; 64 x
 *            max_blocks always bounds it).  For a decode batch (no
 *            request with more than one query row), 0 < max_ctx <= 8192 adds
 *            room for per-row key areas: the rows are then scored into the
 *            workspace and their top-k selected by a second kernel, instead
 *            of being selected (and, when cut across SMs, merged) inside the
 *            scoring kernel (should a row exceed the bound after all, the
 *            whole batch takes the in-kernel path).  The results are
 *            the same (exact top-k; ties at the k-th score may be broken
 *            differently).  The scoring calls detect the room from their
 *            workspace_bytes argument; the rows take at most 256 MB.
 */
size_t dsa_indexer_workspace_bytes(int T, int H, int R, int64_t max_ctx, int index_topk);

/*
 * Steps 2-3 ([DSA] score, [IC] §二 top-k into the shared buffer): for every
 * query row t in [0, T), score the keys s <= pos(t) of its request,
 *   score = k_scale[s] * sum_h (w[t,h] * q_scale[t,h]) * ReLU(q_fp8[t,h] . k_fp8[s])
 * and write the indices of the index_topk largest into row t of topk_buffer,
 * then -1 up to index_topk.  Rows >= T are not touched.
 *   q_fp8      [T, H, 128] E4M3 bytes; q_scale, w: [T, H] FP32.
 *   k_cache    [num_pages, 8448] uint8, already holding every key s < seq_len.
 *   topk_buffer [max_num_batched_tokens, index_topk] int32, T <= max_num_batched_tokens.
 *   scores_out optional [T, scores_ld] FP32 debug dump: scores_out[t, s] for
 *              every visible key (other entries untouched); NULL in production.
 *   workspace  >= dsa_indexer_workspace_bytes(T, H, R, 0, index_topk) bytes,
 *              256-byte aligned, contents need not be initialised.
 * H must be one of 4, 8, 16, 32, 64, 128 and 1 <= index_topk <= 2048
 * (UNSUPPORTED otherwise).  Errors: INVALID_ARG, UNSUPPORTED,
 * WORKSPACE_TOO_SMALL, CUDA.
 */
int dsa_indexer_score_topk(const uint8_t* q_fp8, const float* q_scale, const float* w, int T,
                           int H, const uint8_t* k_cache, int64_t num_pages,
                           const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                           const int32_t* block_table, int max_blocks, int index_topk,
                           int32_t* topk_buffer, int max_num_batched_tokens, float* scores_out,
                           int64_t scores_ld, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, dsa_stream_t stream);

/*
 * Steps 2-3 over a compressed cache: as dsa_indexer_score_topk, with row t
 * ranking the entries c < (pos(t)+1) / compress_ratio and returning entry
 * numbers; scores_out[t, c] is indexed by entry.  compress_ratio = 1 is
 * dsa_indexer_score_topk.  DSA_STATUS_BAD_METADATA also flags
 * seq_len / compress_ratio > 64 * max_blocks.
 * Errors: as dsa_indexer_score_topk, plus INVALID_ARG for compress_ratio < 1.
 */
int dsa_indexer_score_topk_compressed(const uint8_t* q_fp8, const float* q_scale, const float* w,
                                      int T, int H, const uint8_t* k_cache, int64_t num_pages,
                                      const int32_t* query_start_loc, const int32_t* seq_lens,
                                      int R, const int32_t* block_table, int max_blocks,
                                      int compress_ratio, int index_topk, int32_t* topk_buffer,
                                      int max_num_batched_tokens, float* scores_out,
                                      int64_t scores_ld, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_status, dsa_stream_t stream);

/*
 * Same computation and arguments as dsa_indexer_score_topk (without the debug
 * score dump), but it allocates nothing and takes no workspace argument: it
 * uses a workspace of DSA_NO_ALLOC_WORKSPACE_BYTES compiled into the library
 * as a static device array.  The pages describe no such entry point; it
 * exists for callers that cannot call cudaMalloc or take memory from their
 * host framework at the moment they run the indexer -- e.g. an inference
 * server whose device memory is fully owned by its own pool, a plugin host
 * that forbids allocation inside its enqueue callback, or code running while
 * another component captures the stream into a CUDA graph.
 *   - Memory: every GPU that loads this library holds the array until the
 *     process exits.
 *   - Set-up: the first call on each device looks the array's device address
 *     up (cudaGetSymbolAddress) with that device current and caches it with
 *     the identity of the device's current context; make that first call
 *     before any stream capture.  After a device reset (cudaDeviceReset) the
 *     next call sees a new context and looks the address up again, so make
 *     that call, too, before any capture.
 *   - Errors: the argument checks of dsa_indexer_score_topk, with the same
 *     codes, come first.
 *   - Sharing: all calls share the one array and it keeps the previous call's
 *     contents (each call re-initialises what it needs).  Calls whose kernels
 *     overlap on the GPU (other streams, other threads) race on it: serialise
 *     them.
 *   - Limit: batches needing more than DSA_NO_ALLOC_WORKSPACE_BYTES of
 *     workspace (dsa_indexer_workspace_bytes) return
 *     DSA_ERR_WORKSPACE_TOO_SMALL; use dsa_indexer_score_topk for those.
 */
#define DSA_NO_ALLOC_WORKSPACE_BYTES ((size_t)16 << 20)
int dsa_indexer_score_topk_no_alloc(const uint8_t* q_fp8, const float* q_scale, const float* w,
                                    int T, int H, const uint8_t* k_cache, int64_t num_pages,
                                    const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                                    const int32_t* block_table, int max_blocks, int index_topk,
                                    int32_t* topk_buffer, int max_num_batched_tokens,
                                    int32_t* dev_status, dsa_stream_t stream);

/* Size in bytes of the workspace built into the library for the entry point above. */
size_t dsa_indexer_no_alloc_workspace_bytes(void);

/*
 * Step 4, [IC] §三/§四: 1 if DSA layer `layer_id` is an F layer, 0 if S, <0 on
 * error.  With a pattern (NUL-terminated string of 'F'/'S') the pattern
 * decides and layers at or beyond its length are F; otherwise the layer
 * skips iff max(layer_id - offset + 1, 0) % freq != 0.  Pure host function.
 */
int dsa_layer_is_full(int layer_id, const char* pattern, int freq, int offset);

/* Per-layer inputs of dsa_layer_stack_run; S layers may leave every field NULL.
 * score_begin / score_end: optional cudaEvent_t handles (NULL = none) that are
 * recorded on the stream immediately before this layer's scoring kernel and
 * after its top-k selection (the scoring kernel, and the row-selection kernel
 * when the batch takes that path), so a caller can time scoring + selection
 * inside a larger (or captured) step. */
typedef struct dsa_layer_io {
  const float* k;         /* [T, 128] FP32 new-token keys of this layer */
  const uint8_t* q_fp8;   /* [T, H, 128] E4M3 queries */
  const float* q_scale;   /* [T, H] */
  const float* w;         /* [T, H] head weights */
  uint8_t* k_cache;       /* [num_pages, 8448] this layer's page pool */
  void* score_begin;      /* cudaEvent_t or NULL */
  void* score_end;        /* cudaEvent_t or NULL */
} dsa_layer_io;

/*
 * Steps 1-4 over a layer stack in one call ([IC] §二: F layers write the
 * shared topk buffer; S layers build no indexer and consume what the last F
 * layer wrote in this pass).  The batch plan is built once and reused by all
 * F layers.
 *   layers                HOST array [num_layers] of device-pointer structs.
 *   pattern / freq / offset  as dsa_layer_is_full; the first layer must be F.
 *   per_layer_topk_out    HOST array [num_layers] of device pointers, each
 *                         [T, index_topk] int32 or NULL, or NULL altogether:
 *                         receives rows [0, T) of the buffer as layer l
 *                         consumes it (a copy made after layer l).
 *   slot_mapping          [T] int64 or NULL, from the first F layer.
 * Within an F layer the scoring kernel starts streaming cache pages while the
 * layer's cache write still runs, but only pages whose entries all lie below
 * the request's first new position (seq_len - q_len); so a physical page that
 * receives a new key in this call must hold no earlier position of another
 * request (the paged-cache convention: only full pages are shared).
 * Errors: as dsa_indexer_score_topk, plus INVALID_ARG for a bad pattern,
 * freq <= 0, a first layer that is S, or an F layer with a NULL field.
 */
int dsa_layer_stack_run(int num_layers, const char* pattern, int freq, int offset,
                        const dsa_layer_io* layers, int T, int H,
                        const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                        const int32_t* block_table, int max_blocks, int64_t num_pages,
                        int index_topk, int32_t* topk_buffer, int max_num_batched_tokens,
                        int32_t* const* per_layer_topk_out, int64_t* slot_mapping,
                        void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        dsa_stream_t stream);

/*
 * dsa_layer_stack_run over compressed caches: every F layer writes its keys
 * as dsa_indexer_write_k_compressed and scores as
 * dsa_indexer_score_topk_compressed, with one compress_ratio for the stack.
 * Arguments, schedule and errors otherwise as dsa_layer_stack_run.
 */
int dsa_layer_stack_run_compressed(int num_layers, const char* pattern, int freq, int offset,
                                   const dsa_layer_io* layers, int T, int H,
                                   const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                                   const int32_t* block_table, int max_blocks, int64_t num_pages,
                                   int compress_ratio, int index_topk, int32_t* topk_buffer,
                                   int max_num_batched_tokens, int32_t* const* per_layer_topk_out,
                                   int64_t* slot_mapping, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, dsa_stream_t stream);

/* Per-layer inputs of dsa_layer_stack_run_bf16 (BF16 keys and queries). */
typedef struct dsa_layer_io_bf16 {
  const void* k;          /* [T, 128] BF16 new-token keys of this layer */
  const void* q;          /* [T, H, 128] BF16 query rows */
  const float* w;         /* [T, H] head weights */
  uint8_t* k_cache;       /* [num_pages, 8448] this layer's page pool */
  uint8_t* q_fp8;         /* [T, H, 128] scratch: this layer's quantised queries */
  float* q_scale;         /* [T, H] scratch: their scales */
  void* score_begin;      /* cudaEvent_t or NULL */
  void* score_end;        /* cudaEvent_t or NULL */
} dsa_layer_io_bf16;

/*
 * dsa_layer_stack_run with BF16 keys and queries: each F layer's cache write
 * also quantises its query rows into the layer's q_fp8 / q_scale scratch (one
 * launch, dsa_indexer_write_k_bf16), which its scoring kernel then reads.
 * Arguments, schedule and errors as dsa_layer_stack_run.
 */
int dsa_layer_stack_run_bf16(int num_layers, const char* pattern, int freq, int offset,
                             const dsa_layer_io_bf16* layers, int T, int H,
                             const int32_t* query_start_loc, const int32_t* seq_lens, int R,
                             const int32_t* block_table, int max_blocks, int64_t num_pages,
                             int index_topk, int32_t* topk_buffer, int max_num_batched_tokens,
                             int32_t* const* per_layer_topk_out, int64_t* slot_mapping,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             dsa_stream_t stream);

/*
 * ---------------------------------------------------------------------------
 * Sparse MLA attention over the top-k buffer (the consumer of steps 1-4).
 *
 * Sources: [KV] the list above the byte-accounting table (the main KV of a
 * token in one layer is an fp8_ds_mla record of 656 B: a 512-d KV latent and
 * a 64-d RoPE part as 576 FP8 bytes plus 16 B of FP32 scales for each of five
 * 128-element blocks; 656 x 64 = 41,984 B per page) and its page-table passage
 * (the indexer cache and the main KV share slot numbers); [RFC] "RFC:
 * DeepseekV32 模型适配支持" §2.1.3 (the top-k is a 0 / -inf mask on the q.k
 * scores, i.e. attention over the selected tokens only).
 *
 * Record layout (DSA_MLA_RECORD_BYTES per token, 64 records per page row of
 * DSA_MLA_PAGE_BYTES, record of position p at (p % 64) * 656 of page
 * block_table[r, p / 64]): bytes [0, 576) E4M3 codes of [latent | RoPE];
 * bytes [576, 656) 20 FP32 scales, scale j for elements [32 j, 32 j + 32),
 * slots 18 and 19 zero.  Each 32-element group is quantised with the rule of
 * the indexer cache (s = amax / 448, codes E4M3(x / s) RNE, saturating).
 * ---------------------------------------------------------------------------
 */
#define DSA_MLA_DIM 576
#define DSA_MLA_LATENT 512
#define DSA_MLA_RECORD_BYTES 656
#define DSA_MLA_PAGE_BYTES 41984

/*
 * Quantise each new token's 576-vector [latent | RoPE] (FP32 [T, 576], 16-byte
 * aligned) into its record of kv_cache [num_pages, 41984] (this layer's main
 * KV pool), at the slot of the indexer's slot mapping (same block table).
 * slot_mapping [T] int64 or NULL.  Bad pages / metadata: as
 * dsa_indexer_write_k.  Errors: INVALID_ARG, CUDA.
 */
int dsa_mla_write_kv(const float* kv, int T, const int32_t* query_start_loc,
                     const int32_t* seq_lens, int R, const int32_t* block_table, int max_blocks,
                     uint8_t* kv_cache, int64_t num_pages, int64_t* slot_mapping,
                     int32_t* dev_status, dsa_stream_t stream);

/*
 * For every query row t in [0, T) and head h < Hq (absorbed MLA):
 *   out[t, h, :] = sum_s softmax_s(softmax_scale * q[t,h] . key_s) * key_s[0:512]
 *   lse[t, h]    = ln sum_s exp(softmax_scale * q[t,h] . key_s)
 * over the tokens s of row t of topk_indices (entries >= 0 and < seq_len of
 * the row's request; -1 selects nothing), key_s = the dequantised 576-vector
 * of s's record.  A row selecting nothing gives out = 0, lse = -inf.
 *   q            [T, Hq, 576] BF16 (16-byte aligned), 1 <= Hq <= 128.
 *   topk_indices [>= T, index_topk] int32 (the indexer's buffer), index_topk <= 2048.
 *   out          [T, Hq, 512] BF16 (16-byte aligned); lse [T, Hq] FP32 or NULL.
 * Entries >= seq_len set DSA_STATUS_BAD_METADATA and are skipped; tokens on a
 * page outside the pool set DSA_STATUS_BAD_PAGE and contribute zero keys.
 * Computation: keys dequantised to BF16, tensor-core products with FP32
 * accumulation, probabilities rounded to BF16.  Errors: INVALID_ARG,
 * UNSUPPORTED, CUDA.
 */
int dsa_sparse_mla_attention(const void* q, int T, int Hq, const uint8_t* kv_cache,
                             int64_t num_pages, const int32_t* query_start_loc,
                             const int32_t* seq_lens, int R, const int32_t* block_table,
                             int max_blocks, const int32_t* topk_indices, int index_topk,
                             float softmax_scale, void* out, float* lse, int32_t* dev_status,
                             dsa_stream_t stream);

/*
 * Number of kernel launches the last successful call of each entry point on
 * this thread enqueued (for launch accounting by benchmarks).
 */
int dsa_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_INDEXER_H_ */
