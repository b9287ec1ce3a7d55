/*
 * tq.h - TurboQuant-style KV-cache compression and decode attention over the
 * compressed cache, for NVIDIA GB300 (sm_103a).  C ABI of libtq.so.
 *
 * What is computed (sources are cited by page title and section):
 *
 *   Encode, per (token, KV head) vector x of head_dim d
 *   ("TurboQuant+ KV cache compression", Stage 1 and Stage 2 step lists):
 *     n = ||x||, x_hat = x / n;  y = H_d diag(s) x_hat  (seeded random signs s,
 *     orthonormal Walsh-Hadamard H_d);  idx_i = Lloyd-Max index of y_i for the
 *     Gaussian N(0, 1/d) with 2^b levels;  store idx and n.
 *     K formats add the QJL stage: r = y - c[idx], store rnorm = n ||r|| and
 *     sigma_j = [(S r)_j > 0] for an iid N(0, 1) d x d matrix S
 *     ("TurboQuant+ deep dive", section 2.3: sign of the projection).
 *     V formats keep stage 1 only ("TurboQuant+ KV cache compression",
 *     K/V asymmetric strategy).
 *
 *   Decode attention, one query token per sequence:
 *     q_rot = H_d diag(s) q;  Sq = S q_rot;
 *     score_j = scale (n_j <q_rot, c[idx_j]> + rnorm_j sqrt(pi/2)/d <Sq, 2 sigma_j - 1>);
 *     online softmax over the context; V accumulated in the rotated space as
 *     n_j c_V[idx_j], skipping tokens whose weight is below skip_threshold
 *     ("TurboQuant+: 3.8x compression ...", core content item 4, Sparse V);
 *     split-K partials merged by log-sum-exp; out = diag(s) H_d acc / l.
 *
 * Conventions for every function below
 *   - All device pointers are CUDA device (or managed) memory of the device that
 *     was current when the context was created; host pointers are noted "host".
 *   - The caller allocates and owns every buffer: inputs, caches, workspace,
 *     outputs.  The library allocates only the small tables inside a context.
 *   - Device work is enqueued on `stream` (NULL = the legacy default stream) and
 *     is asynchronous; nothing is synchronised unless stated.
 *   - Arguments are validated on the host before any launch; an invalid call
 *     launches nothing and returns TQ_ERR_INVALID_ARG / TQ_ERR_UNSUPPORTED /
 *     TQ_ERR_WORKSPACE.  A failed launch returns TQ_ERR_CUDA.  Nothing aborts,
 *     nothing throws across the ABI.
 *   - Values that only the device can see (sequence lengths, block-table
 *     entries, slot ids) are bounds-checked in the kernels: an offending item is
 *     skipped and a bit is set in the context's device status word, read with
 *     tq_get_status().
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime's stream handle); NULL is the legacy default stream. */
typedef struct CUstream_st* tq_stream_t;

typedef enum tq_status {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,  /* bad pointer, size, format, stride or a device-side bounds flag */
  TQ_ERR_UNSUPPORTED = 2,  /* valid request outside what this build implements (e.g. d = 96) */
  TQ_ERR_WORKSPACE = 3,    /* workspace smaller than tq_decode_workspace_bytes() */
  TQ_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  TQ_ERR_OOM = 5           /* context tables could not be allocated */
} tq_status;

/*
 * Storage formats.  Stage-1 bits and QJL bit per element follow the format
 * table of "TurboQuant+ KV cache compression" (turbo2 = 1+1, turbo3 = 2+1,
 * turbo4 = 3+1); the _MSE variants are the V forms with stage 1 only (turbo4
 * V = 3 bits, same page, K/V asymmetric strategy).  Q8_0 is the pages' int8
 * baseline cache type (absmax / 127 per block of 32, "TurboQuant+ deep dive"
 * section 2.1 with n = 8).  MINMAX is the per-group asymmetric min-max
 * quantiser of "mac-code TurboQuant analysis" section 2.1 (group 64,
 * cache_view.bits = 2, 3 or 4).
 */
typedef enum tq_format {
  TQ_FMT_TURBO2 = 0,
  TQ_FMT_TURBO3 = 1,
  TQ_FMT_TURBO4 = 2,
  TQ_FMT_TURBO2_MSE = 3,
  TQ_FMT_TURBO3_MSE = 4,
  TQ_FMT_TURBO4_MSE = 5,
  TQ_FMT_Q8_0 = 6,
  TQ_FMT_MINMAX = 7
} tq_format;

/*
 * Byte layout of one stored vector (one token of one KV head of one layer).
 * Each vector has a payload and a header, kept in two separate arrays.
 *
 *   turbo (K and V): each coordinate i has a w-bit code, w = b (+1 for K):
 *     bits [0, b) = Lloyd-Max index (ascending level order), bit b = QJL sign
 *     (K only, 1 = positive projection).  Codes are packed little-endian,
 *     coordinate i at bit offset w*i of the payload; so every group of 32
 *     coordinates ("block-32") fills exactly w 32-bit words.
 *     payload = d*w/8 bytes.  header: K = {fp16 n, fp16 rnorm}, V = {fp16 n}.
 *   q8_0: payload = d int8 values; header = d/32 fp16 scales (block order).
 *   minmax: codes of `bits` bits packed as for turbo; header = d/64 pairs
 *     {fp16 scale, fp16 zero} (group order).
 *
 * Cache view: a 4-D array of vectors [n_layers][num_pages][n_kv_heads][page_size].
 * The vector at (layer, page, head, p) has index
 *     v = ((layer * num_pages + page) * n_kv_heads + head) * page_size + p
 * and lives at payload + v * tq_payload_bytes(), header + v * tq_header_bytes().
 * Token slot t of a layer means page = t / page_size, p = t % page_size, so a
 * contiguous cache of capacity C per sequence is the view with page_size = C
 * and page = sequence index (block_table = NULL in tq_decode_attention).
 */
typedef struct tq_cache_view {
  int32_t format;      /* tq_format */
  int32_t head_dim;    /* d: 64, 128 or 256 */
  int32_t n_kv_heads;  /* H >= 1 */
  int32_t page_size;   /* tokens per page >= 1 */
  int64_t num_pages;   /* pages per layer >= 1 */
  int32_t n_layers;    /* layers held by this view >= 1 */
  int32_t bits;        /* TQ_FMT_MINMAX only: 2, 3 or 4; ignored otherwise */
  void* payload;       /* device, 16-byte aligned */
  void* header;        /* device, 4-byte aligned */
} tq_cache_view;

typedef struct tq_context tq_context;

/* ---- sizes and names (host, pure functions) ---- */

const char* tq_status_string(tq_status s);
const char* tq_format_name(tq_format f);
/* Payload / header bytes of one vector; 0 for an invalid (format, head_dim, bits). */
size_t tq_payload_bytes(tq_format f, int head_dim, int bits);
size_t tq_header_bytes(tq_format f, int head_dim, int bits);
/* payload + header, the compressed bytes of one vector. */
size_t tq_vector_bytes(tq_format f, int head_dim, int bits);

/* ---- host math ---- */

/*
 * Lloyd-Max quantiser for N(0, 1/head_dim) with 2^bits levels, bits in 1..4
 * ("TurboQuant+ KV cache compression", Stage 1 step 3: optimal codebook for the
 * Gaussian precomputed with Lloyd's algorithm).  Iterated in double precision:
 * boundaries = midpoints, centroids = conditional means of their cells, until no
 * centroid moves by more than 1e-13 sigma.  Writes (host) centroids[2^bits] and
 * boundaries[2^bits - 1], ascending, rounded to float (boundaries are the
 * double midpoints rounded once).  head_dim >= 1.
 */
tq_status tq_codebook_build(int bits, int head_dim, float* centroids, float* boundaries);

/*
 * Default random tables, counter based (SplitMix64 of Steele, Lea and Flood,
 * evaluated at counter (seed << 32) + k).  seed < 2^32.
 *   signs[i] = -1 if the top bit of SplitMix64(c_i) is set else +1   (host int8 [d])
 *   S[j*d + i] = sqrt(-2 ln u1) cos(2 pi u2), u = ((SplitMix64(c) >> 11) + 1) 2^-53
 *                at counters 2(j*d+i), 2(j*d+i)+1, computed in double, rounded
 *                to float                                           (host float [d*d])
 */
tq_status tq_signs_generate(uint32_t seed, int head_dim, int8_t* signs);
tq_status tq_qjl_matrix_generate(uint32_t seed, int head_dim, float* S);

/* ---- context: the per-head_dim tables on the current device ---- */

/*
 * Creates a context for one head_dim (64, 128 or 256) on the current device:
 * the sign diagonal, the QJL matrix S (row j = projection j) and the turbo
 * codebooks for 1, 2 and 3 bits.  `signs` (host int8 [d], +-1) and `qjl` (host
 * float [d*d]) may be NULL, in which case the default generators are used with
 * wht_seed / qjl_seed; when given they are copied.  Synchronous.  The context
 * is immutable afterwards (except its status word) and may be used from any
 * stream of that device.  Returns TQ_ERR_UNSUPPORTED for other head_dim.
 */
tq_status tq_context_create(int head_dim, uint32_t wht_seed, uint32_t qjl_seed,
                            const int8_t* signs, const float* qjl, tq_context** out);
tq_status tq_context_destroy(tq_context* ctx);

/*
 * Copies the context's tables to host memory (any pointer may be NULL):
 * signs int8 [d]; qjl float [d*d]; centroids float [3][8] and boundaries
 * float [3][7] for bits 1, 2, 3 (unused entries zero).  Synchronous.
 */
tq_status tq_context_get_tables(const tq_context* ctx, int8_t* signs, float* qjl,
                                float* centroids, float* boundaries);

/*
 * Reads and clears the context's device status word (synchronises the device).
 * *flags (host, may be NULL) receives the bits: 1 = a sequence length above
 * max_ctx or the view's capacity was clamped, 2 = a block-table entry out of
 * [0, num_pages) was skipped, 4 = a slot id out of range was skipped, 8 = a
 * bounded wait for the tensor cores ran out (the results of that call are not
 * valid).  Returns TQ_ERR_INVALID_ARG if any bit was set, else TQ_OK.
 */
tq_status tq_get_status(tq_context* ctx, uint32_t* flags);

/* ---- encode ---- */

/*
 * Compresses fp16 K and/or V vectors into cache views (either pair may be NULL,
 * not both).  Input element (l, t, h, i) of K is
 *     k[l * in_layer_stride + t * in_token_stride + h * d + i]
 * for l < n_layers, t < n_tokens, h < n_kv_heads of the view, i < d (same for V);
 * strides are in elements and heads are contiguous d-vectors.  k and v must be
 * 16-byte aligned and both strides multiples of 8 elements (the inputs are read
 * with 16-byte loads), else TQ_ERR_INVALID_ARG.  Layer l of the
 * input goes to layer layer_begin + l of the view.  Token t goes to slot
 * slots[t] (device int64 [n_tokens]) when `slots` is non-NULL, else to slot
 * slot_begin + t; a slot outside [0, num_pages * page_size) is skipped and
 * flagged.  K views take any format except the _MSE ones; V views take any
 * format; both views must share head_dim and n_kv_heads with the context's d.
 * Turbo K: stage 1 + QJL; turbo _MSE: stage 1; Q8_0; MINMAX.
 */
tq_status tq_encode_kv(const tq_context* ctx,
                       const tq_cache_view* k_view, const void* k,
                       const tq_cache_view* v_view, const void* v,
                       int layer_begin, int n_layers, int n_tokens,
                       int64_t in_layer_stride, int64_t in_token_stride,
                       const int64_t* slots, int64_t slot_begin,
                       tq_stream_t stream);

/* ---- decode attention ---- */

/*
 * Bytes of workspace tq_decode_attention needs for these sizes (split-K
 * partials plus the rotated queries).  Depends only on its arguments and on the
 * context's device.
 */
size_t tq_decode_workspace_bytes(const tq_context* ctx, int n_layers, int batch,
                                 int n_q_heads, int max_ctx);

/*
 * One decode step of attention for `batch` sequences over n_layers layers.
 *   q:   device [n_layers][batch][n_q_heads][d], fp32 (q_is_fp16 = 0) or fp16 (1).
 *   out: device float [n_layers][batch][n_q_heads][d].
 *   Layer l reads layer layer_begin + l of k_view and v_view.
 *   Query head h reads KV head h / (n_q_heads / n_kv_heads); n_q_heads must be
 *   a multiple of n_kv_heads.
 *   seq_lens: device int32 [batch]; sequence b attends to its tokens [0, seq_lens[b]).
 *   max_ctx: host upper bound on every seq_lens[b] (sizes the split-K grid).
 *   block_table: device int32 [batch][max_blocks_per_seq] mapping logical page
 *     t / page_size of sequence b to a physical page, or NULL for page = b.
 *   softmax_scale: the logit scale (1/sqrt(d) in the usual model).
 *   skip_threshold: V terms whose weight exp(s - running max) is below it are
 *     not accumulated (Sparse V); 0 keeps every term.  The softmax denominator
 *     keeps every token.
 *   workspace: device scratch of tq_decode_workspace_bytes() bytes, 256-byte
 *     aligned; its contents are undefined after the call (the combine drops the
 *     split partials from L2 without writing them back).
 *   K formats: turbo (with or without QJL) or Q8_0.  V formats: turbo _MSE or
 *   Q8_0.  A sequence of length 0 yields zeros.
 *   The call is three kernels on `stream`: the query prologue, the split-K
 *   attention (launched as a programmatic dependent of the prologue) and the
 *   combine (a dependent of the attention); work queued after it on the stream
 *   sees the finished result, as after any kernel.
 */
tq_status tq_decode_attention(const tq_context* ctx,
                              const void* q, int q_is_fp16,
                              int n_layers, int batch, int n_q_heads,
                              const tq_cache_view* k_view, const tq_cache_view* v_view,
                              int layer_begin,
                              const int32_t* seq_lens, int max_ctx,
                              const int32_t* block_table, int max_blocks_per_seq,
                              float softmax_scale, float skip_threshold,
                              void* workspace, size_t workspace_bytes,
                              float* out, tq_stream_t stream);

/*
 * tq_decode_attention without a caller workspace, for callers that cannot
 * allocate device memory when they run decode attention (a process whose
 * device memory is all reserved by its own pool, code inside an allocator
 * callback, a plug-in that only receives its inputs and outputs).  The paper
 * has no counterpart: this is a deployment variant of the same computation.
 *
 * Same arguments and result as tq_decode_attention minus the workspace pair.
 * The workspace is a fixed 16 MiB array inside libtq.so (every GPU that loads
 * the library keeps it until exit); a call whose tq_decode_workspace_bytes()
 * exceeds 16 MiB returns TQ_ERR_WORKSPACE and launches nothing.  The first call
 * on a device looks the array's device address up (with that device current)
 * and should come before any stream capture; the address is kept for the life
 * of the process, so the entry point must not be used on a device after
 * cudaDeviceReset (the library's module, and the array with it, is gone).  All
 * calls share the array: calls that overlap on the GPU race.  The context's
 * device must be current.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
tq_status tq_decode_attention_static(const tq_context* ctx,
                                     const void* q, int q_is_fp16,
                                     int n_layers, int batch, int n_q_heads,
                                     const tq_cache_view* k_view, const tq_cache_view* v_view,
                                     int layer_begin,
                                     const int32_t* seq_lens, int max_ctx,
                                     const int32_t* block_table, int max_blocks_per_seq,
                                     float softmax_scale, float skip_threshold,
                                     float* out, tq_stream_t stream);

/* ---- per-layer views: a K and a V format per layer ---- */

/*
 * Layer policies that give some layers another format, as in Boundary V ("TurboQuant+: 3.8x
 * compression ...", core content item 3: q8_0 V on the first 2 and last 2 layers, turbo2 V
 * elsewhere; "TurboQuant+ deep dive", section 3.2, layer-wise V strategy), or asymmetric K/V
 * pairs per layer (same page's item 2; deep dive section 3.1), are expressed with one view per
 * layer: layer l is stored at layer k_view_layers[l] of k_views[l] (host arrays [n_layers]) and
 * at layer v_view_layers[l] of v_views[l].  Views may repeat (a view holding several layers).
 * Every layer's views must share head_dim (the context's) and n_kv_heads; the K and V views of a
 * layer must share page_size and num_pages.
 */

/*
 * tq_encode_kv over per-layer views: input layer l (at k + l * in_layer_stride elements, same for
 * v) is encoded into layer k_view_layers[l] of k_views[l] (and v_*).  k_views (with k_view_layers
 * and k) or v_views (with v_view_layers and v) may be NULL, not both.  Every layer is validated
 * before anything is launched; then runs of consecutive layers that share their views at
 * consecutive view layers are encoded by one call of tq_encode_kv each.  Errors as tq_encode_kv.
 */
tq_status tq_encode_kv_layers(const tq_context* ctx,
                              const tq_cache_view* k_views, const int32_t* k_view_layers,
                              const tq_cache_view* v_views, const int32_t* v_view_layers, int n_layers,
                              const void* k, const void* v, int n_tokens,
                              int64_t in_layer_stride, int64_t in_token_stride,
                              const int64_t* slots, int64_t slot_begin, tq_stream_t stream);

/*
 * tq_decode_attention over per-layer views, in one call: q, out, seq_lens, block_table, the scale,
 * the skip threshold and the workspace as for tq_decode_attention (layer l of q and out is query
 * layer l), the workspace sized by tq_decode_workspace_bytes(ctx, n_layers, batch, n_q_heads,
 * max_ctx).  Every layer is validated before anything is launched (TQ_ERR_INVALID_ARG /
 * TQ_ERR_UNSUPPORTED / TQ_ERR_WORKSPACE as for tq_decode_attention; more than 65535 layers or
 * view layers: TQ_ERR_UNSUPPORTED); then the layers are grouped by their (K view, V view) pair,
 * wherever they sit, and each group (128 layers at most per launch) runs the decode kernels once,
 * with the split plan tq_decode_attention would take for that group alone when it fits in the
 * workspace, else the whole call's.  The result then equals tq_decode_attention run on each group.
 */
tq_status tq_decode_attention_layers(const tq_context* ctx, const void* q, int q_is_fp16,
                                     int n_layers, int batch, int n_q_heads,
                                     const tq_cache_view* k_views, const int32_t* k_view_layers,
                                     const tq_cache_view* v_views, const int32_t* v_view_layers,
                                     const int32_t* seq_lens, int max_ctx,
                                     const int32_t* block_table, int max_blocks_per_seq,
                                     float softmax_scale, float skip_threshold,
                                     void* workspace, size_t workspace_bytes,
                                     float* out, tq_stream_t stream);

/* ---- chunked-prefill attention ---- */

/* Bytes of workspace tq_prefill_attention needs (the prepared queries). */
size_t tq_prefill_workspace_bytes(const tq_context* ctx, int n_tokens, int n_q_heads);

/*
 * Attention of a prefill chunk over the compressed cache ("TurboQuant+: 3.8x compression ...",
 * core content item 1: prefill reads the quantised cache).  The chunk's n_tokens tokens sit at
 * positions start .. start + n_tokens - 1 of one sequence and are already encoded into the cache
 * (tq_encode_kv); chunk token i attends to the cached tokens 0 .. start + i (causal, its own
 * token included), with the same compressed-domain scores as tq_decode_attention (q rotated once,
 * n_j <q', c[idx_j]> + rnorm_j sqrt(pi/2)/d <S q', sign_j>) and no Sparse V.
 *   q:   device [n_tokens][n_q_heads][d], fp32 (q_is_fp16 = 0) or fp16 (1).
 *   out: device float [n_tokens][n_q_heads][d].
 *   Query head h reads KV head h / (n_q_heads / n_kv_heads).
 *   The sequence: layer `layer` of k_view and v_view; block_table (device int32 [max_blocks],
 *   logical page -> physical page) or NULL for page `seq` of a contiguous cache.
 *   workspace: device, tq_prefill_workspace_bytes() bytes, 256-byte aligned.
 * This build: head_dim 128, K turbo2/3/4 (with the QJL stage), V turbo2/3/4_mse; other formats or
 * head_dims return TQ_ERR_UNSUPPORTED.  The products run on the fifth-generation tensor cores.
 * A block-table entry out of range sets status bit 2, and its keys are left out.
 */
tq_status tq_prefill_attention(const tq_context* ctx, const void* q, int q_is_fp16, int n_tokens, int n_q_heads,
                               const tq_cache_view* k_view, const tq_cache_view* v_view, int layer, int seq,
                               const int32_t* block_table, int max_blocks, int start, float softmax_scale,
                               void* workspace, size_t workspace_bytes, float* out, tq_stream_t stream);

/* ---- dequantize (reconstruction; test and debugging path) ---- */

/*
 * Reconstructs n slots of one layer of a view into out (device float
 * [n][n_kv_heads][d]) in the original, unrotated space.  Slot t = slots[t]
 * (device int64 [n]) or slot_begin + t.  Turbo: n diag(s) H c[idx], plus for K
 * formats with include_qjl != 0 the QJL vector-form residual
 * diag(s) H (rnorm sqrt(pi/2)/d S^T (2 sigma - 1)).  Q8_0: q * scale.
 * MINMAX: q * scale + zero.  Skipped (out-of-range) slots are written as zeros.
 */
tq_status tq_dequantize(const tq_context* ctx, const tq_cache_view* view, int layer,
                        const int64_t* slots, int64_t slot_begin, int n,
                        int include_qjl, float* out, tq_stream_t stream);

/* ---- persistence of a compressed cache (host; out of the hot path) ---- */

/*
 * A compressed cache saved to disk and read back ("mac-code TurboQuant analysis",
 * section 2.4: the compressed arrays are serialised with a small JSON metadata
 * record; here both go into one file).  File layout:
 *   the 9 bytes "TQCACHE1\n";
 *   one JSON object on one line followed by "\n", with the keys version, format,
 *     format_id, head_dim, n_kv_heads, page_size, num_pages, n_layers, bits,
 *     payload_bytes, header_bytes, wht_seed, qjl_seed, tables_hash (16 hex
 *     digits), data_hash (16 hex digits) and layout;
 *   zero bytes up to the next multiple of 4096;
 *   the view's payload array (all its layers, in the view's own order), then its
 *     header array.
 * tables_hash is FNV-1a 64 over head_dim (int32), the sign diagonal (int8 [d]),
 * the QJL matrix (float [d*d]) and the codebook tables (float [3][8], [3][7]) of
 * the context; data_hash is FNV-1a 64 over the two arrays as 64-bit
 * little-endian words, taken in blocks of 64 MiB per array (each block's trailing
 * bytes one at a time).  Codes are only meaningful with the tables they were made
 * with, so a load checks tables_hash against its context.
 */

/* FNV-1a 64 hash of the context's tables (the file's tables_hash). */
tq_status tq_context_tables_hash(const tq_context* ctx, uint64_t* hash);

/*
 * Writes every layer of `view` to `path` (created or replaced: written to
 * path + ".partial" and renamed on success).  host_memory = 0: the view's arrays
 * are device memory of the current device (the device is synchronised, the
 * arrays are copied through a host buffer of at most 64 MiB); 1: host memory.
 * ctx (may be NULL: seeds and tables_hash are then written as 0) supplies the
 * seeds and the tables hash; its head_dim must match the view's.  Synchronous.
 * Errors: TQ_ERR_INVALID_ARG (bad view, I/O failure), TQ_ERR_OOM, TQ_ERR_CUDA.
 */
tq_status tq_cache_save(const tq_context* ctx, const tq_cache_view* view, int host_memory, const char* path);

/*
 * Reads the geometry of a file written by tq_cache_save: format, head_dim,
 * n_kv_heads, page_size, num_pages, n_layers and bits into *geometry (payload and
 * header set to NULL), the tables hash into *tables_hash (may be NULL), so that a
 * caller can allocate the view to load into.  TQ_ERR_INVALID_ARG if the file is
 * missing or not such a file.
 */
tq_status tq_cache_file_info(const char* path, tq_cache_view* geometry, uint64_t* tables_hash);

/*
 * Reads a file written by tq_cache_save into `view`, whose format, head_dim,
 * n_kv_heads, page_size, num_pages, n_layers and bits must equal the file's
 * (host_memory as for tq_cache_save).  With a context, the file's tables_hash
 * must equal the context's.  The data hash is checked after the copy; on any
 * mismatch (geometry, tables, size, trailing bytes, data hash) the call returns
 * TQ_ERR_INVALID_ARG, and when the data hash alone fails the view already holds
 * the file's (corrupt) bytes.  Synchronous.
 */
tq_status tq_cache_load(const tq_context* ctx, const tq_cache_view* view, int host_memory, const char* path);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
