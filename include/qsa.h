/*
 * qsa.h - C ABI of libqsa: QSA gather-GQA sparse attention over a ragged,
 * paged KV cache, as hand-written CUDA kernels for GB300 (sm_103a).
 *
 * The operation is the one the MAX kernel page "QSASparseAttentionRaggedPaged"
 * documents ("Gather-GQA over the token indices a QSA selection names"; its
 * "Tensor shapes" list, the `execute` method's parameters and arguments, and
 * its "Raises" clause):
 *
 *   for each query row r of sequence b (input_row_offsets[b] <= r < [b+1]),
 *   each kv head h in [0, num_kv_heads) and each i in [0, group):
 *     n   = min(max(counts[r], 0), selection_width)
 *     p_j = token_indices[r, j]  for j < n       (entries at or past counts
 *                                                 are never read)
 *     K_j = kv_blocks[page, 0, layer_idx, p_j % page_size, h, :]
 *     V_j = kv_blocks[page, 1, layer_idx, p_j % page_size, h, :]
 *           with page = kv_lookup_table[b, p_j / page_size]
 *     output[r, h*group + i, :] = softmax_j(scale * q[r, h*group+i, :] . K_j) . V_j
 *
 * Conventions the page leaves open and this library fixes:
 *   - axis 1 of kv_blocks is K at index 0 and V at index 1;
 *   - query head h*group+i reads kv head h (consecutive query heads share);
 *   - no causal mask: exactly the listed positions are attended;
 *   - n == 0 (counts <= 0) writes a zero row; counts > selection_width is
 *     clamped to selection_width; a repeated index is its own softmax term;
 *   - a position outside [0, cache_lengths[b] + rows_b) inside the valid
 *     prefix (or a page-table entry >= num_pages) is skipped and recorded in
 *     the library's device status word (see qsa_read_device_status); it is
 *     never dereferenced;
 *   - FP8 is e4m3fn and scale-free: stored bytes are the values themselves.
 *
 * Memory, ownership, errors:
 *   - every qsa_tensor `data` is a DEVICE pointer on the current CUDA device,
 *     contiguous row-major (kv_blocks: its page axis is `page_stride`
 *     elements apart); the caller owns every buffer and the stream, and must
 *     keep them alive until the work enqueued on `stream` has finished.
 *   - calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  No call reads device memory on the host, synchronises
 *     or copies device->host, so they can be captured in a CUDA graph once the
 *     split-K workspace is sized (qsa_reserve_workspace).
 *   - argument problems are reported before anything is launched, as a
 *     non-zero qsa_status ("Raises: Error if the operand shapes disagree with
 *     the parameters"); nothing falls back to another implementation.
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QSA_API __attribute__((visibility("default")))
#else
#define QSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types.  QSA_F8E4M3 is FP8 e4m3fn (bias 7, no infinities, max 448). */
typedef enum qsa_dtype {
  QSA_F32 = 0,
  QSA_BF16 = 1,
  QSA_F8E4M3 = 2,
  QSA_U32 = 3,
  QSA_I32 = 4
} qsa_dtype;

/* A tensor descriptor: device pointer, element type (qsa_dtype), rank and
 * shape.  Unused trailing shape entries are ignored. */
typedef struct qsa_tensor {
  void* data;
  int32_t dtype;
  int32_t ndim;
  int64_t shape[6];
} qsa_tensor;

typedef enum qsa_status {
  QSA_OK = 0,
  QSA_ERR_NULL = 1,        /* a needed pointer is NULL */
  QSA_ERR_SHAPE = 2,       /* ranks or extents disagree with each other or with group */
  QSA_ERR_DTYPE = 3,       /* an operand has the wrong element type */
  QSA_ERR_UNSUPPORTED = 4, /* a legal combination this build has no kernel for */
  QSA_ERR_ARG = 5,         /* a scalar argument is out of range (layer_idx, page_stride, ...) */
  QSA_ERR_CUDA = 6         /* a CUDA runtime call failed (launch, allocation) */
} qsa_status;

/* Bits of the device status word. */
#define QSA_STATUS_BAD_INDEX 1u /* a position inside counts outside [0, kv_len) */
#define QSA_STATUS_BAD_PAGE 2u  /* p / page_size >= max_pages or a table entry >= num_pages */
#define QSA_STATUS_BAD_ROW 4u   /* a query row owned by no sequence (bad input_row_offsets) */
#define QSA_STATUS_TIMEOUT 8u   /* a kernel gave up waiting for its own copies (never expected) */

/*
 * qsa_sparse_attention_ragged_paged - one layer of QSA sparse attention.
 *
 *   output            [total_q, num_q_heads, head_dim]  F32 or BF16, written
 *   q                 [total_q, num_q_heads, head_dim]  same type as kv_blocks
 *   input_row_offsets [batch + 1]                       U32, ragged query offsets
 *                     (nondecreasing, [0] == 0, [batch] == total_q)
 *   kv_blocks         [num_pages, 2, num_layers, page_size, num_kv_heads, head_dim]
 *                     F32, BF16 or F8E4M3; read only
 *   page_stride       elements from one page to the next; -1 = packed
 *                     (2*num_layers*page_size*num_kv_heads*head_dim);
 *                     otherwise >= that packed size
 *   cache_lengths     [batch]              U32, keys cached per sequence before
 *                     this step; the cache already holds this step's rows, so
 *                     sequence b has cache_lengths[b] + rows_b valid positions
 *   kv_lookup_table   [batch, max_pages]   U32, logical page -> physical page
 *   max_prompt_length host scalar: max new rows of any sequence (a hint only)
 *   max_cache_length  host scalar: max cache_lengths entry (a hint only)
 *   layer_idx         layer of kv_blocks to read, < num_layers
 *   token_indices     [total_q, selection_width] I32, positions within the
 *                     row's own sequence, valid entries first
 *   counts            [total_q]            I32, valid entries per row
 *   scale             multiplies q.K before the softmax
 *   group             query heads per kv head (num_q_heads == group*num_kv_heads)
 *   stream            cudaStream_t to enqueue on
 *
 * Kernel coverage: output F32 or BF16; head_dim 64 or 128.  BF16 and F8E4M3
 * with head_dim 128 run on the persistent tensor-core kernel (group 1..16),
 * or, when its units (total_q * num_kv_heads / H, H = 4, 2 or 1, the largest
 * that divides num_kv_heads) are under a quarter of the SM count, on the
 * per-(row, kv head) tensor-core kernel with split-K; the rest on the
 * CUDA-core kernel (group 1..8 or 16).
 *
 * Prefill-like BF16 calls (head_dim 128, group 4, 8 or 16, a power-of-two
 * page_size >= 8, on average at least R = 128 / group rows per sequence and
 * max_cache_length + max_prompt_length <= (128 / min(group, 8)) *
 * selection_width) run on the
 * row-group kernel: 2 R consecutive rows of a sequence share one CTA per kv
 * head, which loads the sequence's pages tile by tile once for all of them
 * and masks each row to its own positions.  It reads K and V at every
 * position of a tile some row of the group selects from.  Scores of keys a
 * row did not select are masked, and V rows of keys no row of the group
 * selects are zeroed before use, so a non-finite K anywhere, or a non-finite
 * V at a position no row of the group selects, does not reach the output.  A
 * non-finite V at a position another row of the same group selects does
 * reach the rows that did not select it (as 0 x that value): for such caches
 * force kernel 3 (qsa_options.kernel = 3).  Its workspace (one bitmap of max_cache_length +
 * max_prompt_length bits and one flag per row) comes from the same
 * per-stream workspace as split-K.  Rows that repeat a position, or whose
 * sequence is longer than the hints say, are served exactly by that
 * kernel's CUDA-core path.  Device pointers must be 16-byte aligned, and
 * page_stride * element size a multiple of 16 bytes.  kv_blocks may span up
 * to 64 GiB.
 *
 * Differences from the page's signature: page_stride, max_prompt_length and
 * max_cache_length are host scalars (the page passes them as device tensors),
 * so a call never needs a device->host read.
 *
 * When more than one CTA shares a (row, kv head), the call uses a split-K
 * workspace owned by the library, one per (device, stream), grown on demand
 * with cudaMalloc; call qsa_reserve_workspace with qsa_plan's figure first to
 * keep allocation off the hot path and out of graph capture.  Calls on the
 * same stream are ordered; calls on different streams use different
 * workspaces.
 */
QSA_API qsa_status qsa_sparse_attention_ragged_paged(
    qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets, qsa_tensor kv_blocks,
    int64_t page_stride, qsa_tensor cache_lengths, qsa_tensor kv_lookup_table,
    uint32_t max_prompt_length, uint32_t max_cache_length, uint32_t layer_idx,
    qsa_tensor token_indices, qsa_tensor counts, float scale, int32_t group, void* stream);

/* Launch controls for tests and measurement.  Zero fields mean "choose". */
typedef struct qsa_options {
  int32_t kernel;    /* 0 auto, 1 CUDA-core kernel, 2 tensor-core kernel with one
                        CTA per (row, kv head[, split]), 3 persistent stream-K
                        tensor-core kernel (the default where it applies), 4
                        row-group kernel (see "Kernel coverage"; only the
                        entry points that take max_prompt_length and
                        max_cache_length, and qsa_plan_ex, can run it) */
  int32_t splits;    /* kernel 2: 0 auto, else CTAs per (row, kv head) */
  int32_t ctas;      /* kernel 3: 0 auto (one per SM), else the persistent grid size */
  int32_t block_lists; /* qsa_plan only: nonzero plans a qsa_msa_attention_ragged_paged
                          call (block lists run kernel 2's variant with tile copies,
                          whose occupancy differs); other entry points ignore it */
  int32_t heads_per_unit; /* kernel 3: 0 auto, else the adjacent kv heads one unit gathers
                             together (1, 2, 4 or 8, dividing num_kv_heads; 8 needs group <= 8) */
  int32_t test_stall;  /* tests only: nonzero makes kernel 3's producers issue no K/V
                          copies and every wait give up after a few thousand polls, so
                          the call ends early with QSA_STATUS_TIMEOUT and an undefined
                          output; no copy is in flight when a CTA gives up */
  int32_t tcgen05;     /* kernel 2: 0 auto, 1 the tcgen05 consumer (BF16: scores and output
                          accumulate in tensor memory; the stage layout of tile copies),
                          -1 the mma.sync consumer */
  int32_t reserved[1];
} qsa_options;

/* Same as qsa_sparse_attention_ragged_paged, with explicit launch controls
 * (NULL = defaults).  A forced kernel that cannot run the case returns
 * QSA_ERR_UNSUPPORTED. */
QSA_API qsa_status qsa_sparse_attention_ragged_paged_ex(
    qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets, qsa_tensor kv_blocks,
    int64_t page_stride, qsa_tensor cache_lengths, qsa_tensor kv_lookup_table,
    uint32_t max_prompt_length, uint32_t max_cache_length, uint32_t layer_idx,
    qsa_tensor token_indices, qsa_tensor counts, float scale, int32_t group, void* stream,
    const qsa_options* options);

/*
 * qsa_msa_attention_ragged_paged - block-sparse attention: the selection is a
 * list of whole blocks per (kv head, query row) instead of token positions
 * (MAX page "Struct_msa_attention_ragged_paged": "Gathers topk KV blocks per
 * (kv head, query token) using the block ids in d_indices"; its Args list).
 *
 *   d_indices  [num_kv_heads, total_q, topk] I32, block ids per (kv head, row)
 *
 * Every other argument is as for qsa_sparse_attention_ragged_paged (no
 * token_indices or counts).  For row r of sequence b, kv head h and each of
 * its query heads, the attended keys are the slots s of each listed block
 * beta = d_indices[h, r, e] (positions beta*page_size + s, page
 * kv_lookup_table[b, beta]) whose position is <= the row's own position
 * cache_lengths[b] + (r - input_row_offsets[b]).  Readings where the page is
 * silent: a block is one page of the row's own sequence; beta < 0 marks an
 * unused slot; the position rule is the page's per-token causal masking for
 * prefill and speculative decode and, for one new token per sequence, exactly
 * "every cached key" (its decode path has no mask); a repeated block counts
 * twice; nothing attended gives a zero row; a listed block with no page
 * (beta >= max_pages, or a table entry >= num_pages) is skipped and sets
 * QSA_STATUS_BAD_PAGE.
 *
 * Runs on the per-(row, kv head) tensor-core kernel with split-K: BF16 or
 * F8E4M3 with head_dim 128, group <= 16, output F32 or BF16 (the page's op
 * always writes BF16).  `options` may set splits (kernel must be 0 or 2).
 * Differences from the page's signature: cache_row_offsets,
 * total_context_length and msa_scalar_args are not taken (the first two follow
 * from cache_lengths, the scalars are host-known), and max_prompt_length /
 * max_cache_length are host hints as above.
 */
QSA_API qsa_status qsa_msa_attention_ragged_paged(
    qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets, qsa_tensor kv_blocks,
    int64_t page_stride, qsa_tensor cache_lengths, qsa_tensor kv_lookup_table,
    uint32_t max_prompt_length, uint32_t max_cache_length, uint32_t layer_idx,
    qsa_tensor d_indices, float scale, int32_t group, void* stream, const qsa_options* options);

/*
 * qsa_latent_attention_ragged_paged - latent sparse attention: every query
 * row attends its sliding window and its listed compressed entries, with
 * per-head sinks (MAX page "latent_sparse_attention_ragged_paged": "Attends
 * every query row to its window keys and its listed compressed entries"; its
 * window, comp_indices, attn_sink and two-cache parameters).
 *
 *   output, q           [total_q, num_heads, 128]  (BF16 or F8E4M3 q; output F32/BF16)
 *   input_row_offsets   [batch + 1] U32
 *   swa_blocks          [pages, 2, num_layers, page_size, 1, 128]: the window
 *                       cache, paged by token position (swa_page_stride,
 *                       swa_cache_lengths [batch] U32: the row position is
 *                       swa_cache_lengths[b] + (r - input_row_offsets[b]),
 *                       swa_lookup_table [batch, max_pages] U32)
 *   comp_blocks         [pages2, 2, num_layers2, page_size2, 1, 128]: the
 *                       compressed cache, paged by entry (comp_page_stride)
 *   comp_cache_lengths  DEVICE pointer, [batch] U32 entries per sequence
 *   comp_lookup_table   DEVICE pointer, [batch, comp_max_pages] U32
 *   layer_idx           layer of both caches
 *   comp_indices        DEVICE pointer, [total_q, num_comp] I32 entry ids,
 *                       -1 = unused slot
 *   attn_sink           DEVICE pointer, [num_heads] F32 sink logits
 * (the per-row and per-sequence arrays of the compressed cache are plain
 * pointers with their extents given alongside, so that no descriptor is
 * passed after the eighth argument register)
 *   window              tokens: a row at pos sees positions max(0, pos -
 *                       window + 1) .. pos
 *
 * For query head h of row r: softmax over the scores scale * q.K of the
 * window keys and the listed entries plus one extra term attn_sink[h] that
 * has no value, then the weighted sum of V.  Readings where the page is
 * silent: both caches hold K at axis-1 index 0 and V at 1 with one latent
 * head shared by every query head; the sink logit is not scaled and only
 * enlarges the denominator; a repeated entry counts twice; an entry at or
 * past comp_cache_lengths[b] is skipped and sets QSA_STATUS_BAD_INDEX; a row
 * with nothing attended is zero.  num_heads <= 16 or a multiple of 16 (each
 * group of 16 query heads is one unit reading the latent head); each cache
 * below 32 GiB; runs on the per-(row, head group) tensor-core kernel with
 * split-K (options: kernel 0 or 2, splits).
 */
QSA_API qsa_status qsa_latent_attention_ragged_paged(
    qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets, qsa_tensor swa_blocks,
    int64_t swa_page_stride, qsa_tensor swa_cache_lengths, qsa_tensor swa_lookup_table,
    qsa_tensor comp_blocks, int64_t comp_page_stride, const uint32_t* comp_cache_lengths,
    const uint32_t* comp_lookup_table, int64_t comp_max_pages, uint32_t layer_idx,
    const int32_t* comp_indices, int64_t num_comp, const float* attn_sink, int32_t window, float scale,
    void* stream, const qsa_options* options);

/*
 * qsa_compress_keys_paged - block-key compression of raw QSA index keys
 * (MAX page "QSACompressKeysPaged": "Pools a paged group of raw QSA index
 * keys into dense block keys"; its tensor shapes, its gamma / freqs_cis /
 * key_counts arguments and its ratio, rotary_dim and eps parameters).
 *
 *   block_keys       [batch * max_blocks, head_dim]  F32 or BF16, written
 *   gamma            [head_dim] same type (k_layernorm weight)
 *   freqs_cis        [positions, rotary_dim] F32 or BF16: cos, sin pairs
 *   key_counts       [batch] I32, raw keys per sequence, this step included
 *   kv_blocks        [num_pages, 2, num_layers, page_size, 1, head_dim]
 *                    same type as block_keys; K at axis-1 index 0 is read
 *   page_stride, cache_lengths [batch] U32 (shape-checked only),
 *   kv_lookup_table, max_prompt_length, max_cache_length, layer_idx as for
 *   qsa_sparse_attention_ragged_paged
 *   ratio            raw keys per block (1 .. 64)
 *   rotary_dim       channels the rotation covers (even, <= head_dim)
 *   eps              RMS-norm epsilon (>= 0)
 *
 * Computes, for block i of sequence b (max_blocks = rows / batch): x = mean of
 * raw keys i*ratio .. i*ratio + ratio - 1 (raw key j is kv_blocks[page
 * kv_lookup_table[b, j / page_size], 0, layer_idx, j % page_size, 0, :]);
 * y = x / sqrt(mean(x^2) + eps) * gamma; channel pairs (2k, 2k+1) below
 * rotary_dim turned by freqs_cis[i, 2k] (cos) and [i, 2k+1] (sin).  Readings
 * where the page is silent: the pooling is a mean over complete blocks only
 * (rows of incomplete or missing blocks are zero), the order is pool, norm,
 * rotate, and the rotary position of a block is its index.  A raw key with no
 * page is skipped: its block's row is zero and QSA_STATUS_BAD_PAGE is set.
 * head_dim 128 or 256; f32 arithmetic; block_keys, gamma and kv_blocks
 * 16-byte aligned.
 */
QSA_API qsa_status qsa_compress_keys_paged(
    qsa_tensor block_keys, qsa_tensor gamma, qsa_tensor freqs_cis, qsa_tensor key_counts,
    qsa_tensor kv_blocks, int64_t page_stride, qsa_tensor cache_lengths, qsa_tensor kv_lookup_table,
    uint32_t max_prompt_length, uint32_t max_cache_length, uint32_t layer_idx, int32_t ratio,
    int32_t rotary_dim, float eps, void* stream);

/* Describes the launch a call with these extents would make, without
 * launching: kernel (1 .. 4, as qsa_options.kernel), CTAs per (row, kv head)
 * along the selection, total CTAs and workspace bytes.  dtype is the
 * q / kv_blocks element type.  Host only; reads no device memory (it queries
 * the current device's SM count and the kernel's occupancy).  Without the
 * batch, page size and length hints it never plans kernel 4: use qsa_plan_ex
 * for the plan of a qsa_sparse_attention_ragged_paged call. */
QSA_API qsa_status qsa_plan(int32_t dtype, int64_t total_q, int64_t num_kv_heads, int64_t head_dim,
                    int64_t selection_width, int32_t group, const qsa_options* options, int32_t* kernel,
                    int32_t* splits, int64_t* ctas, size_t* workspace_bytes);

/* qsa_plan with every host-known extent of a qsa_sparse_attention_ragged_paged
 * call: batch (cache_lengths' extent, >= 1 when total_q > 0), page_size
 * (kv_blocks' axis 3, >= 1) and the two length hints as the call passes them.
 * Its kernel and workspace figure are those of that call. */
QSA_API qsa_status qsa_plan_ex(int32_t dtype, int64_t total_q, int64_t batch, int64_t num_kv_heads,
                    int64_t head_dim, int64_t page_size, int64_t selection_width, int32_t group,
                    uint32_t max_prompt_length, uint32_t max_cache_length, const qsa_options* options,
                    int32_t* kernel, int32_t* splits, int64_t* ctas, size_t* workspace_bytes);

/* Makes sure the split-K workspace of (current device, stream) holds at least
 * `bytes` bytes (allocating and zeroing it if not).  Blocking; not for the
 * hot path or inside stream capture. */
QSA_API qsa_status qsa_reserve_workspace(void* stream, size_t bytes);

/* Frees every workspace and status word this library allocated on the
 * current device (after synchronising the device). */
QSA_API qsa_status qsa_release_device_state(void);

/* Reads (and with clear != 0 also zeroes) the current device's status word,
 * a bitwise OR of QSA_STATUS_* flags raised by kernels since the last clear.
 * Synchronises `stream`; for tests and debugging, not the hot path. */
QSA_API qsa_status qsa_read_device_status(void* stream, int32_t clear, uint32_t* flags);

/* Bytes of the fixed device scratch used by
 * qsa_sparse_attention_ragged_paged_noalloc (16 MiB). */
#define QSA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * qsa_sparse_attention_ragged_paged_noalloc - the same operation, arguments
 * and result as qsa_sparse_attention_ragged_paged, for callers that cannot
 * let a library allocate device memory: an engine that reserves nearly all of
 * the GPU's memory for its own pools at start-up and passes plugins only
 * buffers it owns, or a latency-bound loop that cannot take the device-wide
 * synchronisation cudaMalloc/cudaFree imply.  This entry point is a library
 * addition with no counterpart among the operations the method describes.
 *
 * It never calls cudaMalloc, cudaFree or any allocating routine.  It always
 * runs the persistent stream-K tensor-core kernel, so q / kv_blocks must be
 * BF16 or F8E4M3 with head_dim 128 (else QSA_ERR_UNSUPPORTED).  That kernel's
 * scratch (records of (row, kv-head group) units that two or more CTAs share,
 * and their arrival tickets) lives in a fixed array of
 * QSA_NOALLOC_SCRATCH_BYTES inside the library's device image, which every
 * GPU that loads the library holds until the process exits.  A call whose
 * scratch would not fit (roughly total_q * num_kv_heads beyond a few million)
 * returns QSA_ERR_UNSUPPORTED with the sizes in qsa_last_error_message, before
 * anything is enqueued.
 *
 *   status_flags  optional DEVICE pointer to a uint32 (4-byte aligned) that
 *                 kernels OR QSA_STATUS_* bits into; the caller zeroes and
 *                 reads it.  NULL sends the bits to a word in the scratch that
 *                 nothing reports.  qsa_read_device_status does not see
 *                 either.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * scratch array's device address once and keeps it; make that first call
 * before any stream capture begins.  qsa_release_device_state forgets the
 * address (a device reset drops it), and the call after it looks it up again,
 * so that call too must come before any capture.  Each call then enqueues a
 * clear of the tickets and the kernel on `stream`.  Argument errors are
 * reported before any CUDA call.
 *
 * Every call on a device uses the same scratch, which keeps what the last
 * call left there: calls whose GPU work overlaps (different streams, or
 * different host threads without ordering between their streams) race on it
 * and may produce wrong outputs.  Order such calls on one stream or with
 * events.
 */
QSA_API qsa_status qsa_sparse_attention_ragged_paged_noalloc(
    qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets, qsa_tensor kv_blocks,
    int64_t page_stride, qsa_tensor cache_lengths, qsa_tensor kv_lookup_table,
    uint32_t max_prompt_length, uint32_t max_cache_length, uint32_t layer_idx,
    qsa_tensor token_indices, qsa_tensor counts, float scale, int32_t group, void* stream,
    uint32_t* status_flags);

/* Human-readable name of a status code (static storage). */
QSA_API const char* qsa_status_string(qsa_status status);

/* Message describing the last non-OK status returned to this thread
 * (thread-local storage, valid until this thread's next call). */
QSA_API const char* qsa_last_error_message(void);

/* Library version, (major << 16) | minor. */
QSA_API int32_t qsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
