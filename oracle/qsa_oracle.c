/*
 * CPU oracle for QSA gather-GQA sparse attention over a ragged, paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition the CUDA path is checked against.  Only the tests, the smoke
 * check and the bench's CPU-baseline leg may load it; the product library
 * never links or calls it, and it shares no code, header or table with it.
 *
 * What it computes (QSASparseAttentionRaggedPaged, "Gather-GQA over the token
 * indices a QSA selection names", with the tensor shapes listed on that page):
 *
 *   for each query row r of sequence b (input_row_offsets[b] <= r < [b+1]),
 *   each kv head h and each of the `group` query heads i that share it:
 *     n   = min(max(counts[r], 0), selection_width)   valid entries come first
 *     p_j = token_indices[r, j]                        j < n, never read past n
 *     K_j = kv_blocks[page(b, p_j), 0, layer_idx, p_j % page_size, h, :]
 *     V_j = kv_blocks[page(b, p_j), 1, layer_idx, p_j % page_size, h, :]
 *     page(b, p) = kv_lookup_table[b, p / page_size], pages page_stride
 *                  elements apart (or packed when page_stride == -1)
 *     s_j = scale * sum_d q[r, h*group + i, d] * K_j[d]
 *     out[r, h*group + i, :] = sum_j softmax(s)_j * V_j
 *
 * Everything is float64; inputs are decoded exactly from their storage type
 * (IEEE binary32, bfloat16, or scale-free FP8 e4m3fn).  Readings taken where
 * the page is silent: axis 1 of kv_blocks is K at 0 and V at 1; query head
 * h*group+i uses kv head h; no causal mask is applied (the selection alone
 * decides what is attended); an empty selection gives a zero row; an index
 * outside [0, cache_lengths[b] + rows_b) inside the valid prefix is a
 * precondition violation and makes the oracle fail.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 2 };

enum {
  ORACLE_OK = 0,
  ORACLE_BAD_ARGUMENT = 1,
  ORACLE_INDEX_OUT_OF_RANGE = 2,
  ORACLE_BAD_PAGE = 3,
  ORACLE_BAD_ROW = 4,
  ORACLE_NO_MEMORY = 5
};

/* IEEE binary32 element -> double (exact). */
static double decode_f32(const void* base, int64_t i) {
  float f;
  memcpy(&f, (const unsigned char*)base + 4 * i, 4);
  return (double)f;
}

/* bfloat16 element -> double (exact): the upper 16 bits of a binary32. */
static double decode_bf16(const void* base, int64_t i) {
  uint16_t h;
  uint32_t w;
  float f;
  memcpy(&h, (const unsigned char*)base + 2 * i, 2);
  w = (uint32_t)h << 16;
  memcpy(&f, &w, 4);
  return (double)f;
}

/* FP8 e4m3fn element -> double (exact), from the format's definition:
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * S.1111.111 is NaN, exponent 0 is subnormal (m/8 * 2^-6). */
static double decode_e4m3(const void* base, int64_t i) {
  unsigned b = ((const unsigned char*)base)[i];
  int sign = (b >> 7) & 1;
  int e = (b >> 3) & 15;
  int m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

static double decode(int dtype, const void* base, int64_t i) {
  if (dtype == ORACLE_F32) return decode_f32(base, i);
  if (dtype == ORACLE_BF16) return decode_bf16(base, i);
  return decode_e4m3(base, i);
}

/*
 * Computes the attention output for the query rows listed in `rows`
 * (n_rows of them) into out[n_rows, num_q_heads, head_dim] (float64).
 * All arrays are host memory, contiguous, row-major, shaped as the
 * QSASparseAttentionRaggedPaged page lists; kv_blocks pages are `page_stride`
 * elements apart (-1 = packed).  On an index error *bad_row receives the row.
 */
int qsa_oracle_sparse_attention(
    double* out, const int64_t* rows, int64_t n_rows,
    const void* q, int q_dtype, int64_t total_q, int64_t num_q_heads, int64_t head_dim,
    const uint32_t* input_row_offsets, int64_t batch,
    const void* kv_blocks, int kv_dtype, int64_t num_pages, int64_t page_stride,
    int64_t num_layers, int64_t page_size, int64_t num_kv_heads,
    const uint32_t* cache_lengths, const uint32_t* kv_lookup_table, int64_t max_pages,
    int64_t layer_idx, const int32_t* token_indices, int64_t selection_width,
    const int32_t* counts, double scale, int64_t group, int64_t* bad_row) {
  int64_t packed_page, pitch, ri;
  double* s;
  double* w;

  *bad_row = -1;
  if (group <= 0 || num_kv_heads <= 0 || num_q_heads != group * num_kv_heads) return ORACLE_BAD_ARGUMENT;
  if (layer_idx < 0 || layer_idx >= num_layers) return ORACLE_BAD_ARGUMENT;
  if (q_dtype != kv_dtype || q_dtype < 0 || q_dtype > 2) return ORACLE_BAD_ARGUMENT;
  packed_page = 2 * num_layers * page_size * num_kv_heads * head_dim;
  if (page_stride != -1 && page_stride < packed_page) return ORACLE_BAD_ARGUMENT;
  pitch = (page_stride == -1) ? packed_page : page_stride;

  s = (double*)malloc(sizeof(double) * (size_t)(selection_width > 0 ? selection_width : 1));
  w = (double*)malloc(sizeof(double) * (size_t)(selection_width > 0 ? selection_width : 1));
  if (!s || !w) {
    free(s);
    free(w);
    return ORACLE_NO_MEMORY;
  }

  for (ri = 0; ri < n_rows; ++ri) {
    int64_t r = rows[ri];
    int64_t b = -1, k, kv_len, n, h, i, j, d;

    if (r < 0 || r >= total_q) goto bad_row_exit;
    /* the sequence that owns row r: input_row_offsets[b] <= r < input_row_offsets[b+1] */
    for (k = 0; k < batch; ++k)
      if ((int64_t)input_row_offsets[k] <= r && r < (int64_t)input_row_offsets[k + 1]) {
        b = k;
        break;
      }
    if (b < 0) goto bad_row_exit;
    /* the cache already holds this step's rows of sequence b */
    kv_len = (int64_t)cache_lengths[b] + ((int64_t)input_row_offsets[b + 1] - (int64_t)input_row_offsets[b]);

    n = counts[r];
    if (n < 0) n = 0;
    if (n > selection_width) n = selection_width;

    for (h = 0; h < num_kv_heads; ++h) {
      for (i = 0; i < group; ++i) {
        int64_t head = h * group + i;
        int64_t q_off = (r * num_q_heads + head) * head_dim;
        double* o = out + (ri * num_q_heads + head) * head_dim;
        double m = -INFINITY, z = 0.0;

        for (d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (n == 0) continue; /* empty selection: zero row */

        /* scores s_j = scale * q . K_j over the valid prefix only */
        for (j = 0; j < n; ++j) {
          int64_t p = token_indices[r * selection_width + j];
          int64_t logical_page, page, slot, k_off;
          double dot = 0.0;
          if (p < 0 || p >= kv_len) {
            *bad_row = r;
            free(s);
            free(w);
            return ORACLE_INDEX_OUT_OF_RANGE;
          }
          logical_page = p / page_size;
          slot = p % page_size;
          if (logical_page >= max_pages) goto bad_page_exit;
          page = (int64_t)kv_lookup_table[b * max_pages + logical_page];
          if (page >= num_pages) goto bad_page_exit;
          k_off = page * pitch + ((0 * num_layers + layer_idx) * page_size + slot) * num_kv_heads * head_dim +
                  h * head_dim;
          for (d = 0; d < head_dim; ++d) dot += decode(q_dtype, q, q_off + d) * decode(kv_dtype, kv_blocks, k_off + d);
          s[j] = scale * dot;
        }
        /* softmax over the n scores (max-subtracted, natural exponent) */
        for (j = 0; j < n; ++j)
          if (s[j] > m || isnan(s[j])) m = s[j];
        for (j = 0; j < n; ++j) {
          w[j] = exp(s[j] - m);
          z += w[j];
        }
        /* out = sum_j softmax_j * V_j */
        for (j = 0; j < n; ++j) {
          int64_t p = token_indices[r * selection_width + j];
          int64_t page = (int64_t)kv_lookup_table[b * max_pages + p / page_size];
          int64_t v_off = page * pitch +
                          ((1 * num_layers + layer_idx) * page_size + p % page_size) * num_kv_heads * head_dim +
                          h * head_dim;
          double a = w[j] / z;
          for (d = 0; d < head_dim; ++d) o[d] += a * decode(kv_dtype, kv_blocks, v_off + d);
        }
      }
    }
    continue;
  bad_page_exit:
    *bad_row = r;
    free(s);
    free(w);
    return ORACLE_BAD_PAGE;
  bad_row_exit:
    *bad_row = r;
    free(s);
    free(w);
    return ORACLE_BAD_ROW;
  }
  free(s);
  free(w);
  return ORACLE_OK;
}

/* Decodes `n` elements of storage type `dtype` to float64 (exact). */
void qsa_oracle_decode(double* out, const void* src, int dtype, int64_t n) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = decode(dtype, src, i);
}

/*
 * Block-sparse (MSA-style) variant: Struct_msa_attention_ragged_paged,
 * "Gathers topk KV blocks per (kv head, query token) using the block ids in
 * d_indices" ([n_kv_heads, num_rows, topk] int32), decode with no mask,
 * prefill and speculative decode causal per token.
 *
 * Readings taken where the page is silent: a block is one page of the row's
 * own sequence, block id beta names logical page beta (positions beta*P ..
 * beta*P + P - 1, physical page kv_lookup_table[b, beta]); a negative id is
 * an unused slot; a position attends when it is <= the row's position
 * pos = cache_lengths[b] + (r - input_row_offsets[b]) (for one new token per
 * sequence this is exactly "every cached key", so decode needs no mask); a
 * repeated id is attended twice; a row with nothing attended is zero.  An id
 * whose first position is <= pos but that has no page-table entry or names a
 * page outside kv_blocks is a precondition violation.
 */
int qsa_oracle_msa_attention(
    double* out, const int64_t* rows, int64_t n_rows,
    const void* q, int dtype, int64_t total_q, int64_t num_q_heads, int64_t head_dim,
    const uint32_t* input_row_offsets, int64_t batch,
    const void* kv_blocks, int64_t num_pages, int64_t page_stride,
    int64_t num_layers, int64_t page_size, int64_t num_kv_heads,
    const uint32_t* cache_lengths, const uint32_t* kv_lookup_table, int64_t max_pages,
    int64_t layer_idx, const int32_t* d_indices, int64_t topk, double scale, int64_t group,
    int64_t* bad_row) {
  int64_t packed_page, pitch, ri, cap;
  double* s;
  int64_t* koff;

  *bad_row = -1;
  if (group <= 0 || num_kv_heads <= 0 || num_q_heads != group * num_kv_heads) return ORACLE_BAD_ARGUMENT;
  if (layer_idx < 0 || layer_idx >= num_layers || dtype < 0 || dtype > 2 || topk < 0) return ORACLE_BAD_ARGUMENT;
  packed_page = 2 * num_layers * page_size * num_kv_heads * head_dim;
  if (page_stride != -1 && page_stride < packed_page) return ORACLE_BAD_ARGUMENT;
  pitch = (page_stride == -1) ? packed_page : page_stride;

  cap = topk * page_size > 0 ? topk * page_size : 1;
  s = (double*)malloc(sizeof(double) * (size_t)cap);
  koff = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
  if (!s || !koff) {
    free(s);
    free(koff);
    return ORACLE_NO_MEMORY;
  }

  for (ri = 0; ri < n_rows; ++ri) {
    int64_t r = rows[ri];
    int64_t b = -1, k, pos, h, i, d;

    if (r < 0 || r >= total_q) goto msa_bad_row;
    for (k = 0; k < batch; ++k)
      if ((int64_t)input_row_offsets[k] <= r && r < (int64_t)input_row_offsets[k + 1]) {
        b = k;
        break;
      }
    if (b < 0) goto msa_bad_row;
    pos = (int64_t)cache_lengths[b] + (r - (int64_t)input_row_offsets[b]);

    for (h = 0; h < num_kv_heads; ++h) {
      /* the attended keys of (row, kv head): K-row element offsets, in list order */
      int64_t n = 0, j, e;
      for (e = 0; e < topk; ++e) {
        int64_t beta = d_indices[(h * total_q + r) * topk + e], sl;
        if (beta < 0) continue; /* unused slot */
        for (sl = 0; sl < page_size; ++sl) {
          int64_t p = beta * page_size + sl, page;
          if (p > pos) break; /* causal: later positions of the block are not attended */
          if (beta >= max_pages) goto msa_bad_page;
          page = (int64_t)kv_lookup_table[b * max_pages + beta];
          if (page >= num_pages) goto msa_bad_page;
          koff[n++] = page * pitch + ((0 * num_layers + layer_idx) * page_size + sl) * num_kv_heads * head_dim +
                      h * head_dim;
        }
      }
      for (i = 0; i < group; ++i) {
        int64_t head = h * group + i;
        int64_t q_off = (r * num_q_heads + head) * head_dim;
        double* o = out + (ri * num_q_heads + head) * head_dim;
        double m = -INFINITY, z = 0.0;
        for (d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (n == 0) continue;
        for (j = 0; j < n; ++j) {
          double dot = 0.0;
          for (d = 0; d < head_dim; ++d) dot += decode(dtype, q, q_off + d) * decode(dtype, kv_blocks, koff[j] + d);
          s[j] = scale * dot;
          if (s[j] > m || isnan(s[j])) m = s[j];
        }
        for (j = 0; j < n; ++j) z += exp(s[j] - m);
        for (j = 0; j < n; ++j) {
          /* V sits num_layers * page_size * num_kv_heads * head_dim after K */
          int64_t v_off = koff[j] + num_layers * page_size * num_kv_heads * head_dim;
          double a = exp(s[j] - m) / z;
          for (d = 0; d < head_dim; ++d) o[d] += a * decode(dtype, kv_blocks, v_off + d);
        }
      }
    }
    continue;
  msa_bad_page:
    *bad_row = r;
    free(s);
    free(koff);
    return ORACLE_BAD_PAGE;
  msa_bad_row:
    *bad_row = r;
    free(s);
    free(koff);
    return ORACLE_BAD_ROW;
  }
  free(s);
  free(koff);
  return ORACLE_OK;
}

/*
 * Block-key compression: QSACompressKeysPaged ("Pools a paged group of raw QSA
 * index keys into dense block keys"; tensor shapes block_keys
 * [batch * max_blocks, head_dim], gamma [head_dim], freqs_cis [positions,
 * rotary_dim], key_counts [batch], kv_blocks [num_pages, 2, num_layers,
 * page_size, 1, head_dim]; parameters ratio, rotary_dim, eps).
 *
 * Readings taken where the page is silent (the page names the steps -
 * pooling by `ratio`, the k_layernorm weight gamma with rms_norm_eps, the
 * rotary table - but not their order or exact form):
 *   raw key j of sequence b (j < key_counts[b]) is
 *     kv_blocks[kv_lookup_table[b, j / page_size], 0, layer_idx, j % page_size, 0, :];
 *   block i (i < max_blocks = rows of block_keys / batch) covers raw keys
 *     i*ratio .. i*ratio + ratio - 1 and exists when all of them do; the rows
 *     of missing blocks are zero;
 *   x = mean of the block's raw keys; y_d = x_d / sqrt(mean_d x_d^2 + eps) * gamma_d;
 *   the channel pairs (2k, 2k+1) below rotary_dim turn by the angle whose
 *     cosine and sine are freqs_cis[i, 2k] and freqs_cis[i, 2k+1] (the block's
 *     index is its position); channels at or past rotary_dim pass through.
 * Keys, gamma and the output share one element type; freqs_cis has its own.
 * Parity unpinned against the pages on the step order and the rotary
 * position: the tests pin each step's arithmetic, not which order was meant.
 */
int qsa_oracle_compress_keys(double* out, int64_t batch, int64_t max_blocks, int64_t head_dim,
                             const void* gamma, const void* freqs, int freq_dtype, int64_t positions,
                             int64_t rotary_dim, const int32_t* key_counts, const void* kv_blocks, int dtype,
                             int64_t num_pages, int64_t page_stride, int64_t num_layers, int64_t page_size,
                             const uint32_t* kv_lookup_table, int64_t max_pages, int64_t layer_idx, int64_t ratio,
                             double eps) {
  int64_t pitch, b, i, d, j;
  double* x;
  if (ratio <= 0 || head_dim <= 0 || rotary_dim < 0 || rotary_dim > head_dim || (rotary_dim & 1)) return ORACLE_BAD_ARGUMENT;
  if (layer_idx < 0 || layer_idx >= num_layers) return ORACLE_BAD_ARGUMENT;
  pitch = page_stride == -1 ? 2 * num_layers * page_size * head_dim : page_stride;
  x = (double*)malloc(sizeof(double) * (size_t)head_dim);
  if (!x) return ORACLE_NO_MEMORY;
  for (b = 0; b < batch; ++b) {
    int64_t nblk = key_counts[b] > 0 ? key_counts[b] / ratio : 0;
    for (i = 0; i < max_blocks; ++i) {
      double* o = out + (b * max_blocks + i) * head_dim;
      double ss = 0.0, inv;
      for (d = 0; d < head_dim; ++d) o[d] = 0.0;
      if (i >= nblk) continue;
      if (rotary_dim > 0 && i >= positions) {
        free(x);
        return ORACLE_BAD_ARGUMENT;
      }
      for (d = 0; d < head_dim; ++d) x[d] = 0.0;
      for (j = i * ratio; j < (i + 1) * ratio; ++j) {
        int64_t lp = j / page_size, page, off;
        if (lp >= max_pages) {
          free(x);
          return ORACLE_BAD_PAGE;
        }
        page = (int64_t)kv_lookup_table[b * max_pages + lp];
        if (page >= num_pages) {
          free(x);
          return ORACLE_BAD_PAGE;
        }
        off = page * pitch + ((0 * num_layers + layer_idx) * page_size + j % page_size) * head_dim;
        for (d = 0; d < head_dim; ++d) x[d] += decode(dtype, kv_blocks, off + d);
      }
      for (d = 0; d < head_dim; ++d) {
        x[d] /= (double)ratio;
        ss += x[d] * x[d];
      }
      inv = 1.0 / sqrt(ss / (double)head_dim + eps);
      for (d = 0; d < head_dim; ++d) o[d] = x[d] * inv * decode(dtype, gamma, d);
      for (d = 0; d + 1 < rotary_dim; d += 2) {
        double c = decode(freq_dtype, freqs, i * rotary_dim + d), s = decode(freq_dtype, freqs, i * rotary_dim + d + 1);
        double a = o[d], e = o[d + 1];
        o[d] = a * c - e * s;
        o[d + 1] = a * s + e * c;
      }
    }
  }
  free(x);
  return ORACLE_OK;
}

/*
 * Latent sparse attention: latent_sparse_attention_ragged_paged ("Attends
 * every query row to its window keys and its listed compressed entries"): a
 * sliding window of `window` tokens (a query at pos sees positions
 * max(0, pos - window + 1) .. pos) from a cache paged by token position, the
 * entries comp_indices[r, :] (-1 marks an unused slot) from a cache paged by
 * entry, both with one latent head shared by all query heads, and per-head
 * sink logits attn_sink.
 *
 * Readings taken where the page is silent: each cache stores K at axis-1
 * index 0 and V at index 1 like the paged KV caches of the other ops; the
 * row's position is swa_cache_lengths[b] + (r - input_row_offsets[b]); a sink
 * is one more softmax term with logit attn_sink[h] (not scaled) and no value,
 * so it only enlarges the denominator; a repeated entry counts twice; an
 * entry at or past comp_cache_lengths[b] is a precondition violation.
 */
int qsa_oracle_latent_attention(
    double* out, const int64_t* rows, int64_t n_rows,
    const void* q, int dtype, int64_t total_q, int64_t num_heads, int64_t head_dim,
    const uint32_t* input_row_offsets, int64_t batch,
    const void* swa_blocks, int64_t swa_pages, int64_t swa_stride, int64_t swa_layers, int64_t swa_page_size,
    const uint32_t* swa_cache_lengths, const uint32_t* swa_table, int64_t swa_max_pages,
    const void* comp_blocks, int64_t comp_pages, int64_t comp_stride, int64_t comp_layers, int64_t comp_page_size,
    const uint32_t* comp_cache_lengths, const uint32_t* comp_table, int64_t comp_max_pages,
    int64_t layer_idx, const int32_t* comp_indices, int64_t num_comp, const float* attn_sink,
    int64_t window, double scale, int64_t* bad_row) {
  int64_t swa_pitch, comp_pitch, ri, cap;
  double* s;
  int64_t* koff;
  int* src;

  *bad_row = -1;
  if (dtype < 0 || dtype > 2 || window < 0 || num_comp < 0) return ORACLE_BAD_ARGUMENT;
  if (layer_idx < 0 || layer_idx >= swa_layers || layer_idx >= comp_layers) return ORACLE_BAD_ARGUMENT;
  swa_pitch = swa_stride == -1 ? 2 * swa_layers * swa_page_size * head_dim : swa_stride;
  comp_pitch = comp_stride == -1 ? 2 * comp_layers * comp_page_size * head_dim : comp_stride;
  cap = window + num_comp > 0 ? window + num_comp : 1;
  s = (double*)malloc(sizeof(double) * (size_t)cap);
  koff = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
  src = (int*)malloc(sizeof(int) * (size_t)cap);
  if (!s || !koff || !src) {
    free(s);
    free(koff);
    free(src);
    return ORACLE_NO_MEMORY;
  }
  for (ri = 0; ri < n_rows; ++ri) {
    int64_t r = rows[ri], b = -1, k, pos, n = 0, p, e, h, d, j;
    if (r < 0 || r >= total_q) goto lat_bad_row;
    for (k = 0; k < batch; ++k)
      if ((int64_t)input_row_offsets[k] <= r && r < (int64_t)input_row_offsets[k + 1]) {
        b = k;
        break;
      }
    if (b < 0) goto lat_bad_row;
    pos = (int64_t)swa_cache_lengths[b] + (r - (int64_t)input_row_offsets[b]);
    /* window keys, oldest first */
    for (p = pos - window + 1; p <= pos; ++p) {
      int64_t lp, page;
      if (p < 0) continue;
      lp = p / swa_page_size;
      if (lp >= swa_max_pages) goto lat_bad_page;
      page = (int64_t)swa_table[b * swa_max_pages + lp];
      if (page >= swa_pages) goto lat_bad_page;
      koff[n] = page * swa_pitch + ((0 * swa_layers + layer_idx) * swa_page_size + p % swa_page_size) * head_dim;
      src[n++] = 0;
    }
    /* listed compressed entries */
    for (k = 0; k < num_comp; ++k) {
      int64_t lp, page;
      e = comp_indices[r * num_comp + k];
      if (e < 0) continue;
      if (e >= (int64_t)comp_cache_lengths[b]) {
        *bad_row = r;
        free(s);
        free(koff);
        free(src);
        return ORACLE_INDEX_OUT_OF_RANGE;
      }
      lp = e / comp_page_size;
      if (lp >= comp_max_pages) goto lat_bad_page;
      page = (int64_t)comp_table[b * comp_max_pages + lp];
      if (page >= comp_pages) goto lat_bad_page;
      koff[n] = page * comp_pitch + ((0 * comp_layers + layer_idx) * comp_page_size + e % comp_page_size) * head_dim;
      src[n++] = 1;
    }
    for (h = 0; h < num_heads; ++h) {
      int64_t q_off = (r * num_heads + h) * head_dim;
      double* o = out + (ri * num_heads + h) * head_dim;
      double m = (double)attn_sink[h], z;
      for (d = 0; d < head_dim; ++d) o[d] = 0.0;
      for (j = 0; j < n; ++j) {
        const void* base = src[j] ? comp_blocks : swa_blocks;
        double dot = 0.0;
        for (d = 0; d < head_dim; ++d) dot += decode(dtype, q, q_off + d) * decode(dtype, base, koff[j] + d);
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
      }
      z = exp((double)attn_sink[h] - m); /* the sink: denominator only */
      for (j = 0; j < n; ++j) z += exp(s[j] - m);
      for (j = 0; j < n; ++j) {
        const void* base = src[j] ? comp_blocks : swa_blocks;
        int64_t v_off = koff[j] + (src[j] ? comp_layers * comp_page_size : swa_layers * swa_page_size) * head_dim;
        double a = exp(s[j] - m) / z;
        for (d = 0; d < head_dim; ++d) o[d] += a * decode(dtype, base, v_off + d);
      }
    }
    continue;
  lat_bad_page:
    *bad_row = r;
    free(s);
    free(koff);
    free(src);
    return ORACLE_BAD_PAGE;
  lat_bad_row:
    *bad_row = r;
    free(s);
    free(koff);
    free(src);
    return ORACLE_BAD_ROW;
  }
  free(s);
  free(koff);
  free(src);
  return ORACLE_OK;
}
