// Device helpers shared by libqsa's kernels: row -> sequence lookup, position
// -> cache row translation through the page table, and the end of a
// (row, kv head) unit (cross-warp softmax merge, split-K partials and the
// fused last-CTA combine).
#pragma once

#include <cuda_bf16.h>
#include <math_constants.h>
#include <stdint.h>

#include "qsa_internal.cuh"

namespace qsa {

constexpr uint32_t kInvalidOff = 0xFFFFFFFFu;

struct RowInfo {
  int b;           // owning sequence
  int64_t kv_len;  // valid positions of that sequence: cache_lengths[b] + rows_b
  int n;           // valid selection entries: clamp(counts[r], 0, W) (W with block lists)
  bool ok;         // r belongs to a sequence
};

// Block-wide (every thread must call): finds the sequence b with
// input_row_offsets[b] <= r < input_row_offsets[b + 1] by counting the
// offsets [1, batch] that are <= r (the offsets are nondecreasing), one
// coalesced pass per blockDim.x sequences.
__device__ __forceinline__ RowInfo row_info(const Params& p, int r) {
  int c = 0;
  for (int base = 1; base <= p.batch; base += blockDim.x) {
    const int k = base + (int)threadIdx.x;
    const int pred = (k <= p.batch) && (__ldg(p.row_offsets + k) <= (uint32_t)r);
    c += __syncthreads_count(pred);
  }
  RowInfo ri;
  ri.b = c;
  ri.ok = false;
  ri.kv_len = 0;
  ri.n = 0;
  if (c < p.batch) {
    const uint32_t o0 = __ldg(p.row_offsets + c), o1 = __ldg(p.row_offsets + c + 1);
    if (o0 <= (uint32_t)r && (uint32_t)r < o1) {
      ri.ok = true;
      ri.kv_len = (int64_t)__ldg(p.cache_lengths + c) + (int64_t)(o1 - o0);
      ri.n = p.counts ? min(max(__ldg(p.counts + r), 0), p.W) : p.W;  // no counts with block lists
    }
  }
  return ri;
}

// Warp-wide (every lane of the warp must call, with the same r): the sequence
// b with input_row_offsets[b] <= r < input_row_offsets[b + 1], or batch when r
// is at or past input_row_offsets[batch].  A 32-ary search of the
// nondecreasing offsets with no block barrier: one round of loads while batch
// <= 32, and a 32x narrower range per further round.  It keeps
// offsets[lo] <= r < offsets[hi] (offsets[batch + 1] read as +inf and
// offsets[0] taken to be <= r; the caller checks both ends of the row
// against the loaded offsets).
__device__ __forceinline__ int row_sequence_warp(const Params& p, int r) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = p.batch + 1;
  while (hi - lo > 1) {
    const int span = hi - lo - 1;  // candidates lo + 1 .. hi - 1
    const int m = span > 32 ? lo + 1 + (int)(((int64_t)lane * span) >> 5) : lo + 1 + lane;
    const bool valid = m < hi;
    const bool le = valid && __ldg(p.row_offsets + m) <= (uint32_t)r;
    const int c = __popc(__ballot_sync(0xffffffffu, le));  // lanes 0 .. c-1 hold candidates <= r
    const int m_lo = __shfl_sync(0xffffffffu, m, c > 0 ? c - 1 : 0);
    const int m_hi = __shfl_sync(0xffffffffu, m, c < 32 ? c : 31);
    const bool hi_valid = __shfl_sync(0xffffffffu, valid, c < 32 ? c : 31);
    // the range shrinks every round, whatever the offsets hold
    if (c > 0) lo = m_lo;
    hi = (c < 32 && hi_valid) ? m_hi : (c > 0 ? hi : lo + 1);
  }
  return lo;
}

// First half of a position's translation: range checks and the logical page.
// Returns the logical page, or -1 (and sets a status bit) when the position
// cannot be read.
__device__ __forceinline__ int64_t logical_page(const Params& p, int64_t kv_len, int32_t pos, uint32_t& bad) {
  if (pos < 0 || (int64_t)pos >= kv_len) {
    bad |= QSA_STATUS_BAD_INDEX;
    return -1;
  }
  const uint32_t lp = (uint32_t)pos / (uint32_t)p.P;
  if (lp >= (uint32_t)p.max_pages) {
    bad |= QSA_STATUS_BAD_PAGE;
    return -1;
  }
  return (int64_t)lp;
}

// Second half: the K row of (page, slot, kv head) in 16-byte units from the
// kv_blocks base, or kInvalidOff when the table entry names no page.
__device__ __forceinline__ uint32_t k_row_offset16(const Params& p, uint32_t page, int32_t pos, int h, uint32_t& bad) {
  if (page >= p.num_pages) {
    bad |= QSA_STATUS_BAD_PAGE;
    return kInvalidOff;
  }
  const int64_t off = (int64_t)page * p.page_pitch_bytes + p.k_layer_bytes +
                      (int64_t)((uint32_t)pos % (uint32_t)p.P) * p.slot_bytes + (int64_t)h * p.head_bytes;
  return (uint32_t)(off >> 4);
}

__device__ __forceinline__ void store_out(const Params& p, int64_t idx, float v) {
  if (p.out_bf16)
    reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(p.out)[idx] = v;
}

// The latent mode's sink of query head `head`, as a denominator term relative
// to the running max M of the base-2 scores: 2^(sink * log2(e) - M) (0 when
// there are no sinks).  The sink is one more softmax term without a value.
__device__ __forceinline__ float sink_term(const Params& p, int head, float M) {
  if (!p.sinks) return 0.f;
  return exp2f(__ldg(p.sinks + head) * 1.4426950408889634f - M);
}

// The split-K tail once this CTA's partial (o[G][D], m[G], l[G] at
// ws_partial + ((r * nkv + h) * splits + split) * partial_stride) is stored:
// the unit's ticket, and the merge of all partials by the last CTA to
// arrive (no CTA ever waits for another), which also re-arms the ticket.
// `scratch` is shared memory for 2 * kMaxSplits * group floats.
__device__ __forceinline__ void merge_split_partials(const Params& p, int r, int h, bool row_ok, float* scratch) {
  const int G = p.group, D = p.D;
  const int64_t out_base = ((int64_t)r * p.nq + (int64_t)h * G) * D;
  const int unit = r * p.nkv + h;
  const int S = p.splits;
  const int64_t stride = partial_stride(G, D);
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    const uint32_t t = atomicAdd(p.ws_ticket + unit, 1u);
    s_last = (t == (uint32_t)(S - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* base = p.ws_partial + (int64_t)unit * S * stride;
  // (1) every split's max and sum into shared memory, all loads in flight at once
  float* s_m = scratch;               // [S][G]
  float* s_w = scratch + kMaxSplits * G;  // [S][G]: weight of split s for head i
  for (int k = threadIdx.x; k < S * G; k += blockDim.x) {
    const int s = k / G, i = k - s * G;
    s_m[k] = __ldcg(base + s * stride + G * D + i);
    s_w[k] = __ldcg(base + s * stride + G * D + G + i);
  }
  __syncthreads();
  // (2) per head: global max, denominator, and each split's normalised weight
  for (int i = threadIdx.x; i < G; i += blockDim.x) {
    float M = -CUDART_INF_F;
    for (int s = 0; s < S; ++s) M = fmaxf(M, s_m[s * G + i]);
    float L = 0.f;
    if (M != -CUDART_INF_F)
      for (int s = 0; s < S; ++s) L += s_w[s * G + i] * exp2f(s_m[s * G + i] - M);
    const bool live = row_ok && M != -CUDART_INF_F;
    if (live) L += sink_term(p, h * G + i, M);
    for (int s = 0; s < S; ++s) s_w[s * G + i] = live ? exp2f(s_m[s * G + i] - M) / L : 0.f;
  }
  __syncthreads();
  // (3) output: four channels per thread, every split's float4 in flight together
  for (int q4 = threadIdx.x; q4 < G * D / 4; q4 += blockDim.x) {
    const int idx = q4 * 4, i = idx / D;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int s = 0; s < S; ++s) {
      const float w = s_w[s * G + i];
      const float4 o = __ldcg(reinterpret_cast<const float4*>(base + s * stride + idx));
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
    store_out(p, out_base + idx, acc.x);
    store_out(p, out_base + idx + 1, acc.y);
    store_out(p, out_base + idx + 2, acc.z);
    store_out(p, out_base + idx + 3, acc.w);
  }
  if (threadIdx.x == 0) p.ws_ticket[unit] = 0u;
}

// Finishes one (row r, kv head h) unit from NW per-warp softmax states held in
// shared memory: sm_m[w*GP + i] (running max of the base-2 scores),
// sm_l[w*GP + i] (sum of exponentials) and sm_o[(w*GP + i)*D + d]
// (unnormalised output), for query heads i < group.
//
// With one CTA per unit it writes output[r, h*group + i, :].  With split-K it
// stores this CTA's merged partial, and the last CTA of the unit to arrive
// (an atomic ticket; no CTA ever waits for another) merges all partials and
// writes the output, then re-arms the ticket for the next call.  `scratch`
// is shared memory for 2 * kMaxSplits * group floats (split-K only).
template <int NW>
__device__ __forceinline__ void finish_unit(const Params& p, int r, int h, int split, bool row_ok, const float* sm_m,
                                            const float* sm_l, const float* sm_o, int GP, float* scratch) {
  const int G = p.group, D = p.D;
  const int64_t out_base = ((int64_t)r * p.nq + (int64_t)h * G) * D;
  if (p.splits == 1) {
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
      const int i = idx / D, d = idx - i * D;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * GP + i]);
      float val = 0.f;
      if (row_ok && M != -CUDART_INF_F) {
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float e = exp2f(sm_m[w * GP + i] - M);
          L += sm_l[w * GP + i] * e;
          O += sm_o[(w * GP + i) * D + d] * e;
        }
        val = O / (L + sink_term(p, h * G + i, M));
      }
      store_out(p, out_base + idx, val);
    }
    return;
  }

  // split-K: partial layout per (unit, split): o[G][D], m[G], l[G]
  const int unit = r * p.nkv + h;
  const int S = p.splits;
  const int64_t stride = partial_stride(G, D);
  float* part = p.ws_partial + ((int64_t)unit * S + split) * stride;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int i = idx / D, d = idx - i * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w * GP + i]);
    float L = 0.f, O = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float e = exp2f(sm_m[w * GP + i] - M);
        L += sm_l[w * GP + i] * e;
        O += sm_o[(w * GP + i) * D + d] * e;
      }
    }
    part[idx] = O;
    if (d == 0) {
      part[G * D + i] = M;
      part[G * D + G + i] = L;
    }
  }
  merge_split_partials(p, r, h, row_ok, scratch);
}

}  // namespace qsa
