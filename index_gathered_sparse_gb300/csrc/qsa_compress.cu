// Block-key compression (QSACompressKeysPaged: "Pools a paged group of raw
// QSA index keys into dense block keys"; its tensor shapes and its gamma /
// freqs_cis / ratio / rotary_dim / eps parameters).
//
// One CTA per chunk of raw key rows (32 KB of them, at least 64; whole
// blocks of one sequence): the CTA stages the rows in shared memory with 16-byte
// cp.async, all copies in flight at once, so a chunk costs two dependent
// trips (counts and page table, then the rows).  Then each warp pools a
// block, RMS-normalises it with a warp-shuffle sum of squares (lane l holds
// channels l*4 .. l*4 + 3 of each 128-channel chunk), scales by gamma, turns
// the channel pairs below rotary_dim (both members of a pair sit in one lane)
// and writes the row.  Memory-bound: ratio rows in, one row out.
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "qsa.h"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

template <int ELEM>
__device__ __forceinline__ void load_chunk(const unsigned char* src, float (&v)[4]);

// 4 consecutive elements (bf16: 8 bytes, f32: 16 bytes)
template <>
__device__ __forceinline__ void load_chunk<kBF16>(const unsigned char* src, float (&v)[4]) {
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
  v[0] = __uint_as_float(w.x << 16);
  v[1] = __uint_as_float(w.x & 0xFFFF0000u);
  v[2] = __uint_as_float(w.y << 16);
  v[3] = __uint_as_float(w.y & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ void load_chunk<kF32>(const unsigned char* src, float (&v)[4]) {
  const float4 w = __ldg(reinterpret_cast<const float4*>(src));
  v[0] = w.x;
  v[1] = w.y;
  v[2] = w.z;
  v[3] = w.w;
}

template <int ELEM>
__device__ __forceinline__ float load_one(const unsigned char* base, int64_t i) {
  if constexpr (ELEM == kBF16)
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(base) + i) << 16);
  else
    return __ldg(reinterpret_cast<const float*>(base) + i);
}

template <int ELEM>
__device__ __forceinline__ void store_chunk(unsigned char* dst, const float (&v)[4]) {
  if constexpr (ELEM == kBF16) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

constexpr int kWarpsPerCta = 8;
// raw key rows a CTA stages: 32 KB worth, and at least 64 (ratio <= 64)
__host__ __device__ constexpr int rows_per_cta(int row_bytes) { return 32768 / row_bytes > 64 ? 32768 / row_bytes : 64; }

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool live) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(live ? 16u : 0u));
}

// One CTA per chunk of C = NROWS / ratio consecutive blocks of one sequence:
// its threads copy the chunk's raw key rows (C * ratio <= NROWS, all copies in
// flight) into shared memory, then each warp pools, normalises and turns
// blocks w, w + 8, ... of the chunk from there.
template <int ELEM, int FREQ, int CPL>
__global__ void __launch_bounds__(kWarpsPerCta * 32) compress_kernel(const CompressParams p) {
  constexpr int EB = ELEM == kBF16 ? 2 : 4;
  constexpr int NCH = CPL / 4;
  constexpr int D = 32 * CPL;
  constexpr int ROWB = D * EB, CPR = ROWB / 16;  // bytes and 16-byte chunks per row
  constexpr int NROWS = rows_per_cta(ROWB);
  extern __shared__ __align__(16) unsigned char s_rows[];  // [NROWS][ROWB]
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = max(1, NROWS / p.ratio);
  const int chunks = (p.max_blocks + C - 1) / C;
  const int b = blockIdx.x / chunks, i0 = (blockIdx.x - b * chunks) * C;
  const int i1 = min(i0 + C, p.max_blocks);
  const int kc = __ldg(p.key_counts + b);
  const int nblk = min(kc > 0 ? kc / p.ratio : 0, i1);  // complete blocks of this sequence below i1
  const uint32_t* trow = p.table + (int64_t)b * p.max_pages;
  if (tid == 0) s_bad = 0;
  // ---- the chunk's raw rows of complete blocks into shared memory ----
  const int rows = max(0, nblk - i0) * p.ratio;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(s_rows);
  bool bad = false;
  for (int q = tid; q < rows * CPR; q += kWarpsPerCta * 32) {
    const int row = q / CPR, ch = q - row * CPR;
    const int64_t j = (int64_t)i0 * p.ratio + row, lp = j / p.P;
    const uint32_t page = lp < p.max_pages ? __ldg(trow + lp) : 0xFFFFFFFFu;
    const bool live = page < p.num_pages;
    bad |= !live;
    const unsigned char* src =
        live ? p.kv + (int64_t)page * p.page_pitch_bytes + p.k_layer_bytes + (j - lp * p.P) * p.slot_bytes + ch * 16 : p.kv;
    cp_async16_zfill(sbase + row * ROWB + ch * 16, src, live);
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  // ---- one block per warp at a time ----
  for (int i = i0 + warp; i < i1; i += kWarpsPerCta) {
    unsigned char* orow = p.out + ((int64_t)b * p.max_blocks + i) * ROWB;
    float y[NCH][4];
#pragma unroll
    for (int c = 0; c < NCH; ++c) y[c][0] = y[c][1] = y[c][2] = y[c][3] = 0.f;
    // a block with a raw key that has no page is written as zeros (flagged below)
    bool row_bad = false;
    if (i < nblk && s_bad) {
      // which rows failed is not kept: recheck this block's pages
      for (int k = 0; k < p.ratio; ++k) {
        const int64_t j = (int64_t)i * p.ratio + k, lp = j / p.P;
        row_bad |= !(lp < p.max_pages && __ldg(trow + lp) < p.num_pages);
      }
    }
    if (i < nblk && !row_bad) {
      float acc[NCH][4];
#pragma unroll
      for (int c = 0; c < NCH; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
      const unsigned char* r0 = s_rows + (i - i0) * p.ratio * ROWB;
      for (int k = 0; k < p.ratio; ++k)
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          float v[4];
          const unsigned char* src = r0 + k * ROWB + (c * 128 + lane * 4) * EB;
          if constexpr (ELEM == kBF16) {
            const uint2 w = *reinterpret_cast<const uint2*>(src);
            v[0] = __uint_as_float(w.x << 16);
            v[1] = __uint_as_float(w.x & 0xFFFF0000u);
            v[2] = __uint_as_float(w.y << 16);
            v[3] = __uint_as_float(w.y & 0xFFFF0000u);
          } else {
            const float4 w = *reinterpret_cast<const float4*>(src);
            v[0] = w.x;
            v[1] = w.y;
            v[2] = w.z;
            v[3] = w.w;
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[c][e] += v[e];
        }
      const float inv_r = 1.f / (float)p.ratio;
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[c][e] *= inv_r;
          ss += acc[c][e] * acc[c][e];
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = 1.f / sqrtf(ss / (float)D + p.eps);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int ch = c * 128 + lane * 4;
        float g[4];
        load_chunk<ELEM>(p.gamma + ch * EB, g);
#pragma unroll
        for (int e = 0; e < 4; ++e) y[c][e] = acc[c][e] * inv * g[e];
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          if (ch + e < p.rotary_dim) {
            const int64_t f = (int64_t)i * p.rotary_dim + ch + e;
            const float cs = load_one<FREQ>(p.freqs, f), sn = load_one<FREQ>(p.freqs, f + 1);
            const float a = y[c][e], z = y[c][e + 1];
            y[c][e] = a * cs - z * sn;
            y[c][e + 1] = a * sn + z * cs;
          }
        }
      }
    }
    if (row_bad && lane == 0) atomicOr(p.status, QSA_STATUS_BAD_PAGE);
#pragma unroll
    for (int c = 0; c < NCH; ++c) store_chunk<ELEM>(orow + (c * 128 + lane * 4) * EB, y[c]);
  }
}

template <int ELEM, int FREQ>
cudaError_t launch_compress_t(const CompressParams& p, int cpl, cudaStream_t s) {
  const int row_bytes = 32 * cpl * (ELEM == kBF16 ? 2 : 4), nrows = rows_per_cta(row_bytes);
  const int C = std::max(1, nrows / p.ratio);
  const int64_t ctas = (int64_t)p.batch * ((p.max_blocks + C - 1) / C);
  if (ctas == 0) return cudaSuccess;
  const int smem = nrows * row_bytes;
  if (cpl == 4) {
    compress_kernel<ELEM, FREQ, 4><<<(unsigned)ctas, kWarpsPerCta * 32, smem, s>>>(p);
  } else if (cpl == 8) {
    // 64 rows of 256 f32 channels exceed the default 48 KB (the attribute is per device)
    if (smem > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(compress_kernel<ELEM, FREQ, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
    }
    compress_kernel<ELEM, FREQ, 8><<<(unsigned)ctas, kWarpsPerCta * 32, smem, s>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress(const CompressParams& p, int elem, int freq_elem, int head_dim, cudaStream_t s) {
  const int cpl = head_dim / 32;
  if (elem == kBF16)
    return freq_elem == kBF16 ? launch_compress_t<kBF16, kBF16>(p, cpl, s) : launch_compress_t<kBF16, kF32>(p, cpl, s);
  return freq_elem == kBF16 ? launch_compress_t<kF32, kBF16>(p, cpl, s) : launch_compress_t<kF32, kF32>(p, cpl, s);
}

}  // namespace qsa
