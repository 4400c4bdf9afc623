// Block-key compression (QSACompressKeysPaged: "Pools a paged group of raw
// QSA index keys into dense block keys"; its tensor shapes and its gamma /
// freqs_cis / ratio / rotary_dim / eps parameters).
//
// One warp per output row (sequence b, block i): lane l holds channels
// [l*CPL, l*CPL + CPL) of head_dim = 32*CPL.  The warp reads the block's
// `ratio` raw keys (one coalesced head_dim row each, all loads in flight),
// averages them, RMS-normalises with a warp-shuffle sum of squares, scales by
// gamma, turns the channel pairs below rotary_dim (both members of a pair sit
// in one lane) and writes the row.  Memory-bound: ratio rows in, one row out.
#include <cuda_bf16.h>
#include <stdint.h>

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

// CPL channels per lane = head_dim / 32, in chunks of 4.
template <int ELEM, int FREQ, int CPL>
__global__ void __launch_bounds__(kWarpsPerCta * 32) compress_kernel(const CompressParams p) {
  constexpr int EB = ELEM == kBF16 ? 2 : 4;
  constexpr int NCH = CPL / 4;
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (w >= (int64_t)p.batch * p.max_blocks) return;
  const int b = (int)(w / p.max_blocks), i = (int)(w - (int64_t)b * p.max_blocks);
  const int D = 32 * CPL;
  unsigned char* orow = p.out + w * D * EB;
  const int kc = __ldg(p.key_counts + b);
  const int nblk = kc > 0 ? kc / p.ratio : 0;
  float acc[NCH][4];
#pragma unroll
  for (int c = 0; c < NCH; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
  bool live = i < nblk;
  if (live) {
    const int64_t j0 = (int64_t)i * p.ratio;
    // the block's raw keys, four rows in flight at a time
    for (int k0 = 0; k0 < p.ratio; k0 += 4) {
      float v[4][NCH][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t j = j0 + k0 + k;
        bool ok = k0 + k < p.ratio;
        const unsigned char* row = nullptr;
        if (ok) {
          const int64_t lp = j / p.P;
          const uint32_t page = lp < p.max_pages ? __ldg(p.table + (int64_t)b * p.max_pages + lp) : 0xFFFFFFFFu;
          if (page >= p.num_pages) {
            ok = false;
            live = false;
          } else {
            row = p.kv + (int64_t)page * p.page_pitch_bytes + p.k_layer_bytes + (j - lp * p.P) * p.slot_bytes;
          }
        }
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          if (ok) {
            load_chunk<ELEM>(row + (c * 128 + lane * 4) * EB, v[k][c]);
          } else {
            v[k][c][0] = v[k][c][1] = v[k][c][2] = v[k][c][3] = 0.f;
          }
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[c][e] += v[k][c][e];
    }
    if (!live && lane == 0) atomicOr(p.status, QSA_STATUS_BAD_PAGE);
  }
  live = __all_sync(0xffffffffu, live);
  float y[NCH][4];
  if (live) {
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
  } else {
#pragma unroll
    for (int c = 0; c < NCH; ++c) y[c][0] = y[c][1] = y[c][2] = y[c][3] = 0.f;
  }
#pragma unroll
  for (int c = 0; c < NCH; ++c) store_chunk<ELEM>(orow + (c * 128 + lane * 4) * EB, y[c]);
}

template <int ELEM, int FREQ>
cudaError_t launch_compress_t(const CompressParams& p, int cpl, cudaStream_t s) {
  const int64_t rows = (int64_t)p.batch * p.max_blocks;
  if (rows == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + kWarpsPerCta - 1) / kWarpsPerCta);
  switch (cpl) {
    case 2: break;  // head_dim 64: two channels per lane does not fill a 4-chunk
    case 4: compress_kernel<ELEM, FREQ, 4><<<grid, kWarpsPerCta * 32, 0, s>>>(p); return cudaGetLastError();
    case 8: compress_kernel<ELEM, FREQ, 8><<<grid, kWarpsPerCta * 32, 0, s>>>(p); return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_compress(const CompressParams& p, int elem, int freq_elem, int head_dim, cudaStream_t s) {
  const int cpl = head_dim / 32;
  if (elem == kBF16)
    return freq_elem == kBF16 ? launch_compress_t<kBF16, kBF16>(p, cpl, s) : launch_compress_t<kBF16, kF32>(p, cpl, s);
  return freq_elem == kBF16 ? launch_compress_t<kF32, kBF16>(p, cpl, s) : launch_compress_t<kF32, kF32>(p, cpl, s);
}

}  // namespace qsa
