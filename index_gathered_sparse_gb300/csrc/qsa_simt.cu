// CUDA-core kernel for QSA gather-GQA sparse attention (QSASparseAttentionRaggedPaged:
// "Gather-GQA over the token indices a QSA selection names").
//
// One CTA of 4 warps per (query row, kv head).  Warps take the row's selected
// positions U at a time, round-robin (the page's `unroll`: gathered keys
// loaded before any is consumed): lanes 0..U-1 translate one position each
// (index, then page-table entry, all U in flight together), then every lane
// loads its head_dim/32 slice of all U K and V rows before the first is
// used.  Per key the warp forms the `group` dot products with warp-shuffle
// sums, updates a base-2 online softmax per query head and accumulates the V
// row.  The four warp states are merged in shared memory at the end.  This kernel
// serves FP32 (whose 1e-4 tolerance rules out TF32 tensor cores) and every
// (dtype, head_dim, group) the tensor-core kernel does not cover.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "qsa_device.cuh"

namespace qsa {
namespace {

// Loads this lane's EPL consecutive elements of a row (lane * EPL onwards) as floats.
template <int ELEM, int EPL>
__device__ __forceinline__ void load_slice(const unsigned char* row, int lane, float (&x)[EPL]) {
  if constexpr (ELEM == kF32) {
    const float* f = reinterpret_cast<const float*>(row) + lane * EPL;
    if constexpr (EPL == 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(f));
      x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
    } else {
      const float2 v = __ldg(reinterpret_cast<const float2*>(f));
      x[0] = v.x, x[1] = v.y;
    }
  } else if constexpr (ELEM == kBF16) {
    const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(row) + lane * EPL;
    if constexpr (EPL == 4) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(e));
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
      x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
    } else {
      const unsigned v = __ldg(reinterpret_cast<const unsigned*>(e));
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
      x[0] = a.x, x[1] = a.y;
    }
  } else {
    const unsigned char* e = row + lane * EPL;
    if constexpr (EPL == 4) {
      const unsigned v = __ldg(reinterpret_cast<const unsigned*>(e));
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xFFFFu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v >> 16), __NV_E4M3);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      x[0] = a.x, x[1] = a.y, x[2] = b.x, x[3] = b.y;
    } else {
      const unsigned short v = __ldg(reinterpret_cast<const unsigned short*>(e));
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      x[0] = a.x, x[1] = a.y;
    }
  }
}

template <int ELEM>
__device__ __forceinline__ float load_elem(const unsigned char* base, int64_t i) {
  if constexpr (ELEM == kF32) return __ldg(reinterpret_cast<const float*>(base) + i);
  if constexpr (ELEM == kBF16) return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(base) + i));
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)__ldg(base + i), __NV_E4M3);
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

template <int ELEM, int D, int G>
__global__ void __launch_bounds__(128) simt_kernel(const Params p) {
  constexpr int NW = 4, EPL = D / 32;
  __shared__ float sq[G * D];
  __shared__ float sm_m[NW * G], sm_l[NW * G];
  __shared__ float sm_o[NW * G * D];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int h = blockIdx.x % p.nkv;
  const int r = p.total_q - 1 - (int)(blockIdx.x / p.nkv);  // latest rows (longest selections) first
  const RowInfo ri = row_info(p, r);

  const int64_t q_base = ((int64_t)r * p.nq + (int64_t)h * G) * D;
  for (int idx = tid; idx < G * D; idx += blockDim.x) sq[idx] = load_elem<ELEM>(p.q, q_base + idx);
  __syncthreads();
  float qr[G][EPL];
#pragma unroll
  for (int i = 0; i < G; ++i)
#pragma unroll
    for (int e = 0; e < EPL; ++e) qr[i][e] = sq[i * D + lane * EPL + e];

  float m[G], l[G], acc[G][EPL];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    m[i] = -CUDART_INF_F;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[i][e] = 0.f;
  }

  uint32_t bad = ri.ok ? 0u : QSA_STATUS_BAD_ROW;
  const int32_t* idx_row = p.indices + (int64_t)r * p.W;
  // keys in flight per warp: 8, or 4 when the group's accumulators are large
  constexpr int U = G * EPL <= 32 ? 8 : 4;
  for (int j0 = warp * U; j0 < ri.n; j0 += NW * U) {
    // lane u < U translates key j0 + u (entries past counts are never read)
    uint32_t off = kInvalidOff;
    if (lane < U && j0 + lane < ri.n) {
      const int32_t pos = __ldg(idx_row + j0 + lane);
      const int64_t lp = logical_page(p, ri.kv_len, pos, bad);
      if (lp >= 0) off = k_row_offset16(p, __ldg(p.table + (int64_t)ri.b * p.max_pages + lp), pos, h, bad);
    }
    uint32_t offs[U];
    float k[U][EPL], v[U][EPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      offs[u] = __shfl_sync(0xffffffffu, off, u);
      if (offs[u] != kInvalidOff) {
        const unsigned char* krow = p.kv + (int64_t)offs[u] * 16;
        load_slice<ELEM, EPL>(krow, lane, k[u]);
        load_slice<ELEM, EPL>(krow + p.v_minus_k_bytes, lane, v[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (offs[u] == kInvalidOff) continue;  // (the same in every lane)
#pragma unroll
      for (int i = 0; i < G; ++i) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dot = fmaf(qr[i][e], k[u][e], dot);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const float s = dot * p.scale_log2;
        const float mn = fmaxf(m[i], s);
        const float alpha = exp2f(m[i] - mn);
        const float pe = exp2f(s - mn);
        l[i] = l[i] * alpha + pe;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[i][e] = fmaf(acc[i][e], alpha, pe * v[u][e]);
        m[i] = mn;
      }
    }
  }
  bad = __reduce_or_sync(0xffffffffu, bad);  // the translating lanes' flags
  if (bad && lane == 0) atomicOr(p.status, bad);

#pragma unroll
  for (int i = 0; i < G; ++i) {
    if (lane == 0) {
      sm_m[warp * G + i] = m[i];
      sm_l[warp * G + i] = l[i];
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_o[(warp * G + i) * D + lane * EPL + e] = acc[i][e];
  }
  __syncthreads();
  finish_unit<NW>(p, r, h, 0, ri.ok, sm_m, sm_l, sm_o, G, nullptr);  // never split
}

template <int ELEM, int D>
cudaError_t launch_d(const Params& p, cudaStream_t s) {
  const dim3 grid((unsigned)((int64_t)p.total_q * p.nkv)), block(128);
  switch (p.group) {
    case 1: simt_kernel<ELEM, D, 1><<<grid, block, 0, s>>>(p); break;
    case 2: simt_kernel<ELEM, D, 2><<<grid, block, 0, s>>>(p); break;
    case 3: simt_kernel<ELEM, D, 3><<<grid, block, 0, s>>>(p); break;
    case 4: simt_kernel<ELEM, D, 4><<<grid, block, 0, s>>>(p); break;
    case 5: simt_kernel<ELEM, D, 5><<<grid, block, 0, s>>>(p); break;
    case 6: simt_kernel<ELEM, D, 6><<<grid, block, 0, s>>>(p); break;
    case 7: simt_kernel<ELEM, D, 7><<<grid, block, 0, s>>>(p); break;
    case 8: simt_kernel<ELEM, D, 8><<<grid, block, 0, s>>>(p); break;
    case 16: simt_kernel<ELEM, D, 16><<<grid, block, 0, s>>>(p); break;
    default:
      return cudaErrorInvalidValue;  // the host only sends groups 1..8 and 16 here
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt(const Params& p, int elem, cudaStream_t s) {
  if (p.total_q == 0 || p.nkv == 0) return cudaSuccess;
  if (elem == kF32) return p.D == 64 ? launch_d<kF32, 64>(p, s) : launch_d<kF32, 128>(p, s);
  if (elem == kBF16) return p.D == 64 ? launch_d<kBF16, 64>(p, s) : launch_d<kBF16, 128>(p, s);
  return p.D == 64 ? launch_d<kE4M3, 64>(p, s) : launch_d<kE4M3, 128>(p, s);
}

}  // namespace qsa
