// Tensor-core kernel for QSA gather-GQA sparse attention, BF16 and FP8 e4m3
// caches, head_dim 128 (QSASparseAttentionRaggedPaged: "Gather-GQA over the
// token indices a QSA selection names"; its `group`, `warps` and `unroll`
// parameters: query heads per kv head, warps per CTA, gathered keys loaded
// before any is consumed).
//
// Shape of the work.  One (query row, kv head) attends `group` query heads to
// n gathered rows: S = Q K^T with Q only group x 128 and K n x 128.  So the
// gathered keys are the MMA's M dimension and the group's query heads its N:
//     S^T[16 keys x 8 heads]   = K[16 x 128] . Q^T            (mma m16n8k16 bf16 /
//                                                               m16n8k32 e4m3)
//     O^T[128 x 8 heads]      += V^T[128 x 16 keys] . P^T      (mma m16n8k16 bf16 / f16)
// Groups of up to 8 heads use one 8-wide N tile, up to 16 two.  The S^T
// accumulator turns into the P^T operand with two movmatrix transposes per
// N tile, so scores never leave registers.  FP8 V is widened to f16 in
// registers (exact) after a transposing ldmatrix; P is f16 there.
//
// Memory.  CTA = 4 warps = one (row, kv head) unit, or one band of its
// selection under split-K.  A prologue translates the band's positions into
// 16-byte cache-row offsets once (page table lookups overlapped 8 deep per
// thread) and keeps them in shared memory.  Gathered K and V rows then stream
// through a cp.async ring of 64-key stages (16 keys per warp) with
// STAGES - 1 stages in flight; rows are padded by 16 bytes in shared memory
// so ldmatrix is conflict-free.  Skipped keys (past the band, or positions
// that fail the range checks) are zero-filled by cp.async and masked to -inf.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "qsa_device.cuh"

namespace qsa {

template <int KIND>
struct MmaCfg {
  static constexpr int D = 128;
  static constexpr int ELEM = KIND == kBF16 ? 2 : 1;
  static constexpr int ROWB = D * ELEM;            // bytes of one K or V row
  static constexpr int SROW = ROWB + 16;           // padded shared-memory row
  static constexpr int TILE = kMmaTile;            // keys per stage
  static constexpr int KV_BYTES = TILE * SROW;     // the K (or V) half of a stage
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int STAGES = KIND == kBF16 ? 3 : 4;
  static constexpr int CPR = ROWB / 16;            // 16-byte chunks per row
  static constexpr int KSTEPS = KIND == kBF16 ? 8 : 4;  // MMA k-steps over head_dim for S
  static constexpr int SMEM = STAGES * STAGE_BYTES + kMmaMaxBand * 4;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_e4m3(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// Two e4m3 bytes (low byte first) -> f16x2 with the low byte in the low half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two_bytes, __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

template <int KIND, int NT>
__global__ void __launch_bounds__(kMmaThreads, 2) mma_kernel(const Params p) {
  using C = MmaCfg<KIND>;
  constexpr int NW = kMmaThreads / 32;
  constexpr int GP = 8 * NT;  // padded query heads
  extern __shared__ __align__(128) unsigned char smem[];
  uint32_t* s_off = reinterpret_cast<uint32_t*>(smem + C::STAGES * C::STAGE_BYTES);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;

  // CTA -> (kv head, split, row): kv heads of one row are adjacent in the grid
  // (their K/V rows sit side by side in a cache slot), rows run latest first.
  int cta = blockIdx.x;
  const int h = cta % p.nkv;
  cta /= p.nkv;
  const int split = cta % p.splits;
  const int r = p.total_q - 1 - cta / p.splits;

  const RowInfo ri = row_info(p, r);
  const bool block_sel = p.blocks != nullptr;
  const bool latent = p.comp != nullptr;
  const int j0 = split * p.band;
  const int n_row = block_sel || latent ? p.W : ri.n;  // block and latent lists are masked per key instead
  const int band_n = ri.ok ? max(0, min(n_row - j0, p.band)) : 0;
  uint32_t bad = ri.ok ? 0u : QSA_STATUS_BAD_ROW;

  // ---- translate the band's positions into K-row offsets (16-byte units) ----
  {
    const int32_t* idx_row = p.indices + (int64_t)r * p.W + j0;
    const int32_t* blk_row = p.blocks + ((int64_t)h * p.total_q + r) * p.topk;
    // the row's own position, for the block lists' causal rule and the window
    const int64_t pos_q =
        (block_sel || latent) && ri.ok ? (int64_t)__ldg(p.cache_lengths + ri.b) + r - (int64_t)__ldg(p.row_offsets + ri.b) : 0;
    const uint32_t* trow = p.table + (int64_t)ri.b * p.max_pages;
    for (int k0 = 0; k0 < band_n; k0 += kMmaThreads * 8) {
      int32_t pos[8];
      int64_t lp[8];
      uint32_t page[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * kMmaThreads + tid;
        if (block_sel) {
          // slot (j0 + k) % P of listed block (j0 + k) / P; -1 when unused or
          // after the row's position (never attended, not an error)
          const int j = j0 + k;
          const int32_t beta = k < band_n ? __ldg(blk_row + j / p.P) : -1;
          const int64_t q = (int64_t)beta * p.P + (j - (j / p.P) * p.P);
          pos[u] = beta >= 0 && q <= pos_q ? (int32_t)q : -1;
        } else if (latent) {
          // window key j (position pos - window + 1 + j; -1 before the start of
          // the sequence), then entry j - window of the compressed list
          const int j = j0 + k;
          if (k >= band_n) pos[u] = -1;
          else if (j < p.window) pos[u] = pos_q - p.window + 1 + j >= 0 ? (int32_t)(pos_q - p.window + 1 + j) : -1;
          else pos[u] = __ldg(p.comp + (int64_t)r * p.num_comp + (j - p.window));
        } else {
          pos[u] = k < band_n ? __ldg(idx_row + k) : 0;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * kMmaThreads + tid;
        const bool skip = (block_sel || latent) && pos[u] < 0;
        const bool entry = latent && j0 + k >= p.window;  // in the compressed cache
        if (entry && k < band_n && !skip) {
          const int64_t ent = pos[u];
          if (ent >= (int64_t)__ldg(p.cache_lengths2 + ri.b)) {
            bad |= QSA_STATUS_BAD_INDEX;
            lp[u] = -1;
          } else if (ent / p.P2 >= p.max_pages2) {
            bad |= QSA_STATUS_BAD_PAGE;
            lp[u] = -1;
          } else {
            lp[u] = ent / p.P2;
          }
          page[u] = lp[u] >= 0 ? __ldg(p.table2 + (int64_t)ri.b * p.max_pages2 + lp[u]) : 0u;
        } else {
          lp[u] = k < band_n && !skip ? logical_page(p, ri.kv_len, pos[u], bad) : -1;
          page[u] = lp[u] >= 0 ? __ldg(trow + lp[u]) : 0u;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * kMmaThreads + tid;
        if (k >= band_n) continue;
        if (latent && j0 + k >= p.window && lp[u] >= 0) {
          if (page[u] >= p.num_pages2) {
            bad |= QSA_STATUS_BAD_PAGE;
            s_off[k] = kInvalidOff;
          } else {
            const int64_t ent = pos[u];
            const int64_t off = (int64_t)page[u] * p.page_pitch_bytes2 + p.k_layer_bytes2 + (ent - lp[u] * p.P2) * p.slot_bytes2;
            s_off[k] = (uint32_t)(off >> 4) | 0x80000000u;  // bit 31: the compressed cache
          }
        } else {
          s_off[k] = lp[u] >= 0 ? k_row_offset16(p, page[u], pos[u], h, bad) : kInvalidOff;
        }
      }
    }
  }
  if (bad) atomicOr(p.status, bad);

  // ---- Q^T fragments (the MMA B operand), zero for padded heads ----
  uint32_t qf[NT][C::KSTEPS][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = nt * 8 + gid;
    const bool live = head < p.group;
    const unsigned char* qrow = p.q + (((int64_t)r * p.nq + (int64_t)h * p.group + (live ? head : 0)) * C::D) * C::ELEM;
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      // bf16: k-step of 16 elements, thread pair (2 tig, 2 tig + 1) and +8
      // e4m3: k-step of 32 elements, thread quad (4 tig .. 4 tig + 3) and +16
      const int e0 = KIND == kBF16 ? ks * 16 + 2 * tig : ks * 32 + 4 * tig;
      const int e1 = KIND == kBF16 ? e0 + 8 : e0 + 16;
      qf[nt][ks][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + e0 * C::ELEM)) : 0u;
      qf[nt][ks][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + e1 * C::ELEM)) : 0u;
    }
  }
  __syncthreads();  // s_off complete

  const int ntiles = (band_n + C::TILE - 1) / C::TILE;
  auto issue = [&](int t) {
    unsigned char* sb = smem + (t % C::STAGES) * C::STAGE_BYTES;
    constexpr int TOTAL = C::TILE * 2 * C::CPR;
#pragma unroll
    for (int i = 0; i < TOTAL / kMmaThreads; ++i) {
      const int c = i * kMmaThreads + tid;
      const int key = c / (2 * C::CPR);
      const int w = c - key * (2 * C::CPR);
      const int kv = w / C::CPR, ch = w - kv * C::CPR;
      const int kk = t * C::TILE + key;
      const uint32_t off = kk < band_n ? s_off[kk] : kInvalidOff;
      const bool live = off != kInvalidOff;
      // bit 31 of a live offset names the latent mode's compressed cache
      const bool second = live && (off & 0x80000000u);
      const unsigned char* base = second ? p.kv2 : p.kv;
      const int64_t vk = second ? p.v_minus_k_bytes2 : p.v_minus_k_bytes;
      const unsigned char* src = live ? base + (int64_t)(off & 0x7FFFFFFFu) * 16 + (kv ? vk : 0) + ch * 16 : p.kv;
      cp_async16(smem_addr(sb + kv * C::KV_BYTES + key * C::SROW + ch * 16), src, live ? 16u : 0u);
    }
  };

#pragma unroll
  for (int s = 0; s < C::STAGES - 1; ++s) {
    if (s < ntiles) issue(s);
    cp_async_commit();
  }

  float m_run[NT][2], l_run[NT][2];
  float o[8][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
  }

  // per-lane ldmatrix row / column: non-transposed A (K) and transposed A (V^T)
  const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8, a_col = ((lane >> 4) & 1) * 16;
  const int t_row = (lane & 7) + ((lane >> 4) & 1) * 8, t_col = ((lane >> 3) & 1) * 16;

  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<C::STAGES - 2>();
    __syncthreads();
    if (t + C::STAGES - 1 < ntiles) issue(t + C::STAGES - 1);
    cp_async_commit();

    const unsigned char* sb = smem + (t % C::STAGES) * C::STAGE_BYTES;
    const int kA = t * C::TILE + warp * 16 + gid, kB = kA + 8;
    const bool vA = kA < band_n && s_off[kA] != kInvalidOff;
    const bool vB = kB < band_n && s_off[kB] != kInvalidOff;
    if (!__any_sync(0xffffffffu, vA || vB)) continue;
    const uint32_t kbase = smem_addr(sb) + warp * 16 * C::SROW;
    const uint32_t vbase = smem_addr(sb + C::KV_BYTES) + warp * 16 * C::SROW;

    // S^T = K Q^T over head_dim
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      uint32_t a[4];
      ldsm_x4(kbase + a_row * C::SROW + ks * 32 + a_col, a);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if constexpr (KIND == kBF16)
          mma_bf16(s[nt], a, qf[nt][ks][0], qf[nt][ks][1]);
        else
          mma_e4m3(s[nt], a, qf[nt][ks][0], qf[nt][ks][1]);
      }
    }

    // online softmax (base 2) per query head; this thread holds keys gid and
    // gid + 8 of heads nt*8 + 2*tig + {0, 1}
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float pv[4];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float x0 = vA ? s[nt][c] * p.scale_log2 : -CUDART_INF_F;
        const float x1 = vB ? s[nt][2 + c] * p.scale_log2 : -CUDART_INF_F;
        float mx = fmaxf(x0, x1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m_run[nt][c], mx);
        const float muse = mnew == -CUDART_INF_F ? 0.f : mnew;
        const float alpha = exp2f(m_run[nt][c] - muse);
        const float p0 = exp2f(x0 - muse), p1 = exp2f(x1 - muse);
        l_run[nt][c] = l_run[nt][c] * alpha + p0 + p1;
        m_run[nt][c] = mnew;
        pv[c] = p0;
        pv[2 + c] = p1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][nt][c] *= alpha;
          o[mt][nt][2 + c] *= alpha;
        }
      }
      // P^T as the B operand: transpose the two 8x8 halves (keys 0-7, 8-15)
      const uint32_t top = KIND == kBF16 ? pack_bf16(pv[0], pv[1]) : pack_f16(pv[0], pv[1]);
      const uint32_t bot = KIND == kBF16 ? pack_bf16(pv[2], pv[3]) : pack_f16(pv[2], pv[3]);
      pb[nt][0] = movmatrix_t(top);
      pb[nt][1] = movmatrix_t(bot);
    }

    // O^T += V^T P^T
    if constexpr (KIND == kBF16) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t a[4];
        ldsm_x4_t(vbase + t_row * C::SROW + mt * 32 + t_col, a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(o[mt][nt], a, pb[nt][0], pb[nt][1]);
      }
    } else {
      // e4m3 rows are read as byte pairs: a transposing ldmatrix hands this
      // thread (key 2tig, 2tig+1) x (d 2gid, 2gid+1) of each 16-byte column
      // block; output rows of an M tile are d = 16mt + 2gid (row gid) and
      // 16mt + 2gid + 1 (row gid + 8).
#pragma unroll
      for (int pr = 0; pr < 4; ++pr) {
        uint32_t r4[4];
        ldsm_x4_t(vbase + t_row * C::SROW + pr * 32 + t_col, r4);
        uint32_t a_even[4], a_odd[4];
        const uint32_t s0 = __byte_perm(r4[0], 0, 0x3120), s1 = __byte_perm(r4[1], 0, 0x3120);
        const uint32_t s2 = __byte_perm(r4[2], 0, 0x3120), s3 = __byte_perm(r4[3], 0, 0x3120);
        a_even[0] = e4m3x2_to_f16x2(s0 & 0xFFFFu);
        a_even[1] = e4m3x2_to_f16x2(s0 >> 16);
        a_even[2] = e4m3x2_to_f16x2(s2 & 0xFFFFu);
        a_even[3] = e4m3x2_to_f16x2(s2 >> 16);
        a_odd[0] = e4m3x2_to_f16x2(s1 & 0xFFFFu);
        a_odd[1] = e4m3x2_to_f16x2(s1 >> 16);
        a_odd[2] = e4m3x2_to_f16x2(s3 & 0xFFFFu);
        a_odd[3] = e4m3x2_to_f16x2(s3 >> 16);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_f16(o[2 * pr][nt], a_even, pb[nt][0], pb[nt][1]);
          mma_f16(o[2 * pr + 1][nt], a_odd, pb[nt][0], pb[nt][1]);
        }
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // the ring is drained; its shared memory now holds the warp states

  float* sm_o = reinterpret_cast<float*>(smem);  // [NW][GP][D]
  float* sm_m = sm_o + NW * GP * C::D;
  float* sm_l = sm_m + NW * GP;
  float* scratch = sm_l + NW * GP;  // split-K merge: 2 * kMaxSplits * group floats
  static_assert((NW * GP * C::D + 2 * NW * GP + 2 * kMaxSplits * GP) * 4 <= C::STAGES * C::STAGE_BYTES,
                "epilogue buffers must fit in the drained ring");
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float l = l_run[nt][c];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      const int head = nt * 8 + 2 * tig + c;
      if (gid == 0) {
        sm_m[warp * GP + head] = m_run[nt][c];
        sm_l[warp * GP + head] = l;
      }
    }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int head = nt * 8 + 2 * tig + (c & 1);
        const int d = KIND == kBF16 ? mt * 16 + gid + (c >> 1) * 8 : mt * 16 + 2 * gid + (c >> 1);
        sm_o[(warp * GP + head) * C::D + d] = o[mt][nt][c];
      }
  __syncthreads();
  finish_unit<NW>(p, r, h, split, ri.ok, sm_m, sm_l, sm_o, GP, scratch);
}

template <int KIND, int NT>
cudaError_t launch_mma_nt(const Params& p, cudaStream_t s) {
  using C = MmaCfg<KIND>;
  static int configured_mask = 0;  // one bit per device (up to 32)
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(configured_mask & (1 << (dev & 31)))) {
    const cudaError_t e = cudaFuncSetAttribute(mma_kernel<KIND, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured_mask |= 1 << (dev & 31);
  }
  const int64_t ctas = (int64_t)p.total_q * p.nkv * p.splits;
  if (ctas == 0) return cudaSuccess;
  mma_kernel<KIND, NT><<<(unsigned)ctas, kMmaThreads, C::SMEM, s>>>(p);
  return cudaGetLastError();
}

template <int KIND>
int mma_occupancy(int group) {
  using C = MmaCfg<KIND>;
  int n = 0;
  if (group <= 8) {
    cudaFuncSetAttribute(mma_kernel<KIND, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mma_kernel<KIND, 1>, kMmaThreads, C::SMEM);
  } else {
    cudaFuncSetAttribute(mma_kernel<KIND, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mma_kernel<KIND, 2>, kMmaThreads, C::SMEM);
  }
  return n > 0 ? n : 1;
}

}  // namespace qsa
