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
// 16-byte cache-row offsets once, in three dependent trips to memory (row
// search, counts and Q; list entries; page table), and keeps them in shared
// memory.  Gathered K and V rows then stream through a ring of 64-key stages
// (16 keys per warp) with STAGES - 1 stages in flight.  Two variants:
//   - 16-byte cp.async per row chunk into rows padded by 16 bytes (ldmatrix
//     is conflict-free); skipped keys (past the band, or positions that fail
//     the range checks) are zero-filled and masked to -inf;
//   - for block lists, TILES: a tile of 64 consecutive slots of one page is
//     one TMA tile copy per 128-byte line of K and of V into a 128-byte-
//     swizzled layout, completing on a per-stage mbarrier; other tiles take
//     16-byte copies into the same layout.
// The bands of a unit merge through distributed shared memory when they form
// one thread-block cluster (2 to 8 bands), else through a workspace ticket.
// BF16 tile copies on grids of many waves use two stages (three CTAs per SM);
// latent rows whose 16-head groups come in fours run one CTA for four groups,
// a warp per group over every key (each key gathered once per row).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "qsa_device.cuh"
#include "qsa_umma.cuh"

namespace qsa {

// TILES: the variant with tile copies (block lists, whose tiles are mostly
// whole pages) and the 128-byte-swizzled stage layout they write; without,
// 16-byte copies only into rows padded by 16 bytes (no tile-copy code in the
// loop, which measurably slows the per-row path).  SHALLOW (BF16 tile copies
// only): two stages instead of three, so three CTAs fit on an SM, for grids
// of many waves whose gathers mostly hit L2.
template <int KIND, bool TILES, bool SHALLOW = false, bool UMMA = false>
struct MmaCfg {
  static constexpr int D = 128;
  static constexpr int ELEM = KIND == kBF16 ? 2 : 1;
  static constexpr int ROWB = D * ELEM;            // bytes of one K or V row
  static constexpr int LINES = ROWB / 128;         // 128-byte lines per row
  static constexpr int TILE = kMmaTile;            // keys per stage
  static constexpr int LINE_BYTES = TILE * 128;    // one line of every key of a stage (swizzled layout)
  static constexpr int SROW = ROWB + 16;           // padded shared-memory row (16-byte copies only)
  static constexpr int KV_BYTES = TILES ? LINES * LINE_BYTES : TILE * SROW;  // the K (or V) half of a stage
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int STAGES = KIND == kBF16 ? (SHALLOW ? 2 : 3) : 4;
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int CPR = ROWB / 16;            // 16-byte chunks per row
  static constexpr int KSTEPS = KIND == kBF16 ? 8 : 4;  // MMA k-steps over head_dim for S
  static constexpr int MAXT = kMmaMaxBand / TILE;  // most tiles of a band
  // ring (1024-byte aligned with tile copies: the 128-byte swizzle repeats
  // every 8 lines), band offsets, and with tile copies one barrier per stage
  // and the tile-copy coordinates
  // tcgen05 consumer (UMMA, tile-copy layout only): the query heads as a
  // 128-byte-swizzled K-major tile (16 rows x 128 elements), right after the
  // ring, and a small block after the tile records (reductions, barriers,
  // the tensor-memory address)
  static constexpr int QBYTES = UMMA ? 16 * 128 * ELEM : 0;
  static constexpr int UMISC = UMMA ? 1024 : 0;
  static constexpr int SMEM = TILES ? 1024 + RING + QBYTES + kMmaMaxBand * 4 + STAGES * 8 + MAXT * 8 + UMISC
                                    : RING + kMmaMaxBand * 4;
  static_assert(!UMMA || (TILES && KIND == kBF16), "the tcgen05 consumer reads the BF16 tile-copy layout");
};

// Shared-memory layout of a stage's K (or V) half: line x of key k's row
// (x < LINES) sits at x * TILE * 128 + k * 128, and its 16-byte chunk c at
// chunk c XOR (k mod 8) inside that line: the 128-byte swizzle a TMA tile
// copy applies, which also keeps ldmatrix's eight 16-byte rows in eight
// different bank groups.
__device__ __forceinline__ uint32_t swz_off(int k, int chunk) {
  return (uint32_t)((chunk >> 3) * (kMmaTile * 128) + k * 128 + (((chunk & 7) ^ (k & 7)) << 4));
}

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

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of `bar` with this parity; false after kSpinLimit polls
// (each poll may block for a while in hardware), which never happens unless a
// copy was lost.
constexpr int kSpinLimit = 1 << 20;
// The poll limit of a test-only call whose producers issue no copies: its
// waits give up quickly instead of after kSpinLimit polls.
constexpr int kStallSpins = 4096;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int limit = kSpinLimit) {
  for (int i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// The same bounded wait as one asm statement (its loop stays out of the
// compiler's view of the surrounding loop): 1 when the phase completed, 0
// after kSpinLimit polls.  Kernel 2's tile-copy helpers carry no memory
// clobber: the stage is read only by volatile asm (ldmatrix), which keeps
// its order, and written only after a __syncthreads.
__device__ __forceinline__ uint32_t mbar_wait_asm(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      " .reg .pred p;\n"
      " .reg .u32 n;\n"
      " mov.u32 n, %3;\n"
      "WAIT:\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " @p bra.uni DONE;\n"
      " sub.u32 n, n, 1;\n"
      " setp.ne.u32 p, n, 0;\n"
      " @p bra.uni WAIT;\n"
      "DONE:\n"
      " selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSpinLimit));
  return ok;
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
// One-dimensional bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// The arrive fires on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
// Tiled TMA copy of one box of a 5-D tensor map into this CTA's shared
// memory, completing on `bar` (the map is a __grid_constant__ kernel parameter).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* map, int c0, int c1, int c2, int c3, int c4,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], "
      "[%7];\n" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar));
}
__device__ __forceinline__ void tile_fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::); }
__device__ __forceinline__ void tile_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes));
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

// 2^x with the hardware approximation (PTX ex2.approx.ftz: relative error
// near 2^-22, results below 2^-126 flushed to zero, 2^-inf = 0), for the
// softmax terms 2^(s - max) <= 1 of the main loops.
__device__ __forceinline__ float exp2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// Four e4m3 bytes [b0 b1 b2 b3] -> f16x2 (b0, b1) and f16x2 (b2, b3), each
// conversion reading a 16-bit half of the word directly.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four_bytes, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(four_bytes));
}

// ---- thread-block cluster: barrier and distributed shared memory ----
// All threads of every CTA of the cluster arrive; writes before the barrier
// are visible cluster-wide after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// End of a (row r, kv head h) unit, or of band `split` of it, from NW
// per-warp softmax states in shared memory: sm_m[w*GP + i] (running max of
// the base-2 scores), sm_l[w*GP + i] (sum of exponentials) and
// sm_o[(w*GP + i)*D + d] (unnormalised output), query heads i < group.
// First one thread per head merges the warps' maxima and sums and keeps each
// warp's weight (s_e: NW*GP + 2*GP floats of shared memory); then every
// output element is a weighted sum of NW values, four channels per thread.
//   - one band (splits == 1): writes output[r, h*group + i, :];
//   - bands merged through the workspace: stores this band's partial and
//     runs the ticket merge (the last band to arrive merges);
//   - bands of one thread-block cluster (CTA rank = band): keeps the partial
//     o[G][D], m[G], l[G] in its own shared memory (`part`); after a cluster
//     barrier every CTA reads all bands' maxima and sums, and the o values
//     of its 1/S slice of the output, through distributed shared memory and
//     writes that slice; a second barrier keeps each partial alive until
//     the other CTAs have read it.  No global workspace, fence or ticket.
template <int NW>
__device__ __forceinline__ void finish_unit_mma(const Params& p, int r, int h, int split, bool row_ok,
                                                const float* sm_m, const float* sm_l, const float* sm_o, int GP,
                                                float* scratch, float* part, float* s_e) {
  const int G = p.group, D = p.D, S = p.splits;
  float* s_M = s_e + NW * GP;
  float* s_L = s_M + GP;
  // one thread per (head, warp), NW adjacent lanes per head
  static_assert(NW == 4, "four warp states per head");
  const int wid = threadIdx.x >> 5;
  if (wid < (G * NW + 31) / 32) {
    const int i = threadIdx.x >> 2, w = threadIdx.x & 3;
    const bool on = i < G;
    const float m = on ? sm_m[w * GP + i] : -CUDART_INF_F;
    float M = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
    const float e = M == -CUDART_INF_F ? 0.f : exp2f(m - M);
    float L = on ? sm_l[w * GP + i] * e : 0.f;
    L += __shfl_xor_sync(0xffffffffu, L, 1);
    L += __shfl_xor_sync(0xffffffffu, L, 2);
    if (on) {
      s_e[w * GP + i] = e;
      if (w == 0) {
        s_M[i] = M;
        s_L[i] = L;
      }
    }
  }
  __syncthreads();
  const int n4 = G * D / 4;
  const int64_t out_base = ((int64_t)r * p.nq + (int64_t)h * G) * D;
  if (S == 1) {
    for (int q4 = threadIdx.x; q4 < n4; q4 += blockDim.x) {
      const int idx = q4 * 4, i = idx / D, d = idx - i * D;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float e = s_e[w * GP + i];
        const float4 o = *reinterpret_cast<const float4*>(sm_o + (w * GP + i) * D + d);
        acc.x = fmaf(e, o.x, acc.x);
        acc.y = fmaf(e, o.y, acc.y);
        acc.z = fmaf(e, o.z, acc.z);
        acc.w = fmaf(e, o.w, acc.w);
      }
      const float M = s_M[i];
      const bool live = row_ok && M != -CUDART_INF_F;
      const float den = live ? s_L[i] + sink_term(p, h * G + i, M) : 1.f;
      store_out(p, out_base + idx, live ? acc.x / den : 0.f);
      store_out(p, out_base + idx + 1, live ? acc.y / den : 0.f);
      store_out(p, out_base + idx + 2, live ? acc.z / den : 0.f);
      store_out(p, out_base + idx + 3, live ? acc.w / den : 0.f);
    }
    return;
  }
  // this band's partial: o[G][D], m[G], l[G]
  float* dst = p.cluster ? part : p.ws_partial + ((int64_t)(r * p.nkv + h) * S + split) * partial_stride(G, D);
  for (int q4 = threadIdx.x; q4 < n4; q4 += blockDim.x) {
    const int idx = q4 * 4, i = idx / D, d = idx - i * D;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float e = s_e[w * GP + i];
      const float4 o = *reinterpret_cast<const float4*>(sm_o + (w * GP + i) * D + d);
      acc.x = fmaf(e, o.x, acc.x);
      acc.y = fmaf(e, o.y, acc.y);
      acc.z = fmaf(e, o.z, acc.z);
      acc.w = fmaf(e, o.w, acc.w);
    }
    *reinterpret_cast<float4*>(dst + idx) = acc;
  }
  for (int i = threadIdx.x; i < G; i += blockDim.x) {
    dst[G * D + i] = s_M[i];
    dst[G * D + G + i] = s_L[i];
  }
  if (!p.cluster) {
    merge_split_partials(p, r, h, row_ok, scratch);
    return;
  }
  cluster_sync_all();
  const uint32_t part_a = smem_addr(part);
  // every band's max and sum, one thread per (head, band): SP adjacent lanes
  // per head (SP = S rounded up to a power of two), reduced by shuffles
  float* s_w = scratch;  // [S][G]: weight of band s for head i
  {
    const int SP = S <= 2 ? 2 : S <= 4 ? 4 : 8;
    if (wid < (G * SP + 31) / 32) {
      const int i = threadIdx.x / SP, sb = threadIdx.x - i * SP;
      const bool on = i < G && sb < S;
      const float m = on ? ld_cluster_f32(cluster_map(part_a + (uint32_t)(G * D + i) * 4u, (uint32_t)sb)) : -CUDART_INF_F;
      const float l = on ? ld_cluster_f32(cluster_map(part_a + (uint32_t)(G * D + G + i) * 4u, (uint32_t)sb)) : 0.f;
      float M = m;
      for (int o = 1; o < SP; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float e = M == -CUDART_INF_F ? 0.f : exp2f(m - M);
      float L = l * e;
      for (int o = 1; o < SP; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      const bool live = row_ok && M != -CUDART_INF_F;
      if (live) L += sink_term(p, h * G + (i < G ? i : 0), M);
      if (on) s_w[sb * G + i] = live ? e / L : 0.f;
    }
  }
  __syncthreads();
  const int q_lo = split * n4 / S, q_hi = (split + 1) * n4 / S;
  for (int q4 = q_lo + (int)threadIdx.x; q4 < q_hi; q4 += blockDim.x) {
    const int idx = q4 * 4, i = idx / D;
    // every band's four values in flight at once
    float4 o[kMaxClusterSplits];
#pragma unroll
    for (int s = 0; s < kMaxClusterSplits; ++s)
      if (s < S) o[s] = ld_cluster_f32x4(cluster_map(part_a + (uint32_t)idx * 4u, (uint32_t)s));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kMaxClusterSplits; ++s)
      if (s < S) {
        const float w = s_w[s * G + i];
        acc.x = fmaf(w, o[s].x, acc.x);
        acc.y = fmaf(w, o[s].y, acc.y);
        acc.z = fmaf(w, o[s].z, acc.z);
        acc.w = fmaf(w, o[s].w, acc.w);
      }
    store_out(p, out_base + idx, acc.x);
    store_out(p, out_base + idx + 1, acc.y);
    store_out(p, out_base + idx + 2, acc.z);
    store_out(p, out_base + idx + 3, acc.w);
  }
  cluster_sync_all();
}

// GROUPS (latent mode, one band): a CTA serves NW query-head groups of one
// row that read the same keys; warp w owns group w over every key of a tile
// (all NW 16-key slices) and writes its heads from registers, so each key is
// gathered once per row instead of once per group.
//
// UMMA (BF16, tile-copy layout): the scores and the output accumulate in
// tensor memory through tcgen05 MMAs issued by one thread, on the stage bytes
// as the copies left them (the 128-byte-swizzled layout is the tensor cores'
// K-major layout for K and, read transposed, their MN-major layout for V^T):
//     S^T[64 keys x GP]  = K[64 x 128] . Q^T      (M = 64, one lane per key)
//     O^T[128 x 16]     += V^T[128 x 64] . P^T    (M = 128, one lane per channel)
// The four warps turn S^T into P^T (one key per lane); the running maximum is
// one reference per head for the whole CTA, moved only when a tile's maximum
// passes it by more than 8 (base 2), and O^T is rescaled in tensor memory
// then.  P^T goes into the stage's first 2 KB, whose K rows q.K has consumed.
template <int KIND, int NT, bool TILES, bool SHALLOW, bool GROUPS, bool UMMA = false>
__global__ void __launch_bounds__(kMmaThreads, 2) mma_kernel(const __grid_constant__ Params p) {
  using C = MmaCfg<KIND, TILES, SHALLOW, UMMA>;
  constexpr int NW = kMmaThreads / 32;
  constexpr int GP = 8 * NT;  // padded query heads
  static_assert(!UMMA || !GROUPS, "the tcgen05 consumer serves one head group per CTA");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = TILES ? smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u) : smem_raw;  // the stage ring
  unsigned char* q_tile = smem + C::RING;  // UMMA: the query heads, K-major, 128-byte swizzle (1024-byte aligned)
  uint32_t* s_off = reinterpret_cast<uint32_t*>(smem + C::RING + C::QBYTES);
  uint64_t* s_full = reinterpret_cast<uint64_t*>(s_off + kMmaMaxBand);  // TILES: one barrier per stage
  int2* s_tile = reinterpret_cast<int2*>(s_full + C::STAGES);           // TILES: tile copy (page, first slot) or (-1, 0)
  // UMMA: per-warp maxima and sums [NW][16], the barriers of q.K (two S^T
  // buffers) and p.V, the tensor-memory base
  float* u_red = reinterpret_cast<float*>(s_tile + C::MAXT);
  uint64_t* u_bar = reinterpret_cast<uint64_t*>(u_red + NW * 16);
  uint32_t* u_tmem = reinterpret_cast<uint32_t*>(u_bar + 3);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  if (TILES && tid == 0) {
    // a stage's barrier completes a phase when a tile copy into it landed
    // (16-byte copies complete through per-thread cp.async groups instead)
    for (int k = 0; k < C::STAGES; ++k) mbar_init(smem_addr(&s_full[k]), 1);
    if (UMMA) {  // q.K of even and of odd tiles, p.V: one tcgen05 commit per phase
      mbar_init(smem_addr(&u_bar[0]), 1);
      mbar_init(smem_addr(&u_bar[1]), 1);
      mbar_init(smem_addr(&u_bar[2]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if constexpr (UMMA) {
    // 64 tensor-memory columns: two S^T buffers at 0 and 16, O^T in [32, 48)
    if (warp == 0) {
      tmem_alloc(smem_addr(u_tmem), 64);
      tmem_relinquish();
      tc_fence_before();  // the address is read after the translation's barriers
    }
  }

  // CTA -> (split, kv head, row): the bands of one unit are adjacent in the
  // grid (one thread-block cluster when they merge through distributed shared
  // memory), then the kv heads of one row (their K/V rows sit side by side in
  // a cache slot); rows run latest first.
  int cta = blockIdx.x;
  const int split = cta % p.splits;
  cta /= p.splits;
  const int h = cta % p.nkv;
  const int qh = GROUPS ? h * NW + warp : h;  // the query-head group of this thread's heads
  const int r = p.total_q - 1 - cta / p.nkv;
  const bool block_sel = p.blocks != nullptr;
  const bool latent = p.comp != nullptr;
  const int j0 = split * p.band;

  // The translation takes three dependent trips to memory, each issuing all
  // the loads it can: (1) counts[r], the Q fragments and the search for the
  // row's sequence; (2) the sequence's offsets and cache length, and the
  // band's list entries (index entries after counts, block ids, compressed
  // entries); (3) the page-table entries.

  // ---- trip 1 ----
  const int cnt = block_sel || latent ? p.W : __ldg(p.counts + r);
  if constexpr (UMMA) {
    // the group's query heads as rows of a K-major 128-byte-swizzled tile
    // (rows past the group zero): the B operand of q.K
    for (int i = tid; i < 16 * 16; i += kMmaThreads) {
      const int n = i >> 4, c = i & 15;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (n < p.group)
        v = __ldg(reinterpret_cast<const uint4*>(p.q + (((int64_t)r * p.nq + (int64_t)qh * p.group + n) * C::D + c * 8) * C::ELEM));
      *reinterpret_cast<uint4*>(q_tile + (c >> 3) * (16 * 128) + (n >> 3) * 1024 + (n & 7) * 128 + (((c & 7) ^ (n & 7)) << 4)) = v;
    }
  }
  // Q^T fragments (the mma.sync B operand), zero for padded heads
  uint32_t qf[NT][C::KSTEPS][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if constexpr (UMMA) break;
    const int head = nt * 8 + gid;
    const bool live = head < p.group;
    const unsigned char* qrow = p.q + (((int64_t)r * p.nq + (int64_t)qh * p.group + (live ? head : 0)) * C::D) * C::ELEM;
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
  const int b = row_sequence_warp(p, r);

  // ---- trip 2 ----
  const bool in_batch = b < p.batch;
  const uint32_t o0 = in_batch ? __ldg(p.row_offsets + b) : 0u;
  const uint32_t o1 = in_batch ? __ldg(p.row_offsets + b + 1) : 0u;
  const uint32_t cl = in_batch ? __ldg(p.cache_lengths + b) : 0u;
  const bool row_ok = in_batch && o0 <= (uint32_t)r && (uint32_t)r < o1;
  const int64_t kv_len = (int64_t)cl + (int64_t)(o1 - o0);
  const int64_t pos_q = (int64_t)cl + (int64_t)r - (int64_t)o0;  // the row's own position (when row_ok)
  // keys of the band: valid index entries (counts clamped to [0, W]), or the
  // whole block / latent list (masked per key); none when the row is not in a sequence
  const int n_row = block_sel || latent ? p.W : min(max(cnt, 0), p.W);
  const int band_n = max(0, min(n_row - j0, p.band));
  const int band_keys = row_ok ? band_n : 0;
  uint32_t bad = row_ok ? 0u : QSA_STATUS_BAD_ROW;
  const uint32_t* trow = p.table + (int64_t)(in_batch ? b : 0) * p.max_pages;

  if (block_sel) {
    // one page-table lookup per listed block that meets the band, kept in
    // the (still unused) stage ring; then every key's offset from its block
    int32_t* s_beta = reinterpret_cast<int32_t*>(smem);
    uint32_t* s_page = reinterpret_cast<uint32_t*>(smem) + (kMmaMaxBand + 2);
    const int jb0 = j0 / p.P;
    const int nbk = band_n > 0 ? (j0 + band_n - 1) / p.P - jb0 + 1 : 0;
    const int32_t* blk_row = p.blocks + ((int64_t)h * p.total_q + r) * p.topk;
    for (int t = tid; t < nbk; t += kMmaThreads) {
      const int32_t beta = __ldg(blk_row + jb0 + t);  // trip 2
      const bool in_table = in_batch && beta >= 0 && beta < p.max_pages;
      s_beta[t] = beta;
      s_page[t] = in_table ? __ldg(trow + beta) : kInvalidOff;  // trip 3
    }
    __syncthreads();
    for (int k = tid; k < band_keys; k += kMmaThreads) {
      const int j = j0 + k, jb = j / p.P;
      const int32_t beta = s_beta[jb - jb0];
      // slot j % P of block beta; -1 blocks and positions after the row's own
      // are never attended (not an error)
      const int64_t q = (int64_t)beta * p.P + (j - jb * p.P);
      uint32_t off = kInvalidOff;
      if (beta >= 0 && q <= pos_q) {
        if (beta >= p.max_pages)
          bad |= QSA_STATUS_BAD_PAGE;
        else
          off = k_row_offset16(p, s_page[jb - jb0], (int32_t)q, h, bad);
      }
      s_off[k] = off;
      if (TILES && k % C::TILE == 0) s_tile[k / C::TILE] = make_int2((int)s_page[jb - jb0], j - jb * p.P);
    }
  } else {
    // ---- translate the band's positions into K-row offsets (16-byte units) ----
    const int32_t* idx_row = p.indices + (int64_t)r * p.W + j0;
    for (int k0 = 0; k0 < band_n; k0 += kMmaThreads * 8) {
      int32_t pos[8];
      int64_t lp[8];
      uint32_t page[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * kMmaThreads + tid;
        if (latent) {
          // window key j (position pos - window + 1 + j; -1 before the start of
          // the sequence), then entry j - window of the compressed list
          const int j = j0 + k;
          if (k >= band_n) pos[u] = -1;
          else if (j < p.window) pos[u] = pos_q - p.window + 1 + j >= 0 ? (int32_t)(pos_q - p.window + 1 + j) : -1;
          else pos[u] = __ldg(p.comp + (int64_t)r * p.num_comp + (j - p.window));
        } else {
          pos[u] = k < band_n ? __ldg(idx_row + k) : 0;  // entries past counts are never read
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * kMmaThreads + tid;
        const bool live = row_ok && k < band_n && !(latent && pos[u] < 0);
        const bool entry = latent && j0 + k >= p.window;  // in the compressed cache
        if (entry && live) {
          const int64_t ent = pos[u];
          if (ent >= (int64_t)__ldg(p.cache_lengths2 + b)) {
            bad |= QSA_STATUS_BAD_INDEX;
            lp[u] = -1;
          } else if (ent / p.P2 >= p.max_pages2) {
            bad |= QSA_STATUS_BAD_PAGE;
            lp[u] = -1;
          } else {
            lp[u] = ent / p.P2;
          }
          page[u] = lp[u] >= 0 ? __ldg(p.table2 + (int64_t)b * p.max_pages2 + lp[u]) : 0u;
        } else {
          lp[u] = live ? logical_page(p, kv_len, pos[u], bad) : -1;
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
          if (TILES && k % C::TILE == 0) s_tile[k / C::TILE] = make_int2((int)page[u], (int)((uint32_t)pos[u] % (uint32_t)p.P));
        }
      }
    }
  }
  if (bad) atomicOr(p.status, bad);
  __syncthreads();  // s_off complete

  // Tiles whose 64 keys are consecutive slots of one page of the first cache
  // (page-aligned runs, whole blocks) load with one TMA tile copy per 128-byte
  // line of K and of V; the others with 16-byte copies per row.
  const int ntiles = (band_keys + C::TILE - 1) / C::TILE;
  uint32_t tma_mask = 0;  // bit t: tile t is a tile copy (a band has at most 32 tiles)
  if constexpr (TILES) {
  if (p.tma) {
    const uint32_t sstep = (uint32_t)(p.slot_bytes >> 4);
    for (int t = warp; t < ntiles; t += NW) {
      const uint32_t base = s_off[t * C::TILE];
      const bool ok = (t + 1) * C::TILE <= band_keys && base != kInvalidOff && !(base & 0x80000000u) &&
                      s_off[t * C::TILE + lane] == base + (uint32_t)lane * sstep &&
                      s_off[t * C::TILE + 32 + lane] == base + (uint32_t)(32 + lane) * sstep;
      // consecutive offsets are consecutive slots of one page (a page holds
      // more than P slots of one plane); the translation recorded the page
      // and slot of the tile's first key
      if (!__all_sync(0xffffffffu, ok) && lane == 0) s_tile[t] = make_int2(-1, 0);
    }
  } else {
    for (int t = tid; t < ntiles; t += kMmaThreads) s_tile[t] = make_int2(-1, 0);
  }
  __syncthreads();
  static_assert(C::MAXT <= 32, "tile mask");
  if (p.tma)
    for (int t = 0; t < ntiles; ++t) tma_mask |= (s_tile[t].x >= 0 ? 1u : 0u) << t;
  }

  const int hc = p.head_bytes ? h : 0;  // the unit's head in the cache (the latent cache has one)
  // stages that received a tile copy, and the parity of each stage's next
  // tile-copy phase (identical in every thread): a give-up drains them
  uint32_t tma_used = 0, tma_next = 0;
  auto issue = [&](int t) {
    unsigned char* sb = smem + (t % C::STAGES) * C::STAGE_BYTES;
    const uint32_t bar = smem_addr(&s_full[t % C::STAGES]);
    if (TILES && (tma_mask >> t & 1u)) {
      tma_used |= 1u << (t % C::STAGES);
      tma_next ^= 1u << (t % C::STAGES);
      if (tid == 0) {
        const int2 tc = s_tile[t];
        tile_fence_proxy_async();  // earlier generic accesses of the stage before the async-proxy writes
        tile_expect_tx(bar, C::STAGE_BYTES);
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
          for (int x = 0; x < C::LINES; ++x)
            tma_load_5d(smem_addr(sb + kv * C::KV_BYTES + x * C::LINE_BYTES), &p.tmap, 0, hc * C::LINES + x, tc.y,
                        kv ? p.tma_plane_v : p.tma_plane_k, tc.x, bar);
      }
      return;
    }
    constexpr int TOTAL = C::TILE * 2 * C::CPR;
#pragma unroll
    for (int i = 0; i < TOTAL / kMmaThreads; ++i) {
      const int c = i * kMmaThreads + tid;
      const int key = c / (2 * C::CPR);
      const int w = c - key * (2 * C::CPR);
      const int kv = w / C::CPR, ch = w - kv * C::CPR;
      const int kk = t * C::TILE + key;
      const uint32_t off = kk < band_keys ? s_off[kk] : kInvalidOff;
      const bool live = off != kInvalidOff;
      // bit 31 of a live offset names the latent mode's compressed cache
      const bool second = live && (off & 0x80000000u);
      const unsigned char* base = second ? p.kv2 : p.kv;
      const int64_t vk = second ? p.v_minus_k_bytes2 : p.v_minus_k_bytes;
      const unsigned char* src = live ? base + (int64_t)(off & 0x7FFFFFFFu) * 16 + (kv ? vk : 0) + ch * 16 : p.kv;
      const uint32_t dst = TILES ? swz_off(key, ch) : (uint32_t)(key * C::SROW + ch * 16);
      cp_async16(smem_addr(sb + kv * C::KV_BYTES) + dst, src, live ? 16u : 0u);
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

  // per-lane ldmatrix rows: non-transposed A (K) and transposed A (V^T), and
  // the swizzle term of each lane's 16-byte chunk (its row mod 8, and which
  // chunk of the pair it reads)
  const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int t_row = (lane & 7) + ((lane >> 4) & 1) * 8;
  const uint32_t kx16 = (uint32_t)(((lane & 7) ^ ((lane >> 4) & 1)) << 4);
  const uint32_t vx16 = (uint32_t)(((lane & 7) ^ ((lane >> 3) & 1)) << 4);
  bool timed_out = false;
  uint32_t tma_phase = 0;  // bit s: parity of the next tile-copy phase of stage s

  // UMMA state: the tensor-memory base, each head's reference maximum (the
  // same in every thread) and this thread's key's share of each head's sum
  uint32_t tmem = 0;
  int issued = 0, issued_qk = 0;  // tiles whose p.V / q.K were issued (the same in every thread)
  float m_ref[GP], l_part[GP];
  if constexpr (UMMA) {
    tc_fence_after();  // the allocation's address, published by the translation's barriers
    tmem = *u_tmem;
#pragma unroll
    for (int n = 0; n < GP; ++n) {
      m_ref[n] = -CUDART_INF_F;
      l_part[n] = 0.f;
    }
  }

  if constexpr (UMMA) {
    // Pipeline, per tile t (every thread, uniform control flow):
    //   A  tile t + 1's bytes landed -> q.K(t + 1) into the other S^T buffer
    //      (the tensor cores run it during this tile's softmax)
    //   B  S^T(t) read; p.V(t - 1) done (O^T stable, its stage free)
    //   D  tile t + 2 copied into the stage tile t - 1 used
    //   B' when a key passes its head's reference by more than 8, the exact
    //      tile maxima move the references and O^T is rescaled; P^T(t) written
    //   C  p.V(t)
    // S^T buffer b (tiles of parity b) has its own barrier, so no wait can
    // see a later phase of it; p.V's barrier is waited for tile t - 1 before
    // p.V(t) is issued.  Ring of three stages: the copies of tile t + 1 are
    // the newest when step A waits for them.
    static_assert(C::STAGES == 3, "the pipeline's copy waits assume three stages");
    constexpr uint32_t kO = 32;  // O^T columns; S^T buffers at 0 and 16
    auto wait_tile = [&](int t) -> bool {  // this thread's copies of tile t, visible to the tensor cores
      cp_async_wait<0>();
      fence_proxy_async_smem();
      bool ok = true;
      if (TILES && (tma_mask >> t & 1u)) {
        const int st = t % C::STAGES;
        ok = mbar_wait_asm(smem_addr(&s_full[st]), (tma_phase >> st) & 1u) != 0;
        tma_phase ^= 1u << st;
      }
      return ok;
    };
    auto issue_qk = [&](int t) {  // thread 0
      const uint32_t kb = smem_addr(smem + (t % C::STAGES) * C::STAGE_BYTES);
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks)
        umma_f16(tmem + (uint32_t)((t & 1) * 16),
                 smem_desc(kb + (uint32_t)((ks >> 2) * C::LINE_BYTES + (ks & 3) * 32), 16, 1024, kSwizzle128),
                 smem_desc(smem_addr(q_tile) + (uint32_t)((ks >> 2) * 2048 + (ks & 3) * 32), 16, 1024, kSwizzle128),
                 instr_desc(64, GP, 1, 0, 0), ks > 0);
      umma_commit(smem_addr(&u_bar[t & 1]));
    };
    if (ntiles > 0) {
      if (__syncthreads_or(!wait_tile(0))) {
        timed_out = true;
      } else {
        if (tid == 0) issue_qk(0);
        issued_qk = 1;
      }
    }
    for (int t = 0; t < ntiles && !timed_out; ++t) {
      const unsigned char* sb = smem + (t % C::STAGES) * C::STAGE_BYTES;
      const uint32_t kb = smem_addr(sb), vb = kb + (uint32_t)C::KV_BYTES;
      // A
      if (t + 1 < ntiles) {
        if (__syncthreads_or(!wait_tile(t + 1))) {
          timed_out = true;
          break;
        }
        if (tid == 0) issue_qk(t + 1);
        ++issued_qk;
      }
      // B: scores of key k in lane (k / 16) * 32 + k % 16
      bool lost = !mbar_wait_asm(smem_addr(&u_bar[t & 1]), (uint32_t)((t >> 1) & 1));
      tc_fence_after();
      float sv[GP];
      const uint32_t srow = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)((t & 1) * 16);
      if constexpr (GP == 8) tmem_ld8(srow, sv);
      else tmem_ld16(srow, sv);
      if (t > 0) lost |= !mbar_wait_asm(smem_addr(&u_bar[2]), (uint32_t)((t - 1) & 1));
      // D: the stage of tile t - 1 (its p.V is done) takes tile t + 2, whose
      // copies then overlap this tile's softmax and p.V (after a give-up it
      // is left alone: the stage may still be read)
      if (t + C::STAGES - 1 < ntiles && !lost) issue(t + C::STAGES - 1);
      cp_async_commit();
      const int kk = t * C::TILE + warp * 16 + (lane & 15);
      const bool valid = lane < 16 && kk < band_keys && s_off[kk] != kInvalidOff;
      bool want = false;
#pragma unroll
      for (int n = 0; n < GP; ++n) {
        sv[n] = valid && n < p.group ? sv[n] * p.scale_log2 : -CUDART_INF_F;
        want |= sv[n] > m_ref[n] + 8.f;
      }
      if (__syncthreads_or(want || lost)) {
        // the tile's maxima per head, across the warps; every thread moves the
        // references it passes by more than 8 the same way
#pragma unroll
        for (int n = 0; n < GP; ++n) {
          float mx = sv[n];
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          if (lane == 0) u_red[warp * 16 + n] = mx;
        }
        __syncthreads();
        float alpha[GP];
        bool moved = false;
#pragma unroll
        for (int n = 0; n < GP; ++n) {
          const float mt = fmaxf(fmaxf(u_red[n], u_red[16 + n]), fmaxf(u_red[32 + n], u_red[48 + n]));
          alpha[n] = 1.f;
          if (mt > m_ref[n] + 8.f) {
            alpha[n] = m_ref[n] == -CUDART_INF_F ? 0.f : exp2f(m_ref[n] - mt);
            m_ref[n] = mt;
            moved = true;
          }
          l_part[n] *= alpha[n];
        }
        if (moved && t > 0) {
          // O^T (this warp's 32 channels, 16 head columns) to the new references
          float ov[16];
          tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + kO, ov);
#pragma unroll
          for (int n = 0; n < GP; ++n) ov[n] *= alpha[n];
          tmem_st16(tmem + ((uint32_t)(warp * 32) << 16) + kO, ov);
          tmem_wait_st();
        }
        __syncthreads();  // u_red is read by every thread before the next tile writes it
      }
#pragma unroll
      for (int n = 0; n < GP; ++n) {
        const float pn = exp2_fast(sv[n] - (m_ref[n] == -CUDART_INF_F ? 0.f : m_ref[n]));
        l_part[n] += pn;
        sv[n] = pn;
      }
      // P^T, MN-major without swizzle, over the stage's first 2 KB (q.K(t)
      // has read those K rows): key k's 16 head values at (k / 8) * 256 +
      // (k % 8) * 16 (heads 0..7) and +128 (heads 8..15)
      if (lane < 16) {
        const int k = warp * 16 + lane;
        unsigned char* pr = const_cast<unsigned char*>(sb) + (k >> 3) * 256 + (k & 7) * 16;
        *reinterpret_cast<uint4*>(pr) =
            make_uint4(pack_bf16(sv[0], sv[1]), pack_bf16(sv[2], sv[3]), pack_bf16(sv[4], sv[5]), pack_bf16(sv[6], sv[7]));
        uint4 hi = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (GP == 16)
          hi = make_uint4(pack_bf16(sv[8], sv[9]), pack_bf16(sv[10], sv[11]), pack_bf16(sv[12], sv[13]),
                          pack_bf16(sv[14], sv[15]));
        *reinterpret_cast<uint4*>(pr + 128) = hi;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (__syncthreads_or(lost)) {
        timed_out = true;
        break;
      }
      // C: p.V, 4 K steps of 16 keys; O^T in columns [32, 48), lane = channel
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < C::TILE / 16; ++ks)
          umma_f16(tmem + kO, smem_desc(vb + (uint32_t)(ks * 2048), (uint32_t)C::LINE_BYTES, 1024, kSwizzle128),
                   smem_desc(kb + (uint32_t)(ks * 512), 256, 128, kSwizzleNone), instr_desc(128, 16, 1, 1, 1),
                   t > 0 || ks > 0);
        umma_commit(smem_addr(&u_bar[2]));
      }
      ++issued;
    }
  } else
  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<C::STAGES - 2>();  // this thread's 16-byte copies of tile t
    __syncthreads();  // everyone's copies of tile t landed; every warp is done with tile t - 1
    if (t + C::STAGES - 1 < ntiles) issue(t + C::STAGES - 1);
    cp_async_commit();
    if (TILES && (tma_mask >> t & 1u)) {
      const int st = t % C::STAGES;
      if (!mbar_wait_asm(smem_addr(&s_full[st]), (tma_phase >> st) & 1u)) timed_out = true;
      tma_phase ^= 1u << st;
    }

    const unsigned char* sb = smem + (t % C::STAGES) * C::STAGE_BYTES;
#pragma unroll 1
    for (int sl = 0; sl < (GROUPS ? NW : 1); ++sl) {
    const int kw = GROUPS ? sl : warp;  // the 16-key slice of the tile this warp scores
    const int kA = t * C::TILE + kw * 16 + gid, kB = kA + 8;
    const bool vA = kA < band_keys && s_off[kA] != kInvalidOff;
    const bool vB = kB < band_keys && s_off[kB] != kInvalidOff;
    if (!__any_sync(0xffffffffu, vA || vB)) continue;
    constexpr uint32_t RS = TILES ? 128u : (uint32_t)C::SROW;  // row stride of a stage half
    const uint32_t krow = smem_addr(sb) + (uint32_t)(kw * 16 + a_row) * RS;
    const uint32_t vrow = smem_addr(sb + C::KV_BYTES) + (uint32_t)(kw * 16 + t_row) * RS;

    // S^T = K Q^T over head_dim
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < C::KSTEPS; ++ks) {
      uint32_t a[4];
      if constexpr (TILES)
        ldsm_x4(krow + (uint32_t)((ks >> 2) * C::LINE_BYTES) + ((uint32_t)((2 * (ks & 3)) << 4) ^ kx16), a);
      else
        ldsm_x4(krow + ks * 32 + ((lane >> 4) & 1) * 16, a);
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
        const float alpha = exp2_fast(m_run[nt][c] - muse);
        const float p0 = exp2_fast(x0 - muse), p1 = exp2_fast(x1 - muse);
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
        if constexpr (TILES)
          ldsm_x4_t(vrow + (uint32_t)((mt >> 2) * C::LINE_BYTES) + ((uint32_t)((2 * (mt & 3)) << 4) ^ vx16), a);
        else
          ldsm_x4_t(vrow + mt * 32 + ((lane >> 3) & 1) * 16, a);
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
        if constexpr (TILES)
          ldsm_x4_t(vrow + ((uint32_t)((2 * pr) << 4) ^ vx16), r4);
        else
          ldsm_x4_t(vrow + pr * 32 + ((lane >> 3) & 1) * 16, r4);
        uint32_t a_even[4], a_odd[4];
        const uint32_t s0 = __byte_perm(r4[0], 0, 0x3120), s1 = __byte_perm(r4[1], 0, 0x3120);
        const uint32_t s2 = __byte_perm(r4[2], 0, 0x3120), s3 = __byte_perm(r4[3], 0, 0x3120);
        e4m3x4_to_f16x2x2(s0, a_even[0], a_even[1]);
        e4m3x4_to_f16x2x2(s2, a_even[2], a_even[3]);
        e4m3x4_to_f16x2x2(s1, a_odd[0], a_odd[1]);
        e4m3x4_to_f16x2x2(s3, a_odd[2], a_odd[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_f16(o[2 * pr][nt], a_even, pb[nt][0], pb[nt][1]);
          mma_f16(o[2 * pr + 1][nt], a_odd, pb[nt][0], pb[nt][1]);
        }
      }
    }
    }  // slices
  }
  float u_o[16];  // UMMA: O^T of this thread's channel (tid), one value per head column
  if constexpr (UMMA) {
    // p.V of the last tile done (its commit also covers every earlier MMA, so
    // after a give-up nothing of ours is still running either, unless this
    // bounded wait gives up too); then every head's sum over all key lanes,
    // and the tensor memory handed back
    if (issued > 0 && !mbar_wait_asm(smem_addr(&u_bar[2]), (uint32_t)((issued - 1) & 1))) timed_out = true;
    if (timed_out && issued_qk > issued)  // a q.K issued after the last p.V
      mbar_wait_asm(smem_addr(&u_bar[(issued_qk - 1) & 1]), (uint32_t)(((issued_qk - 1) >> 1) & 1));
    tc_fence_after();
    if (issued > 0) {
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 32u, u_o);
    } else {
#pragma unroll
      for (int n = 0; n < 16; ++n) u_o[n] = 0.f;
    }
#pragma unroll
    for (int n = 0; n < GP; ++n) {
      float l = l_part[n];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (lane == 0) u_red[warp * 16 + n] = l;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
  }
  if (timed_out) {
    atomicOr(p.status, QSA_STATUS_TIMEOUT);
    // a tile copy whose wait gave up may still be landing: wait again
    // (bounded) for each stage's last tile-copy phase before the ring is reused
    if (TILES && tid == 0)
      for (int st = 0; st < C::STAGES; ++st)
        if ((tma_used >> st) & 1u) mbar_wait_asm(smem_addr(&s_full[st]), ((tma_next >> st) & 1u) ^ 1u);
  }
  cp_async_wait<0>();
  __syncthreads();  // the ring is drained; its shared memory now holds the warp states

  if constexpr (GROUPS) {
    // this warp holds the whole softmax state of its group's heads: sums
    // across its key lanes, then the output straight from registers
    const int64_t ob = ((int64_t)r * p.nq + (int64_t)qh * p.group) * C::D;
    float inv[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float l = l_run[nt][c];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int head = nt * 8 + 2 * tig + c;
        const float M = m_run[nt][c];
        const bool live = row_ok && head < p.group && M != -CUDART_INF_F;
        inv[nt][c] = live ? 1.f / (l + sink_term(p, qh * p.group + head, M)) : 0.f;
      }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int head = nt * 8 + 2 * tig + (c & 1);
          const int d = KIND == kBF16 ? mt * 16 + gid + (c >> 1) * 8 : mt * 16 + 2 * gid + (c >> 1);
          if (head < p.group) store_out(p, ob + (int64_t)head * C::D + d, o[mt][nt][c] * inv[nt][c & 1]);
        }
    return;
  }

  float* sm_o = reinterpret_cast<float*>(smem);  // [NW][GP][D]
  float* sm_m = sm_o + NW * GP * C::D;
  float* sm_l = sm_m + NW * GP;
  float* scratch = sm_l + NW * GP;  // split-K merge: 2 * kMaxSplits * group floats
  float* part = scratch + 2 * kMaxSplits * GP;  // cluster merge: this band's o[G][D], m[G], l[G]
  float* s_e = part + GP * (C::D + 2);          // per-warp weights, merged max and sum
  static_assert((NW * GP * C::D + 2 * NW * GP + 2 * kMaxSplits * GP + GP * (C::D + 2) + NW * GP + 2 * GP) * 4 <=
                    C::STAGES * C::STAGE_BYTES,
                "epilogue buffers must fit in the drained ring");
  if constexpr (UMMA) {
    // one softmax state (the CTA's), as warp state 0 beside three empty ones
    static_assert(kMmaThreads == C::D, "one thread per channel");
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
      for (int n = 0; n < GP; ++n) sm_o[(w * GP + n) * C::D + tid] = w == 0 ? u_o[n] : 0.f;
    if (tid == 0)
#pragma unroll
      for (int n = 0; n < GP; ++n) {
        sm_m[n] = m_ref[n];
        sm_l[n] = u_red[n] + u_red[16 + n] + u_red[32 + n] + u_red[48 + n];
#pragma unroll
        for (int w = 1; w < NW; ++w) {
          sm_m[w * GP + n] = -CUDART_INF_F;
          sm_l[w * GP + n] = 0.f;
        }
      }
    __syncthreads();
    finish_unit_mma<NW>(p, r, h, split, row_ok, sm_m, sm_l, sm_o, GP, scratch, part, s_e);
    return;
  }
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
  finish_unit_mma<NW>(p, r, h, split, row_ok, sm_m, sm_l, sm_o, GP, scratch, part, s_e);
}

template <int KIND, int NT, bool TILES, bool SHALLOW, bool GROUPS = false, bool UMMA = false>
cudaError_t launch_mma_t(const Params& p, cudaStream_t s) {
  using C = MmaCfg<KIND, TILES, SHALLOW, UMMA>;
  static std::atomic<unsigned char> configured[kMaxTrackedDevices] = {};
  const cudaError_t e = ensure_dynamic_smem(configured, mma_kernel<KIND, NT, TILES, SHALLOW, GROUPS, UMMA>, C::SMEM);
  if (e != cudaSuccess) return e;
  const int64_t ctas = (int64_t)p.total_q * p.nkv * p.splits;
  if (ctas == 0) return cudaSuccess;
  if (p.cluster) {
    // the bands of one unit form one cluster (splits <= kMaxClusterSplits)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)p.splits;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mma_kernel<KIND, NT, TILES, SHALLOW, GROUPS, UMMA>, p);
  }
  mma_kernel<KIND, NT, TILES, SHALLOW, GROUPS, UMMA><<<(unsigned)ctas, kMmaThreads, C::SMEM, s>>>(p);
  return cudaGetLastError();
}
template <int KIND, int NT>
cudaError_t launch_mma_nt(const Params& p, cudaStream_t s) {
  if (p.umma) {  // the tcgen05 consumer: BF16, the tile-copy layout (tile copies where p.tma)
    if constexpr (KIND == kBF16) return launch_mma_t<KIND, NT, true, false, false, true>(p, s);
    return cudaErrorInvalidValue;
  }
  if (!p.tma) {
    if constexpr (NT == 2)
      if (p.groups) return launch_mma_t<KIND, NT, false, false, true>(p, s);
    return launch_mma_t<KIND, NT, false, false>(p, s);
  }
  // (groups of up to 8 heads: with two N tiles the registers allow two CTAs anyway)
  if constexpr (KIND == kBF16 && NT == 1)
    if (p.shallow) return launch_mma_t<KIND, NT, true, true>(p, s);
  return launch_mma_t<KIND, NT, true, false>(p, s);
}

// Clusters of `splits` CTAs of the tensor-core kernel that can be resident
// at once on the device (0 when such a cluster cannot be placed).
template <int KIND, int NT, bool TILES, bool UMMA = false>
int mma_max_clusters_nt(int splits) {
  using C = MmaCfg<KIND, TILES, false, UMMA>;
  if (cudaFuncSetAttribute(mma_kernel<KIND, NT, TILES, false, false, UMMA>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)splits);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)splits;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mma_kernel<KIND, NT, TILES, false, false, UMMA>, &cfg) != cudaSuccess) {
    cudaGetLastError();  // a refused query is not a launch error
    return 0;
  }
  return n;
}
template <int KIND>
int mma_max_clusters(int group, int splits, bool tiles, bool umma = false) {
  if constexpr (KIND == kBF16)
    if (umma) return group <= 8 ? mma_max_clusters_nt<KIND, 1, true, true>(splits) : mma_max_clusters_nt<KIND, 2, true, true>(splits);
  if (tiles) return group <= 8 ? mma_max_clusters_nt<KIND, 1, true>(splits) : mma_max_clusters_nt<KIND, 2, true>(splits);
  return group <= 8 ? mma_max_clusters_nt<KIND, 1, false>(splits) : mma_max_clusters_nt<KIND, 2, false>(splits);
}

template <int KIND, int NT, bool TILES, bool UMMA = false>
int mma_occupancy_nt() {
  using C = MmaCfg<KIND, TILES, false, UMMA>;
  int n = 0;
  cudaFuncSetAttribute(mma_kernel<KIND, NT, TILES, false, false, UMMA>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, mma_kernel<KIND, NT, TILES, false, false, UMMA>, kMmaThreads, C::SMEM);
  return n > 0 ? n : 1;
}
template <int KIND>
int mma_occupancy(int group, bool tiles, bool umma = false) {
  if constexpr (KIND == kBF16)
    if (umma) return group <= 8 ? mma_occupancy_nt<KIND, 1, true, true>() : mma_occupancy_nt<KIND, 2, true, true>();
  if (tiles) return group <= 8 ? mma_occupancy_nt<KIND, 1, true>() : mma_occupancy_nt<KIND, 2, true>();
  return group <= 8 ? mma_occupancy_nt<KIND, 1, false>() : mma_occupancy_nt<KIND, 2, false>();
}

}  // namespace qsa
