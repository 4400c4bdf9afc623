// Kernel 4: row groups over page tiles (BF16 caches, head_dim 128, group 4,
// 8 or 16).
//
// The operation is the gather-GQA attention of the QSASparseAttentionRaggedPaged
// page ("Gather-GQA over the token indices a QSA selection names"): for each
// query row, kv head and query head of its group, softmax(scale q.K_sel) V_sel
// over exactly the positions the row lists.  Rows of one prefill sequence list
// heavily overlapping positions, so this kernel serves R = 128 / group
// consecutive rows of a sequence together: their R x group query heads of one
// kv head are the 128 rows of a tensor-core tile, and the kernel walks the
// sequence's positions in tiles of 128 (whole pages, loaded once by TMA),
// skipping tiles no row of the group selects.  Scores of keys a row did not
// list are masked out before the softmax, so every row still attends exactly
// its own positions:
//
//   S = Q . K^T    (M = 128 query heads x rows, N = 128 keys, K = 128 channels)
//   P = 2^(scale log2(e) S - m) on the row's own keys, 0 elsewhere
//   O += P . V     (M = 128, N = 128 channels, K = 128 keys)
//
// Both contractions run on the fifth-generation tensor cores (tcgen05): Q and
// the K/V tiles in 128-byte-swizzled shared memory, S, P and O in tensor
// memory.  A first kernel turns each row's list into a bitmap over its
// sequence's positions (dropping and flagging positions that cannot be read,
// as every kernel of the library does) and flags rows that repeat a position:
// a repeated index is its own softmax term, which a bitmap cannot count, so a
// group with such a row takes an exact CUDA-core path instead.
//
// CTA = (group of rows, kv head); 6 warps:
//   warp 0      producer: the group's mask words of each tile from the bitmaps,
//               empty tiles skipped, page-table lookups, TMA tile copies of K
//               and V (page 0 stands in for pages past the sequence or named
//               by no page: none of their keys is selected), three stages
//   warp 1      one thread issues the MMAs: S(i) = Q.K(i)^T, then O += P(i-1).V(i-1)
//   warps 2..5  softmax of the 128 accumulator rows (one thread per row), with
//               a lazy running maximum: O is rescaled only when a row's maximum
//               grows by more than 2^8; they also zero the V rows of keys no
//               row of the group selects (so 0 x non-finite never reaches O)
//               and write the output.
// Tensor memory: S double-buffered (2 x 128 columns), O (128), P
// double-buffered (2 x 64 columns of packed bf16 pairs) = 512 columns.
#include "qsa_mma.cuh"

namespace qsa {
namespace {

constexpr int kRgThreads = 192;
constexpr int kRgStages = 3;
constexpr uint32_t kRgHalf = 16384;           // 64 channels (128 B) x 128 rows, 128-byte swizzle
constexpr uint32_t kRgTileBytes = 2 * kRgHalf;  // Q, or one K or V tile
constexpr uint32_t kRgStageBytes = 2 * kRgTileBytes;
constexpr uint32_t kRgStageOff = kRgTileBytes;  // after Q

struct TileHdr {
  int32_t pos0;          // first position of the tile
  int32_t end;           // 1: the unit has no more tiles
  int32_t pad[2];
  uint32_t any[4];       // keys some row of the group selects
  uint32_t mask[32][4];  // per row of the group: the keys it selects
};
constexpr uint32_t kRgHdrOff = kRgStageOff + kRgStages * kRgStageBytes;
constexpr uint32_t kRgBarOff = kRgHdrOff + kRgStages * (uint32_t)sizeof(TileHdr);
// barriers: full[3], done[3], s_full[2], p_full[2], q_full -> 11 x 8 B, then misc words
constexpr int kBarFull = 0, kBarDone = 3, kBarS = 6, kBarP = 8, kBarQ = 10;
constexpr uint32_t kRgMiscOff = kRgBarOff + 128;
constexpr uint32_t kRgSmemBytes = kRgMiscOff + 32 * 4;
constexpr uint32_t kRgSmemAlloc = kRgSmemBytes + 1024;  // the 1024-byte alignment of the swizzled tiles
static_assert(kRgSmemAlloc <= 232448, "kernel 4's shared memory exceeds the per-CTA limit");
static_assert(sizeof(TileHdr) % 16 == 0, "tile headers must stay 16-byte aligned");

// TMEM columns
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;

// S = Q.K^T: A (Q) and B (K) K-major; O = P.V: A (P) in tensor memory, B (V) MN-major.
constexpr uint32_t kIdescQK = instr_desc(128, 128, 1, 0, 0);
constexpr uint32_t kIdescPV = instr_desc(128, 128, 1, 0, 1);

struct GroupInfo {
  int b, row0, nrows;
  int64_t kv_len;
};

// Block-wide (every thread calls it): group gi of the call, where the rows of
// sequence b form ceil(rows_b / R) groups of R consecutive rows, sequence by
// sequence.  b < 0 when gi is past the last group.  `scratch` holds at least
// blockDim.x / 32 + 2 words of shared memory.
__device__ GroupInfo group_info(const Params& p, int gi, int R, int* scratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int* found = scratch + nw;
  if (threadIdx.x == 0) found[0] = -1;
  __syncthreads();
  int base = 0;
  for (int c0 = 0; c0 < p.batch; c0 += blockDim.x) {
    const int b = c0 + (int)threadIdx.x;
    int ng = 0;
    if (b < p.batch) {
      const uint32_t o0 = __ldg(p.row_offsets + b), o1 = __ldg(p.row_offsets + b + 1);
      ng = o1 > o0 ? (int)((o1 - o0 + (uint32_t)R - 1) / (uint32_t)R) : 0;
    }
    int x = ng;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < nw; ++w) {
      const int t = scratch[w];
      if (w < warp) before += t;
      total += t;
    }
    const int incl = base + before + x;
    if (ng > 0 && incl - ng <= gi && gi < incl) {
      found[0] = b;
      found[1] = gi - (incl - ng);
    }
    base += total;
    __syncthreads();
  }
  GroupInfo g;
  g.b = found[0];
  g.row0 = g.nrows = 0;
  g.kv_len = 0;
  if (g.b >= 0) {
    const uint32_t o0 = __ldg(p.row_offsets + g.b), o1 = __ldg(p.row_offsets + g.b + 1);
    g.row0 = (int)o0 + found[1] * R;
    g.nrows = min(R, (int)o1 - g.row0);
    g.kv_len = (int64_t)__ldg(p.cache_lengths + g.b) + (int64_t)(o1 - o0);
  }
  __syncthreads();  // `found` is reused by the caller
  return g;
}

// One CTA per query row: the bitmap of the row's readable selected positions
// over its sequence's kv_len positions, and the row's flags.  Rows owned by no
// sequence get a zero output row and QSA_STATUS_BAD_ROW, as in every kernel.
__global__ void __launch_bounds__(256) rg_bitmap_kernel(const Params p) {
  extern __shared__ uint32_t bm[];
  const int r = blockIdx.x;
  const RowInfo ri = row_info(p, r);
  if (!ri.ok) {
    const int64_t n = (int64_t)p.nq * p.D, o = (int64_t)r * n;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) store_out(p, o + i, 0.f);
    if (threadIdx.x == 0) {
      atomicOr(p.status, QSA_STATUS_BAD_ROW);
      p.rg_flags[r] = 0;
    }
    return;
  }
  if (ri.kv_len > (int64_t)p.rg_capw * 32) {
    if (threadIdx.x == 0) p.rg_flags[r] = kRgOverflow;
    return;
  }
  const int words = (int)((ri.kv_len + 31) >> 5);
  for (int w = threadIdx.x; w < words; w += blockDim.x) bm[w] = 0u;
  __syncthreads();
  uint32_t bad = 0;
  int dup = 0;
  const int32_t* idx = p.indices + (int64_t)r * p.W;
  for (int j = threadIdx.x; j < ri.n; j += blockDim.x) {
    const int32_t pos = __ldg(idx + j);
    if (logical_page(p, ri.kv_len, pos, bad) < 0) continue;
    const uint32_t bit = 1u << (pos & 31);
    if (atomicOr(&bm[pos >> 5], bit) & bit) dup = 1;
  }
  dup = __syncthreads_or(dup);
  uint32_t* out = p.rg_bits + (int64_t)r * p.rg_capw;
  for (int w = threadIdx.x; w < words; w += blockDim.x) out[w] = bm[w];
  if (bad) atomicOr(p.status, bad);
  if (threadIdx.x == 0) p.rg_flags[r] = dup ? kRgDup : 0;
}

// The exact path of a group with a flagged row: warp w serves rows w, w + 6,
// ... of the group, its `group` query heads on kv head h, walking the row's
// list in order (repeats included) with an online softmax per head; lane l
// holds channels 4l .. 4l + 3.
__device__ void rg_exact(const Params& p, const GroupInfo& gr, int h) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int G = p.group;
  for (int rl = warp; rl < gr.nrows; rl += nw) {
    const int r = gr.row0 + rl;
    const int n = min(max(__ldg(p.counts + r), 0), p.W);
    float qv[16][4], acc[16][4], m[16], l[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      m[i] = -CUDART_INF_F;
      l[i] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) qv[i][c] = acc[i][c] = 0.f;
      if (i < G) {
        const __nv_bfloat16* qp =
            reinterpret_cast<const __nv_bfloat16*>(p.q) + ((int64_t)r * p.nq + (int64_t)h * G + i) * 128 + 4 * lane;
#pragma unroll
        for (int c = 0; c < 4; ++c) qv[i][c] = __bfloat162float(qp[c]);
      }
    }
    uint32_t bad = 0;
    const int32_t* idx = p.indices + (int64_t)r * p.W;
    for (int j = 0; j < n; ++j) {
      const int32_t pos = __ldg(idx + j);
      const int64_t lp = logical_page(p, gr.kv_len, pos, bad);
      if (lp < 0) continue;
      const uint32_t page = __ldg(p.table + (int64_t)gr.b * p.max_pages + lp);
      const uint32_t off16 = k_row_offset16(p, page, pos, h, bad);
      if (off16 == kInvalidOff) continue;
      const unsigned char* kp = p.kv + (int64_t)off16 * 16 + 8 * lane;
      const uint2 kr = *reinterpret_cast<const uint2*>(kp);
      const uint2 vr = *reinterpret_cast<const uint2*>(kp + p.v_minus_k_bytes);
      float kf[4], vf[4];
      {
        const __nv_bfloat162 k01 = *reinterpret_cast<const __nv_bfloat162*>(&kr.x);
        const __nv_bfloat162 k23 = *reinterpret_cast<const __nv_bfloat162*>(&kr.y);
        const __nv_bfloat162 v01 = *reinterpret_cast<const __nv_bfloat162*>(&vr.x);
        const __nv_bfloat162 v23 = *reinterpret_cast<const __nv_bfloat162*>(&vr.y);
        kf[0] = __low2float(k01); kf[1] = __high2float(k01); kf[2] = __low2float(k23); kf[3] = __high2float(k23);
        vf[0] = __low2float(v01); vf[1] = __high2float(v01); vf[2] = __low2float(v23); vf[3] = __high2float(v23);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i >= G) break;
        float d = qv[i][0] * kf[0] + qv[i][1] * kf[1] + qv[i][2] * kf[2] + qv[i][3] * kf[3];
#pragma unroll
        for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        const float s = d * p.scale_log2;
        const float mn = fmaxf(m[i], s);
        const float a = m[i] == -CUDART_INF_F ? 0.f : exp2f(m[i] - mn);
        const float e = exp2f(s - mn);
        l[i] = l[i] * a + e;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = acc[i][c] * a + e * vf[c];
        m[i] = mn;
      }
    }
    if (bad && lane == 0) atomicOr(p.status, bad);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i >= G) break;
      const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
      const int64_t o = ((int64_t)r * p.nq + (int64_t)h * G + i) * 128 + 4 * lane;
#pragma unroll
      for (int c = 0; c < 4; ++c) store_out(p, o + c, acc[i][c] * inv);
    }
  }
}

// A wait whose outcome every lane of the warp shares: when any lane gives up,
// all do, so no lane is left alone at a later warp-wide vote or tcgen05 access.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 x = __floats2bfloat162_rn(a, b);  // low half: a
  return *reinterpret_cast<const uint32_t*>(&x);
}

__global__ void __launch_bounds__(kRgThreads, 1) rg_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.rg_rows, G = p.group;
  const int h = (int)(blockIdx.x % (uint32_t)p.nkv), gi = (int)(blockIdx.x / (uint32_t)p.nkv);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRgBarOff);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kRgMiscOff);  // [0] tmem base, [8..] scratch
  TileHdr* hdr = reinterpret_cast<TileHdr*>(smem + kRgHdrOff);
  const uint32_t sQ = smem_addr(smem), sStage = sQ + kRgStageOff;
  auto bar = [&](int k) { return smem_addr(&bars[k]); };

  const GroupInfo gr = group_info(p, gi, R, reinterpret_cast<int*>(misc + 8));
  if (gr.b < 0) return;  // past the call's groups (the grid is sized for the most there can be)
  int flagged = 0;
  for (int i = tid; i < gr.nrows; i += blockDim.x) flagged |= __ldg(p.rg_flags + gr.row0 + i);
  if (__syncthreads_or(flagged)) {
    rg_exact(p, gr, h);
    return;
  }

  if (tid == 0) {
    for (int k = 0; k < 3; ++k) {
      mbar_init(bar(kBarFull + k), 1);
      mbar_init(bar(kBarDone + k), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(kBarS + k), 1);
      mbar_init(bar(kBarP + k), 128);
    }
    mbar_init(bar(kBarQ), 128);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(misc), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = misc[0];
  volatile uint32_t* abort_flag = misc + 1;
  if (tid == 0) *abort_flag = 0;
  __syncthreads();
  auto give_up = [&]() {
    *abort_flag = 1;
    atomicOr(p.status, QSA_STATUS_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    const int NT = (int)((gr.kv_len + 127) >> 7);
    const int words_valid = (int)((gr.kv_len + 31) >> 5);  // bitmap words the first kernel wrote
    const int nw = R * 4;
    const uint32_t* bits = p.rg_bits + (int64_t)gr.row0 * p.rg_capw;
    const int BR = p.rg_box;  // slots per copy: min(P, 128)
    const int np = 128 / BR;  // copies per line of a tile
    auto load_words = [&](int t, uint32_t (&wv)[4]) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int w = lane + 32 * k, row = w >> 2, wi = t * 4 + (w & 3);
        wv[k] = 0u;
        if (w < nw && row < gr.nrows && wi < words_valid) wv[k] = __ldg(bits + (int64_t)row * p.rg_capw + wi);
      }
    };
    uint32_t nxt[4] = {0u, 0u, 0u, 0u};
    if (NT > 0) load_words(0, nxt);
    int i = 0;
    bool ok = true;
    for (int t = 0; t < NT && ok; ++t) {
      uint32_t cur[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) cur[k] = nxt[k];
      if (t + 1 < NT) load_words(t + 1, nxt);
      if (!__any_sync(0xffffffffu, (cur[0] | cur[1] | cur[2] | cur[3]) != 0u)) continue;
      const int s = i % kRgStages;
      if (i >= kRgStages && !warp_wait(bar(kBarDone + s), (uint32_t)((i / kRgStages - 1) & 1))) {
        ok = false;
        break;
      }
      // the physical page of each copy.  A copy past the sequence, or whose
      // table entry names no page, reads page 0 instead: none of its keys is
      // selected (the first kernel dropped positions past the sequence, bits
      // on a bad page are cleared below), so its scores are masked and its V
      // rows zeroed before use.
      const int64_t pos0 = (int64_t)t * 128;
      int phys = 0;
      bool badpage = false;
      if (lane < np) {
        const int64_t lp = pos0 / p.P + (BR < 128 ? lane : 0);
        if (lp < p.max_pages && lp * p.P < gr.kv_len) {
          const uint32_t e = __ldg(p.table + (int64_t)gr.b * p.max_pages + lp);
          if (e < p.num_pages)
            phys = (int)e;
          else
            badpage = true;
        }
      }
      const uint32_t badm = __ballot_sync(0xffffffffu, badpage);
      if (badm) {
        // selected keys on a page the table does not name: dropped and flagged
        const int part = lane & 3;
        uint32_t kill = 0u;
        for (int k = 0; k < np; ++k) {
          if (!((badm >> k) & 1u)) continue;
          const int k0 = BR < 128 ? k * BR : 0, k1 = BR < 128 ? k0 + BR : 128;
          const int a = max(k0, part * 32), e = min(k1, part * 32 + 32);
          if (a < e) kill |= (e - a == 32 ? 0xFFFFFFFFu : ((1u << (e - a)) - 1u)) << (a - part * 32);
        }
        bool had = false;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          had |= (cur[k] & kill) != 0u;
          cur[k] &= ~kill;
        }
        if (__any_sync(0xffffffffu, had) && lane == 0) atomicOr(p.status, QSA_STATUS_BAD_PAGE);
      }
      TileHdr& th = hdr[s];
      uint32_t any = 0u;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int w = lane + 32 * k;
        if (w < nw) th.mask[w >> 2][w & 3] = cur[k];
        any |= cur[k];
      }
      any |= __shfl_xor_sync(0xffffffffu, any, 4);
      any |= __shfl_xor_sync(0xffffffffu, any, 8);
      any |= __shfl_xor_sync(0xffffffffu, any, 16);
      if (lane < 4) th.any[lane] = any;
      if (lane == 0) {
        th.pos0 = (int32_t)pos0;
        th.end = 0;
      }
      __syncwarp();
      const uint32_t fb = bar(kBarFull + s);
      if (lane == 0) {
        tile_fence_proxy_async();
        mbar_arrive_expect_tx(fb, 2 * kRgTileBytes);
      }
      __syncwarp();
      if (lane < np) {
        const uint32_t dst = sStage + (uint32_t)s * kRgStageBytes + (uint32_t)(BR < 128 ? lane * BR * 128 : 0);
        const int slot = BR < 128 ? 0 : (int)(pos0 % p.P);
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
          for (int x = 0; x < 2; ++x)
            tma_load_5d(dst + kv * kRgTileBytes + x * kRgHalf, &p.tmap, 0, h * 2 + x, slot,
                        kv ? p.tma_plane_v : p.tma_plane_k, phys, fb);
      }
      ++i;
    }
    if (ok) {
      // end of the unit
      const int s = i % kRgStages;
      if (i >= kRgStages && !warp_wait(bar(kBarDone + s), (uint32_t)((i / kRgStages - 1) & 1))) ok = false;
      if (ok && lane == 0) {
        hdr[s].end = 1;
        mbar_arrive(bar(kBarFull + s));
      }
    }
    if (!ok) {
      if (lane == 0) give_up();
      // copies in flight land before the CTA leaves
      for (int j = max(0, i - kRgStages); j < i; ++j)
        if (!warp_wait(bar(kBarFull + j % kRgStages), (uint32_t)((j / kRgStages) & 1))) break;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      uint32_t last_bar = 0, last_phase = 0;
      bool ok = mbar_wait(bar(kBarQ), 0);
      int i = 0;
      auto pv = [&](int j) -> bool {
        if (!mbar_wait(bar(kBarP + (j & 1)), (uint32_t)((j >> 1) & 1))) return false;
        tc_fence_after();
        const uint32_t vbase = sStage + (uint32_t)(j % kRgStages) * kRgStageBytes + kRgTileBytes;
        const uint32_t pcol = tm + kColP + (uint32_t)(j & 1) * 64;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_f16_ts(tm + kColO, pcol + ks * 8, smem_desc(vbase + ks * 2048, kRgHalf, 1024, kSwizzle128), kIdescPV,
                      j > 0 || ks > 0);
        umma_commit(bar(kBarDone + j % kRgStages));
        last_bar = bar(kBarDone + j % kRgStages);
        last_phase = (uint32_t)((j / kRgStages) & 1);
        return true;
      };
      while (ok) {
        const int s = i % kRgStages;
        if (!mbar_wait(bar(kBarFull + s), (uint32_t)((i / kRgStages) & 1))) {
          ok = false;
          break;
        }
        if (*reinterpret_cast<volatile int32_t*>(&hdr[s].end)) break;
        tc_fence_after();
        const uint32_t kbase = sStage + (uint32_t)s * kRgStageBytes;
        const uint32_t sc = tm + kColS + (uint32_t)(i & 1) * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (uint32_t)(ks >> 2) * kRgHalf + (uint32_t)(ks & 3) * 32;
          umma_f16(sc, smem_desc(sQ + off, 16, 1024, kSwizzle128), smem_desc(kbase + off, 16, 1024, kSwizzle128),
                   kIdescQK, ks > 0);
        }
        umma_commit(bar(kBarS + (i & 1)));
        last_bar = bar(kBarS + (i & 1));
        last_phase = (uint32_t)((i >> 1) & 1);
        if (i > 0 && !pv(i - 1)) {
          ok = false;
          break;
        }
        ++i;
      }
      if (ok && i > 0) ok = pv(i - 1);
      if (!ok) {
        give_up();
        if (last_bar) mbar_wait(last_bar, last_phase);  // the tensor cores finish what was issued
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;  // accumulator row = TMEM lane
    const int rl = m / G, hq = m % G;   // row of the group, query head of kv head h
    const bool live = rl < gr.nrows;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    {
      // this row of Q, 128-byte-swizzled K-major (zeros past the group's rows)
      const uint4* src =
          live ? reinterpret_cast<const uint4*>(p.q + ((int64_t)(gr.row0 + rl) * p.nq + (int64_t)h * G + hq) * 256)
               : nullptr;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (live) v = __ldg(src + c);
        const uint32_t dst = sQ + (uint32_t)(c >> 3) * kRgHalf + (uint32_t)m * 128 + ((uint32_t)((c & 7) ^ (m & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kBarQ));
    }
    float m_ref = -CUDART_INF_F, l = 0.f;
    int i = 0;
    bool ok = true;
    for (;;) {
      const int s = i % kRgStages;
      if (!warp_wait(bar(kBarFull + s), (uint32_t)((i / kRgStages) & 1))) {
        ok = false;
        break;
      }
      if (*reinterpret_cast<volatile int32_t*>(&hdr[s].end)) break;
      if (!warp_wait(bar(kBarS + (i & 1)), (uint32_t)((i >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[128];
      const uint32_t sc = tm + lane_off + kColS + (uint32_t)(i & 1) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(sc + c * 32, x + c * 32);
      const uint4 mk = *reinterpret_cast<const uint4*>(&hdr[s].mask[rl < R ? rl : 0][0]);
      const uint32_t mw[4] = {mk.x, mk.y, mk.z, mk.w};
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float v = ((mw[c] >> j) & 1u) ? x[c * 32 + j] * p.scale_log2 : -CUDART_INF_F;
          x[c * 32 + j] = v;
          mx = fmaxf(mx, v);
        }
      // lazy running maximum: move it only when this tile's maximum exceeds it by 2^8
      const bool need = mx > m_ref + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float mnew = need ? mx : m_ref;
        const float f = need ? (m_ref == -CUDART_INF_F ? 0.f : exp2_fast(m_ref - mnew)) : 1.f;
        if (i > 0 && __any_sync(0xffffffffu, need && l > 0.f)) {
          // O holds every earlier tile once the previous P.V is done
          if (!warp_wait(bar(kBarDone + (i - 1) % kRgStages), (uint32_t)(((i - 1) / kRgStages) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t oc = tm + lane_off + kColO;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float o[32];
            uint32_t w[32];
            tmem_ld32(oc + c * 32, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(o[j] * f);
            tmem_st32(oc + c * 32, w);
          }
          tmem_wait_st();
        }
        l *= f;
        m_ref = mnew;
      }
      const float mr = m_ref == -CUDART_INF_F ? 0.f : m_ref;
      uint32_t pk[64];
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float p0 = exp2_fast(x[2 * j] - mr), p1 = exp2_fast(x[2 * j + 1] - mr);
        sum += p0 + p1;
        pk[j] = pack_bf16(p0, p1);
      }
      l += sum;
      // P(i) goes where P(i - 2) was: that P.V must be done
      if (i >= 2 && !warp_wait(bar(kBarDone + (i - 2) % kRgStages), (uint32_t)(((i - 2) / kRgStages) & 1))) {
        ok = false;
        break;
      }
      const uint32_t pc = tm + lane_off + kColP + (uint32_t)(i & 1) * 64;
      tmem_st32(pc, pk);
      tmem_st32(pc + 32, pk + 32);
      tmem_wait_st();
      // V rows of keys no row of the group selects (other positions, slots past
      // the sequence) are zeroed, so 0 x non-finite never reaches O
      if (!((hdr[s].any[m >> 5] >> (m & 31)) & 1u)) {
        const uint32_t vrow = sStage + (uint32_t)s * kRgStageBytes + kRgTileBytes + (uint32_t)m * 128;
#pragma unroll
        for (int x2 = 0; x2 < 2; ++x2)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};\n" ::"r"(vrow + x2 * kRgHalf + c * 16), "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarP + (i & 1)));
      ++i;
    }
    // epilogue: O / l for this row (tiles i; zero when the row attended nothing)
    bool have = i > 0 && ok;
    if (have && !warp_wait(bar(kBarDone + (i - 1) % kRgStages), (uint32_t)(((i - 1) / kRgStages) & 1))) {
      ok = false;
      have = false;
    }
    if (!ok && lane == 0) give_up();
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int64_t orow = ((int64_t)(gr.row0 + rl) * p.nq + (int64_t)h * G + hq) * 128;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float o[32];
      if (__any_sync(0xffffffffu, have)) tmem_ld32(tm + lane_off + kColO + c * 32, o);
      if (!live) continue;
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = have ? o[j] * inv : 0.f;
      if (p.out_bf16) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + orow + c * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_uint4(pack_bf16(o[8 * k], o[8 * k + 1]), pack_bf16(o[8 * k + 2], o[8 * k + 3]),
                              pack_bf16(o[8 * k + 4], o[8 * k + 5]), pack_bf16(o[8 * k + 6], o[8 * k + 7]));
      } else {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow + c * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

std::atomic<unsigned char> g_rg_smem_set[kMaxTrackedDevices];
std::atomic<unsigned char> g_rg_bitmap_smem_set[kMaxTrackedDevices];

}  // namespace

cudaError_t launch_rowgroup(const Params& p, cudaStream_t stream) {
  if (p.total_q <= 0) return cudaSuccess;
  cudaError_t e = ensure_dynamic_smem(g_rg_bitmap_smem_set, rg_bitmap_kernel, kRgMaxCapWords * 4);
  if (e != cudaSuccess) return e;
  e = ensure_dynamic_smem(g_rg_smem_set, rg_kernel, (int)kRgSmemAlloc);
  if (e != cudaSuccess) return e;
  rg_bitmap_kernel<<<p.total_q, 256, (size_t)p.rg_capw * 4, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t ctas = (int64_t)p.rg_groups * p.nkv;
  if (ctas <= 0) return cudaSuccess;
  rg_kernel<<<(unsigned)ctas, kRgThreads, kRgSmemAlloc, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qsa
