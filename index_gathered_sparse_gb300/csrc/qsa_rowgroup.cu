// Kernel 4: row groups over page tiles (BF16 caches, head_dim 128, group 4,
// 8 or 16).
//
// The operation is the gather-GQA attention of the QSASparseAttentionRaggedPaged
// page ("Gather-GQA over the token indices a QSA selection names"): for each
// query row, kv head and query head of its group, softmax(scale q.K_sel) V_sel
// over exactly the positions the row lists.  Rows of one prefill sequence list
// heavily overlapping positions, so this kernel serves R = 256 / group
// consecutive rows of a sequence together: their R x group query heads of one
// kv head are the rows of two 128-row tensor-core tiles, and the kernel walks
// the sequence's positions in tiles of 128 keys (whole pages, loaded once by
// TMA for both), skipping tiles no row of the group selects.  Scores of keys
// a row did not list are masked out before the softmax, so every row still
// attends exactly its own positions:
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
// CTA = (group of rows, kv head): R = 256 / group rows, whose 256 query
// heads form two 128-row accumulator tiles A (the first R / 2 rows) and B
// sharing every K/V tile.  11 warps:
//   warp 0      producer: the group's mask words of each tile from the bitmaps,
//               empty tiles skipped, page-table lookups, TMA tile copies of K
//               and V (page 0 stands in for pages past the sequence or named
//               by no page: none of their keys is selected), two stages with
//               separate K and V arrivals
//   warp 10     once a tile's V has landed, zeroes the V rows of keys no row
//               of the group selects (so a non-finite value there cannot
//               reach O as 0 x value) before P.V may read them; a non-finite
//               V at a key another row of the group selects still reaches the
//               rows that did not select it, as 0 x value
//   warp 1      one thread issues the MMAs in the order
//               QK_A(i) QK_B(i) PV_A(i) QK_A(i+1) PV_B(i) QK_B(i+1) ...,
//               so each softmax warpgroup works while the tensor cores serve
//               the other tile
//   warps 2..5  softmax of tile A (one thread per accumulator row), warps
//   6..9        of tile B: a lazy running maximum (O is rescaled only when a
//               row's maximum grows by more than 2^8), one read of S per
//               tile (the second 64 columns load while the first are
//               processed), P written back over the scores it replaces
//               (keys 2j, 2j + 1 in column j), and the output.
// Tensor memory: S_A, S_B (128 columns each, P_A / P_B in their first 64
// columns as packed bf16 pairs), O_A, O_B (128 each) = 512 columns.  P_X(i)
// overwrites S_X(i) after it is read, and QK_X(i+1) overwrites P_X(i) only
// after PV_X(i), issued before it by the same thread (tensor-core operations
// of one thread execute in issue order).
#include "qsa_mma.cuh"

namespace qsa {
namespace {

constexpr int kRgThreads = 352;
constexpr int kRgStages = 2;
constexpr uint32_t kRgHalf = 16384;           // 64 channels (128 B) x 128 rows, 128-byte swizzle
constexpr uint32_t kRgTileBytes = 2 * kRgHalf;  // a Q tile, or one K or V tile
constexpr uint32_t kRgStageBytes = 2 * kRgTileBytes;
constexpr uint32_t kRgStageOff = 2 * kRgTileBytes;  // after Q_A, Q_B

struct TileHdr {
  int32_t pos0;          // first position of the tile
  int32_t end;           // 1: the unit has no more tiles
  int32_t pad[2];
  uint32_t any[4];       // keys some row of the group selects
  uint32_t mask[64][4];  // per row of the group (at most 64): the keys it selects
};
constexpr uint32_t kRgHdrOff = kRgStageOff + kRgStages * kRgStageBytes;
constexpr uint32_t kRgBarOff = kRgHdrOff + kRgStages * (uint32_t)sizeof(TileHdr);
// barriers: full_k[2], full_v[2], kv_free[2], s_full[2], p_full[2], o_done[2], q_full, v_ready[2] -> 15 x 8 B
constexpr int kBarK = 0, kBarV = 2, kBarFree = 4, kBarS = 6, kBarP = 8, kBarO = 10, kBarQ = 12, kBarVR = 13;
constexpr uint32_t kRgMiscOff = kRgBarOff + 128;
constexpr uint32_t kRgSmemBytes = kRgMiscOff + 32 * 4;
constexpr uint32_t kRgSmemAlloc = kRgSmemBytes + 1024;  // the 1024-byte alignment of the swizzled tiles
static_assert(kRgSmemAlloc <= 232448, "kernel 4's shared memory exceeds the per-CTA limit");
static_assert(sizeof(TileHdr) % 16 == 0, "tile headers must stay 16-byte aligned");

// TMEM columns of tile X (0 = A, 1 = B)
constexpr uint32_t kColS = 0, kColO = 256;

// S = Q.K^T: A (Q) and B (K) K-major; O = P.V: A (P) in tensor memory, B (V) MN-major.
constexpr uint32_t kIdescQK = instr_desc(128, 128, 1, 0, 0);
constexpr uint32_t kIdescPV = instr_desc(128, 128, 1, 0, 1);

struct GroupInfo {
  int b, row0, nrows;
  int64_t kv_len;
};

// Block-wide (every thread calls it): group gi of the call, where the rows of
// sequence b form ceil(rows_b / R) groups of R consecutive rows.  Sequences
// are numbered longest first (when batch <= blockDim.x; in sequence order
// otherwise), so the CTAs with the most tiles start in the first waves and the
// last wave holds short ones.  b < 0 when gi is past the last group.
// `scratch` holds at least blockDim.x / 32 + 2 words of shared memory, `big`
// 12 blockDim.x bytes (8-byte aligned).
__device__ GroupInfo group_info(const Params& p, int gi, int R, int* scratch, unsigned char* big) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int* found = scratch + nw;
  if (threadIdx.x == 0) found[0] = -1;
  const bool longest_first = p.batch <= (int)blockDim.x;
  int* ord = reinterpret_cast<int*>(big + 8 * blockDim.x);
  if (longest_first) {
    uint64_t* len = reinterpret_cast<uint64_t*>(big);
    const int b = threadIdx.x;
    uint64_t mine = 0;
    if (b < p.batch) {
      const uint32_t o0 = __ldg(p.row_offsets + b), o1 = __ldg(p.row_offsets + b + 1);
      mine = (uint64_t)__ldg(p.cache_lengths + b) + (o1 > o0 ? (uint64_t)(o1 - o0) : 0u);
      len[b] = mine;
    }
    __syncthreads();
    if (b < p.batch) {
      int rank = 0;  // sequences longer than b, or as long and earlier
      for (int k = 0; k < p.batch; ++k) {
        const uint64_t v = len[k];
        rank += (v > mine || (v == mine && k < b)) ? 1 : 0;
      }
      ord[rank] = b;
    }
  }
  __syncthreads();
  int base = 0;
  for (int c0 = 0; c0 < p.batch; c0 += blockDim.x) {
    const int t = c0 + (int)threadIdx.x;
    const int b = t < p.batch ? (longest_first ? ord[t] : t) : p.batch;
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
  // each thread a contiguous chunk of the list: bits of consecutive entries
  // in one word are gathered in a register and set with one atomic (lists
  // are usually sorted, with runs of adjacent positions); a bit already set,
  // locally or in the bitmap, is a repeated position
  const int chunk = (ri.n + (int)blockDim.x - 1) / (int)blockDim.x;
  const int j0 = (int)threadIdx.x * chunk, j1 = min(ri.n, j0 + chunk);
  int word = -1;
  uint32_t acc = 0u;
  for (int j = j0; j < j1; ++j) {
    const int32_t pos = __ldg(idx + j);
    if (logical_page(p, ri.kv_len, pos, bad) < 0) continue;
    const uint32_t bit = 1u << (pos & 31);
    if ((pos >> 5) != word) {
      if (word >= 0 && (atomicOr(&bm[word], acc) & acc)) dup = 1;
      word = pos >> 5;
      acc = 0u;
    }
    if (acc & bit) dup = 1;
    acc |= bit;
  }
  if (word >= 0 && (atomicOr(&bm[word], acc) & acc)) dup = 1;
  dup = __syncthreads_or(dup);
  uint32_t* out = p.rg_bits + (int64_t)r * p.rg_capw;
  for (int w = threadIdx.x; w < words; w += blockDim.x) out[w] = bm[w];
  if (bad) atomicOr(p.status, bad);
  if (threadIdx.x == 0) p.rg_flags[r] = dup ? kRgDup : 0;
}

// The exact path of a group with a flagged row: the warps take (row, up to 8
// query heads on kv head h) items in turn, walking the row's list in order
// (repeats included) with an online softmax per head; lane l holds channels
// 4l .. 4l + 3.
__device__ void rg_exact(const Params& p, const GroupInfo& gr, int h) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int G = p.group;
  // (row, chunk of up to 8 query heads) items, one per warp at a time
  const int chunks = (G + 7) / 8;
  for (int item = warp; item < gr.nrows * chunks; item += nw) {
    const int rl = item / chunks, h0 = (item % chunks) * 8, hn = min(8, G - h0);
    const int r = gr.row0 + rl;
    const int n = min(max(__ldg(p.counts + r), 0), p.W);
    float qv[8][4], acc[8][4], m[8], l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      m[i] = -CUDART_INF_F;
      l[i] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) qv[i][c] = acc[i][c] = 0.f;
      if (i < hn) {
        const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                  ((int64_t)r * p.nq + (int64_t)h * G + h0 + i) * 128 + 4 * lane;
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
      for (int i = 0; i < 8; ++i) {
        if (i >= hn) break;
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
    for (int i = 0; i < 8; ++i) {
      if (i >= hn) break;
      const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
      const int64_t o = ((int64_t)r * p.nq + (int64_t)h * G + h0 + i) * 128 + 4 * lane;
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

// 32 lanes x 64 columns of 32 bits, issued without its wait: the words are
// the tile's only after tmem_wait_ld64 on the same array, whose operands tie
// every later use of them to the wait
__device__ __forceinline__ void tmem_ld64_issue(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld64(uint32_t (&r)[64]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63]) : : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 x = __floats2bfloat162_rn(a, b);  // low half: a
  return *reinterpret_cast<const uint32_t*>(&x);
}

// 352 threads, one CTA per SM (its shared memory).  Eleven warps put three on
// three of the SM's four sub-partitions, whose register files hold 16 Ki
// registers each: at most 168 registers a thread.
__global__ void __launch_bounds__(kRgThreads, 1) rg_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.rg_rows, G = p.group;
  const int h = (int)(blockIdx.x % (uint32_t)p.nkv), gi = (int)(blockIdx.x / (uint32_t)p.nkv);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRgBarOff);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kRgMiscOff);  // [0] tmem base, [1] abort, [8..] scratch
  TileHdr* hdr = reinterpret_cast<TileHdr*>(smem + kRgHdrOff);
  const uint32_t sQ = smem_addr(smem), sStage = sQ + kRgStageOff;
  auto bar = [&](int k) { return smem_addr(&bars[k]); };

  // (the K/V stages are free scratch until the group is known)
  const GroupInfo gr = group_info(p, gi, R, reinterpret_cast<int*>(misc + 8), smem + kRgStageOff);
  if (gr.b < 0) return;  // past the call's groups (the grid is sized for the most there can be)
  int flagged = 0;
  for (int i = tid; i < gr.nrows; i += blockDim.x) flagged |= __ldg(p.rg_flags + gr.row0 + i);
  if (__syncthreads_or(flagged)) {
    rg_exact(p, gr, h);
    return;
  }

  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(kBarK + k), 1);
      mbar_init(bar(kBarV + k), 1);
      mbar_init(bar(kBarFree + k), 1);
      mbar_init(bar(kBarS + k), 1);
      mbar_init(bar(kBarP + k), 128);
      mbar_init(bar(kBarO + k), 1);
      mbar_init(bar(kBarVR + k), 1);
    }
    mbar_init(bar(kBarQ), 256);
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
    const int nw = R * 4;                                    // mask words of a tile (at most 256)
    const uint32_t* bits = p.rg_bits + (int64_t)gr.row0 * p.rg_capw;
    const int BR = p.rg_box;  // slots per copy: min(P, 128)
    const int np = 128 / BR;  // copies per line of a tile
    auto load_words = [&](int t, uint32_t (&wv)[8]) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int w = lane + 32 * k, row = w >> 2, wi = t * 4 + (w & 3);
        wv[k] = 0u;
        if (w < nw && row < gr.nrows && wi < words_valid) wv[k] = __ldg(bits + (int64_t)row * p.rg_capw + wi);
      }
    };
    // table entry of page `lane` of tile t (in_seq: the page holds positions of
    // the sequence and the table has it), fetched a tile ahead like the mask
    // words so no dependent load stands between a free stage and its copies
    auto load_page = [&](int t, uint32_t& e, bool& in_seq) {
      e = 0u;
      in_seq = false;
      if (lane < np) {
        const int64_t lp = (int64_t)t * 128 / p.P + (BR < 128 ? lane : 0);
        in_seq = lp < p.max_pages && lp * p.P < gr.kv_len;
        if (in_seq) e = __ldg(p.table + (int64_t)gr.b * p.max_pages + lp);
      }
    };
    uint32_t nxt[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    uint32_t pe_nxt = 0u;
    bool pin_nxt = false;
    if (NT > 0) {
      load_words(0, nxt);
      load_page(0, pe_nxt, pin_nxt);
    }
    int i = 0;
    bool ok = true;
    for (int t = 0; t < NT && ok; ++t) {
      uint32_t cur[8], o = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        cur[k] = nxt[k];
        o |= cur[k];
      }
      const uint32_t pe = pe_nxt;
      const bool pin = pin_nxt;
      if (t + 1 < NT) {
        load_words(t + 1, nxt);
        load_page(t + 1, pe_nxt, pin_nxt);
      }
      if (!__any_sync(0xffffffffu, o != 0u)) continue;
      const int s = i % kRgStages;
      if (i >= kRgStages && !warp_wait(bar(kBarFree + s), (uint32_t)((i / kRgStages - 1) & 1))) {
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
      if (pin) {
        if (pe < p.num_pages)
          phys = (int)pe;
        else
          badpage = true;
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
        for (int k = 0; k < 8; ++k) {
          had |= (cur[k] & kill) != 0u;
          cur[k] &= ~kill;
        }
        if (__any_sync(0xffffffffu, had) && lane == 0) atomicOr(p.status, QSA_STATUS_BAD_PAGE);
      }
      TileHdr& th = hdr[s];
      uint32_t any = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
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
      const uint32_t kb = bar(kBarK + s), vb = bar(kBarV + s);
      if (lane == 0) {
        tile_fence_proxy_async();
        mbar_arrive_expect_tx(kb, kRgTileBytes);
        mbar_arrive_expect_tx(vb, kRgTileBytes);
      }
      __syncwarp();
      if (lane < np) {
        const uint32_t dst = sStage + (uint32_t)s * kRgStageBytes + (uint32_t)(BR < 128 ? lane * BR * 128 : 0);
        const int slot = BR < 128 ? 0 : (int)(pos0 % p.P);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          tma_load_5d(dst + x * kRgHalf, &p.tmap, 0, h * 2 + x, slot, p.tma_plane_k, phys, kb);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          tma_load_5d(dst + kRgTileBytes + x * kRgHalf, &p.tmap, 0, h * 2 + x, slot, p.tma_plane_v, phys, vb);
      }
      ++i;
    }
    if (ok) {
      // end of the unit: a header with no copies, on the K barrier
      const int s = i % kRgStages;
      if (i >= kRgStages && !warp_wait(bar(kBarFree + s), (uint32_t)((i / kRgStages - 1) & 1))) ok = false;
      if (ok && lane == 0) {
        hdr[s].end = 1;
        mbar_arrive(bar(kBarK + s));
      }
    }
    if (!ok) {
      if (lane == 0) give_up();
      // copies in flight land before the CTA leaves
      for (int j = max(0, i - kRgStages); j < i; ++j) {
        if (!warp_wait(bar(kBarK + j % kRgStages), (uint32_t)((j / kRgStages) & 1))) break;
        if (!warp_wait(bar(kBarV + j % kRgStages), (uint32_t)((j / kRgStages) & 1))) break;
      }
    }
  } else if (warp == 10) {
    // V fix-up: once tile i's V has landed, zero the rows of keys no row of
    // the group selects, then let P.V read it
    for (int i = 0;; ++i) {
      const int s = i % kRgStages;
      if (!warp_wait(bar(kBarK + s), (uint32_t)((i / kRgStages) & 1))) {
        if (lane == 0) give_up();
        break;
      }
      if (*reinterpret_cast<volatile int32_t*>(&hdr[s].end)) break;
      if (!warp_wait(bar(kBarV + s), (uint32_t)((i / kRgStages) & 1))) {
        if (lane == 0) give_up();
        break;
      }
      const uint32_t vt = sStage + (uint32_t)s * kRgStageBytes + kRgTileBytes;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int k = lane + 32 * c;
        if ((hdr[s].any[c] >> lane) & 1u) continue;
#pragma unroll
        for (int x2 = 0; x2 < 2; ++x2)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};\n" ::"r"(vt + x2 * kRgHalf + (uint32_t)k * 128 + q * 16),
                         "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarVR + s));
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      uint32_t last_bar = 0, last_phase = 0;
      // descriptors of the tile bases, computed once: a step's descriptor
      // adds its byte offset / 16 to the start-address field (bits 0..13),
      // which cannot carry (shared addresses stay below 256 KB).  This thread
      // shares its sub-partition with two softmax warps: the fewer
      // instructions between its MMAs, the sooner the tensor pipe is fed.
      const uint64_t dq0 = smem_desc(sQ, 16, 1024, kSwizzle128);
      const uint64_t dk0 = smem_desc(sStage, 16, 1024, kSwizzle128);
      const uint64_t dv0 = smem_desc(sStage + kRgTileBytes, kRgHalf, 1024, kSwizzle128);
      auto qk = [&](int X, int i) {
        const uint64_t dk = dk0 + (uint64_t)((i % kRgStages) * (kRgStageBytes >> 4));
        const uint64_t dq = dq0 + (uint64_t)(X * (kRgTileBytes >> 4));
        const uint32_t sc = tm + kColS + (uint32_t)X * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off16 = ((uint32_t)(ks >> 2) * kRgHalf + (uint32_t)(ks & 3) * 32) >> 4;
          umma_f16(sc, dq + off16, dk + off16, kIdescQK, ks > 0);
        }
        umma_commit(bar(kBarS + X));
        last_bar = bar(kBarS + X);
        last_phase = (uint32_t)(i & 1);
      };
      auto pv = [&](int X, int i) -> bool {
        if (!mbar_wait(bar(kBarP + X), (uint32_t)(i & 1))) return false;
        tc_fence_after();
        const uint64_t dv = dv0 + (uint64_t)((i % kRgStages) * (kRgStageBytes >> 4));
        const uint32_t pcol = tm + kColS + (uint32_t)X * 128;  // P_X over the first 64 columns of S_X
        const uint32_t oc = tm + kColO + (uint32_t)X * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_f16_ts(oc, pcol + ks * 8, dv + (uint64_t)(ks * (2048 >> 4)), kIdescPV, i > 0 || ks > 0);
        umma_commit(bar(kBarO + X));
        last_bar = bar(kBarO + X);
        last_phase = (uint32_t)(i & 1);
        return true;
      };
      // waits for tile i's K copy; false at the end of the unit (or on a give-up)
      auto next_k = [&](int i, bool& ok) -> bool {
        const int s = i % kRgStages;
        if (!mbar_wait(bar(kBarK + s), (uint32_t)((i / kRgStages) & 1))) {
          ok = false;
          return false;
        }
        if (*reinterpret_cast<volatile int32_t*>(&hdr[s].end)) return false;
        tc_fence_after();
        return true;
      };
      bool ok = mbar_wait(bar(kBarQ), 0);
      int i = 0;
      bool more = ok && next_k(0, ok);
      if (more) {
        qk(0, 0);
        qk(1, 0);
      }
      while (more && ok) {
        const int s = i % kRgStages;
        if (!mbar_wait(bar(kBarVR + s), (uint32_t)((i / kRgStages) & 1)) || !pv(0, i)) {
          ok = false;
          break;
        }
        more = next_k(i + 1, ok);
        if (!ok) break;
        if (more) qk(0, i + 1);  // after PV_A(i), which reads P_A in these columns
        if (!pv(1, i)) {
          ok = false;
          break;
        }
        umma_commit(bar(kBarFree + s));  // both P.V of tile i issued: its stage is free once they are done
        last_bar = bar(kBarFree + s);
        last_phase = (uint32_t)((i / kRgStages) & 1);
        if (more) qk(1, i + 1);
        ++i;
      }
      if (!ok) {
        give_up();
        if (last_bar) mbar_wait(last_bar, last_phase);  // the tensor cores finish what was issued
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    // warp w serves accumulator rows 32 (w & 3) .. + 31 of tile X = (w - 2) / 4
    // (the TMEM lanes its position in the warpgroup may access)
    const int X = (warp - 2) >> 2, quarter = warp & 3;
    const int m = quarter * 32 + lane;               // accumulator row = TMEM lane
    const int rl = X * (R >> 1) + m / G, hq = m % G;  // row of the group, query head of kv head h
    const bool live = rl < gr.nrows;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t sc = tm + lane_off + kColS + (uint32_t)X * 128;
    const uint32_t oc = tm + lane_off + kColO + (uint32_t)X * 128;
    {
      // this row of Q into tile X, 128-byte-swizzled K-major (zeros past the group's rows)
      const uint4* src =
          live ? reinterpret_cast<const uint4*>(p.q + ((int64_t)(gr.row0 + rl) * p.nq + (int64_t)h * G + hq) * 256)
               : nullptr;
      const uint32_t qb = sQ + (uint32_t)X * kRgTileBytes;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (live) v = __ldg(src + c);
        if (p.scale_log2 < 0.f) {
          v.x ^= 0x80008000u;
          v.y ^= 0x80008000u;
          v.z ^= 0x80008000u;
          v.w ^= 0x80008000u;
        }
        const uint32_t dst = qb + (uint32_t)(c >> 3) * kRgHalf + (uint32_t)m * 128 + ((uint32_t)((c & 7) ^ (m & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kBarQ));
    }
    // the softmax runs on raw scores times c = |scale log2(e)| (at least
    // 1e-30, so a zero scale still gives -inf x c = -inf on masked keys); a
    // negative scale is applied by negating Q, which is exact
    const float c_log2 = fmaxf(fabsf(p.scale_log2), 1e-30f);
    float m_ref = -CUDART_INF_F, l = 0.f;
    int i = 0;
    bool ok = true;
    for (;;) {
      const int s = i % kRgStages;
      if (!warp_wait(bar(kBarK + s), (uint32_t)((i / kRgStages) & 1))) {
        ok = false;
        break;
      }
      if (*reinterpret_cast<volatile int32_t*>(&hdr[s].end)) break;
      if (!warp_wait(bar(kBarS + X), (uint32_t)(i & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint4 mk = *reinterpret_cast<const uint4*>(&hdr[s].mask[rl][0]);
      const uint32_t mw[4] = {mk.x, mk.y, mk.z, mk.w};
      // One pass over S, half by half (keys 64 hf .. + 63): keys this row did
      // not select read as -inf; the half's maximum over eight independent
      // chains (raw scores; c >= 0); the reference moves when that maximum
      // exceeds it by more than 2^8 (or there was none yet), rescaling O, the
      // sum and, for the second half, the first half's P already in tensor
      // memory; then p = 2^(c s - m) in one FFMA and one ex2 per key (masked
      // keys: 0), written as bf16 pairs over columns 32 hf .. + 31 of S_X,
      // which that half has read.
      float sa[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sa[k] = 0.f;
      auto move_ref = [&](float mxh, int hf) -> bool {
        const bool need = mxh > m_ref + 8.f;
        if (!__any_sync(0xffffffffu, need)) return true;
        const bool seen = m_ref != -CUDART_INF_F;  // O holds nonzero terms only then
        const float mnew = need ? mxh : m_ref;
        const float f = need ? (seen ? exp2_fast(m_ref - mnew) : 0.f) : 1.f;
        if (i > 0 && __any_sync(0xffffffffu, need && seen)) {
          // O holds every earlier tile once the previous P.V is done
          if (!warp_wait(bar(kBarO + X), (uint32_t)((i - 1) & 1))) return false;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {  // 16 columns at a time: the scores stay live across it
            float o[16];
            tmem_ld16(oc + c * 16, o);
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] *= f;
            tmem_st16(oc + c * 16, o);
          }
        }
        if (hf == 1 && __any_sync(0xffffffffu, need && seen)) {
          // the first half's P was taken against the old reference
          tmem_wait_st();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            float pw[16];
            tmem_ld16(sc + c * 16, pw);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const uint32_t b = __float_as_uint(pw[j]);
              pw[j] = __uint_as_float(pack_bf16(__uint_as_float(b << 16) * f, __uint_as_float(b & 0xFFFF0000u) * f));
            }
            tmem_st16(sc + c * 16, pw);
          }
        }
        tmem_wait_st();
#pragma unroll
        for (int k = 0; k < 8; ++k) sa[k] *= f;
        l *= f;
        m_ref = mnew;
        return true;
      };
      auto half_pass = [&](int hf, const uint32_t (&xr)[64]) -> bool {
        const uint32_t w0 = mw[2 * hf], w1 = mw[2 * hf + 1];
        float x[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(xr[j]);
        float mxa[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mxa[k] = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          x[j] = (((j < 32 ? w0 : w1) >> (j & 31)) & 1u) ? x[j] : -CUDART_INF_F;
          mxa[j & 7] = fmaxf(mxa[j & 7], x[j]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) mxa[k] = fmaxf(mxa[k], mxa[k + 4]);
        const float mxr = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3]));
        if (!move_ref(mxr == -CUDART_INF_F ? -CUDART_INF_F : mxr * c_log2, hf)) return false;
        const float nm = m_ref == -CUDART_INF_F ? 0.f : -m_ref;
#pragma unroll
        for (int q = 0; q < 2; ++q) {  // 32 keys at a time, so x is consumed as P is stored
          float pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float p0 = exp2_fast(fmaf(x[32 * q + 2 * j], c_log2, nm));
            const float p1 = exp2_fast(fmaf(x[32 * q + 2 * j + 1], c_log2, nm));
            sa[(2 * j) & 7] += p0;
            sa[(2 * j + 1) & 7] += p1;
            pk[j] = __uint_as_float(pack_bf16(p0, p1));
          }
          tmem_st16(sc + hf * 32 + 16 * q, pk);
        }
        return true;
      };
      // the second half's scores load while the first half is processed
      uint32_t xr0[64], xr1[64];
      tmem_ld64_issue(sc, xr0);
      tmem_wait_ld64(xr0);
      tmem_ld64_issue(sc + 64, xr1);
      if (!half_pass(0, xr0)) {
        ok = false;
        break;
      }
      tmem_wait_ld64(xr1);
      if (!half_pass(1, xr1)) {
        ok = false;
        break;
      }
      tmem_wait_st();
      l += ((sa[0] + sa[1]) + (sa[2] + sa[3])) + ((sa[4] + sa[5]) + (sa[6] + sa[7]));
      tc_fence_before();
      mbar_arrive(bar(kBarP + X));
      ++i;
    }
    // epilogue: O / l for this row (tiles i; zero when the row attended nothing)
    bool have = i > 0 && ok;
    if (have && !warp_wait(bar(kBarO + X), (uint32_t)((i - 1) & 1))) {
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
      if (__any_sync(0xffffffffu, have)) tmem_ld32(oc + c * 32, o);
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
