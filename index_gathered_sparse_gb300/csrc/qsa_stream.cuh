// Persistent stream-K kernel for QSA gather-GQA sparse attention, BF16 and FP8
// e4m3 caches, head_dim 128 (QSASparseAttentionRaggedPaged: "Gather-GQA over
// the token indices a QSA selection names"; its `warps` and `unroll`
// parameters: warps per CTA, gathered keys loaded before any is consumed).
//
// Work.  A unit is one query row and a group of HPU adjacent kv heads (4 when
// num_kv_heads allows): the K rows of those heads are HPU*256 B (BF16) or
// HPU*128 B (FP8) contiguous in a cache slot, so one translated position
// feeds HPU heads with one contiguous read.  A unit has as many key tiles as
// its row's count fills (one, empty, when the count is 0); the launch has one
// CTA per SM, and CTA c processes the contiguous range [c*R/G, (c+1)*R/G) of
// all R tiles (stream-K; G = min(CTAs, R)), found by a block scan of the counts at the start,
// so the load is balanced to a tile and at most the first and the last unit
// of a range are shared with other CTAs.  The rows are numbered in an
// interleaved order that keeps all CTAs on neighbouring rows.  When there
// are no more units than CTAs, the split skips the scan and counts W / TILE
// tiles for every unit instead (tiles past a count are skipped).
//
// Roles.  The first PW warps produce (four, or eight for units of one or two
// heads with one 8-head N tile), the last NC consume (eight, two per kv head,
// for units of four heads with one N tile, else four), linked per stage by a
// "full" and an "empty" mbarrier.  Producers fetch everything a tile needs in hops
// spaced H = STAGES - 1 producer iterations apart, so each hop has landed when
// the next one reads it and nothing waits on a dependent load in steady state:
//     unit meta (counts, cache_lengths)   ~ H + 1 units ahead of the index hop
//     indices  (token_indices)            3H + 1 tiles ahead of the K/V hop's
//     page     (kv_lookup_table entries)  2H + 1 tiles ahead         ... tile
//     offsets  (computed from both)        H + 1 tiles ahead
// and the K/V rows by 16-byte cp.async (zero-filled for slots without a valid
// key), each producer thread arriving on the stage's full barrier when its
// copies land.  Consumers own heads (WPH = NC / HPU warps per head split a
// tile's keys) and run the keys-on-M / heads-on-N mma.sync scheme: S^T = K Q^T,
// online softmax in base 2, P^T by movmatrix, O^T += V^T P^T; they release each
// stage on its empty barrier.  A unit's end merges the consumer warps in
// shared memory and writes the output, or, for a shared unit, a partial
// record; after its range each CTA arrives on the shared units' tickets and
// the last arrival merges the records (no CTA ever waits for another).
#pragma once

#include "qsa_mma.cuh"

namespace qsa {

template <int KIND, int NT, int HPU>
struct StreamCfg {
  static constexpr int D = 128;
  static constexpr int ELEM = KIND == kBF16 ? 2 : 1;
  static constexpr int ROWB = D * ELEM;             // one head's K (or V) row
  static constexpr int KEYB = HPU * ROWB;           // a unit's K (or V) bytes per key, contiguous
  static constexpr int SROW = KEYB + 16;            // padded shared-memory row (conflict-free ldmatrix)
  // Consumer warps: eight for units of four heads with one 8-head N tile (two
  // per kv head, splitting each tile's keys, so that two dependent
  // MMA/softmax chains share each SM sub-partition) or of eight heads (one per
  // head); else four.
  static constexpr int NC = (NT == 1 && HPU >= 4) ? 8 : 4;
  static constexpr int CT = NC * 32;                // consumer threads
  static constexpr int WPH = NC / HPU;              // warps per head
  // two warps per head merge their softmax states pairwise through shared
  // memory (half of head_dim at a time) into the first warp's registers
  static constexpr bool PAIR = NC == 8 && WPH == 2;
  // keys per stage: 64 KB of K+V when each warp owns a head (no epilogue
  // buffer competes for shared memory), else 32 KB
  static constexpr int TILE = stream_tile(ELEM, HPU);
  static constexpr int KPW = TILE / WPH;            // keys per warp per tile
  static constexpr int MSL = KPW / 16;              // 16-key MMA slices per warp per tile
  static constexpr int KV_BYTES = TILE * SROW;
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int GP = 8 * NT;                 // padded query heads per kv head
  static constexpr int KSTEPS = KIND == kBF16 ? 8 : 4;
  static constexpr int CPK = 2 * KEYB / 16;         // 16-byte chunks per key (K and V)
  static constexpr int CHUNKS = TILE * CPK;         // per stage
  static constexpr int RT = TILE <= 32 ? 32 : 16;   // tile-record ring (positions, pages, offsets)
  static constexpr int MR = 64;                     // unit-meta ring
  static constexpr int MAXOFF = 1024;               // input_row_offsets entries kept in shared memory
  // Warps that share a head merge through shared memory; a warp that owns its
  // head writes straight from registers and needs no epilogue buffer.
  static constexpr int EPI_FLOATS = PAIR ? 4 * GP * (D / 2) + 2 * 4 * GP : WPH > 1 ? 4 * GP * D + 2 * 4 * GP : 0;
  static constexpr int FIXED = EPI_FLOATS * 4 + 3 * RT * TILE * 4 + MR * 32 + MAXOFF * 4;
  static constexpr int STAGES_FIT = (232448 - FIXED) / STAGE_BYTES;
  static constexpr int STAGES_CAP = TILE <= 32 ? 8 : 5;
  static constexpr int STAGES = STAGES_FIT < STAGES_CAP ? STAGES_FIT : STAGES_CAP;
  static constexpr int H = STAGES - 1;
  static constexpr int SMEM = STAGES * STAGE_BYTES + FIXED;
  // Producer warps: eight when the consumers fit the 168 registers a thread of
  // a 384-thread CTA gets (one 8-head N tile), else four; more producers keep
  // more copies in flight while some of them translate.
  static constexpr int PW = NT == 1 && NC == 4 ? 8 : 4;
  static constexpr int PT = PW * 32;
  static constexpr int THREADS = PT + CT;
  // K/V copies: one bulk copy per key chunk when chunks are 512 B or more (a
  // warp pays a fixed issue time per bulk copy), else 16-byte cp.async, whose
  // outstanding copies are limited per thread.
  static constexpr bool BULK = KEYB >= 512;
  static constexpr int FULL_ARRIVALS = BULK ? PW : PT + 1;
  static_assert(CHUNKS % PT == 0, "stage copy split over the producer warps");
  static_assert(KPW % 16 == 0, "warp key slices are 16 keys");
  // producers run up to STAGES tiles ahead of consumers with hops up to 3H+1
  // tiles further; the consumers still read a tile's offsets and meta then
  static_assert(2 * H + 1 + STAGES < RT, "tile-record ring too small");
  static_assert(3 * H + 1 + STAGES + H + 2 < MR, "unit-meta ring too small");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(STAGES >= 3, "stage ring");
  static_assert(WPH >= 1 && NC % HPU == 0, "every head has whole consumer warps");
  static_assert(HPU < 8 || NT == 1, "eight-head units take one 8-head N tile");
};

// Barrier over the `n` threads of one role (id 1: producers, id 2: consumers).
__device__ __forceinline__ void role_sync(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }
// The same barrier, returning whether any of the role's threads passed true.
__device__ __forceinline__ bool role_any(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.or.pred po, %2, %3, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// A cursor over this CTA's tiles: unit u (its row r, kv-head group hg, valid
// count n and last tile jl inside the range), tile j, ordinal o.  Every thread
// of a role holds the same cursor values, so branches on them are uniform.
struct TileCursor {
  int u, j, o, r, hg, n, jl;
  bool live;
};

// Order of the rows in the tile numbering: the transpose of a row-major
// matrix with `cols` columns, so that a CTA's contiguous range takes rows c,
// c + cols, c + 2*cols, ... and all CTAs move through neighbouring rows
// together.  Rows of one sequence read overlapping cache positions, which
// then stay in L2 between them.  Columns 0..rem-1 hold ni rows, the rest
// ni - 1.  row(k) is the row index (before the reversal below) at position k.
struct RowOrder {
  int cols, ni, rem;
  __device__ __forceinline__ RowOrder(int total_q, int ctas) {
    cols = max(1, min(ctas, total_q));
    ni = (total_q + cols - 1) / cols;
    rem = total_q - (ni - 1) * cols;
  }
  __device__ __forceinline__ int row(int k) const {
    const int big = rem * ni;
    int c, i;
    if (k < big) {
      c = k / ni;
      i = k - c * ni;
    } else {
      const int k2 = k - big;
      c = rem + k2 / (ni - 1);
      i = k2 - (c - rem) * (ni - 1);
    }
    return i * cols + c;
  }
};

// Query row of unit u: row total_q - 1 - ord.row(u / NG) of the order in use.
static __device__ __noinline__ int unit_row(const Params& p, const StreamPlan& sp, int u) {
  const RowOrder ro(p.total_q, sp.G);
  return p.total_q - 1 - ro.row(u / sp.NG);
}

// This CTA's share of the key tiles: R tiles in all, its range [t0, t1), the
// units holding t0 and t1 - 1 and the tile numbers where those units start
// and end.
struct SplitRange {
  int64_t R, t0, t1;
  int G;  // CTAs with work: min(launched CTAs, R), so that no range is empty
  int u_first, u_last;
  int64_t P_first, P_first_end, P_last, P_last_end;
};

// Block-wide (every thread of the CTA, before any role split): position q of
// the row order (row total_q - 1 - rorder.row(q)) has NG units of RT = max(1, ceil(n / TILE))
// tiles each, n = clamp(counts, 0, W); each thread sums a chunk of rows, a
// block scan places the chunks, and the threads whose chunks hold t0 and
// t1 - 1 locate them.  The counts are first read coalesced into `s_tiles`
// (room for `cap` rows; longer batches read them in place).  `s_scan` holds
// 16 int64.
template <int TILE, int NTH>
__device__ __forceinline__ SplitRange split_range(const Params& p, const StreamPlan& sp, const RowOrder& rorder,
                                                  long long* s_scan, int32_t* s_tiles, int cap) {
  constexpr int NW = NTH / 32;
  static_assert(NW <= 16, "scan scratch");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int total_q = p.total_q, NG = sp.NG;
  auto tiles = [&](int c) { const int n = min(max(c, 0), p.W); return n > 0 ? (n + TILE - 1) / TILE : 1; };
  const bool cached = total_q <= cap;
  if (cached) {
    for (int base = 0; base < total_q; base += 8 * NTH) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = base + i * NTH + tid;
        v[i] = q < total_q ? __ldg(p.counts + (total_q - 1 - rorder.row(q))) : 0;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = base + i * NTH + tid;
        if (q < total_q) s_tiles[q] = tiles(v[i]);
      }
    }
    __syncthreads();
  }
  const int ch = (total_q + NTH - 1) / NTH;
  const int q0 = min(tid * ch, total_q), q1 = min(q0 + ch, total_q);
  auto tiles_of = [&](int q) -> int64_t {
    return cached ? s_tiles[q] : tiles(__ldg(p.counts + (total_q - 1 - rorder.row(q))));
  };
  int64_t mine = 0;
  for (int q = q0; q < q1; ++q) mine += tiles_of(q);
  int64_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < NW ? s_scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    __syncwarp();
    if (lane < NW) s_scan[lane] = w;
  }
  __syncthreads();
  const int64_t before = (warp ? s_scan[warp - 1] : 0) + incl - mine;  // tiles of the rows before this chunk
  SplitRange rg;
  rg.R = (int64_t)NG * s_scan[NW - 1];
  rg.G = (int)min((int64_t)sp.G, rg.R);
  rg.t0 = blockIdx.x < rg.G ? (int64_t)blockIdx.x * rg.R / rg.G : 0;
  rg.t1 = blockIdx.x < rg.G ? ((int64_t)blockIdx.x + 1) * rg.R / rg.G : 0;
  __syncthreads();  // s_scan now receives the result
  if (rg.t0 < rg.t1) {
    int64_t s = (int64_t)NG * before;
    const int64_t e = s + (int64_t)NG * mine;
    const int64_t a = rg.t0, b = rg.t1 - 1;
    if ((a >= s && a < e) || (b >= s && b < e)) {
      for (int q = q0; q < q1; ++q) {
        const int64_t rt = tiles_of(q), w = (int64_t)NG * rt;
        if (a >= s && a < s + w) {
          const int64_t hg = (a - s) / rt;
          s_scan[0] = (int64_t)q * NG + hg;
          s_scan[1] = s + hg * rt;
          s_scan[2] = s + (hg + 1) * rt;
        }
        if (b >= s && b < s + w) {
          const int64_t hg = (b - s) / rt;
          s_scan[3] = (int64_t)q * NG + hg;
          s_scan[4] = s + hg * rt;
          s_scan[5] = s + (hg + 1) * rt;
        }
        s += w;
      }
    }
  }
  __syncthreads();
  rg.u_first = (int)s_scan[0];
  rg.P_first = s_scan[1];
  rg.P_first_end = s_scan[2];
  rg.u_last = (int)s_scan[3];
  rg.P_last = s_scan[4];
  rg.P_last_end = s_scan[5];
  return rg;
}

// The split without a scan: every unit counts VT tiles (those past its count
// are skipped), R = U * VT, CTA c takes [c*R/G, (c+1)*R/G).
__device__ __forceinline__ SplitRange even_range(const StreamPlan& sp) {
  SplitRange rg;
  rg.R = sp.T;
  rg.G = (int)min((int64_t)sp.G, sp.T);
  rg.t0 = blockIdx.x < rg.G ? (int64_t)blockIdx.x * rg.R / rg.G : 0;
  rg.t1 = blockIdx.x < rg.G ? ((int64_t)blockIdx.x + 1) * rg.R / rg.G : 0;
  rg.u_first = (int)(rg.t0 / sp.VT);
  rg.u_last = rg.t1 > rg.t0 ? (int)((rg.t1 - 1) / sp.VT) : rg.u_first;
  rg.P_first = (int64_t)rg.u_first * sp.VT;
  rg.P_first_end = rg.P_first + sp.VT;
  rg.P_last = (int64_t)rg.u_last * sp.VT;
  rg.P_last_end = rg.P_last + sp.VT;
  return rg;
}

template <int KIND, int NT, int HPU, bool SCAN>
__global__ void __launch_bounds__(StreamCfg<KIND, NT, HPU>::THREADS, 1) stream_kernel(const Params p, const StreamPlan sp) {
  using C = StreamCfg<KIND, NT, HPU>;
  constexpr int H = C::H, S = C::STAGES, TILE = C::TILE, RT = C::RT, MR = C::MR, GP = C::GP;
  static_assert((RT & (RT - 1)) == 0 && (MR & (MR - 1)) == 0, "rings are powers of two");
  extern __shared__ __align__(128) unsigned char smem[];
  // epilogue buffer [4][GP][D] + m[4][GP] + l[4][GP] (warps sharing a head)
  float* epi_buf = reinterpret_cast<float*>(smem + S * C::STAGE_BYTES);
  int32_t* s_pos = reinterpret_cast<int32_t*>(epi_buf + C::EPI_FLOATS);  // [RT][TILE]
  uint32_t* s_page = reinterpret_cast<uint32_t*>(s_pos + RT * TILE); // [RT][TILE]
  uint32_t* s_off = s_page + RT * TILE;                               // [RT][TILE]
  // unit meta [MR][MW]: count, clen, b, rows_b (and, with the scan, the row)
  constexpr int MW = SCAN ? 8 : 4;
  int32_t* s_meta = reinterpret_cast<int32_t*>(s_off + RT * TILE);
  uint32_t* s_rowoff = reinterpret_cast<uint32_t*>(s_meta + MR * 8);  // [MAXOFF]
  __shared__ int s_merge[2];
  __shared__ long long s_scan[16];  // the work split's scan and its result
  // stage landed: one expect-tx arrival per producer warp (bulk copies), or one
  // cp.async arrival per producer thread plus one release arrival
  __shared__ __align__(8) uint64_t s_full[S];
  __shared__ __align__(8) uint64_t s_empty[S];   // stage consumed: one arrival per consumer warp

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
  constexpr int PT = C::PT;
  const int rw = warp < C::PW ? warp : warp - C::PW;  // warp within its role
  const int VT = sp.VT;
  // Work split over the tiles that hold keys.  Unit u (row r = total_q-1-u/NG)
  // has RT(r) = max(1, ceil(clamp(counts[r], 0, W) / TILE)) tiles; tiles are
  // numbered unit after unit (P_u = tiles before unit u, R = all of them) and
  // CTA c takes [c*R/G, (c+1)*R/G).  Every CTA scans the counts itself.
  if (warp < C::PW && p.batch + 1 <= C::MAXOFF)  // lands during the scan
    for (int k = tid; k <= p.batch; k += C::PT) cp_async4(smem_addr(&s_rowoff[k]), p.row_offsets + k);
  SplitRange rg;
  if constexpr (SCAN) {
    const RowOrder ro(p.total_q, sp.G);
    rg = split_range<TILE, C::THREADS>(p, sp, ro, s_scan, reinterpret_cast<int32_t*>(smem), S * C::STAGE_BYTES / 4);
    fence_proxy_async_smem();  // the scan's writes to the stage ring before any copy into it
  } else {
    rg = even_range(sp);
  }
  if (rg.t0 >= rg.t1) {
    cp_async_wait_all();
    return;
  }
  const int u_first = rg.u_first, u_last = rg.u_last;
  const int jlo_first = (int)(rg.t0 - rg.P_first);  // first tile of the first unit in range
  const int jhi_last = (int)(rg.t1 - rg.P_last);    // end tile of the last unit in range
  // the rest of the scanned split is needed only at shared units' ends: keep
  // it in shared memory (published by the barrier after the mbarrier set-up)
  __shared__ SplitRange s_rg;
  if (SCAN && tid == 0) s_rg = rg;
  if (tid == 0) {
    for (int k = 0; k < S; ++k) {
      mbar_init(smem_addr(&s_full[k]), C::FULL_ARRIVALS);
      mbar_init(smem_addr(&s_empty[k]), C::NC);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();  // the last block-wide barrier: the roles part here

  auto mslot = [&](int u) { return ((u - u_first) & (MR - 1)) * MW; };
  // tile j of unit u: jl = last tile inside the range that holds keys (or the
  // first tile in range when none does: that unit still gets one empty tile)
  auto unit_jl = [&](int u, int n) {
    const int jlo = u == u_first ? jlo_first : 0, jhi = u == u_last ? jhi_last : VT;
    return max(jlo, min(jhi, (n + TILE - 1) / TILE) - 1);
  };
  auto unit_n = [&](int u) {
    const int m = mslot(u);
    return s_meta[m + 2] < 0 ? 0 : min(max(s_meta[m + 0], 0), p.W);
  };
  auto keys_in = [&](int n, int j) { return min(max(n - j * TILE, 0), TILE); };

  if (warp < C::PW) {
    // =====================================================================
    // producers
    // =====================================================================
    uint32_t bad = 0;
    // query row of unit u (computed once per unit by thread 0, which
    // publishes it in the unit meta)
    const RowOrder rorder(p.total_q, SCAN ? sp.G : p.total_q);  // the identity without the scan
    auto row_of = [&](int u) {
      if constexpr (SCAN) return p.total_q - 1 - rorder.row(u / sp.NG);
      else return p.total_q - 1 - u / sp.NG;
    };
    auto find_seq = [&](int r) -> int {  // sequence of row r, -1 when no sequence owns it
      const bool in_smem = p.batch + 1 <= C::MAXOFF;
      auto off = [&](int k) { return in_smem ? s_rowoff[k] : __ldg(p.row_offsets + k); };
      int lo = 0, hi = p.batch;  // largest b in [0, batch] with off[b] <= r
      if (off(0) > (uint32_t)r) return -1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off(mid) <= (uint32_t)r) lo = mid; else hi = mid - 1;
      }
      if (lo >= p.batch || (uint32_t)r >= off(lo + 1)) return -1;
      return lo;
    };
    // unit meta in two parts: the row's count (needs nothing), then its
    // sequence, that sequence's rows and cached length (needs the offsets)
    auto issue_meta_count = [&](int u) {  // producer thread 0 only
      const int r = row_of(u), m = mslot(u);
      if constexpr (SCAN) s_meta[m + 4] = r;  // the unit's query row, for the other producers and the consumers
      cp_async4(smem_addr(&s_meta[m + 0]), p.counts + r);
    };
    auto issue_meta_seq = [&](int u) {  // producer thread 0 only
      const int m = mslot(u), r = SCAN ? s_meta[m + 4] : row_of(u);
      const int b = find_seq(r);
      s_meta[m + 2] = b;
      if (b >= 0) {
        const bool in_smem = p.batch + 1 <= C::MAXOFF;
        s_meta[m + 3] = (int32_t)((in_smem ? s_rowoff[b + 1] : __ldg(p.row_offsets + b + 1)) -
                                  (in_smem ? s_rowoff[b] : __ldg(p.row_offsets + b)));
        cp_async4(smem_addr(&s_meta[m + 1]), p.cache_lengths + b);
      } else {
        s_meta[m + 1] = 0;
        s_meta[m + 3] = 0;
        bad |= QSA_STATUS_BAD_ROW;
      }
    };
    auto issue_meta = [&](int u) {
      issue_meta_count(u);
      issue_meta_seq(u);
    };
    int meta_issued = u_first, meta_landed = u_first;
    int hist[H];  // meta_issued at the end of each of the last H iterations
    auto issue_meta_upto = [&](int u) {
      u = min(u, u_last);
      if (u < meta_issued) return;
      if (tid == 0)
        for (int v = meta_issued; v <= u; ++v) issue_meta(v);
      meta_issued = u + 1;
    };
    auto ensure_meta = [&](int u) {  // makes unit u's meta readable (a full wait when it has not landed)
      if (u >= meta_issued) issue_meta_upto(u);
      if (u >= meta_landed) {
        cp_async_wait_all();
        role_sync(1, PT);
        meta_landed = meta_issued;
#pragma unroll
        for (int k = 0; k < H; ++k) hist[k] = meta_issued;
      }
    };
    auto enter = [&](TileCursor& c, int u) {
      ensure_meta(u);
      c.u = u;
      const int q = u / sp.NG;
      c.r = SCAN ? s_meta[mslot(u) + 4] : p.total_q - 1 - q;
      c.hg = u - q * sp.NG;
      c.n = unit_n(u);
      c.jl = unit_jl(u, c.n);
      c.j = u == u_first ? jlo_first : 0;
    };
    auto advance = [&](TileCursor& c) {
      ++c.o;
      if (c.j < c.jl) ++c.j;
      else if (c.u < u_last) enter(c, c.u + 1);
      else c.live = false;
    };
    // hops: indices on warp 1, page entries on warp 2, offsets on warp 3,
    // K/V copies on all four producer warps
    auto idx_hop = [&](const TileCursor& c) {
      if (rw != 1) return;
      const int kt = keys_in(c.n, c.j), slot = (c.o & (RT - 1)) * TILE;
      const int32_t* src = p.indices + (int64_t)c.r * p.W + c.j * TILE;
      for (int k = lane; k < kt; k += 32) cp_async4(smem_addr(&s_pos[slot + k]), src + k);
    };
    auto page_hop = [&](const TileCursor& c) {
      if (rw != 2) return;
      const int kt = keys_in(c.n, c.j), slot = (c.o & (RT - 1)) * TILE;
      if (kt == 0) return;
      const int m = mslot(c.u);
      const int64_t kvl = (int64_t)(uint32_t)s_meta[m + 1] + (int64_t)s_meta[m + 3];
      const uint32_t* trow = p.table + (int64_t)s_meta[m + 2] * p.max_pages;
      for (int k = lane; k < kt; k += 32) {
        const int32_t pos = s_pos[slot + k];
        uint32_t so = kInvalidOff;
        if (pos < 0 || (int64_t)pos >= kvl) {
          bad |= QSA_STATUS_BAD_INDEX;
        } else {
          const uint32_t lp = p.log2P >= 0 ? (uint32_t)pos >> p.log2P : (uint32_t)pos / (uint32_t)p.P;
          if (lp >= (uint32_t)p.max_pages) {
            bad |= QSA_STATUS_BAD_PAGE;
          } else {
            cp_async4(smem_addr(&s_page[slot + k]), trow + lp);
            so = (uint32_t)pos - lp * (uint32_t)p.P;  // slot within the page
          }
        }
        s_off[slot + k] = so;
      }
    };
    auto off_hop = [&](const TileCursor& c) {
      if (rw != 3) return;
      const int kt = keys_in(c.n, c.j), slot = (c.o & (RT - 1)) * TILE;
      const int64_t head0 = p.k_layer_bytes + (int64_t)c.hg * HPU * p.head_bytes;
      for (int k = lane; k < kt; k += 32) {
        const uint32_t so = s_off[slot + k];
        if (so == kInvalidOff) continue;
        const uint32_t page = s_page[slot + k];
        if (page >= p.num_pages) {
          bad |= QSA_STATUS_BAD_PAGE;
          s_off[slot + k] = kInvalidOff;
        } else {
          s_off[slot + k] =
              (uint32_t)(((int64_t)page * p.page_pitch_bytes + head0 + (int64_t)so * p.slot_bytes) >> 4);
        }
      }
    };
    // this thread's fixed role in a stage copy: key offset, K or V, 16-byte chunk
    constexpr int KPI = PT / C::CPK;  // keys per copy round
    const int my_key = tid / C::CPK, my_w = tid - my_key * C::CPK;
    const int my_kv = my_w / (C::CPK / 2), my_ch = my_w - my_kv * (C::CPK / 2);
    const int64_t my_src = (my_kv ? p.v_minus_k_bytes : 0) + my_ch * 16;
    const int my_dst = my_kv * C::KV_BYTES + my_key * C::SROW + my_ch * 16;
    // K/V of a tile into its stage, once the consumers have released it;
    // false when that wait gave up.  Slots without a valid key hold zeros:
    // their scores are masked, but 0 * NaN would not vanish.
    // Thread 0 waits until the consumers have released the stage of K/V tile
    // c (the other producers learn of it, or of a give-up, at the next
    // producer barrier); false after a give-up.
    auto stage_free = [&](const TileCursor& c) -> bool {
      if (tid != 0 || c.o < S) return true;
      return mbar_wait(smem_addr(&s_empty[c.o % S]), (uint32_t)((c.o / S - 1) & 1), p.stall ? kStallSpins : kSpinLimit);
    };
    auto kv_hop = [&](const TileCursor& c) {
      if (p.stall) return;  // (tests) no copy and no arrival: the consumers' waits give up
      const int kt = keys_in(c.n, c.j), slot = (c.o & (RT - 1)) * TILE, st = c.o % S;
      const uint32_t bar = smem_addr(&s_full[st]);
      if constexpr (C::BULK) {
        // producer warp w moves keys w, w + PW, ...: lane j copies key j's K
        // row and lane KPWARP + j its V row (one bulk copy each); lane 0 then
        // arrives with the bytes to expect (and so also publishes the tile's
        // offsets and the unit meta, written before the last producer barrier)
        constexpr int KPWARP = (TILE + C::PW - 1) / C::PW;
        static_assert((KPWARP & (KPWARP - 1)) == 0 && 2 * KPWARP <= 32, "one copy per lane");
        unsigned char* sb = smem + st * C::STAGE_BYTES;
        const int j = lane & (KPWARP - 1), half = lane / KPWARP;
        const int key = rw + C::PW * j;
        const bool mine = lane < 2 * KPWARP && key < TILE;
        const bool v = mine && key < kt && s_off[slot + key] != kInvalidOff;
        const uint32_t nv = __popc(__ballot_sync(0xffffffffu, v));
        if (mine && !v && half == 1) {
          // a slot without a valid key: zero V (its score is masked, but 0 * NaN
          // would not vanish); this lane also fills the row when it is valid,
          // so its own proxy fence orders these writes before that copy
          uint4* row = reinterpret_cast<uint4*>(sb + C::KV_BYTES + key * C::SROW);
          for (int q = 0; q < C::KEYB / 16; ++q) row[q] = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(bar, nv * (uint32_t)C::KEYB);
        __syncwarp();
        if (v) {
          const unsigned char* src = p.kv + (int64_t)s_off[slot + key] * 16 + (half ? p.v_minus_k_bytes : 0);
          bulk_g2s(smem_addr(sb + half * C::KV_BYTES + key * C::SROW), src, C::KEYB, bar);
        }
      } else {
        const uint32_t sbase = smem_addr(smem + st * C::STAGE_BYTES) + my_dst;
#pragma unroll 4
        for (int i = 0; i < TILE / KPI; ++i) {
          const int key = i * KPI + my_key;
          const uint32_t off = key < kt ? s_off[slot + key] : kInvalidOff;
          const bool live = off != kInvalidOff;
          cp_async16(sbase + i * KPI * C::SROW, live ? p.kv + (int64_t)off * 16 + my_src : p.kv, live ? 16u : 0u);
        }
        cp_async_mbar_arrive(bar);
        // publishes this tile's offsets (consumers mask with them) and every unit
        // meta written so far: all were written before the last producer barrier
        if (tid == 0) mbar_arrive(bar);
      }
    };

    // prologue: offsets and the first counts, then the sequences' meta
    // together with the first index hops (which need only counts), then page
    // entries, then K/V
    const int u_pro = min(u_first + H + 1, u_last);
    if (tid == 0)  // (the row offsets were issued before the split)
      for (int v = u_first; v <= u_pro; ++v) issue_meta_count(v);
    cp_async_wait_all();
    role_sync(1, PT);
    if (tid == 0)
      for (int v = u_first; v <= u_pro; ++v) issue_meta_seq(v);
    meta_issued = u_pro + 1;
    role_sync(1, PT);  // the sequence ids are plain stores; cached lengths land with the index hops
    meta_landed = meta_issued;
#pragma unroll
    for (int k = 0; k < H; ++k) hist[k] = meta_issued;
    TileCursor ci;
    ci.o = 0;
    ci.live = true;
    enter(ci, u_first);
    TileCursor cpg = ci, cof = ci, ckv = ci;
    for (int n = 0; n <= 2 * H && ci.live; ++n) {
      idx_hop(ci);
      advance(ci);
    }
    cp_async_wait_all();
    role_sync(1, PT);
    for (int n = 0; n <= H && cpg.live; ++n) {
      page_hop(cpg);
      advance(cpg);
    }
    cp_async_wait_all();
    role_sync(1, PT);
    off_hop(cof);
    advance(cof);
    // main loop: one K/V tile per iteration; the hop for the tile t + 1 + kH
    // lands k iterations later
    bool aborted = false;
    while (ckv.live) {
      cp_async_wait<H - 1>();
      const bool lost = !stage_free(ckv);
      if (role_any(1, PT, lost)) {  // one barrier per tile: hops landed, stage free
        aborted = true;
        break;
      }
      meta_landed = max(meta_landed, hist[H - 1]);
      kv_hop(ckv);
      advance(ckv);
      if (cof.live) {
        off_hop(cof);
        advance(cof);
      }
      if (cpg.live) {
        page_hop(cpg);
        advance(cpg);
      }
      if (ci.live) {
        idx_hop(ci);
        issue_meta_upto(ci.u + H + 1);
        advance(ci);
      }
      cp_async_commit();
#pragma unroll
      for (int k = H - 1; k > 0; --k) hist[k] = hist[k - 1];
      hist[0] = meta_issued;
    }
    cp_async_wait_all();  // no copy of ours may land after we leave
    if (aborted) {
      bad |= QSA_STATUS_TIMEOUT;
      // Bulk copies are not covered by the wait above: before leaving, wait
      // (bounded again) for the last STAGES tiles' full barriers, whose phases
      // complete when their bytes have landed (phases complete in order, so
      // earlier uses of a stage are then done too).  A test stall issued none.
      if (C::BULK && !p.stall && tid == 0)
        for (int o = max(0, ckv.o - S); o < ckv.o; ++o)
          if (!mbar_wait(smem_addr(&s_full[o % S]), (uint32_t)((o / S) & 1))) break;
    }
    if (bad) atomicOr(p.status, bad);
    return;
  }

  // =========================================================================
  // consumers
  // =========================================================================
  const int hh = rw / C::WPH, kp = rw % C::WPH;
  auto cta_of = [&](int64_t x) {  // owner of tile x
    if constexpr (SCAN) return (int)(((x + 1) * s_rg.G - 1) / s_rg.R);
    else return (int)(((x + 1) * sp.G - 1) / sp.T);
  };
  // tiles before unit u and before u + 1, for the first and last unit in range
  // (the only ones another CTA can share)
  auto unit_lo = [&](int u) -> int64_t {
    if constexpr (SCAN) return u == u_first ? s_rg.P_first : s_rg.P_last;
    else return (int64_t)u * VT;
  };
  auto unit_hi = [&](int u) -> int64_t {
    if constexpr (SCAN) return u == u_last ? s_rg.P_last_end : s_rg.P_first_end;
    else return (int64_t)(u + 1) * VT;
  };
  auto first_cta = [&](int u) { return cta_of(unit_lo(u)); };
  auto contributors = [&](int u) {
    if (SCAN && u != u_first && u != u_last) return 1;
    return cta_of(unit_hi(u) - 1) - first_cta(u) + 1;
  };
  // A shared unit's partial records: two per CTA, slot 0 for the CTA's first
  // unit and slot 1 for its last.  Every contributor after a unit's first
  // starts its range inside that unit, so only the first one can hold the
  // unit in slot 1 (when its range starts before the unit).
  auto own_record = [&](int u) { return p.ws_partial + ((int64_t)2 * blockIdx.x + (u == u_first ? 0 : 1)) * sp.rec_floats; };
  auto record_of = [&](int c0, int c, int u) {  // contributor c0 + c of unit u
    int slot = 0;
    if (c == 0) {
      const int64_t start = SCAN ? (int64_t)c0 * s_rg.R / s_rg.G : (int64_t)c0 * sp.T / sp.G;
      slot = start == unit_lo(u) ? 0 : 1;
    }
    return p.ws_partial + ((int64_t)2 * (c0 + c) + slot) * sp.rec_floats;
  };
  const int ctid = tid - PT;
  // the epilogue buffer, or, when there is none, the stage ring, which only the
  // final merge of shared units uses, after every stage has been consumed
  float* epi = C::EPI_FLOATS ? epi_buf : reinterpret_cast<float*>(smem);

  uint32_t qf[NT][C::KSTEPS][2], qn[NT][C::KSTEPS][2];
  auto load_q = [&](int u, int r, uint32_t (&dst)[NT][C::KSTEPS][2]) {
    const int h = (u - (u / sp.NG) * sp.NG) * HPU + hh;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int head = nt * 8 + gid;
      const bool live = head < p.group;
      const unsigned char* qrow =
          p.q + (((int64_t)r * p.nq + (int64_t)h * p.group + (live ? head : 0)) * C::D) * C::ELEM;
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        const int e0 = KIND == kBF16 ? ks * 16 + 2 * tig : ks * 32 + 4 * tig;
        const int e1 = KIND == kBF16 ? e0 + 8 : e0 + 16;
        dst[nt][ks][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + e0 * C::ELEM)) : 0u;
        dst[nt][ks][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + e1 * C::ELEM)) : 0u;
      }
    }
  };
  float m_run[NT][2], l_run[NT][2], o[8][NT][4];
  auto reset_state = [&]() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    }
  };
  const int a_row = (lane & 7) + ((lane >> 3) & 1) * 8, a_col = ((lane >> 4) & 1) * 16;
  const int t_row = (lane & 7) + ((lane >> 4) & 1) * 8, t_col = ((lane >> 3) & 1) * 16;

  // A tile of this warp: its MSL 16-key slices.  The scores of every slice
  // come first (independent MMA chains), then one softmax update over all of
  // the warp's keys in the tile (one max reduction and one rescale of O per
  // tile, not per slice), then P.V for every slice; the stage is released
  // after the last V read.
  constexpr int MSL = C::MSL;
  constexpr bool TWO_CHAINS = MSL == 1;  // a lone slice splits its K steps over two accumulators
  auto consume_tile = [&](int kt, int ord) {
    const uint32_t empty = smem_addr(&s_empty[ord % S]);
    const int slot = (ord & (RT - 1)) * TILE;
    const unsigned char* sb = smem + (ord % S) * C::STAGE_BYTES;
    bool vA[MSL], vB[MSL], any[MSL];
    float sc[MSL][NT][4];
#pragma unroll
    for (int sl = 0; sl < MSL; ++sl) {
      const int k0 = kp * C::KPW + sl * 16;
      const int kA = k0 + gid, kB = kA + 8;
      vA[sl] = kA < kt && s_off[slot + kA] != kInvalidOff;
      vB[sl] = kB < kt && s_off[slot + kB] != kInvalidOff;
      any[sl] = __any_sync(0xffffffffu, vA[sl] || vB[sl]);
      float s2[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[sl][nt][c] = s2[nt][c] = 0.f;
      if (any[sl]) {
        const uint32_t kbase = smem_addr(sb) + k0 * C::SROW + hh * C::ROWB + a_row * C::SROW + a_col;
        uint32_t kf[C::KSTEPS][4];
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS; ++ks) ldsm_x4(kbase + ks * 32, kf[ks]);
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS; ++ks)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float (&acc)[4] = (TWO_CHAINS && (ks & 1)) ? s2[nt] : sc[sl][nt];
            if constexpr (KIND == kBF16) mma_bf16(acc, kf[ks], qf[nt][ks][0], qf[nt][ks][1]);
            else mma_e4m3(acc, kf[ks], qf[nt][ks][0], qf[nt][ks][1]);
          }
        if constexpr (TWO_CHAINS) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[sl][nt][c] += s2[nt][c];
        }
      }
    }
    bool any_tile = false;
#pragma unroll
    for (int sl = 0; sl < MSL; ++sl) any_tile |= any[sl];
    uint32_t pb[MSL][NT][2];
    if (any_tile) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pv[MSL][4];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float mx = -CUDART_INF_F;
#pragma unroll
          for (int sl = 0; sl < MSL; ++sl) {
            sc[sl][nt][c] = vA[sl] ? sc[sl][nt][c] * p.scale_log2 : -CUDART_INF_F;
            sc[sl][nt][2 + c] = vB[sl] ? sc[sl][nt][2 + c] * p.scale_log2 : -CUDART_INF_F;
            mx = fmaxf(mx, fmaxf(sc[sl][nt][c], sc[sl][nt][2 + c]));
          }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(m_run[nt][c], mx);
          const float muse = mnew == -CUDART_INF_F ? 0.f : mnew;
          const float alpha = exp2_fast(m_run[nt][c] - muse);
          float lsum = 0.f;
#pragma unroll
          for (int sl = 0; sl < MSL; ++sl) {
            const float p0 = exp2_fast(sc[sl][nt][c] - muse), p1 = exp2_fast(sc[sl][nt][2 + c] - muse);
            pv[sl][c] = p0;
            pv[sl][2 + c] = p1;
            lsum += p0 + p1;
          }
          l_run[nt][c] = l_run[nt][c] * alpha + lsum;
          m_run[nt][c] = mnew;
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              o[mt][nt][c] *= alpha;
              o[mt][nt][2 + c] *= alpha;
            }
          }
        }
#pragma unroll
        for (int sl = 0; sl < MSL; ++sl) {
          const uint32_t top = KIND == kBF16 ? pack_bf16(pv[sl][0], pv[sl][1]) : pack_f16(pv[sl][0], pv[sl][1]);
          const uint32_t bot = KIND == kBF16 ? pack_bf16(pv[sl][2], pv[sl][3]) : pack_f16(pv[sl][2], pv[sl][3]);
          pb[sl][nt][0] = movmatrix_t(top);
          pb[sl][nt][1] = movmatrix_t(bot);
        }
      }
#pragma unroll
      for (int sl = 0; sl < MSL; ++sl) {
        if (!any[sl]) continue;
        const int k0 = kp * C::KPW + sl * 16;
        const uint32_t vbase = smem_addr(sb + C::KV_BYTES) + k0 * C::SROW + hh * C::ROWB + t_row * C::SROW + t_col;
        if constexpr (KIND == kBF16) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a[4];
            ldsm_x4_t(vbase + mt * 32, a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16(o[mt][nt], a, pb[sl][nt][0], pb[sl][nt][1]);
          }
        } else {
#pragma unroll
          for (int pr = 0; pr < 4; ++pr) {
            // e4m3 rows are read as byte pairs: the transposing ldmatrix hands this
            // thread (key 2tig, 2tig+1) x (d 2gid, 2gid+1) of each 16-byte column
            // block; output rows of an M tile are d = 16mt + 2gid and 16mt + 2gid + 1
            uint32_t r4[4];
            ldsm_x4_t(vbase + pr * 32, r4);
            uint32_t ae[4], ao[4];
            const uint32_t q0 = __byte_perm(r4[0], 0, 0x3120), q1 = __byte_perm(r4[1], 0, 0x3120);
            const uint32_t q2 = __byte_perm(r4[2], 0, 0x3120), q3 = __byte_perm(r4[3], 0, 0x3120);
            e4m3x4_to_f16x2x2(q0, ae[0], ae[1]);
            e4m3x4_to_f16x2x2(q2, ae[2], ae[3]);
            e4m3x4_to_f16x2x2(q1, ao[0], ao[1]);
            e4m3x4_to_f16x2x2(q3, ao[2], ao[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              mma_f16(o[2 * pr][nt], ae, pb[sl][nt][0], pb[sl][nt][1]);
              mma_f16(o[2 * pr + 1][nt], ao, pb[sl][nt][0], pb[sl][nt][1]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty);
  };

  // End of unit u: output (unit owned by this CTA) or this CTA's partial
  // record.  A warp that owns its head writes from registers; warps sharing a
  // head merge in shared memory first.
  uint32_t first_ticket = 0xFFFFFFFFu;  // consumer thread 0: ticket taken for u_first
  int pend_last = -1;                   // shared unit still to arrive on at the end
  auto finish = [&](int u, bool row_ok) {
    const int G = p.group, D = C::D;
    const int q = u / sp.NG;
    const int r = SCAN ? s_meta[mslot(u) + 4] : p.total_q - 1 - q, hg = u - q * sp.NG;
    const bool own = contributors(u) == 1;
    float* rec = own ? nullptr : own_record(u);
    const int64_t stride = partial_stride(G, D);
    float lsum[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float l = l_run[nt][c];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        lsum[nt][c] = l;
      }
    if constexpr (C::PAIR) {
      // the second warp of each head hands its (m, l, O) to the first, half
      // of head_dim per round; the first rescales both to the common max
      float* bo = epi;                     // [4][GP][D/2]
      float* bm = epi + 4 * GP * (D / 2);  // [4][GP]
      float* bl = bm + 4 * GP;             // [4][GP]
      float a0[NT][2], a1[NT][2];
      if (kp == 1 && gid == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            bm[hh * GP + nt * 8 + 2 * tig + c] = m_run[nt][c];
            bl[hh * GP + nt * 8 + 2 * tig + c] = lsum[nt][c];
          }
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        if (kp == 1) {
#pragma unroll
          for (int mt = half * 4; mt < half * 4 + 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const int head = nt * 8 + 2 * tig + (c4 & 1);
                const int d = (KIND == kBF16 ? mt * 16 + gid + (c4 >> 1) * 8 : mt * 16 + 2 * gid + (c4 >> 1)) - half * (D / 2);
                bo[(hh * GP + head) * (D / 2) + d] = o[mt][nt][c4];
              }
        }
        role_sync(2, C::CT);
        if (kp == 0) {
          if (half == 0) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int head = nt * 8 + 2 * tig + c;
                const float m1 = bm[hh * GP + head], l1 = bl[hh * GP + head];
                const float M = fmaxf(m_run[nt][c], m1);
                a0[nt][c] = M == -CUDART_INF_F ? 0.f : exp2f(m_run[nt][c] - M);
                a1[nt][c] = M == -CUDART_INF_F ? 0.f : exp2f(m1 - M);
                lsum[nt][c] = lsum[nt][c] * a0[nt][c] + l1 * a1[nt][c];
                m_run[nt][c] = M;
              }
          }
#pragma unroll
          for (int mt = half * 4; mt < half * 4 + 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const int head = nt * 8 + 2 * tig + (c4 & 1);
                const int d = (KIND == kBF16 ? mt * 16 + gid + (c4 >> 1) * 8 : mt * 16 + 2 * gid + (c4 >> 1)) - half * (D / 2);
                o[mt][nt][c4] = o[mt][nt][c4] * a0[nt][c4 & 1] + bo[(hh * GP + head) * (D / 2) + d] * a1[nt][c4 & 1];
              }
        }
        role_sync(2, C::CT);
      }
    }
    if constexpr (C::WPH == 1 || C::PAIR) {
      const int h = hg * HPU + hh;
      const int64_t out0 = ((int64_t)r * p.nq + (int64_t)h * G) * D;
      float* part = own ? nullptr : rec + hh * stride;
      if (!C::PAIR || kp == 0)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int head = nt * 8 + 2 * tig + c;
          if (head >= G) continue;
          const bool live = row_ok && m_run[nt][c] != -CUDART_INF_F;
          const float inv = live ? 1.f / lsum[nt][c] : 0.f;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int hi = 0; hi < 2; ++hi) {
              const int d = KIND == kBF16 ? mt * 16 + gid + hi * 8 : mt * 16 + 2 * gid + hi;
              const float v = o[mt][nt][2 * hi + c];
              if (own) store_out(p, out0 + (int64_t)head * D + d, live ? v * inv : 0.f);
              else part[head * D + d] = v;
            }
          if (!own && gid == 0) {
            part[G * D + head] = m_run[nt][c];
            part[G * D + G + head] = lsum[nt][c];
          }
        }
    } else {
      float* sm_o = epi;
      float* sm_m = epi + 4 * GP * C::D;
      float* sm_l = sm_m + 4 * GP;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          if (gid == 0) {
            sm_m[rw * GP + nt * 8 + 2 * tig + c] = m_run[nt][c];
            sm_l[rw * GP + nt * 8 + 2 * tig + c] = lsum[nt][c];
          }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int head = nt * 8 + 2 * tig + (c & 1);
            const int d = KIND == kBF16 ? mt * 16 + gid + (c >> 1) * 8 : mt * 16 + 2 * gid + (c >> 1);
            sm_o[(rw * GP + head) * C::D + d] = o[mt][nt][c];
          }
      role_sync(2, C::CT);
      const int64_t out0 = ((int64_t)r * p.nq + (int64_t)hg * HPU * G) * D;
      for (int idx = ctid; idx < HPU * G * D; idx += C::CT) {
        const int h2 = idx / (G * D), rem = idx - h2 * G * D, i = rem / D, d = rem - i * D;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < C::WPH; ++k) M = fmaxf(M, sm_m[(h2 * C::WPH + k) * GP + i]);
        float L = 0.f, O = 0.f;
        if (M != -CUDART_INF_F) {
#pragma unroll
          for (int k = 0; k < C::WPH; ++k) {
            const int w = h2 * C::WPH + k;
            const float e = exp2f(sm_m[w * GP + i] - M);
            L += sm_l[w * GP + i] * e;
            O += sm_o[(w * GP + i) * D + d] * e;
          }
        }
        if (own) {
          store_out(p, out0 + idx, row_ok && M != -CUDART_INF_F ? O / L : 0.f);
        } else {
          float* part = rec + h2 * stride;
          part[rem] = O;
          if (d == 0) {
            part[G * D + i] = M;
            part[G * D + G + i] = L;
          }
        }
      }
      role_sync(2, C::CT);  // the epilogue buffer is free again
    }
    if (!own) {
      // publish the partial; arrive on the unit's ticket now when it is this
      // CTA's first unit (the CTA before finishes it late, so it is rarely
      // the last arrival) and keep the answer for the end of the range
      __threadfence();
      role_sync(2, C::CT);
      if (u == u_first && u != u_last) {
        if (ctid == 0) first_ticket = atomicAdd(p.ws_ticket + u, 1u);
      } else {
        pend_last = u;
      }
    }
    reset_state();
  };

  // main loop: wait for a tile, consume it (releasing its stage), finish units
  auto first_rows = [&](int u) { return SCAN ? unit_row(p, sp, u) : p.total_q - 1 - u / sp.NG; };
  load_q(u_first, first_rows(u_first), qf);
  if (u_first < u_last) load_q(u_first + 1, first_rows(u_first + 1), qn);
  reset_state();
  int u = u_first, j = jlo_first, n = 0, jl = 0, ord = 0;
  bool entered = false, row_ok = false, aborted = false;
  while (true) {
    const bool ok = mbar_wait(smem_addr(&s_full[ord % S]), (uint32_t)((ord / S) & 1), p.stall ? kStallSpins : kSpinLimit);
    if (role_any(2, C::CT, !ok)) {  // a give-up by any consumer is every consumer's decision
      aborted = true;
      break;
    }
    if (!entered) {  // the unit's meta was published with its first tile
      n = unit_n(u);
      jl = unit_jl(u, n);
      row_ok = s_meta[mslot(u) + 2] >= 0;
      entered = true;
    }
    consume_tile(keys_in(n, j), ord);
    ++ord;
    if (j < jl) {
      ++j;
      continue;
    }
    finish(u, row_ok);
    if (u >= u_last) break;
    ++u;
    j = 0;
    entered = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int ks = 0; ks < C::KSTEPS; ++ks) {
        qf[nt][ks][0] = qn[nt][ks][0];
        qf[nt][ks][1] = qn[nt][ks][1];
      }
    // unit u + 1's meta (its row) arrived with the first tile of unit u - 1
    if (u + 1 <= u_last) load_q(u + 1, SCAN ? s_meta[mslot(u + 1) + 4] : p.total_q - 1 - (u + 1) / sp.NG, qn);
  }
  if (aborted) {
    // A give-up still arrives on the ticket of every shared unit this CTA
    // contributes to and has not arrived on yet, so that each ticket reads
    // zero again after its last arrival; a ticket this CTA takes last is
    // re-armed without a merge (the call reports QSA_STATUS_TIMEOUT and its
    // output is undefined).
    if (ctid == 0) {
      atomicOr(p.status, QSA_STATUS_TIMEOUT);
      if (contributors(u_first) > 1) {
        const uint32_t t = first_ticket != 0xFFFFFFFFu ? first_ticket : atomicAdd(p.ws_ticket + u_first, 1u);
        if (t == (uint32_t)(contributors(u_first) - 1)) p.ws_ticket[u_first] = 0u;
      }
      if (u_last != u_first && contributors(u_last) > 1 &&
          atomicAdd(p.ws_ticket + u_last, 1u) == (uint32_t)(contributors(u_last) - 1))
        p.ws_ticket[u_last] = 0u;
    }
    return;
  }

  // Shared units: arrive on the last one's ticket, then merge every shared
  // unit this CTA arrived on last (no CTA ever waits for another).
  if (ctid == 0) {
    s_merge[0] = s_merge[1] = -1;
    if (first_ticket != 0xFFFFFFFFu && first_ticket == (uint32_t)(contributors(u_first) - 1)) s_merge[0] = u_first;
    if (pend_last >= 0 && atomicAdd(p.ws_ticket + pend_last, 1u) == (uint32_t)(contributors(pend_last) - 1))
      s_merge[1] = pend_last;
  }
  role_sync(2, C::CT);
  for (int k = 0; k < 2; ++k) {
    const int um = s_merge[k];
    if (um < 0) continue;
    __threadfence();
    const int G = p.group, D = C::D, K = contributors(um), c0 = first_cta(um);
    const int q = um / sp.NG;
    const int r = SCAN ? unit_row(p, sp, um) : p.total_q - 1 - q, hg = um - q * sp.NG;
    const int64_t stride = partial_stride(G, D);
    const float* rec0 = record_of(c0, 0, um);
    const float* rec1 = record_of(c0, 1, um);  // contributors 1.. are 2 * rec_floats apart
    auto rec_c = [&](int c) { return c == 0 ? rec0 : rec1 + (int64_t)2 * (c - 1) * sp.rec_floats; };
    // online merge over the contributors, four records' loads in flight at a time
    for (int q4 = ctid; q4 < HPU * G * D / 4; q4 += C::CT) {
      const int idx = q4 * 4, h2 = idx / (G * D), rem = idx - h2 * G * D, i = rem / D;
      float M = -CUDART_INF_F, L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int cb = 0; cb < K; cb += 4) {
        float mm[4], ll[4];
        float4 oo[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (cb + c < K) {
            const float* part = rec_c(cb + c) + h2 * stride;
            mm[c] = __ldcg(part + G * D + i);
            ll[c] = __ldcg(part + G * D + G + i);
            oo[c] = __ldcg(reinterpret_cast<const float4*>(part + rem));
          } else {
            mm[c] = -CUDART_INF_F;
            ll[c] = 0.f;
            oo[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float Mn = fmaxf(M, mm[c]);
          if (Mn == -CUDART_INF_F) continue;  // nothing seen yet
          const float a = exp2f(M - Mn), b = exp2f(mm[c] - Mn);
          acc.x = acc.x * a + oo[c].x * b;
          acc.y = acc.y * a + oo[c].y * b;
          acc.z = acc.z * a + oo[c].z * b;
          acc.w = acc.w * a + oo[c].w * b;
          L = L * a + ll[c] * b;
          M = Mn;
        }
      }
      const float inv = M != -CUDART_INF_F ? 1.f / L : 0.f;
      const int64_t ob = ((int64_t)r * p.nq + (int64_t)(hg * HPU + h2) * G) * D + rem;
      store_out(p, ob, acc.x * inv);
      store_out(p, ob + 1, acc.y * inv);
      store_out(p, ob + 2, acc.z * inv);
      store_out(p, ob + 3, acc.w * inv);
    }
    if (ctid == 0) p.ws_ticket[um] = 0u;
  }
}

template <int KIND, int NT, int HPU, bool SCAN>
cudaError_t launch_stream_t(const Params& p, const StreamPlan& sp, cudaStream_t s) {
  using C = StreamCfg<KIND, NT, HPU>;
  static std::atomic<unsigned char> configured[kMaxTrackedDevices] = {};
  const cudaError_t e = ensure_dynamic_smem(configured, stream_kernel<KIND, NT, HPU, SCAN>, C::SMEM);
  if (e != cudaSuccess) return e;
  if (sp.G == 0) return cudaSuccess;
  stream_kernel<KIND, NT, HPU, SCAN><<<sp.G, C::THREADS, C::SMEM, s>>>(p, sp);
  return cudaGetLastError();
}

// Instantiations for one element type and one split (each in its own
// translation unit, so that they compile in parallel).
template <int KIND, bool SCAN>
cudaError_t launch_stream_kind(const Params& p, const StreamPlan& sp, cudaStream_t s) {
  const bool nt2 = p.group > 8;
  switch (sp.HPU) {
    case 8: return nt2 ? cudaErrorInvalidValue : launch_stream_t<KIND, 1, 8, SCAN>(p, sp, s);
    case 4: return nt2 ? launch_stream_t<KIND, 2, 4, SCAN>(p, sp, s) : launch_stream_t<KIND, 1, 4, SCAN>(p, sp, s);
    case 2: return nt2 ? launch_stream_t<KIND, 2, 2, SCAN>(p, sp, s) : launch_stream_t<KIND, 1, 2, SCAN>(p, sp, s);
    default: return nt2 ? launch_stream_t<KIND, 2, 1, SCAN>(p, sp, s) : launch_stream_t<KIND, 1, 1, SCAN>(p, sp, s);
  }
}

}  // namespace qsa
