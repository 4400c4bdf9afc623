// Internal declarations shared by libqsa's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "qsa.h"

namespace qsa {

// Everything a kernel needs, resolved on the host from the descriptors.
struct Params {
  void* out;                      // [total_q, nq, D] f32 | bf16
  const unsigned char* q;         // [total_q, nq, D] element bytes
  const uint32_t* row_offsets;    // [batch + 1]
  const unsigned char* kv;        // kv_blocks base
  const uint32_t* cache_lengths;  // [batch]
  const uint32_t* table;          // [batch, max_pages]
  const int32_t* indices;         // [total_q, W]
  const int32_t* counts;          // [total_q]
  uint32_t* status;               // device status word (atomicOr)
  float* ws_partial;              // split-K partials (splits > 1)
  uint32_t* ws_ticket;            // split-K arrival counters, one per (row, kv head)

  int64_t page_pitch_bytes;  // bytes from one page to the next
  int64_t k_layer_bytes;     // byte offset of [page, 0, layer_idx, 0, 0, 0] in a page
  int64_t v_minus_k_bytes;   // byte distance from a K row to its V row
  int64_t slot_bytes;        // num_kv_heads * D * elem
  int64_t head_bytes;        // D * elem

  int32_t total_q, batch, nq, nkv, group, D, P, W, max_pages;
  int32_t log2P;     // log2(page_size) when it is a power of two, else -1
  uint32_t num_pages;
  float scale_log2;  // scale * log2(e): the softmax runs in base 2
  int32_t out_bf16;
  int32_t splits;    // CTAs per (row, kv head)
  int32_t cluster;   // kernel 2, splits > 1: the bands of a unit run as one thread-block
                     // cluster and merge through distributed shared memory (no workspace)
  int32_t band;      // keys per split band (multiple of the key tile)
  // Block-granular selection (kernel 2 only): when `blocks` is set, key j of
  // (row r, kv head h) is slot j % P of logical block
  // blocks[(h * total_q + r) * topk + j / P] (-1: unused), attended when its
  // position is <= the row's position; W == topk * P and indices/counts are
  // unused.
  const int32_t* blocks;  // [nkv, total_q, topk] or nullptr
  int32_t topk;
  // Latent mode (kernel 2 only): when `comp` is set, the key list of row r is
  // its window (positions pos - window + 1 .. pos of the cache above) then
  // the entries comp[r, :] (-1 unused) of a second, entry-paged cache; W ==
  // window + num_comp.  Both caches have one head (head_bytes == 0: every
  // query-head group reads it); offsets into the second cache carry bit 31.
  const int32_t* comp;            // [total_q, num_comp] or nullptr
  const float* sinks;             // [nq] sink logits (natural log units) or nullptr
  const unsigned char* kv2;       // entry-paged cache base
  const uint32_t* table2;         // [batch, max_pages2]
  const uint32_t* cache_lengths2; // [batch] entries per sequence
  int64_t page_pitch_bytes2, k_layer_bytes2, v_minus_k_bytes2, slot_bytes2;
  int32_t num_comp, window, P2, max_pages2;
  uint32_t num_pages2;
  // Kernel 2's tile copies (when tma != 0): a 5-D tiled TMA map of the first
  // cache, innermost first: the elements of a 128-byte line, the lines of a
  // slot (stride 128 B), the P slots of a page (stride slot_bytes), the 2 x L
  // K/V planes (stride P * slot_bytes) and the pages (stride
  // page_pitch_bytes), with a box of one line of 64 slots and the 128-byte
  // swizzle.  tma_plane_k / tma_plane_v: the planes of layer_idx.
  int32_t tma, tma_plane_k, tma_plane_v;
  int32_t shallow;  // BF16 tile copies, group <= 8: the two-stage variant (three CTAs per SM)
  int32_t groups;   // latent mode, one band, group 16: a CTA serves four head groups (nkv = groups / 4)
  int32_t stall;    // kernel 3, tests only: producers issue no K/V copies and waits give up early
  int32_t umma;     // kernel 2: the tcgen05 consumer (BF16, tile-copy layout; tile copies where tma)
  // Kernel 4 (row groups over page tiles): a bitmap of each row's selected
  // positions (bit pos % 32 of word pos / 32), written by its first kernel,
  // and per-row flags (kRgDup, kRgOverflow).  tmap then holds a box of
  // rg_box slots (min(page_size, 128)) instead of kernel 2's 64.
  uint32_t* rg_bits;  // [total_q, rg_capw]
  int32_t* rg_flags;  // [total_q]
  int32_t rg_rows;    // query rows per group: 128 / group
  int32_t rg_capw;    // bitmap words per row (the positions the bitmaps cover / 32)
  int32_t rg_box;     // slots per tile copy
  int32_t rg_groups;  // most groups the call can have (grid size / num_kv_heads)
  CUtensorMap tmap;
};

// Kernel 4's row flags: the row repeats a position, or its sequence has more
// positions than the bitmaps cover.  A group with a flagged row takes the
// kernel's exact CUDA-core path.
constexpr int32_t kRgDup = 1, kRgOverflow = 2;

// Launch plan of the persistent stream-K kernel (computed on the host).
struct StreamPlan {
  int64_t T;          // most key tiles the units can hold (U * VT); the kernel splits the real ones
  int32_t U;          // units: query row x group of HPU kv heads
  int32_t VT;         // most tiles per unit (selection_width / TILE, rounded up)
  int32_t G;          // CTAs (one per SM at most)
  int32_t NG;         // kv-head groups per row (num_kv_heads / HPU)
  int32_t HPU;        // kv heads per unit: 4, 2 or 1
  int32_t rec_floats; // floats of one partial record (HPU heads)
  int32_t scan;       // 1: split the tiles that hold keys (a scan of the counts in
                      // every CTA) in interleaved row order; 0: split all U * VT
                      // tiles in row order, no scan (when U <= G)
};

// Keys per stage of the stream-K kernel for head_dim 128: 64 KB of K+V when
// units have four or eight kv heads (eight consumer warps, no epilogue
// buffer competing for shared memory), else 32 KB.
__host__ __device__ constexpr int stream_tile(int elem_bytes, int hpu) {
  return (hpu >= 4 ? 65536 : 32768) / (2 * hpu * 128 * elem_bytes);
}

// Element type tags.
enum Elem { kF32 = 0, kBF16 = 1, kE4M3 = 2 };

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_simt(const Params& p, int elem, cudaStream_t stream);
cudaError_t launch_mma_bf16(const Params& p, cudaStream_t stream);
cudaError_t launch_mma_e4m3(const Params& p, cudaStream_t stream);
// Block-key compression (one warp per output row).
struct CompressParams {
  unsigned char* out;              // [batch * max_blocks, head_dim], key element type
  const unsigned char* gamma;      // [head_dim]
  const unsigned char* freqs;      // [positions, rotary_dim]
  const int32_t* key_counts;       // [batch]
  const unsigned char* kv;         // kv_blocks base (one kv head)
  const uint32_t* table;           // [batch, max_pages]
  uint32_t* status;                // device status word
  int64_t page_pitch_bytes, k_layer_bytes, slot_bytes;
  int32_t batch, max_blocks, max_pages, P, ratio, rotary_dim;
  uint32_t num_pages;
  float eps;
};
cudaError_t launch_compress(const CompressParams& p, int elem, int freq_elem, int head_dim, cudaStream_t stream);

cudaError_t launch_stream_bf16(const Params& p, const StreamPlan& sp, cudaStream_t stream);
// Kernel 4: the bitmap kernel, then the row-group kernel (BF16, head_dim 128).
cudaError_t launch_rowgroup(const Params& p, cudaStream_t stream);
// Shared memory of kernel 4's bitmap kernel for rg_capw words per row.
constexpr int kRgMaxCapWords = 32768;  // 1 Mi positions, 128 KB
cudaError_t launch_stream_e4m3(const Params& p, const StreamPlan& sp, cudaStream_t stream);
cudaError_t launch_stream_bf16_scan(const Params& p, const StreamPlan& sp, cudaStream_t stream);
cudaError_t launch_stream_e4m3_scan(const Params& p, const StreamPlan& sp, cudaStream_t stream);
// CTAs of the tensor-core kernel that fit on one SM (for the split planner).
// (`tiles`: the variant with tile copies, used for block lists; `umma`: its
// tcgen05 consumer.)
int mma_ctas_per_sm_bf16(int group, bool tiles, bool umma);
int mma_ctas_per_sm_e4m3(int group, bool tiles, bool umma);
// Clusters of `splits` CTAs of the tensor-core kernel resident at once (0: none fit).
int mma_max_clusters_bf16(int group, int splits, bool tiles, bool umma);
int mma_max_clusters_e4m3(int group, int splits, bool tiles, bool umma);

// Floats of one split-K partial: o[group][D], m[group], l[group], padded to a
// multiple of 4 so every partial starts 16-byte aligned.
__host__ __device__ inline int64_t partial_stride(int64_t group, int64_t D) {
  return (group * (D + 2) + 3) / 4 * 4;
}

// Raises a kernel's dynamic shared-memory limit once per device.  `done` holds
// one flag per device ordinal, read and set atomically (host threads may race
// to set the attribute; setting it twice is harmless); ordinals past its end
// set the attribute on every launch.
constexpr int kMaxTrackedDevices = 256;
template <typename Kernel>
cudaError_t ensure_dynamic_smem(std::atomic<unsigned char> (&done)[kMaxTrackedDevices], Kernel kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxTrackedDevices;
  if (tracked && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) done[dev].store(1, std::memory_order_release);
  return e;
}

// Tensor-core kernel limits.
constexpr int kMmaTile = 64;      // keys per pipeline stage (16 per warp)
constexpr int kMmaMaxBand = 2048; // keys one CTA translates up front
constexpr int kMmaThreads = 128;
// Largest split count the fused split-K combine accepts (its per-split
// weights live in shared memory).
constexpr int kMaxSplits = 128;
// Largest split count merged inside one thread-block cluster (the portable
// cluster size).
constexpr int kMaxClusterSplits = 8;

}  // namespace qsa
