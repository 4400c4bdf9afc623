// Host side of libqsa: argument checks, launch planning, per-device state and
// the extern "C" entry points declared in qsa.h.
//
// The checks follow the QSASparseAttentionRaggedPaged page's contract ("Raises:
// Error: If the operand shapes disagree with the parameters"): every mismatch
// is reported before anything is launched, and nothing here reads device
// memory, synchronises or copies device -> host on the call path.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <string>

#include "qsa.h"
#include "qsa_internal.cuh"

namespace {

using qsa::Params;

thread_local std::string g_last_error;

// Drops the cached device address of the allocation-free entry point's
// scratch for one device (defined with that entry point below).
void noalloc_forget_device(int dev);

qsa_status fail(qsa_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

int elem_bytes(int dtype) {
  switch (dtype) {
    case QSA_F32: return 4;
    case QSA_BF16: return 2;
    case QSA_F8E4M3: return 1;
    case QSA_U32: return 4;
    case QSA_I32: return 4;
    default: return 0;
  }
}

int64_t numel(const qsa_tensor& t) {
  int64_t n = 1;
  for (int i = 0; i < t.ndim && i < 6; ++i) n *= t.shape[i];
  return n;
}

const char* dtype_name(int d) {
  switch (d) {
    case QSA_F32: return "F32";
    case QSA_BF16: return "BF16";
    case QSA_F8E4M3: return "F8E4M3";
    case QSA_U32: return "U32";
    case QSA_I32: return "I32";
    default: return "?";
  }
}

// Everything the checks resolve, and the launch plan.
struct Resolved {
  int elem = 0;  // qsa::Elem
  int64_t total_q = 0, nq = 0, D = 0, num_pages = 0, L = 0, P = 0, nkv = 0, batch = 0, max_pages = 0, W = 0;
  int64_t pitch = 0;  // elements between pages
  int out_bf16 = 0;
  int kernel = 0;  // 1 CUDA-core, 2 per-(row, kv head) tensor-core, 3 persistent stream-K, 4 row groups
  // max_cache_length + max_prompt_length as the caller passed them (-1: not
  // given); only kernel 4 depends on them, to size its bitmaps
  int64_t hint_ctx = -1;
  int rg_rows = 0, rg_capw = 0, rg_box = 0;  // kernel 4: rows per group, bitmap words per row, slots per copy
  int64_t rg_groups = 0;                     // kernel 4: most groups the call can have
  int splits = 1;
  int cluster = 0;  // kernel 2: the bands of a unit merge inside one thread-block cluster
  int tiles = 0;    // kernel 2: the variant with tile copies (block lists)
  int umma = 0;     // kernel 2: the tcgen05 consumer (implies the tile-copy layout)
  int groups = 0;   // kernel 2, latent mode: a CTA serves four head groups of a row
  int stall = 0;    // kernel 3, tests only: no K/V copies, early give-up (qsa_options.test_stall)
  int band = 0;
  int64_t ctas = 0;
  size_t ws_partial_bytes = 0, ws_bytes = 0;
  size_t ws_tickets = 0;
  qsa::StreamPlan sp{};
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True when the persistent kernel would have fewer than a quarter as many
// units (row x group of up to four kv heads) as the device has SMs: each unit
// then spreads over many CTAs whose short ranges cannot hide the dependent
// prologue, and the per-(row, kv head) kernel with split-K, several CTAs per
// SM, is faster.
int device_sms();

// Kv heads per unit of the persistent kernel: the forced value, else eight
// when num_kv_heads and group allow and the units still outnumber the SMs
// (prefill-like grids, whose gathers mostly hit L2: a 2 KB BF16 row per key
// moves about 1.5x the L2 bandwidth of a 1 KB one), else the largest of 4,
// 2, 1 that divides num_kv_heads (decode-like grids keep more, smaller units).
int64_t stream_heads_per_unit(const Resolved& R, const qsa_options* opt, int32_t group) {
  if (opt && opt->heads_per_unit > 0) return opt->heads_per_unit;
  if (R.nkv % 8 == 0 && group <= 8) {
    const int sms = device_sms();
    if (sms > 0 && R.total_q * (R.nkv / 8) > sms) return 8;
  }
  return R.nkv % 4 == 0 ? 4 : R.nkv % 2 == 0 ? 2 : 1;
}

bool few_stream_units(const Resolved& R, const qsa_options* opt, int32_t group) {
  const int64_t hpu = stream_heads_per_unit(R, opt, group);
  const int sms = device_sms();
  return sms > 0 && R.total_q * (R.nkv / hpu) * 4 < sms;
}

// Positions kernel 4's bitmaps cover: the hinted longest sequence rounded up
// to whole 128-position tiles.
int64_t rowgroup_positions(const Resolved& R) { return (R.hint_ctx + 127) / 128 * 128; }

// Why kernel 4 cannot run this call (nullptr: it can).  It serves BF16
// caches with head_dim 128, group 4, 8 or 16 (128 / group rows fill the
// tensor-core tile), pages of a power-of-two number of slots, at least 8 (a
// tile copy then starts on a 1024-byte swizzle boundary), and needs the
// length hints to size its bitmaps (at most kRgMaxCapWords words per row).
const char* rowgroup_unfit(const Resolved& R, int32_t group) {
  if (R.hint_ctx < 0)
    return "kernel 4 needs page_size, max_cache_length and max_prompt_length (this entry point has none; "
           "qsa_plan_ex takes them)";
  if (R.elem != qsa::kBF16 || R.D != 128) return "kernel 4 needs BF16 with head_dim 128";
  if (group != 4 && group != 8 && group != 16) return "kernel 4 needs group 4, 8 or 16";
  if (R.P < 8 || (R.P & (R.P - 1))) return "kernel 4 needs a power-of-two page_size of at least 8";
  if (rowgroup_positions(R) / 32 > qsa::kRgMaxCapWords)
    return "kernel 4 covers sequences of at most 1 Mi positions (max_cache_length + max_prompt_length)";
  return nullptr;
}

// Kernel 4 pays when the rows of a sequence are many (prefill) and their
// sequences short enough that walking every position in tiles costs no more
// than the rows' own selections: on average at least 128 / group rows per
// sequence (half the rows of one of its CTAs), and a hinted longest sequence
// of at most 128 / min(group, 8) x selection_width positions (the gathering
// kernels do more math per gathered byte as the group grows, so the bound
// tightens with it up to group 8; at group 16 on chunked prefill, a longest
// sequence of 9 x selection_width, kernel 4 still took 0.83 ms against
// kernel 3's 1.96).  Hints of zero read as "not given" (every sequence would
// then take the kernel's slow exact path).
bool rowgroup_pays(const Resolved& R, int32_t group) {
  const int64_t rows = 128 / group, span = 128 / std::min<int32_t>(group, 8);
  return R.hint_ctx > 0 && R.total_q >= rows * R.batch && R.hint_ctx <= span * R.W;
}

// Picks the kernel for a resolved call: for BF16 and FP8 with head_dim 128
// the persistent tensor-core kernel, or the per-(row, kv head) one when the
// persistent kernel would get few units, or the row-group kernel for
// prefill-like BF16 calls it serves; the CUDA-core kernel otherwise (or as
// forced).
qsa_status choose_kernel(Resolved& R, int32_t group, const qsa_options* opt) {
  const bool mma_ok = (R.elem == qsa::kBF16 || R.elem == qsa::kE4M3) && R.D == 128;
  const bool simt_ok = group <= 8 || group == 16;
  const int want = opt ? opt->kernel : 0;
  if (want == 4) {
    const char* why = rowgroup_unfit(R, group);
    if (why) return fail(QSA_ERR_UNSUPPORTED, why);
    R.kernel = 4;
  } else if (want == 2 || want == 3) {
    if (!mma_ok) return fail(QSA_ERR_UNSUPPORTED, "tensor-core kernels need BF16 or F8E4M3 with head_dim 128");
    R.kernel = want;
  } else if (want == 1) {
    if (!simt_ok) return fail(QSA_ERR_UNSUPPORTED, "CUDA-core kernel runs groups 1..8 and 16");
    R.kernel = 1;
  } else if (want == 0) {
    R.kernel = mma_ok ? 3 : 1;
    if (R.kernel == 3 && few_stream_units(R, opt, group)) R.kernel = 2;
    if (R.kernel == 3 && !(opt && (opt->ctas > 0 || opt->heads_per_unit != 0 || opt->test_stall)) &&
        !rowgroup_unfit(R, group) && rowgroup_pays(R, group))
      R.kernel = 4;
    if (R.kernel == 1 && !simt_ok) return fail(QSA_ERR_UNSUPPORTED, "CUDA-core kernel runs groups 1..8 and 16");
  } else {
    return fail(QSA_ERR_ARG, "options.kernel must be 0, 1, 2, 3 or 4");
  }
  if (opt && (opt->splits < 0 || opt->ctas < 0)) return fail(QSA_ERR_ARG, "options.splits and options.ctas must be >= 0");
  if (R.kernel != 2 && opt && opt->splits > 1) return fail(QSA_ERR_UNSUPPORTED, "only kernel 2 takes options.splits");
  if (R.kernel != 3 && opt && opt->ctas > 0) return fail(QSA_ERR_UNSUPPORTED, "only kernel 3 takes options.ctas");
  if (opt && opt->heads_per_unit != 0) {
    const int h = opt->heads_per_unit;
    if (h != 1 && h != 2 && h != 4 && h != 8) return fail(QSA_ERR_ARG, "options.heads_per_unit must be 0, 1, 2, 4 or 8");
    if (R.kernel != 3) return fail(QSA_ERR_UNSUPPORTED, "only kernel 3 takes options.heads_per_unit");
    if (R.nkv % h) return fail(QSA_ERR_ARG, "options.heads_per_unit must divide num_kv_heads");
    if (h == 8 && group > 8) return fail(QSA_ERR_UNSUPPORTED, "units of eight kv heads need group <= 8");
  }
  if (opt && opt->test_stall && R.kernel != 3) return fail(QSA_ERR_UNSUPPORTED, "only kernel 3 takes options.test_stall");
  if (opt && (opt->tcgen05 < -1 || opt->tcgen05 > 1)) return fail(QSA_ERR_ARG, "options.tcgen05 must be -1, 0 or 1");
  if (opt && opt->tcgen05 == 1) {
    if (R.kernel != 2) return fail(QSA_ERR_UNSUPPORTED, "only kernel 2 takes options.tcgen05");
    if (R.elem != qsa::kBF16) return fail(QSA_ERR_UNSUPPORTED, "the tcgen05 consumer reads BF16 caches");
  }
  return QSA_OK;
}

qsa_status check_args(const qsa_tensor& output, const qsa_tensor& q, const qsa_tensor& offs, const qsa_tensor& kv,
                      int64_t page_stride, const qsa_tensor& cache_lengths, const qsa_tensor& table,
                      uint32_t layer_idx, const qsa_tensor& indices, const qsa_tensor& counts, int32_t group,
                      const qsa_options* opt, Resolved& R) {
  // ranks
  struct {
    const qsa_tensor* t;
    int ndim;
    const char* name;
  } ranks[] = {{&output, 3, "output"},        {&q, 3, "q"},
               {&offs, 1, "input_row_offsets"}, {&kv, 6, "kv_blocks"},
               {&cache_lengths, 1, "cache_lengths"}, {&table, 2, "kv_lookup_table"},
               {&indices, 2, "token_indices"}, {&counts, 1, "counts"}};
  for (auto& x : ranks) {
    if (x.t->ndim != x.ndim)
      return fail(QSA_ERR_SHAPE, std::string(x.name) + ": rank " + std::to_string(x.t->ndim) + ", expected " +
                                     std::to_string(x.ndim));
    for (int i = 0; i < x.ndim; ++i)
      if (x.t->shape[i] < 0) return fail(QSA_ERR_SHAPE, std::string(x.name) + ": negative extent");
  }
  // element types
  if (q.dtype != QSA_F32 && q.dtype != QSA_BF16 && q.dtype != QSA_F8E4M3)
    return fail(QSA_ERR_DTYPE, std::string("q: element type ") + dtype_name(q.dtype) + " is not F32, BF16 or F8E4M3");
  if (kv.dtype != q.dtype)
    return fail(QSA_ERR_DTYPE, std::string("kv_blocks: element type ") + dtype_name(kv.dtype) + " differs from q (" +
                                   dtype_name(q.dtype) + ")");
  if (output.dtype != QSA_F32 && output.dtype != QSA_BF16)
    return fail(QSA_ERR_DTYPE, "output: element type must be F32 or BF16");
  if (offs.dtype != QSA_U32) return fail(QSA_ERR_DTYPE, "input_row_offsets: element type must be U32");
  if (cache_lengths.dtype != QSA_U32) return fail(QSA_ERR_DTYPE, "cache_lengths: element type must be U32");
  if (table.dtype != QSA_U32) return fail(QSA_ERR_DTYPE, "kv_lookup_table: element type must be U32");
  if (indices.dtype != QSA_I32) return fail(QSA_ERR_DTYPE, "token_indices: element type must be I32");
  if (counts.dtype != QSA_I32) return fail(QSA_ERR_DTYPE, "counts: element type must be I32");

  // extents
  R.total_q = q.shape[0];
  R.nq = q.shape[1];
  R.D = q.shape[2];
  R.num_pages = kv.shape[0];
  R.L = kv.shape[2];
  R.P = kv.shape[3];
  R.nkv = kv.shape[4];
  R.batch = cache_lengths.shape[0];
  R.max_pages = table.shape[1];
  R.W = indices.shape[1];
  for (int i = 0; i < 3; ++i)
    if (output.shape[i] != q.shape[i]) return fail(QSA_ERR_SHAPE, "output: shape differs from q");
  if (kv.shape[1] != 2) return fail(QSA_ERR_SHAPE, "kv_blocks: axis 1 must have extent 2 (K, V)");
  if (kv.shape[5] != R.D) return fail(QSA_ERR_SHAPE, "kv_blocks: head_dim differs from q");
  if (group < 1) return fail(QSA_ERR_SHAPE, "group must be >= 1");
  if (R.nkv < 1 || R.nq != (int64_t)group * R.nkv)
    return fail(QSA_ERR_SHAPE, "num_q_heads (" + std::to_string(R.nq) + ") != group (" + std::to_string(group) +
                                   ") * num_kv_heads (" + std::to_string(R.nkv) + ")");
  if (offs.shape[0] != R.batch + 1) return fail(QSA_ERR_SHAPE, "input_row_offsets: extent must be batch + 1");
  if (table.shape[0] != R.batch) return fail(QSA_ERR_SHAPE, "kv_lookup_table: first extent must be batch");
  if (indices.shape[0] != R.total_q) return fail(QSA_ERR_SHAPE, "token_indices: first extent must be total_q");
  if (counts.shape[0] != R.total_q) return fail(QSA_ERR_SHAPE, "counts: extent must be total_q");
  if (R.batch == 0 && R.total_q > 0) return fail(QSA_ERR_SHAPE, "query rows without any sequence (batch == 0)");
  if (R.P < 1 || R.L < 1) return fail(QSA_ERR_SHAPE, "kv_blocks: page_size and num_layers must be >= 1");

  // pointers
  if (!output.data && numel(output)) return fail(QSA_ERR_NULL, "output is NULL");
  if (!q.data && numel(q)) return fail(QSA_ERR_NULL, "q is NULL");
  if (!offs.data) return fail(QSA_ERR_NULL, "input_row_offsets is NULL");
  if (!kv.data && numel(kv)) return fail(QSA_ERR_NULL, "kv_blocks is NULL");
  if (!cache_lengths.data && numel(cache_lengths)) return fail(QSA_ERR_NULL, "cache_lengths is NULL");
  if (!table.data && numel(table)) return fail(QSA_ERR_NULL, "kv_lookup_table is NULL");
  if (!indices.data && numel(indices)) return fail(QSA_ERR_NULL, "token_indices is NULL");
  if (!counts.data && numel(counts)) return fail(QSA_ERR_NULL, "counts is NULL");

  // scalars
  if ((int64_t)layer_idx >= R.L)
    return fail(QSA_ERR_ARG, "layer_idx " + std::to_string(layer_idx) + " >= num_layers " + std::to_string(R.L));
  const int64_t packed = 2 * R.L * R.P * R.nkv * R.D;
  if (page_stride != -1 && page_stride < packed)
    return fail(QSA_ERR_ARG, "page_stride must be -1 (packed) or >= the packed page size " + std::to_string(packed));
  R.pitch = page_stride == -1 ? packed : page_stride;
  R.elem = q.dtype == QSA_F32 ? qsa::kF32 : q.dtype == QSA_BF16 ? qsa::kBF16 : qsa::kE4M3;
  R.out_bf16 = output.dtype == QSA_BF16;
  const int eb = elem_bytes(q.dtype);

  // what this build can run
  if (R.D != 64 && R.D != 128) return fail(QSA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (group > 16) return fail(QSA_ERR_UNSUPPORTED, "group must be <= 16");
  if ((R.pitch * eb) % 16) return fail(QSA_ERR_UNSUPPORTED, "page_stride * element size must be a multiple of 16 bytes");
  if (!aligned16(kv.data) || !aligned16(q.data) || !aligned16(output.data))
    return fail(QSA_ERR_UNSUPPORTED, "q, output and kv_blocks must be 16-byte aligned");
  if (R.num_pages > 0xFFFFFFFFLL) return fail(QSA_ERR_UNSUPPORTED, "more than 2^32 - 1 pages");
  const double kv_bytes = ((double)(R.num_pages > 0 ? R.num_pages - 1 : 0) * R.pitch + packed) * eb;
  if (kv_bytes >= 68719476736.0 - 16.0) return fail(QSA_ERR_UNSUPPORTED, "kv_blocks larger than 64 GiB");
  if (R.total_q > 0x7FFFFFFF || R.W > 0x7FFFFFFF || R.batch > 0x7FFFFFFF || R.max_pages > 0x7FFFFFFF)
    return fail(QSA_ERR_UNSUPPORTED, "an extent exceeds 2^31 - 1");
  if (R.nq * R.D * R.total_q > ((int64_t)1 << 40)) return fail(QSA_ERR_UNSUPPORTED, "q larger than 2^40 elements");

  const qsa_status s = choose_kernel(R, group, opt);
  if (s == QSA_OK && R.kernel == 4 && R.num_pages == 0) {
    // kernel 4 copies whole pages: with no page at all, every position is bad
    // and kernel 3 reports them
    if (opt && opt->kernel == 4) return fail(QSA_ERR_UNSUPPORTED, "kernel 4 needs a cache of at least one page");
    R.kernel = 3;
  }
  return s;
}

// Split-K scratch of one (device, stream): f32 partials (contents never need
// to survive a call) and the per-(row, kv head) arrival tickets, which must
// read 0 at the start of every call: each is zeroed when allocated and re-armed
// by the last CTA that used it, so they live in their own buffer.
struct Workspace {
  void* partial = nullptr;
  size_t partial_bytes = 0;
  uint32_t* tickets = nullptr;
  size_t ticket_count = 0;
};

struct DeviceState {
  uint32_t* status = nullptr;
  std::map<void*, Workspace> workspaces;  // keyed by stream
  int sms = 0;
  int occ[2][2][2][2] = {};  // [bf16, e4m3][nt - 1][tile copies][tcgen05 consumer]
  // resident clusters of s CTAs of the tensor-core kernel ([bf16, e4m3][nt - 1][tile copies][s]; -1 unknown)
  int clusters[2][2][2][2][qsa::kMaxClusterSplits + 1];
  DeviceState() {
    for (auto& a : clusters)
      for (auto& b : a)
        for (auto& c : b)
          for (auto& u : c)
            for (int& d : u) d = -1;
  }
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;

// SM count of the current device (cached per device); 0 when unknown.
int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.sms && cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    st.sms = 0;
  }
  return st.sms;
}

qsa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(QSA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Kernel 2's consumer: the tcgen05 one (scores and output in tensor memory,
// BF16, the tile-copy stage layout) when forced with options.tcgen05 = 1,
// the mma.sync one when forced with -1 or left to choose.
qsa_status choose_consumer(Resolved& R, const qsa_options* opt) {
  const int want = opt ? opt->tcgen05 : 0;
  if (want < -1 || want > 1) return fail(QSA_ERR_ARG, "options.tcgen05 must be -1, 0 or 1");
  R.umma = 0;
  if (want == 1) {
    if (R.kernel != 2) return fail(QSA_ERR_UNSUPPORTED, "only kernel 2 takes options.tcgen05");
    if (R.elem != qsa::kBF16) return fail(QSA_ERR_UNSUPPORTED, "the tcgen05 consumer reads BF16 caches");
    R.umma = 1;
    R.tiles = 1;
  }
  return QSA_OK;
}

// Launch plan of the tensor-core kernel: CTAs per (row, kv head).
qsa_status plan_launch(Resolved& R, int32_t group, const qsa_options* opt, int dev) {
  {
    const qsa_status s = choose_consumer(R, opt);
    if (s != QSA_OK) return s;
  }
  R.splits = 1;
  R.band = qsa::kMmaTile;
  if (R.kernel == 4) {
    // Row groups: 256 / group rows of a sequence per CTA and kv head (two
    // 128-row tensor-core tiles); the sequences' groups number at most
    // ceil(total_q / rows) + batch.  The workspace holds each row's bitmap and
    // its flags.
    R.rg_rows = 256 / group;
    R.rg_capw = (int)(rowgroup_positions(R) / 32);
    R.rg_box = (int)std::min<int64_t>(R.P, 128);
    R.rg_groups = (R.total_q + R.rg_rows - 1) / R.rg_rows + std::min(R.batch, R.total_q);
    R.ctas = R.rg_groups * R.nkv;
    if (R.ctas > 0x7FFFFFFF) return fail(QSA_ERR_UNSUPPORTED, "kernel 4: more than 2^31 - 1 CTAs");
    R.ws_partial_bytes = ((size_t)R.total_q * R.rg_capw * 4 + 255) / 256 * 256 + ((size_t)R.total_q * 4 + 255) / 256 * 256;
    R.ws_tickets = 0;
    R.ws_bytes = R.ws_partial_bytes;
    return QSA_OK;
  }
  if (R.kernel == 1) {
    R.ctas = R.total_q * R.nkv;
    R.ws_bytes = R.ws_partial_bytes = 0;
    return QSA_OK;
  }
  if (R.kernel == 3) {
    // Persistent stream-K: units of HPU adjacent kv heads, TILE keys per
    // 32 KB stage, one CTA per SM over equal ranges of virtual tiles.
    qsa::StreamPlan& sp = R.sp;
    sp.HPU = (int32_t)stream_heads_per_unit(R, opt, group);
    sp.NG = (int32_t)(R.nkv / sp.HPU);
    const int64_t tile = qsa::stream_tile(R.elem == qsa::kBF16 ? 2 : 1, sp.HPU);
    sp.VT = (int32_t)std::max<int64_t>(1, (R.W + tile - 1) / tile);
    sp.U = (int32_t)(R.total_q * sp.NG);
    sp.T = (int64_t)sp.U * sp.VT;
    int64_t G = opt && opt->ctas > 0 ? opt->ctas : 0;
    if (!G) {
      std::lock_guard<std::mutex> lk(g_mu);
      DeviceState& st = g_dev[dev];
      if (!st.sms) {
        const cudaError_t e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
      }
      G = st.sms;
      // Units no more than the SMs: a whole number of CTAs per unit, so that
      // no CTA's range straddles two units and every unit merges the same
      // number of parts (one CTA per unit merges nothing), provided that
      // keeps at least 80 % of the SMs busy (decode, 128 units on 152 SMs:
      // 95 -> 91 us on 128 CTAs).
      if (sp.U > 0 && sp.U <= G) {
        const int64_t whole = (G / sp.U) * sp.U;
        if (5 * whole >= 4 * G) G = whole;
      }
    }
    G = std::min<int64_t>(G, sp.T);
    sp.G = (int32_t)std::max<int64_t>(G, 1);
    // With more units than CTAs, split the tiles that hold keys (the kernel
    // scans the counts); with fewer, each unit spreads over CTAs anyway and
    // the scan's extra dependent read costs more than the balance gains.
    sp.scan = sp.U > sp.G ? 1 : 0;
    sp.rec_floats = (int32_t)(sp.HPU * qsa::partial_stride(group, R.D));
    R.splits = 1;
    R.ctas = sp.G;
    R.ws_partial_bytes = ((size_t)2 * sp.G * sp.rec_floats * 4 + 255) / 256 * 256;
    R.ws_tickets = (size_t)sp.U;
    R.ws_bytes = R.ws_partial_bytes + R.ws_tickets * 4;
    return QSA_OK;
  }
  const int64_t T = qsa::kMmaTile;
  const int64_t min_splits = R.W > 0 ? (R.W + qsa::kMmaMaxBand - 1) / qsa::kMmaMaxBand : 1;
  int64_t splits;
  if (opt && opt->splits > 0) {
    splits = opt->splits;
    if (splits < min_splits)
      return fail(QSA_ERR_ARG, "options.splits below " + std::to_string(min_splits) + " for this selection width");
    if (splits > qsa::kMaxSplits) return fail(QSA_ERR_ARG, "options.splits above " + std::to_string(qsa::kMaxSplits));
  }
  const int kk = R.elem == qsa::kBF16 ? 0 : 1, knt = group <= 8 ? 0 : 1;
  // resident clusters of s bands (s <= kMaxClusterSplits), queried once per device
  auto clusters_of = [&](int64_t s) -> int {
    std::lock_guard<std::mutex> lk(g_mu);
    int& c = g_dev[dev].clusters[kk][knt][R.tiles][R.umma][s];
    if (c < 0)
      c = kk == 0 ? qsa::mma_max_clusters_bf16(group, (int)s, R.tiles != 0, R.umma != 0)
                  : qsa::mma_max_clusters_e4m3(group, (int)s, R.tiles != 0, R.umma != 0);
    return c;
  };
  if (!(opt && opt->splits > 0)) {
    int sms = 0, occ = 0;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      DeviceState& st = g_dev[dev];
      if (!st.sms) {
        const cudaError_t e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
      }
      int& o = st.occ[kk][knt][R.tiles][R.umma];
      if (!o)
        o = kk == 0 ? qsa::mma_ctas_per_sm_bf16(group, R.tiles != 0, R.umma != 0)
                    : qsa::mma_ctas_per_sm_e4m3(group, R.tiles != 0, R.umma != 0);
      sms = st.sms;
      occ = st.occ[kk][knt][R.tiles][R.umma];
    }
    const int64_t units = R.total_q * R.nkv;
    // Wave model: a CTA costs about (kPrologueKeys + keys it gathers); the
    // launch costs waves x that.  Pick the split count that minimises it.
    // Split counts that merge inside a cluster have as many slots as whole
    // clusters fit on the device.
    constexpr int64_t kPrologueKeys = 384;
    const int64_t most = std::max<int64_t>(min_splits, std::min<int64_t>(qsa::kMaxSplits, (R.W + T - 1) / T));
    splits = min_splits;
    double best = -1.0;
    for (int64_t sp = min_splits; units > 0 && sp <= most; ++sp) {
      int64_t slots = (int64_t)sms * occ;
      if (sp > 1 && sp <= qsa::kMaxClusterSplits) {
        const int nc = clusters_of(sp);
        if (nc > 0) slots = (int64_t)nc * sp;
      }
      const int64_t waves = (units * sp + slots - 1) / slots;
      const double cost = (double)waves * (double)(kPrologueKeys + (R.W + sp - 1) / sp);
      if (best < 0 || cost < best) {
        best = cost;
        splits = sp;
      }
    }
  }
  if (R.W > 0) {
    int64_t band = (R.W + splits - 1) / splits;
    band = (band + T - 1) / T * T;
    if (!(opt && opt->splits > 0)) splits = (R.W + band - 1) / band;  // drop bands that start past W
    R.band = (int)band;
  }
  R.splits = (int)splits;
  R.cluster = splits > 1 && splits <= qsa::kMaxClusterSplits && clusters_of(splits) > 0 ? 1 : 0;
  R.ctas = R.total_q * R.nkv * R.splits;
  if (R.splits > 1 && !R.cluster) {
    const int64_t units = R.total_q * R.nkv;
    R.ws_partial_bytes = ((size_t)(units * R.splits * qsa::partial_stride(group, R.D) * 4) + 255) / 256 * 256;
    R.ws_tickets = (size_t)units;
    R.ws_bytes = R.ws_partial_bytes + (size_t)units * 4;
  } else {
    R.ws_bytes = R.ws_partial_bytes = 0;
  }
  return QSA_OK;
}

// Grows (never shrinks) the split-K workspace of (dev, stream) to hold
// `partial_bytes` of partials and `tickets` arrival tickets.  Under the lock.
qsa_status ensure_workspace(DeviceState& st, void* stream, size_t partial_bytes, size_t tickets, Workspace** out) {
  Workspace& ws = st.workspaces[stream];
  const bool grow_p = ws.partial_bytes < partial_bytes, grow_t = ws.ticket_count < tickets;
  if (grow_p || grow_t) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing((cudaStream_t)stream, &cs);
    if (cs != cudaStreamCaptureStatusNone)
      return fail(QSA_ERR_CUDA, "split-K workspace must be reserved (qsa_reserve_workspace) before stream capture");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);  // the old buffers may still be in use
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  }
  if (grow_p) {
    if (ws.partial) cudaFree(ws.partial);
    ws.partial = nullptr;
    ws.partial_bytes = 0;
    cudaError_t e = cudaMalloc(&ws.partial, partial_bytes);
    if (e != cudaSuccess) {
      ws.partial = nullptr;
      return cuda_fail(e, "cudaMalloc(split-K partials)");
    }
    ws.partial_bytes = partial_bytes;
  }
  if (grow_t) {
    if (ws.tickets) cudaFree(ws.tickets);
    ws.tickets = nullptr;
    ws.ticket_count = 0;
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, tickets * sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(split-K tickets)");
    e = cudaMemset(p, 0, tickets * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      cudaFree(p);
      return cuda_fail(e, "cudaMemset(split-K tickets)");
    }
    ws.tickets = static_cast<uint32_t*>(p);
    ws.ticket_count = tickets;
  }
  *out = &ws;
  return QSA_OK;
}

qsa_status ensure_status(DeviceState& st) {
  if (st.status) return QSA_OK;
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, 256);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(status)");
  e = cudaMemset(p, 0, 256);
  if (e != cudaSuccess) {
    cudaFree(p);
    return cuda_fail(e, "cudaMemset(status)");
  }
  st.status = static_cast<uint32_t*>(p);
  return QSA_OK;
}

// Everything after the plan: status word and workspace of (device, stream),
// the kernel parameters, and the launch.  `indices`/`counts` carry a token
// selection, or `blocks`/`topk` a block selection (kernel 2 only).
// The latent mode's second source and sinks (see Params).
// The driver's tensor-map encoder, looked up once through the runtime (no
// link-time dependency on the driver library); null when unavailable.
using TensorMapEncode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                     const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
TensorMapEncode tensor_map_encoder() {
  static const TensorMapEncode fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      f = nullptr;
    }
    return reinterpret_cast<TensorMapEncode>(f);
  }();
  return fn;
}

// Kernel 2's tile copies: encodes the 5-D map of the first cache described
// with qsa::Params::tmap (p.tma = 1), or leaves p.tma = 0 when a tile copy
// cannot describe the layout (pages shorter than a tile, strides that are
// not multiples of 16 bytes, ...): every tile then takes 16-byte copies.
// Kernel 4 asks for boxes of min(page_size, 128) slots and needs the map.
void encode_tile_map(Params& p, const void* kv, int elem, int64_t num_pages, int box_slots = qsa::kMmaTile) {
  p.tma = 0;
  const TensorMapEncode encode = tensor_map_encoder();
  const int64_t plane = (int64_t)p.P * p.slot_bytes;
  if (!encode || elem == qsa::kF32 || p.P < box_slots || p.slot_bytes <= 0 || p.slot_bytes % 128 != 0 ||
      p.k_layer_bytes % plane != 0 || p.v_minus_k_bytes % plane != 0 || p.page_pitch_bytes % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(kv) & 15u) != 0 || num_pages <= 0 || num_pages > 0xFFFFFFFFll)
    return;
  const cuuint64_t dims[5] = {elem == qsa::kBF16 ? 64u : 128u, (cuuint64_t)(p.slot_bytes / 128), (cuuint64_t)p.P,
                              (cuuint64_t)(2 * (p.v_minus_k_bytes / plane)), (cuuint64_t)num_pages};
  const cuuint64_t strides[4] = {128u, (cuuint64_t)p.slot_bytes, (cuuint64_t)plane, (cuuint64_t)p.page_pitch_bytes};
  const cuuint32_t box[5] = {(cuuint32_t)dims[0], 1u, (cuuint32_t)box_slots, 1u, 1u};
  const cuuint32_t estride[5] = {1u, 1u, 1u, 1u, 1u};
  const CUresult r = encode(&p.tmap, elem == qsa::kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
                            const_cast<void*>(kv), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B,
                            // L2 fills as wide as one head's row: 256 B (bf16, both lines are
                            // read) or 128 B (e4m3: a wider fill would bring in the next head's row)
                            elem == qsa::kBF16 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return;
  p.tma = 1;
  p.tma_plane_k = (int32_t)(p.k_layer_bytes / plane);
  p.tma_plane_v = (int32_t)((p.k_layer_bytes + p.v_minus_k_bytes) / plane);
}

struct LatentArgs {
  const int32_t* comp;
  const float* sinks;
  const unsigned char* kv2;
  const uint32_t* table2;
  const uint32_t* cache_lengths2;
  int64_t pitch_bytes2, k_layer_bytes2, v_minus_k_bytes2, slot_bytes2;
  int32_t num_comp, window, P2, max_pages2;
  uint32_t num_pages2;
  // the window cache has one head whatever the number of query-head groups
  int64_t k_layer_bytes1, v_minus_k_bytes1, slot_bytes1;
};

qsa_status launch_planned(Resolved& R, const qsa_tensor& output, const qsa_tensor& q,
                          const qsa_tensor& input_row_offsets, const qsa_tensor& kv_blocks,
                          const qsa_tensor& cache_lengths, const qsa_tensor& kv_lookup_table, uint32_t layer_idx,
                          const int32_t* indices, const int32_t* counts, const int32_t* blocks, int32_t topk,
                          float scale, int32_t group, void* stream, int dev, const LatentArgs* lat = nullptr) {
  qsa_status s = QSA_OK;
  cudaError_t e = cudaSuccess;
  Params p;
  std::memset(&p, 0, sizeof(p));
  {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    s = ensure_status(st);
    if (s != QSA_OK) return s;
    p.status = st.status;
    if (R.ws_bytes > 0) {
      Workspace* ws = nullptr;
      s = ensure_workspace(st, stream, R.ws_partial_bytes, R.ws_tickets, &ws);
      if (s != QSA_OK) return s;
      p.ws_partial = static_cast<float*>(ws->partial);
      p.ws_ticket = ws->tickets;
    }
  }
  const int64_t eb = elem_bytes(q.dtype);
  p.out = output.data;
  p.q = static_cast<const unsigned char*>(q.data);
  p.row_offsets = static_cast<const uint32_t*>(input_row_offsets.data);
  p.kv = static_cast<const unsigned char*>(kv_blocks.data);
  p.cache_lengths = static_cast<const uint32_t*>(cache_lengths.data);
  p.table = static_cast<const uint32_t*>(kv_lookup_table.data);
  p.indices = indices;
  p.counts = counts;
  p.blocks = blocks;
  p.topk = topk;
  p.page_pitch_bytes = R.pitch * eb;
  p.k_layer_bytes = (int64_t)layer_idx * R.P * R.nkv * R.D * eb;
  p.v_minus_k_bytes = R.L * R.P * R.nkv * R.D * eb;
  p.slot_bytes = R.nkv * R.D * eb;
  p.head_bytes = R.D * eb;
  p.total_q = (int32_t)R.total_q;
  p.batch = (int32_t)R.batch;
  p.nq = (int32_t)R.nq;
  p.nkv = (int32_t)R.nkv;
  p.group = group;
  p.D = (int32_t)R.D;
  p.P = (int32_t)R.P;
  p.log2P = -1;
  for (int k = 0; k < 31; ++k)
    if ((int64_t)1 << k == R.P) p.log2P = k;
  p.W = (int32_t)R.W;
  p.max_pages = (int32_t)R.max_pages;
  p.num_pages = (uint32_t)R.num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;  // log2(e): softmax in base 2
  p.out_bf16 = R.out_bf16;
  p.splits = R.splits;
  p.cluster = R.cluster;
  p.groups = R.groups;
  p.stall = R.stall;
  p.umma = R.umma;
  p.band = R.band;
  if (lat) {
    p.comp = lat->comp;
    p.sinks = lat->sinks;
    p.kv2 = lat->kv2;
    p.table2 = lat->table2;
    p.cache_lengths2 = lat->cache_lengths2;
    p.page_pitch_bytes2 = lat->pitch_bytes2;
    p.k_layer_bytes2 = lat->k_layer_bytes2;
    p.v_minus_k_bytes2 = lat->v_minus_k_bytes2;
    p.slot_bytes2 = lat->slot_bytes2;
    p.num_comp = lat->num_comp;
    p.window = lat->window;
    p.P2 = lat->P2;
    p.max_pages2 = lat->max_pages2;
    p.num_pages2 = lat->num_pages2;
    p.k_layer_bytes = lat->k_layer_bytes1;
    p.v_minus_k_bytes = lat->v_minus_k_bytes1;
    p.slot_bytes = lat->slot_bytes1;
    p.head_bytes = 0;  // every query-head group reads the one latent head
  }

  if (R.kernel == 2 && R.tiles) {
    encode_tile_map(p, kv_blocks.data, R.elem, R.num_pages);
    // grids of eight or more CTAs per SM (prefill-like: many waves, gathers
    // mostly from L2) take the two-stage BF16 variant, three CTAs per SM;
    // shorter grids keep three stages
    int sms = 0;
    {
      std::lock_guard<std::mutex> lk(g_mu);
      sms = g_dev[dev].sms;
    }
    p.shallow = !R.umma && R.elem == qsa::kBF16 && sms > 0 && R.ctas >= 8 * (int64_t)sms ? 1 : 0;
  }

  if (R.kernel == 4) {
    p.rg_bits = reinterpret_cast<uint32_t*>(p.ws_partial);
    p.rg_flags = reinterpret_cast<int32_t*>(reinterpret_cast<unsigned char*>(p.ws_partial) +
                                            ((size_t)R.total_q * R.rg_capw * 4 + 255) / 256 * 256);
    p.rg_rows = R.rg_rows;
    p.rg_capw = R.rg_capw;
    p.rg_box = R.rg_box;
    p.rg_groups = (int32_t)R.rg_groups;
    encode_tile_map(p, kv_blocks.data, R.elem, R.num_pages, R.rg_box);
    if (!p.tma) return fail(QSA_ERR_CUDA, "kernel 4: the cache's TMA tensor map could not be encoded");
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (R.kernel == 4)
    e = qsa::launch_rowgroup(p, st);
  else if (R.kernel == 1)
    e = qsa::launch_simt(p, R.elem, st);
  else if (R.kernel == 2)
    e = R.elem == qsa::kBF16 ? qsa::launch_mma_bf16(p, st) : qsa::launch_mma_e4m3(p, st);
  else
    e = R.elem == qsa::kBF16 ? qsa::launch_stream_bf16(p, R.sp, st) : qsa::launch_stream_e4m3(p, R.sp, st);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return QSA_OK;
}

}  // namespace

extern "C" {

qsa_status qsa_sparse_attention_ragged_paged_ex(qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets,
                                                qsa_tensor kv_blocks, int64_t page_stride, qsa_tensor cache_lengths,
                                                qsa_tensor kv_lookup_table, uint32_t max_prompt_length,
                                                uint32_t max_cache_length, uint32_t layer_idx,
                                                qsa_tensor token_indices, qsa_tensor counts, float scale,
                                                int32_t group, void* stream, const qsa_options* options) {
  // Launch-sizing hints: kernel 4 sizes its bitmaps from them (a sequence
  // longer than they say is still served exactly, by that kernel's CUDA-core
  // path); the other kernels use host-known extents only.
  Resolved R;
  R.hint_ctx = (int64_t)max_cache_length + (int64_t)max_prompt_length;
  qsa_status s = check_args(output, q, input_row_offsets, kv_blocks, page_stride, cache_lengths, kv_lookup_table,
                            layer_idx, token_indices, counts, group, options, R);
  if (s != QSA_OK) return s;
  if (R.total_q == 0) return QSA_OK;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  s = plan_launch(R, group, options, dev);
  if (s != QSA_OK) return s;
  R.stall = options && options->test_stall ? 1 : 0;

  return launch_planned(R, output, q, input_row_offsets, kv_blocks, cache_lengths, kv_lookup_table, layer_idx,
                        static_cast<const int32_t*>(token_indices.data), static_cast<const int32_t*>(counts.data),
                        nullptr, 0, scale, group, stream, dev);
}

qsa_status qsa_sparse_attention_ragged_paged(qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets,
                                             qsa_tensor kv_blocks, int64_t page_stride, qsa_tensor cache_lengths,
                                             qsa_tensor kv_lookup_table, uint32_t max_prompt_length,
                                             uint32_t max_cache_length, uint32_t layer_idx, qsa_tensor token_indices,
                                             qsa_tensor counts, float scale, int32_t group, void* stream) {
  return qsa_sparse_attention_ragged_paged_ex(output, q, input_row_offsets, kv_blocks, page_stride, cache_lengths,
                                              kv_lookup_table, max_prompt_length, max_cache_length, layer_idx,
                                              token_indices, counts, scale, group, stream, nullptr);
}

qsa_status qsa_msa_attention_ragged_paged(qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets,
                                          qsa_tensor kv_blocks, int64_t page_stride, qsa_tensor cache_lengths,
                                          qsa_tensor kv_lookup_table, uint32_t max_prompt_length,
                                          uint32_t max_cache_length, uint32_t layer_idx, qsa_tensor d_indices,
                                          float scale, int32_t group, void* stream, const qsa_options* options) {
  (void)max_prompt_length;
  (void)max_cache_length;
  if (d_indices.ndim != 3) return fail(QSA_ERR_SHAPE, "d_indices: rank " + std::to_string(d_indices.ndim) + ", expected 3");
  if (d_indices.dtype != QSA_I32) return fail(QSA_ERR_DTYPE, "d_indices: element type must be I32");
  for (int i = 0; i < 3; ++i)
    if (d_indices.shape[i] < 0) return fail(QSA_ERR_SHAPE, "d_indices: negative extent");
  if (kv_blocks.ndim == 6 && d_indices.shape[0] != kv_blocks.shape[4])
    return fail(QSA_ERR_SHAPE, "d_indices: first extent must be num_kv_heads");
  if (q.ndim == 3 && d_indices.shape[1] != q.shape[0]) return fail(QSA_ERR_SHAPE, "d_indices: second extent must be total_q");
  if (!d_indices.data && numel(d_indices)) return fail(QSA_ERR_NULL, "d_indices is NULL");
  qsa_options opt;
  std::memset(&opt, 0, sizeof(opt));
  if (options) opt = *options;
  if (opt.kernel != 0 && opt.kernel != 2)
    return fail(QSA_ERR_UNSUPPORTED, "block lists run on the per-(row, kv head) tensor-core kernel (options.kernel 2)");
  opt.kernel = 2;
  const int64_t topk = d_indices.shape[2];
  const int64_t P = kv_blocks.ndim == 6 ? kv_blocks.shape[3] : 0;
  if (topk * P > 0x7FFFFFFF) return fail(QSA_ERR_UNSUPPORTED, "topk * page_size exceeds 2^31 - 1");
  // the shared checks see the block list as a token list of topk * page_size
  // keys per row with no counts (stand-ins that are never read)
  qsa_tensor keys = d_indices, cnt = d_indices;
  keys.ndim = 2;
  keys.shape[0] = q.ndim == 3 ? q.shape[0] : 0;
  keys.shape[1] = topk * P;
  cnt.ndim = 1;
  cnt.shape[0] = keys.shape[0];
  cnt.data = output.data;
  if (!keys.data) keys.data = output.data;
  Resolved R;
  qsa_status s = check_args(output, q, input_row_offsets, kv_blocks, page_stride, cache_lengths, kv_lookup_table,
                            layer_idx, keys, cnt, group, &opt, R);
  if (s != QSA_OK) return s;
  if (R.total_q == 0) return QSA_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  R.tiles = 1;  // listed blocks are whole pages: most key tiles are one tile copy
  s = plan_launch(R, group, &opt, dev);
  if (s != QSA_OK) return s;
  return launch_planned(R, output, q, input_row_offsets, kv_blocks, cache_lengths, kv_lookup_table, layer_idx,
                        nullptr, nullptr, static_cast<const int32_t*>(d_indices.data), (int32_t)topk, scale, group,
                        stream, dev);
}

qsa_status qsa_latent_attention_ragged_paged(qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets,
                                             qsa_tensor swa_blocks, int64_t swa_page_stride,
                                             qsa_tensor swa_cache_lengths, qsa_tensor swa_lookup_table,
                                             qsa_tensor comp_blocks, int64_t comp_page_stride,
                                             const uint32_t* comp_cache_lengths, const uint32_t* comp_lookup_table,
                                             int64_t comp_max_pages, uint32_t layer_idx, const int32_t* comp_indices,
                                             int64_t num_comp, const float* attn_sink, int32_t window, float scale,
                                             void* stream, const qsa_options* options) {
  struct {
    const qsa_tensor* t;
    int ndim;
    const char* name;
  } ranks[] = {{&output, 3, "output"}, {&q, 3, "q"}, {&input_row_offsets, 1, "input_row_offsets"},
               {&swa_blocks, 6, "swa_blocks"}, {&swa_cache_lengths, 1, "swa_cache_lengths"},
               {&swa_lookup_table, 2, "swa_lookup_table"}, {&comp_blocks, 6, "comp_blocks"}};
  for (auto& x : ranks) {
    if (x.t->ndim != x.ndim)
      return fail(QSA_ERR_SHAPE, std::string(x.name) + ": rank " + std::to_string(x.t->ndim) + ", expected " +
                                     std::to_string(x.ndim));
    for (int i = 0; i < x.ndim; ++i)
      if (x.t->shape[i] < 0) return fail(QSA_ERR_SHAPE, std::string(x.name) + ": negative extent");
  }
  if (q.dtype != QSA_BF16 && q.dtype != QSA_F8E4M3) return fail(QSA_ERR_UNSUPPORTED, "q must be BF16 or F8E4M3");
  if (swa_blocks.dtype != q.dtype || comp_blocks.dtype != q.dtype)
    return fail(QSA_ERR_DTYPE, "swa_blocks and comp_blocks must have q's element type");
  if (output.dtype != QSA_F32 && output.dtype != QSA_BF16) return fail(QSA_ERR_DTYPE, "output: F32 or BF16");
  if (input_row_offsets.dtype != QSA_U32 || swa_cache_lengths.dtype != QSA_U32 || swa_lookup_table.dtype != QSA_U32)
    return fail(QSA_ERR_DTYPE, "offsets, cache lengths and page tables must be U32");
  if (comp_max_pages < 0 || num_comp < 0) return fail(QSA_ERR_SHAPE, "comp_max_pages and num_comp must be >= 0");
  Resolved R;
  R.elem = q.dtype == QSA_BF16 ? qsa::kBF16 : qsa::kE4M3;
  R.total_q = q.shape[0];
  R.nq = q.shape[1];
  R.D = q.shape[2];
  R.batch = swa_cache_lengths.shape[0];
  R.num_pages = swa_blocks.shape[0];
  R.L = swa_blocks.shape[2];
  R.P = swa_blocks.shape[3];
  R.max_pages = swa_lookup_table.shape[1];
  for (int i = 0; i < 3; ++i)
    if (output.shape[i] != q.shape[i]) return fail(QSA_ERR_SHAPE, "output: shape differs from q");
  if (swa_blocks.shape[1] != 2 || comp_blocks.shape[1] != 2) return fail(QSA_ERR_SHAPE, "caches: axis 1 must be 2 (K, V)");
  if (swa_blocks.shape[4] != 1 || comp_blocks.shape[4] != 1) return fail(QSA_ERR_SHAPE, "caches: one latent head (axis 4 == 1)");
  if (swa_blocks.shape[5] != R.D || comp_blocks.shape[5] != R.D) return fail(QSA_ERR_SHAPE, "caches: head_dim differs from q");
  if (input_row_offsets.shape[0] != R.batch + 1) return fail(QSA_ERR_SHAPE, "input_row_offsets: extent must be batch + 1");
  if (swa_lookup_table.shape[0] != R.batch) return fail(QSA_ERR_SHAPE, "swa_lookup_table: first extent must be batch");
  if (R.batch == 0 && R.total_q > 0) return fail(QSA_ERR_SHAPE, "query rows without any sequence (batch == 0)");
  if (window < 0) return fail(QSA_ERR_ARG, "window must be >= 0");
  if ((int64_t)layer_idx >= R.L || (int64_t)layer_idx >= comp_blocks.shape[2])
    return fail(QSA_ERR_ARG, "layer_idx >= num_layers of a cache");
  if (R.P < 1 || comp_blocks.shape[3] < 1) return fail(QSA_ERR_SHAPE, "page sizes must be >= 1");
  const int64_t eb = elem_bytes(q.dtype), D = R.D, L2 = comp_blocks.shape[2], P2 = comp_blocks.shape[3];
  const int64_t packed1 = 2 * R.L * R.P * D, packed2 = 2 * L2 * P2 * D;
  if ((swa_page_stride != -1 && swa_page_stride < packed1) || (comp_page_stride != -1 && comp_page_stride < packed2))
    return fail(QSA_ERR_ARG, "page_stride must be -1 (packed) or >= the packed page size");
  R.pitch = swa_page_stride == -1 ? packed1 : swa_page_stride;
  const int64_t pitch2 = comp_page_stride == -1 ? packed2 : comp_page_stride;
  if (D != 128) return fail(QSA_ERR_UNSUPPORTED, "head_dim must be 128");
  // query-head groups of up to 16 on the one latent head
  const int64_t group = R.nq <= 16 ? R.nq : 16;
  if (R.nq < 1 || R.nq % group) return fail(QSA_ERR_UNSUPPORTED, "num_heads must be <= 16 or a multiple of 16");
  R.nkv = R.nq / group;
  R.W = (int64_t)window + num_comp;
  R.out_bf16 = output.dtype == QSA_BF16;
  if (R.W > 0x7FFFFFFF || R.total_q > 0x7FFFFFFF || comp_max_pages > 0x7FFFFFFF)
    return fail(QSA_ERR_UNSUPPORTED, "an extent exceeds 2^31 - 1");
  if ((R.pitch * eb) % 16 || (pitch2 * eb) % 16)
    return fail(QSA_ERR_UNSUPPORTED, "page_stride * element size must be a multiple of 16 bytes");
  const double kv1 = ((double)(R.num_pages > 0 ? R.num_pages - 1 : 0) * R.pitch + packed1) * eb;
  const double kv2 = ((double)(comp_blocks.shape[0] > 0 ? comp_blocks.shape[0] - 1 : 0) * pitch2 + packed2) * eb;
  if (kv1 >= 34359738368.0 - 16.0 || kv2 >= 34359738368.0 - 16.0)
    return fail(QSA_ERR_UNSUPPORTED, "a cache larger than 32 GiB");
  if (R.total_q > 0 && (!output.data || !q.data || !input_row_offsets.data || !swa_cache_lengths.data ||
                        !attn_sink || !comp_cache_lengths || (!comp_indices && num_comp) ||
                        (!comp_lookup_table && comp_max_pages) ||
                        (!swa_blocks.data && numel(swa_blocks)) || (!comp_blocks.data && numel(comp_blocks))))
    return fail(QSA_ERR_NULL, "a needed pointer is NULL");
  if (!aligned16(output.data) || !aligned16(q.data) || !aligned16(swa_blocks.data) || !aligned16(comp_blocks.data))
    return fail(QSA_ERR_UNSUPPORTED, "q, output and the caches must be 16-byte aligned");
  qsa_options opt;
  std::memset(&opt, 0, sizeof(opt));
  if (options) opt = *options;
  if (opt.kernel != 0 && opt.kernel != 2) return fail(QSA_ERR_UNSUPPORTED, "latent attention runs on kernel 2");
  if (opt.ctas != 0 || opt.splits < 0) return fail(QSA_ERR_ARG, "only options.splits applies");
  if (opt.tcgen05 == 1) return fail(QSA_ERR_UNSUPPORTED, "latent attention runs on the mma.sync consumer");
  opt.tcgen05 = -1;
  opt.kernel = 2;
  R.kernel = 2;
  if (R.total_q == 0) return QSA_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  qsa_status s = plan_launch(R, (int32_t)group, &opt, dev);
  if (s != QSA_OK) return s;
  // with one band and the 16-head groups in fours, a CTA serves four groups
  // of a row (one gather of each key for the four)
  if (R.splits == 1 && group == 16 && R.nkv % 4 == 0) {
    R.groups = 1;
    R.nkv /= 4;
    R.ctas = R.total_q * R.nkv;
  }
  LatentArgs lat;
  lat.comp = comp_indices;
  lat.sinks = attn_sink;
  lat.kv2 = static_cast<const unsigned char*>(comp_blocks.data);
  lat.table2 = comp_lookup_table;
  lat.cache_lengths2 = comp_cache_lengths;
  lat.pitch_bytes2 = pitch2 * eb;
  lat.k_layer_bytes2 = (int64_t)layer_idx * P2 * D * eb;
  lat.v_minus_k_bytes2 = L2 * P2 * D * eb;
  lat.slot_bytes2 = D * eb;
  lat.num_comp = (int32_t)num_comp;
  lat.window = window;
  lat.P2 = (int32_t)P2;
  lat.max_pages2 = (int32_t)comp_max_pages;
  lat.num_pages2 = (uint32_t)comp_blocks.shape[0];
  lat.k_layer_bytes1 = (int64_t)layer_idx * R.P * D * eb;
  lat.v_minus_k_bytes1 = R.L * R.P * D * eb;
  lat.slot_bytes1 = D * eb;
  return launch_planned(R, output, q, input_row_offsets, swa_blocks, swa_cache_lengths, swa_lookup_table, layer_idx,
                        nullptr, nullptr, nullptr, 0, scale, (int32_t)group, stream, dev, &lat);
}

qsa_status qsa_compress_keys_paged(qsa_tensor block_keys, qsa_tensor gamma, qsa_tensor freqs_cis,
                                   qsa_tensor key_counts, qsa_tensor kv_blocks, int64_t page_stride,
                                   qsa_tensor cache_lengths, qsa_tensor kv_lookup_table, uint32_t max_prompt_length,
                                   uint32_t max_cache_length, uint32_t layer_idx, int32_t ratio, int32_t rotary_dim,
                                   float eps, void* stream) {
  (void)max_prompt_length;
  (void)max_cache_length;
  struct {
    const qsa_tensor* t;
    int ndim;
    const char* name;
  } ranks[] = {{&block_keys, 2, "block_keys"}, {&gamma, 1, "gamma"}, {&freqs_cis, 2, "freqs_cis"},
               {&key_counts, 1, "key_counts"}, {&kv_blocks, 6, "kv_blocks"}, {&cache_lengths, 1, "cache_lengths"},
               {&kv_lookup_table, 2, "kv_lookup_table"}};
  for (auto& x : ranks) {
    if (x.t->ndim != x.ndim)
      return fail(QSA_ERR_SHAPE, std::string(x.name) + ": rank " + std::to_string(x.t->ndim) + ", expected " +
                                     std::to_string(x.ndim));
    for (int i = 0; i < x.ndim; ++i)
      if (x.t->shape[i] < 0) return fail(QSA_ERR_SHAPE, std::string(x.name) + ": negative extent");
  }
  if (kv_blocks.dtype != QSA_F32 && kv_blocks.dtype != QSA_BF16)
    return fail(QSA_ERR_DTYPE, "kv_blocks: the keys must be F32 or BF16");
  if (block_keys.dtype != kv_blocks.dtype || gamma.dtype != kv_blocks.dtype)
    return fail(QSA_ERR_DTYPE, "block_keys and gamma must have the keys' element type");
  if (freqs_cis.dtype != QSA_F32 && freqs_cis.dtype != QSA_BF16) return fail(QSA_ERR_DTYPE, "freqs_cis: F32 or BF16");
  if (key_counts.dtype != QSA_I32) return fail(QSA_ERR_DTYPE, "key_counts: element type must be I32");
  if (cache_lengths.dtype != QSA_U32 || kv_lookup_table.dtype != QSA_U32)
    return fail(QSA_ERR_DTYPE, "cache_lengths and kv_lookup_table must be U32");
  const int64_t batch = key_counts.shape[0], D = kv_blocks.shape[5], L = kv_blocks.shape[2], P = kv_blocks.shape[3];
  if (kv_blocks.shape[1] != 2) return fail(QSA_ERR_SHAPE, "kv_blocks: axis 1 must have extent 2 (K, V)");
  if (kv_blocks.shape[4] != 1) return fail(QSA_ERR_SHAPE, "kv_blocks: the index-key cache has one head (axis 4 == 1)");
  if (block_keys.shape[1] != D || gamma.shape[0] != D) return fail(QSA_ERR_SHAPE, "block_keys / gamma: head_dim differs from kv_blocks");
  if (cache_lengths.shape[0] != batch || kv_lookup_table.shape[0] != batch)
    return fail(QSA_ERR_SHAPE, "cache_lengths / kv_lookup_table: first extent must be batch");
  if (batch == 0 ? block_keys.shape[0] != 0 : block_keys.shape[0] % batch != 0)
    return fail(QSA_ERR_SHAPE, "block_keys: rows must be batch * max_blocks");
  const int64_t max_blocks = batch ? block_keys.shape[0] / batch : 0;
  if (ratio < 1) return fail(QSA_ERR_ARG, "ratio must be >= 1");
  if (ratio > 64) return fail(QSA_ERR_UNSUPPORTED, "ratio above 64 (a CTA stages at most 64 raw keys)");
  if (rotary_dim < 0 || rotary_dim > D || (rotary_dim & 1)) return fail(QSA_ERR_ARG, "rotary_dim must be even and <= head_dim");
  if (rotary_dim > 0 && freqs_cis.shape[1] != rotary_dim) return fail(QSA_ERR_SHAPE, "freqs_cis: second extent must be rotary_dim");
  if (rotary_dim > 0 && freqs_cis.shape[0] < max_blocks)
    return fail(QSA_ERR_SHAPE, "freqs_cis: needs a row per block (positions >= max_blocks)");
  if (!(eps >= 0.f)) return fail(QSA_ERR_ARG, "eps must be >= 0");
  if ((int64_t)layer_idx >= L) return fail(QSA_ERR_ARG, "layer_idx >= num_layers");
  const int eb = elem_bytes(kv_blocks.dtype);
  const int64_t packed = 2 * L * P * D;
  if (page_stride != -1 && page_stride < packed) return fail(QSA_ERR_ARG, "page_stride must be -1 or >= the packed page size");
  const int64_t pitch = page_stride == -1 ? packed : page_stride;
  if (D != 128 && D != 256) return fail(QSA_ERR_UNSUPPORTED, "head_dim must be 128 or 256");
  if ((pitch * eb) % 16) return fail(QSA_ERR_UNSUPPORTED, "page_stride * element size must be a multiple of 16 bytes");
  const int64_t rows = block_keys.shape[0];
  if (rows > 0 && (!block_keys.data || !gamma.data || !key_counts.data || (!kv_lookup_table.data && numel(kv_lookup_table)) ||
                   (!kv_blocks.data && numel(kv_blocks)) || (rotary_dim > 0 && !freqs_cis.data)))
    return fail(QSA_ERR_NULL, "a needed pointer is NULL");
  if (!aligned16(block_keys.data) || !aligned16(gamma.data) || !aligned16(kv_blocks.data))
    return fail(QSA_ERR_UNSUPPORTED, "block_keys, gamma and kv_blocks must be 16-byte aligned");
  if (rows > 0x7FFFFFFF || kv_blocks.shape[0] > 0xFFFFFFFFLL || kv_lookup_table.shape[1] > 0x7FFFFFFF)
    return fail(QSA_ERR_UNSUPPORTED, "an extent exceeds the supported range");
  if (rows == 0) return QSA_OK;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  qsa::CompressParams p;
  std::memset(&p, 0, sizeof(p));
  {
    std::lock_guard<std::mutex> lk(g_mu);
    qsa_status s = ensure_status(g_dev[dev]);
    if (s != QSA_OK) return s;
    p.status = g_dev[dev].status;
  }
  p.out = static_cast<unsigned char*>(block_keys.data);
  p.gamma = static_cast<const unsigned char*>(gamma.data);
  p.freqs = static_cast<const unsigned char*>(freqs_cis.data);
  p.key_counts = static_cast<const int32_t*>(key_counts.data);
  p.kv = static_cast<const unsigned char*>(kv_blocks.data);
  p.table = static_cast<const uint32_t*>(kv_lookup_table.data);
  p.page_pitch_bytes = pitch * eb;
  p.k_layer_bytes = (int64_t)layer_idx * P * D * eb;
  p.slot_bytes = D * eb;
  p.batch = (int32_t)batch;
  p.max_blocks = (int32_t)max_blocks;
  p.max_pages = (int32_t)kv_lookup_table.shape[1];
  p.P = (int32_t)P;
  p.ratio = ratio;
  p.rotary_dim = rotary_dim;
  p.num_pages = (uint32_t)kv_blocks.shape[0];
  p.eps = eps;
  e = qsa::launch_compress(p, kv_blocks.dtype == QSA_BF16 ? qsa::kBF16 : qsa::kF32,
                           freqs_cis.dtype == QSA_BF16 ? qsa::kBF16 : qsa::kF32, (int)D, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return QSA_OK;
}

}  // extern "C"

namespace {

// qsa_plan and qsa_plan_ex: the plan of a call with these extents (batch 0,
// page_size 0 and hint_ctx -1 when the caller does not give them).
qsa_status plan_extents(int32_t dtype, int64_t total_q, int64_t batch, int64_t num_kv_heads, int64_t head_dim,
                        int64_t page_size, int64_t selection_width, int32_t group, int64_t hint_ctx,
                        const qsa_options* options, int32_t* kernel, int32_t* splits, int64_t* ctas,
                        size_t* workspace_bytes) {
  Resolved R;
  if (dtype != QSA_F32 && dtype != QSA_BF16 && dtype != QSA_F8E4M3)
    return fail(QSA_ERR_DTYPE, "dtype must be F32, BF16 or F8E4M3");
  if (total_q < 0 || num_kv_heads < 1 || selection_width < 0 || group < 1 || batch < 0 || page_size < 0)
    return fail(QSA_ERR_SHAPE, "negative or empty extent");
  if (head_dim != 64 && head_dim != 128) return fail(QSA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (group > 16) return fail(QSA_ERR_UNSUPPORTED, "group must be <= 16");
  if (options && options->splits < 0) return fail(QSA_ERR_ARG, "options.splits must be >= 0");
  R.elem = dtype == QSA_F32 ? qsa::kF32 : dtype == QSA_BF16 ? qsa::kBF16 : qsa::kE4M3;
  R.total_q = total_q;
  R.batch = batch;
  R.nkv = num_kv_heads;
  R.D = head_dim;
  R.P = page_size;
  R.W = selection_width;
  R.hint_ctx = hint_ctx;
  qsa_status s = choose_kernel(R, group, options);
  if (s != QSA_OK) return s;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  R.tiles = options && options->block_lists && R.kernel == 2 ? 1 : 0;
  s = plan_launch(R, group, options, dev);
  if (s != QSA_OK) return s;
  if (kernel) *kernel = R.kernel;
  if (splits) *splits = R.splits;
  if (ctas) *ctas = R.ctas;
  if (workspace_bytes) *workspace_bytes = R.ws_bytes;
  return QSA_OK;
}

}  // namespace

extern "C" {

qsa_status qsa_plan(int32_t dtype, int64_t total_q, int64_t num_kv_heads, int64_t head_dim,
                    int64_t selection_width, int32_t group, const qsa_options* options, int32_t* kernel,
                    int32_t* splits, int64_t* ctas, size_t* workspace_bytes) {
  return plan_extents(dtype, total_q, 0, num_kv_heads, head_dim, 0, selection_width, group, -1, options, kernel,
                      splits, ctas, workspace_bytes);
}

qsa_status qsa_plan_ex(int32_t dtype, int64_t total_q, int64_t batch, int64_t num_kv_heads, int64_t head_dim,
                       int64_t page_size, int64_t selection_width, int32_t group, uint32_t max_prompt_length,
                       uint32_t max_cache_length, const qsa_options* options, int32_t* kernel, int32_t* splits,
                       int64_t* ctas, size_t* workspace_bytes) {
  if (total_q > 0 && batch < 1) return fail(QSA_ERR_SHAPE, "query rows without any sequence (batch == 0)");
  if (page_size < 1) return fail(QSA_ERR_SHAPE, "page_size must be >= 1");
  return plan_extents(dtype, total_q, batch, num_kv_heads, head_dim, page_size, selection_width, group,
                      (int64_t)max_cache_length + (int64_t)max_prompt_length, options, kernel, splits, ctas,
                      workspace_bytes);
}

qsa_status qsa_reserve_workspace(void* stream, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  qsa_status s = ensure_status(st);
  if (s != QSA_OK) return s;
  // `bytes` (qsa_plan's figure) covers the partials; size the tickets as if
  // all of it were tickets, which bounds any split of that figure
  Workspace* ws = nullptr;
  return bytes ? ensure_workspace(st, stream, bytes, bytes / sizeof(uint32_t) + 1, &ws) : QSA_OK;
}

qsa_status qsa_release_device_state(void) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  noalloc_forget_device(dev);  // the allocation-free entry point looks its scratch address up again
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) return QSA_OK;
  for (auto& kv : it->second.workspaces) {
    if (kv.second.partial) cudaFree(kv.second.partial);
    if (kv.second.tickets) cudaFree(kv.second.tickets);
  }
  if (it->second.status) cudaFree(it->second.status);
  g_dev.erase(it);
  return QSA_OK;
}

qsa_status qsa_read_device_status(void* stream, int32_t clear, uint32_t* flags) {
  if (!flags) return fail(QSA_ERR_NULL, "flags is NULL");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  uint32_t* status = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    qsa_status s = ensure_status(g_dev[dev]);
    if (s != QSA_OK) return s;
    status = g_dev[dev].status;
  }
  e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  e = cudaMemcpy(flags, status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  if (clear) {
    e = cudaMemset(status, 0, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
  }
  return QSA_OK;
}

const char* qsa_status_string(qsa_status s) {
  switch (s) {
    case QSA_OK: return "QSA_OK";
    case QSA_ERR_NULL: return "QSA_ERR_NULL";
    case QSA_ERR_SHAPE: return "QSA_ERR_SHAPE";
    case QSA_ERR_DTYPE: return "QSA_ERR_DTYPE";
    case QSA_ERR_UNSUPPORTED: return "QSA_ERR_UNSUPPORTED";
    case QSA_ERR_ARG: return "QSA_ERR_ARG";
    case QSA_ERR_CUDA: return "QSA_ERR_CUDA";
    default: return "QSA_ERR_UNKNOWN";
  }
}

const char* qsa_last_error_message(void) { return g_last_error.c_str(); }

int32_t qsa_version(void) { return (0 << 16) | 1; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot let a library call cudaMalloc: an engine that reserves
// nearly all of the device's memory for its own pools (KV cache, activations)
// at start-up and hands plugins only buffers it owns, or a serving loop that
// must not pay cudaMalloc/cudaFree's implicit device synchronisation.  For
// them qsa_sparse_attention_ragged_paged_noalloc runs the persistent stream-K
// kernel with its scratch (shared-unit partial records, arrival tickets and a
// fallback status word) in the fixed array below instead of a per-stream
// workspace.  The array is part of the library's device image, so every GPU
// that loads the library holds it until the process exits.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[QSA_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 64;
constexpr size_t kNoallocStatusBytes = 256;  // [0, 256): status word when the caller passes none

std::mutex g_noalloc_mu;
void* g_noalloc_base[kNoallocMaxDevices];  // device address of g_noalloc_scratch, per device

// Once per device, with that device current: the scratch array's device
// address.  In host code the name g_noalloc_scratch is only a stand-in for
// the symbol, so the address has to be asked for.
qsa_status noalloc_base(int dev, unsigned char** out) {
  // (a device reset drops the image and its symbols: qsa_release_device_state
  // forgets the address, and the next call looks it up again)
  if (dev < 0 || dev >= kNoallocMaxDevices)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_sparse_attention_ragged_paged_noalloc: device ordinal above 63");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_base[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_noalloc_base[dev] = ptr;
  }
  *out = static_cast<unsigned char*>(g_noalloc_base[dev]);
  return QSA_OK;
}

}  // namespace

namespace {

void noalloc_forget_device(int dev) {
  if (dev < 0 || dev >= kNoallocMaxDevices) return;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  g_noalloc_base[dev] = nullptr;
}

}  // namespace

extern "C" qsa_status qsa_sparse_attention_ragged_paged_noalloc(
    qsa_tensor output, qsa_tensor q, qsa_tensor input_row_offsets, qsa_tensor kv_blocks, int64_t page_stride,
    qsa_tensor cache_lengths, qsa_tensor kv_lookup_table, uint32_t max_prompt_length, uint32_t max_cache_length,
    uint32_t layer_idx, qsa_tensor token_indices, qsa_tensor counts, float scale, int32_t group, void* stream,
    uint32_t* status_flags) {
  (void)max_prompt_length;
  (void)max_cache_length;
  // argument errors first, before any CUDA call
  if (reinterpret_cast<uintptr_t>(status_flags) & 3u)
    return fail(QSA_ERR_ARG, "qsa_sparse_attention_ragged_paged_noalloc: status_flags must be 4-byte aligned");
  qsa_options opt;
  std::memset(&opt, 0, sizeof(opt));
  opt.kernel = 3;
  Resolved R;
  qsa_status s = check_args(output, q, input_row_offsets, kv_blocks, page_stride, cache_lengths, kv_lookup_table,
                            layer_idx, token_indices, counts, group, &opt, R);
  if (s != QSA_OK) return s;
  if (R.total_q == 0) return QSA_OK;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  s = plan_launch(R, group, &opt, dev);
  if (s != QSA_OK) return s;
  unsigned char* base = nullptr;
  s = noalloc_base(dev, &base);
  if (s != QSA_OK) return s;

  // scratch layout: status word | partial records | tickets
  const size_t ticket_bytes = (R.ws_tickets * sizeof(uint32_t) + 255) / 256 * 256;
  const size_t need = kNoallocStatusBytes + R.ws_partial_bytes + ticket_bytes;
  if (need > (size_t)QSA_NOALLOC_SCRATCH_BYTES)
    return fail(QSA_ERR_UNSUPPORTED,
                "qsa_sparse_attention_ragged_paged_noalloc: this call needs " + std::to_string(need) +
                    " bytes of scratch (total_q * num_kv_heads too large); the static scratch holds " +
                    std::to_string((size_t)QSA_NOALLOC_SCRATCH_BYTES) + " (use qsa_sparse_attention_ragged_paged)");
  float* partial = reinterpret_cast<float*>(base + kNoallocStatusBytes);
  uint32_t* tickets = reinterpret_cast<uint32_t*>(base + kNoallocStatusBytes + R.ws_partial_bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps whatever the last call left; tickets must start at zero
  e = cudaMemsetAsync(tickets, 0, R.ws_tickets * sizeof(uint32_t), st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static scratch tickets)");

  Params p;
  std::memset(&p, 0, sizeof(p));
  p.status = status_flags ? status_flags : reinterpret_cast<uint32_t*>(base);
  p.ws_partial = partial;
  p.ws_ticket = tickets;
  const int64_t eb = elem_bytes(q.dtype);
  p.out = output.data;
  p.q = static_cast<const unsigned char*>(q.data);
  p.row_offsets = static_cast<const uint32_t*>(input_row_offsets.data);
  p.kv = static_cast<const unsigned char*>(kv_blocks.data);
  p.cache_lengths = static_cast<const uint32_t*>(cache_lengths.data);
  p.table = static_cast<const uint32_t*>(kv_lookup_table.data);
  p.indices = static_cast<const int32_t*>(token_indices.data);
  p.counts = static_cast<const int32_t*>(counts.data);
  p.page_pitch_bytes = R.pitch * eb;
  p.k_layer_bytes = (int64_t)layer_idx * R.P * R.nkv * R.D * eb;
  p.v_minus_k_bytes = R.L * R.P * R.nkv * R.D * eb;
  p.slot_bytes = R.nkv * R.D * eb;
  p.head_bytes = R.D * eb;
  p.total_q = (int32_t)R.total_q;
  p.batch = (int32_t)R.batch;
  p.nq = (int32_t)R.nq;
  p.nkv = (int32_t)R.nkv;
  p.group = group;
  p.D = (int32_t)R.D;
  p.P = (int32_t)R.P;
  p.log2P = -1;
  for (int k = 0; k < 31; ++k)
    if ((int64_t)1 << k == R.P) p.log2P = k;
  p.W = (int32_t)R.W;
  p.max_pages = (int32_t)R.max_pages;
  p.num_pages = (uint32_t)R.num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;  // log2(e): softmax in base 2
  p.out_bf16 = R.out_bf16;
  p.splits = R.splits;
  p.band = R.band;
  e = R.elem == qsa::kBF16 ? qsa::launch_stream_bf16(p, R.sp, st) : qsa::launch_stream_e4m3(p, R.sp, st);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return QSA_OK;
}
