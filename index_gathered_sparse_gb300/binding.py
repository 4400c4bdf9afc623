"""Thin ctypes binding of libqsa (see include/qsa.h): same names as the C ABI.

Only argument marshalling happens here: tensors become ``qsa_tensor``
descriptors (device pointer, element type, shape) and the call goes straight
to the CUDA library.  There is no CPU or PyTorch fallback; a missing library
raises :class:`LibraryMissing`.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqsa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "qsa.h")

QSA_F32, QSA_BF16, QSA_F8E4M3, QSA_U32, QSA_I32 = range(5)
QSA_OK = 0
STATUS_NAMES = {0: "QSA_OK", 1: "QSA_ERR_NULL", 2: "QSA_ERR_SHAPE", 3: "QSA_ERR_DTYPE",
                4: "QSA_ERR_UNSUPPORTED", 5: "QSA_ERR_ARG", 6: "QSA_ERR_CUDA"}
QSA_STATUS_BAD_INDEX, QSA_STATUS_BAD_PAGE, QSA_STATUS_BAD_ROW, QSA_STATUS_TIMEOUT = 1, 2, 4, 8


class qsa_tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 6)]


class qsa_options(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("splits", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("block_lists", ctypes.c_int32), ("heads_per_unit", ctypes.c_int32), ("test_stall", ctypes.c_int32),
                ("tcgen05", ctypes.c_int32), ("reserved", ctypes.c_int32 * 1)]


class LibraryMissing(RuntimeError):
    pass


class QSAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def exported_names() -> list:
    """The entry points include/qsa.h declares."""
    with open(HEADER) as f:
        return re.findall(r"^QSA_API\s+[\w\s\*]+?\b(qsa_\w+)\s*\(", f.read(), flags=re.M)


def load_library():
    """Loads libqsa.so (built by ``index_gathered_sparse_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise LibraryMissing(f"{LIB_PATH} is not built; run index_gathered_sparse_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    T, P, i32, i64, u32 = qsa_tensor, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    common = [T, T, T, T, i64, T, T, u32, u32, u32, T, T, ctypes.c_float, i32, P]
    lib.qsa_sparse_attention_ragged_paged.argtypes = common
    lib.qsa_sparse_attention_ragged_paged.restype = ctypes.c_int
    lib.qsa_sparse_attention_ragged_paged_ex.argtypes = common + [ctypes.POINTER(qsa_options)]
    lib.qsa_sparse_attention_ragged_paged_ex.restype = ctypes.c_int
    lib.qsa_msa_attention_ragged_paged.argtypes = [T, T, T, T, i64, T, T, u32, u32, u32, T, ctypes.c_float, i32, P,
                                                   ctypes.POINTER(qsa_options)]
    lib.qsa_msa_attention_ragged_paged.restype = ctypes.c_int
    lib.qsa_compress_keys_paged.argtypes = [T, T, T, T, T, i64, T, T, u32, u32, u32, i32, i32, ctypes.c_float, P]
    lib.qsa_compress_keys_paged.restype = ctypes.c_int
    lib.qsa_latent_attention_ragged_paged.argtypes = [T, T, T, T, i64, T, T, T, i64, P, P, i64, u32, P, i64, P,
                                                      i32, ctypes.c_float, P, ctypes.POINTER(qsa_options)]
    lib.qsa_latent_attention_ragged_paged.restype = ctypes.c_int
    lib.qsa_plan.argtypes = [i32, i64, i64, i64, i64, i32, ctypes.POINTER(qsa_options), ctypes.POINTER(i32),
                             ctypes.POINTER(i32), ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_size_t)]
    lib.qsa_plan.restype = ctypes.c_int
    lib.qsa_plan_ex.argtypes = [i32, i64, i64, i64, i64, i64, i64, i32, u32, u32, ctypes.POINTER(qsa_options),
                                ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i64),
                                ctypes.POINTER(ctypes.c_size_t)]
    lib.qsa_plan_ex.restype = ctypes.c_int
    lib.qsa_reserve_workspace.argtypes = [P, ctypes.c_size_t]
    lib.qsa_reserve_workspace.restype = ctypes.c_int
    lib.qsa_release_device_state.argtypes = []
    lib.qsa_release_device_state.restype = ctypes.c_int
    lib.qsa_read_device_status.argtypes = [P, i32, ctypes.POINTER(ctypes.c_uint32)]
    lib.qsa_read_device_status.restype = ctypes.c_int
    lib.qsa_status_string.argtypes = [ctypes.c_int]
    lib.qsa_status_string.restype = ctypes.c_char_p
    lib.qsa_last_error_message.argtypes = []
    lib.qsa_last_error_message.restype = ctypes.c_char_p
    lib.qsa_version.argtypes = []
    lib.qsa_version.restype = i32
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != QSA_OK:
        msg = load_library().qsa_last_error_message().decode()
        raise QSAError(status, msg)


_TORCH_CODES = {torch.float32: QSA_F32, torch.bfloat16: QSA_BF16, torch.float8_e4m3fn: QSA_F8E4M3,
                torch.int32: QSA_I32}
if hasattr(torch, "uint32"):
    _TORCH_CODES[torch.uint32] = QSA_U32


def describe(t: Optional[torch.Tensor], code: Optional[int] = None, shape=None) -> qsa_tensor:
    """A qsa_tensor for ``t``; ``code`` overrides the element type (an int32
    tensor may carry U32 bits), ``shape`` the extents."""
    d = qsa_tensor()
    if t is None:
        d.data, d.dtype, d.ndim = None, code if code is not None else 0, len(shape or ())
        for i, s in enumerate(shape or ()):
            d.shape[i] = s
        return d
    d.data = t.data_ptr() if t.numel() else None
    d.dtype = code if code is not None else _TORCH_CODES.get(t.dtype, -1)
    shp = tuple(t.shape) if shape is None else tuple(shape)
    d.ndim = len(shp)
    for i, s in enumerate(shp):
        d.shape[i] = int(s)
    return d


def _u32(t: torch.Tensor) -> qsa_tensor:
    if t.dtype not in (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ()):
        raise TypeError("expected a 32-bit integer tensor for a U32 operand")
    if not t.is_contiguous():
        raise ValueError("U32 operands must be contiguous")
    return describe(t, QSA_U32)


def _contig(t: torch.Tensor, name: str) -> qsa_tensor:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return describe(t)


def _kv_desc(kv: torch.Tensor, page_stride: int) -> qsa_tensor:
    """kv_blocks as a 6-D tensor whose page axis may be padded (stride(0) ==
    page_stride); every inner axis contiguous."""
    if kv.dim() != 6:
        raise ValueError("kv_blocks must be 6-D [num_pages, 2, num_layers, page_size, num_kv_heads, head_dim]")
    inner = kv[0] if kv.shape[0] else kv
    if kv.shape[0] and not inner.is_contiguous():
        raise ValueError("kv_blocks: axes 1..5 must be contiguous")
    packed = 1
    for s in kv.shape[1:]:
        packed *= int(s)
    want = packed if page_stride == -1 else page_stride
    if kv.shape[0] > 1 and kv.stride(0) != want:
        raise ValueError(f"kv_blocks: page stride {kv.stride(0)} disagrees with page_stride {page_stride}")
    return describe(kv)


def qsa_sparse_attention_ragged_paged(output, q, input_row_offsets, kv_blocks, page_stride, cache_lengths,
                                      kv_lookup_table, max_prompt_length, max_cache_length, layer_idx,
                                      token_indices, counts, scale, group, stream=None, *, kernel: int = 0,
                                      splits: int = 0, ctas: int = 0, heads_per_unit: int = 0,
                                      test_stall: int = 0, tcgen05: int = 0) -> None:
    """One layer of QSA sparse attention on the GPU (asynchronous on
    ``stream``, default: PyTorch's current stream), with ``q``'s device
    current.  Raises QSAError on a non-OK status.  ``kernel`` / ``splits`` /
    ``ctas`` / ``heads_per_unit`` / ``tcgen05`` force a launch choice and
    ``test_stall`` drives the give-up path (tests and sweeps; see qsa_options)."""
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    args = [
        _contig(output, "output"), _contig(q, "q"), _u32(input_row_offsets), _kv_desc(kv_blocks, int(page_stride)),
        int(page_stride), _u32(cache_lengths), _u32(kv_lookup_table), int(max_prompt_length),
        int(max_cache_length), int(layer_idx), _contig(token_indices, "token_indices"), _contig(counts, "counts"),
        float(scale), int(group), ctypes.c_void_p(stream),
    ]
    with torch.cuda.device(q.device):  # the library resolves everything on the current device
        if kernel or splits or ctas or heads_per_unit or test_stall or tcgen05:
            opt = qsa_options(kernel=kernel, splits=splits, ctas=ctas, heads_per_unit=heads_per_unit,
                              test_stall=test_stall, tcgen05=tcgen05)
            _check(lib.qsa_sparse_attention_ragged_paged_ex(*args, ctypes.byref(opt)))
        else:
            _check(lib.qsa_sparse_attention_ragged_paged(*args))


def qsa_msa_attention_ragged_paged(output, q, input_row_offsets, kv_blocks, page_stride, cache_lengths,
                                   kv_lookup_table, max_prompt_length, max_cache_length, layer_idx, d_indices,
                                   scale, group, stream=None, *, kernel: int = 0, splits: int = 0,
                                   tcgen05: int = 0) -> None:
    """Block-sparse attention on the GPU: ``d_indices`` [num_kv_heads, total_q,
    topk] int32 lists whole blocks (pages) per (kv head, row); see qsa.h."""
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    if d_indices.dtype != torch.int32:
        raise TypeError("d_indices must be int32")
    opt = qsa_options(kernel=kernel, splits=splits, ctas=0, tcgen05=tcgen05)
    args = (_contig(output, "output"), _contig(q, "q"), _u32(input_row_offsets), _kv_desc(kv_blocks, int(page_stride)),
            int(page_stride), _u32(cache_lengths), _u32(kv_lookup_table), int(max_prompt_length),
            int(max_cache_length), int(layer_idx), _contig(d_indices, "d_indices"), float(scale), int(group),
            ctypes.c_void_p(stream), ctypes.byref(opt))
    with torch.cuda.device(q.device):
        _check(lib.qsa_msa_attention_ragged_paged(*args))


def qsa_compress_keys_paged(block_keys, gamma, freqs_cis, key_counts, kv_blocks, page_stride, cache_lengths,
                            kv_lookup_table, max_prompt_length, max_cache_length, layer_idx, ratio, rotary_dim, eps,
                            stream=None) -> None:
    """Block-key compression on the GPU (see qsa.h): ``block_keys``
    [batch * max_blocks, head_dim] from the raw keys in ``kv_blocks``."""
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(kv_blocks.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    if key_counts.dtype != torch.int32:
        raise TypeError("key_counts must be int32")
    args = (_contig(block_keys, "block_keys"), _contig(gamma, "gamma"), _contig(freqs_cis, "freqs_cis"),
            _contig(key_counts, "key_counts"), _kv_desc(kv_blocks, int(page_stride)), int(page_stride),
            _u32(cache_lengths), _u32(kv_lookup_table), int(max_prompt_length), int(max_cache_length), int(layer_idx),
            int(ratio), int(rotary_dim), float(eps), ctypes.c_void_p(stream))
    with torch.cuda.device(kv_blocks.device):
        _check(lib.qsa_compress_keys_paged(*args))


def qsa_latent_attention_ragged_paged(output, q, input_row_offsets, swa_blocks, swa_page_stride, swa_cache_lengths,
                                      swa_lookup_table, comp_blocks, comp_page_stride, comp_cache_lengths,
                                      comp_lookup_table, layer_idx, comp_indices, attn_sink, window, scale,
                                      stream=None, *, splits: int = 0) -> None:
    """Latent sparse attention on the GPU: sliding window + listed compressed
    entries + per-head sinks (see qsa.h).  The compressed cache's lengths,
    page table and entry lists and the sinks go across as plain pointers."""
    lib = load_library()
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    checks = ((comp_cache_lengths, (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ()), 1),
              (comp_lookup_table, (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ()), 2),
              (comp_indices, (torch.int32,), 2), (attn_sink, (torch.float32,), 1))
    for t, dts, nd in checks:
        if t.dtype not in dts or t.dim() != nd or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("comp_cache_lengths, comp_lookup_table, comp_indices and attn_sink must be contiguous "
                             "CUDA tensors of 32-bit elements with ranks 1, 2, 2 and 1")
    if comp_cache_lengths.numel() != swa_cache_lengths.numel() or comp_lookup_table.shape[0] != swa_cache_lengths.numel():
        raise ValueError("comp_cache_lengths / comp_lookup_table: first extent must be batch")
    if comp_indices.shape[0] != q.shape[0] or attn_sink.numel() != q.shape[1]:
        raise ValueError("comp_indices must have total_q rows and attn_sink num_heads entries")
    opt = qsa_options(kernel=0, splits=splits, ctas=0)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t.numel() else None)
    args = (_contig(output, "output"), _contig(q, "q"), _u32(input_row_offsets), _kv_desc(swa_blocks, int(swa_page_stride)),
            int(swa_page_stride), _u32(swa_cache_lengths), _u32(swa_lookup_table),
            _kv_desc(comp_blocks, int(comp_page_stride)), int(comp_page_stride), ptr(comp_cache_lengths),
            ptr(comp_lookup_table), int(comp_lookup_table.shape[1]), int(layer_idx), ptr(comp_indices),
            int(comp_indices.shape[1]), ptr(attn_sink), int(window), float(scale), ctypes.c_void_p(stream),
            ctypes.byref(opt))
    with torch.cuda.device(q.device):
        _check(lib.qsa_latent_attention_ragged_paged(*args))


def qsa_plan(dtype: int, total_q: int, num_kv_heads: int, head_dim: int, selection_width: int, group: int,
             kernel: int = 0, splits: int = 0, ctas: int = 0, block_lists: bool = False,
             heads_per_unit: int = 0, tcgen05: int = 0, batch=None, page_size=None,
             max_prompt_length=None, max_cache_length=None) -> dict:
    """The launch a call with these extents would make.  With batch,
    page_size and the two length hints (qsa_plan_ex) it is exactly the plan of
    a qsa_sparse_attention_ragged_paged call with those arguments."""
    lib = load_library()
    k, s = ctypes.c_int32(), ctypes.c_int32()
    c, w = ctypes.c_int64(), ctypes.c_size_t()
    opt = qsa_options(kernel=kernel, splits=splits, ctas=ctas, block_lists=int(bool(block_lists)),
                      heads_per_unit=heads_per_unit, tcgen05=tcgen05)
    outs = (ctypes.byref(k), ctypes.byref(s), ctypes.byref(c), ctypes.byref(w))
    if batch is None:
        _check(lib.qsa_plan(dtype, total_q, num_kv_heads, head_dim, selection_width, group, ctypes.byref(opt), *outs))
    else:
        _check(lib.qsa_plan_ex(dtype, total_q, int(batch), num_kv_heads, head_dim, int(page_size), selection_width,
                               group, int(max_prompt_length), int(max_cache_length), ctypes.byref(opt), *outs))
    return {"kernel": k.value, "splits": s.value, "ctas": c.value, "workspace_bytes": w.value}


def qsa_reserve_workspace(nbytes: int, stream=None) -> None:
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    _check(load_library().qsa_reserve_workspace(ctypes.c_void_p(stream), int(nbytes)))


def qsa_release_device_state() -> None:
    _check(load_library().qsa_release_device_state())


def qsa_read_device_status(clear: bool = True, stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    flags = ctypes.c_uint32()
    _check(load_library().qsa_read_device_status(ctypes.c_void_p(stream), int(bool(clear)), ctypes.byref(flags)))
    return flags.value


def qsa_status_string(status: int) -> str:
    return load_library().qsa_status_string(int(status)).decode()


def qsa_version() -> int:
    return load_library().qsa_version()


_noalloc_ready = False


def qsa_sparse_attention_ragged_paged_noalloc(output, q, input_row_offsets, kv_blocks, page_stride, cache_lengths,
                                              kv_lookup_table, max_prompt_length, max_cache_length, layer_idx,
                                              token_indices, counts, scale, group, stream=None,
                                              status_flags: Optional[torch.Tensor] = None) -> None:
    """The allocation-free variant: same operation, enqueued on ``stream``
    with the library's fixed device scratch instead of a cudaMalloc'd
    workspace (persistent stream-K kernel; BF16/F8E4M3 with head_dim 128).
    ``status_flags`` is an optional one-element int32 device tensor that
    receives the QSA_STATUS_* bits.  Calls that overlap on the GPU share the
    scratch and race; the first call on a device should come before any
    stream capture."""
    global _noalloc_ready
    lib = load_library()
    fn = lib.qsa_sparse_attention_ragged_paged_noalloc
    if not _noalloc_ready:
        T, P, i32, i64, u32 = qsa_tensor, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
        fn.argtypes = [T, T, T, T, i64, T, T, u32, u32, u32, T, T, ctypes.c_float, i32, P, P]
        fn.restype = ctypes.c_int
        _noalloc_ready = True
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    flags = None
    if status_flags is not None:
        if status_flags.dtype not in (torch.int32,) + ((torch.uint32,) if hasattr(torch, "uint32") else ()) \
                or status_flags.numel() < 1 or not status_flags.is_cuda:
            raise ValueError("status_flags must be a CUDA tensor of at least one 32-bit integer")
        flags = status_flags.data_ptr()
    args = (_contig(output, "output"), _contig(q, "q"), _u32(input_row_offsets),
            _kv_desc(kv_blocks, int(page_stride)), int(page_stride), _u32(cache_lengths), _u32(kv_lookup_table),
            int(max_prompt_length), int(max_cache_length), int(layer_idx), _contig(token_indices, "token_indices"),
            _contig(counts, "counts"), float(scale), int(group), ctypes.c_void_p(stream), ctypes.c_void_p(flags))
    with torch.cuda.device(q.device):  # the scratch address is looked up on the current device: q's
        _check(fn(*args))
