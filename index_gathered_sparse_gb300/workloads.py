"""Seeded synthetic inputs for QSA gather-GQA sparse attention.

This module only *makes inputs*: ragged query rows, a paged KV cache scattered
through a shuffled page table, and a per-row selection of cache positions.  It
holds none of the attention arithmetic, so both the CPU oracle (through the
tests) and the CUDA path can be fed from it without sharing any code.

Layouts follow the QSASparseAttentionRaggedPaged page ("Tensor shapes"):

* ``q``               ``[total_q, num_q_heads, head_dim]``
* ``input_row_offsets`` ``[batch + 1]`` uint32
* ``kv_blocks``       ``[num_pages, 2, num_layers, page_size, num_kv_heads, head_dim]``
  with ``page_stride`` elements between pages (``-1`` = packed)
* ``cache_lengths``   ``[batch]`` uint32
* ``kv_lookup_table`` ``[batch, max_pages]`` uint32
* ``token_indices``   ``[total_q, selection_width]`` int32, valid entries first
* ``counts``          ``[total_q]`` int32

Element storage is raw: float32 values, bfloat16 *bits* (uint16) or FP8 e4m3fn
*bits* (uint8).  The float -> bf16 / e4m3 encodings are PyTorch's CPU casts
(round to nearest even).

Conventions this generator fixes (the pages leave them open):

* Row ``t`` of sequence ``b`` sits at position ``pos = cache_lengths[b] + t``;
  the cache already holds this step's keys, so positions ``[0, cache_lengths[b]
  + rows_b)`` are valid and a row selects from ``[0, pos]``.
* Axis 1 of ``kv_blocks``: index 0 holds K, index 1 holds V.
* Cache slots that no sequence owns, the layers other than ``layer_idx``, the
  padding between pages and one extra "poison page" are filled with NaN, and
  table entries past a sequence's last page point at the poison page, so any
  stray read shows up as NaN instead of a fault.

Random draw order: the sequence structure (rows, cache lengths) comes from
``default_rng(seed + 1000)`` inside the workload function; then one
``default_rng(seed)`` draws the page permutation -> q -> per sequence K then V
in logical order -> per row (count, indices, tail) in row order.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Callable, List, Optional, Sequence

import numpy as np

DTYPES = ("f32", "bf16", "e4m3")

# NaN bit patterns used to poison every cache byte no selection may read.
_POISON = {"f32": np.uint32(0x7FC00000), "bf16": np.uint16(0x7FC0), "e4m3": np.uint8(0x7F)}
_STORAGE = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}
ELEM_BYTES = {"f32": 4, "bf16": 2, "e4m3": 1}


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 array -> raw storage of ``dtype`` (RNE casts done by PyTorch on CPU)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    import torch

    t = torch.from_numpy(x)
    if dtype == "bf16":
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "e4m3":
        return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    raise ValueError(dtype)


@dataclasses.dataclass
class QSAInputs:
    """One call's worth of inputs, all host numpy arrays in raw storage."""

    name: str
    dtype: str
    out_dtype: str
    q: np.ndarray
    kv_flat: np.ndarray  # raw storage, num_pages * page pitch (+ nothing else)
    kv_shape: tuple  # (num_pages, 2, num_layers, page_size, num_kv_heads, head_dim)
    page_stride: int  # -1 when packed, else elements between pages
    input_row_offsets: np.ndarray
    cache_lengths: np.ndarray
    kv_lookup_table: np.ndarray
    max_prompt_length: int
    max_cache_length: int
    layer_idx: int
    token_indices: np.ndarray
    counts: np.ndarray
    scale: float
    group: int
    poison_page: int
    # logical (unpaged) K and V per sequence, raw storage [kv_len, nkv, D]; kept
    # only on request so independent checks can skip the paging entirely.
    logical_k: Optional[List[np.ndarray]] = None
    logical_v: Optional[List[np.ndarray]] = None

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_q_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_kv_heads(self) -> int:
        return int(self.kv_shape[4])

    @property
    def batch(self) -> int:
        return int(self.cache_lengths.shape[0])

    @property
    def selection_width(self) -> int:
        return int(self.token_indices.shape[1])

    @property
    def page_pitch(self) -> int:
        """Elements from one page to the next."""
        n, two, L, P, nkv, D = self.kv_shape
        return two * L * P * nkv * D if self.page_stride == -1 else self.page_stride

    def kv_view(self) -> np.ndarray:
        """The 6-D ``kv_blocks`` view over ``kv_flat`` (strided when padded)."""
        n, two, L, P, nkv, D = self.kv_shape
        es = self.kv_flat.itemsize
        strides = (self.page_pitch * es, L * P * nkv * D * es, P * nkv * D * es, nkv * D * es, D * es, es)
        return np.lib.stride_tricks.as_strided(self.kv_flat, shape=self.kv_shape, strides=strides)

    def row_sequence(self) -> np.ndarray:
        """Sequence id of every query row (from ``input_row_offsets``)."""
        off = self.input_row_offsets.astype(np.int64)
        return np.repeat(np.arange(self.batch), np.diff(off))

    def valid_counts(self) -> np.ndarray:
        """``counts`` clamped to ``[0, selection_width]``."""
        return np.clip(self.counts.astype(np.int64), 0, self.selection_width)

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move: each selected K and V row once per
        (row, kv head), plus q, the output and the valid indices and counts."""
        ekv = ELEM_BYTES[self.dtype]
        eo = ELEM_BYTES[self.out_dtype]
        n = int(self.valid_counts().sum())
        D = self.head_dim
        return (
            n * self.num_kv_heads * 2 * D * ekv
            + self.total_q * self.num_q_heads * D * (ekv + eo)
            + n * 4
            + self.total_q * 4
        )

    def attended_pairs(self) -> int:
        """(key, kv head) pairs the method attends: every valid entry of every
        row, once per kv head."""
        return int(self.valid_counts().sum()) * self.num_kv_heads

    def algorithmic_flops(self) -> int:
        """Flops of the two contractions: per attended (key, kv head) pair,
        ``group`` query heads x head_dim multiply-adds for q.K and as many
        for p.V (2 flops each)."""
        return 4 * self.group * self.head_dim * self.attended_pairs()

    def distinct_kv_bytes(self) -> int:
        """K and V bytes of the distinct cache positions the selections name,
        counted once per sequence (all kv heads): what a gather must bring
        from DRAM at least once when every repeat hits in L2."""
        n = self.valid_counts()
        seq = self.row_sequence()
        kv_len = self.cache_lengths.astype(np.int64) + np.diff(self.input_row_offsets.astype(np.int64))
        distinct = 0
        for b in range(self.batch):
            rows = np.nonzero(seq == b)[0]
            if rows.size == 0:
                continue
            w = int(n[rows].max())
            sel = self.token_indices[rows, :w].astype(np.int64)
            keep = (np.arange(w)[None, :] < n[rows][:, None]) & (sel >= 0) & (sel < kv_len[b])
            distinct += int(np.unique(sel[keep]).size)
        return distinct * self.num_kv_heads * 2 * self.head_dim * ELEM_BYTES[self.dtype]


# ----------------------------------------------------------------------------
# selection recipes (per row); each returns the valid prefix as int64
# ----------------------------------------------------------------------------

def _sel_uniform_distinct(count_rule: str) -> Callable:
    """Distinct positions drawn uniformly from [0, pos], in random order."""

    def pick(rng, pos, W, P):
        hi = min(W, pos + 1)
        cnt = hi if count_rule == "full" else int(rng.integers(1, hi + 1))
        return rng.choice(pos + 1, size=cnt, replace=False).astype(np.int64)

    return pick


def _sel_local_plus_uniform(local: int = 64) -> Callable:
    """The ``local`` positions nearest pos plus distinct uniform picks from the
    rest of [0, pos]; count = min(W, pos + 1); sorted ascending."""

    def pick(rng, pos, W, P):
        cnt = min(W, pos + 1)
        lo = max(0, pos - local + 1)
        near = np.arange(lo, pos + 1, dtype=np.int64)
        rest = cnt - near.size
        far = rng.choice(lo, size=rest, replace=False).astype(np.int64) if rest > 0 else np.zeros(0, np.int64)
        return np.sort(np.concatenate([far, near]))

    return pick


def _sel_block_runs(runs: int = 64, run_len: int = 64) -> Callable:
    """``runs`` distinct runs of ``run_len`` positions with run-aligned starts,
    always including the run that holds pos, clipped to pos; ascending."""

    def pick(rng, pos, W, P):
        last = pos // run_len
        n_runs = min(runs, last + 1)
        others = rng.choice(last, size=n_runs - 1, replace=False) if n_runs > 1 else np.zeros(0, np.int64)
        starts = np.sort(np.concatenate([others.astype(np.int64), [last]])) * run_len
        idx = (starts[:, None] + np.arange(run_len)[None, :]).reshape(-1)
        return idx[idx <= pos].astype(np.int64)

    return pick


def _tail_const(v: int) -> Callable:
    def fill(rng, n, kv_len):
        return np.full(n, v, dtype=np.int64)

    return fill


def _tail_out_of_range(rng, n, kv_len):
    """Random ints outside [0, kv_len): half >= kv_len, half negative."""
    hi = rng.integers(kv_len, 2**31 - 1, size=n, dtype=np.int64)
    lo = rng.integers(-(2**31), 0, size=n, dtype=np.int64)
    return np.where(rng.random(n) < 0.5, hi, lo)


# ----------------------------------------------------------------------------
# the generic builder
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class WorkloadSpec:
    name: str
    seed: int
    rows: Sequence[int]  # new query rows per sequence
    cache_lengths: Sequence[int]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_layers: int
    layer_idx: int
    dtype: str
    out_dtype: str
    selection_width: int
    select: Callable
    tail: Callable
    page_pad: Optional[int] = None  # extra elements between pages (None = packed)
    scale: Optional[float] = None

    def build(self, keep_logical: bool = False, rng=None) -> QSAInputs:
        return _build(self, keep_logical, rng)


def assemble(name: str, dtype: str, out_dtype: str, q: np.ndarray, logical_k: Sequence[np.ndarray],
             logical_v: Sequence[np.ndarray], rows: Sequence[int], cache_lengths: Sequence[int],
             page_size: int, num_layers: int, layer_idx: int, token_indices: np.ndarray,
             counts: np.ndarray, scale: float, page_perm: Optional[np.ndarray] = None,
             page_pad: Optional[int] = None, keep_logical: bool = False) -> QSAInputs:
    """Pages logical per-sequence K/V (raw storage ``[kv_len_b, nkv, D]``) into
    ``kv_blocks`` through the page assignment ``page_perm`` (identity when None)
    and wraps everything as a :class:`QSAInputs`."""
    B = len(rows)
    rows = np.asarray(rows, dtype=np.int64)
    cache = np.asarray(cache_lengths, dtype=np.int64)
    total_q, nq, D = q.shape
    nkv = int(logical_k[0].shape[1]) if B else 1
    P, L = int(page_size), int(num_layers)
    assert nq % nkv == 0 and 0 <= layer_idx < L
    kv_len = cache + rows
    for b in range(B):
        assert logical_k[b].shape == (kv_len[b], nkv, D) and logical_v[b].shape == (kv_len[b], nkv, D)
    npages = -(-kv_len // P)
    total_pages = int(npages.sum())
    poison_page = total_pages
    num_pages = total_pages + 1
    max_pages = max(1, int(npages.max()) if B else 1)
    perm = np.arange(total_pages) if page_perm is None else np.asarray(page_perm)
    assert perm.shape == (total_pages,)
    table = np.full((B, max_pages), poison_page, dtype=np.uint32)
    start = 0
    for b in range(B):
        table[b, : npages[b]] = perm[start : start + npages[b]]
        start += npages[b]

    packed = 2 * L * P * nkv * D
    page_stride = -1 if page_pad is None else packed + int(page_pad)
    pitch = packed if page_stride == -1 else page_stride
    kv_flat = np.empty(num_pages * pitch, dtype=_STORAGE[dtype])
    kv_flat.view(_POISON[dtype].dtype)[:] = _POISON[dtype]
    es = kv_flat.itemsize
    kv6 = np.lib.stride_tricks.as_strided(
        kv_flat,
        shape=(num_pages, 2, L, P, nkv, D),
        strides=(pitch * es, L * P * nkv * D * es, P * nkv * D * es, nkv * D * es, D * es, es),
    )
    for b in range(B):
        n = int(kv_len[b])
        kb, vb = logical_k[b], logical_v[b]
        full = n // P
        pages = table[b, : npages[b]].astype(np.int64)
        # page by page: fancy indexing through a strided view is far slower
        for i in range(full):
            kv6[pages[i], 0, layer_idx] = kb[i * P : (i + 1) * P]
            kv6[pages[i], 1, layer_idx] = vb[i * P : (i + 1) * P]
        rem = n - full * P
        if rem:
            kv6[pages[full], 0, layer_idx, :rem] = kb[full * P :]
            kv6[pages[full], 1, layer_idx, :rem] = vb[full * P :]

    offsets = np.zeros(B + 1, dtype=np.uint32)
    offsets[1:] = np.cumsum(rows)
    return QSAInputs(
        name=name,
        dtype=dtype,
        out_dtype=out_dtype,
        q=np.ascontiguousarray(q),
        kv_flat=kv_flat,
        kv_shape=(num_pages, 2, L, P, nkv, D),
        page_stride=page_stride,
        input_row_offsets=offsets,
        cache_lengths=cache.astype(np.uint32),
        kv_lookup_table=table,
        max_prompt_length=int(rows.max()) if B else 0,
        max_cache_length=int(cache.max()) if B else 0,
        layer_idx=int(layer_idx),
        token_indices=np.ascontiguousarray(token_indices, dtype=np.int32),
        counts=np.ascontiguousarray(counts, dtype=np.int32),
        scale=float(scale),
        group=nq // nkv,
        poison_page=poison_page,
        logical_k=list(logical_k) if keep_logical else None,
        logical_v=list(logical_v) if keep_logical else None,
    )


def _build(spec: WorkloadSpec, keep_logical: bool, rng) -> QSAInputs:
    if rng is None:
        rng = np.random.default_rng(spec.seed)
    B = len(spec.rows)
    rows = np.asarray(spec.rows, dtype=np.int64)
    cache = np.asarray(spec.cache_lengths, dtype=np.int64)
    nq, nkv, D, P = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.page_size
    W = spec.selection_width
    kv_len = cache + rows
    total_pages = int((-(-kv_len // P)).sum())
    perm = rng.permutation(total_pages)

    total_q = int(rows.sum())
    q = encode(rng.standard_normal((total_q, nq, D), dtype=np.float32), spec.dtype)
    logical_k, logical_v = [], []
    for b in range(B):
        n = int(kv_len[b])
        logical_k.append(encode(rng.standard_normal((n, nkv, D), dtype=np.float32), spec.dtype))
        logical_v.append(encode(rng.standard_normal((n, nkv, D), dtype=np.float32), spec.dtype))

    token_indices = np.empty((total_q, W), dtype=np.int32)
    counts = np.empty(total_q, dtype=np.int32)
    r = 0
    for b in range(B):
        for t in range(int(rows[b])):
            pos = int(cache[b]) + t
            sel = spec.select(rng, pos, W, P)
            assert sel.size <= W
            counts[r] = sel.size
            token_indices[r, : sel.size] = sel
            if sel.size < W:
                token_indices[r, sel.size :] = spec.tail(rng, W - sel.size, int(kv_len[b]))
            r += 1

    scale = spec.scale if spec.scale is not None else 1.0 / math.sqrt(D)
    return assemble(spec.name, spec.dtype, spec.out_dtype, q, logical_k, logical_v, rows, cache, P,
                    spec.num_layers, spec.layer_idx, token_indices, counts, scale, page_perm=perm,
                    page_pad=spec.page_pad, keep_logical=keep_logical)


# ----------------------------------------------------------------------------
# the five workloads (full size by default; keyword overrides shrink them for
# parity tests while keeping each one's structure)
# ----------------------------------------------------------------------------

def tiny_ragged(seed: int = 0) -> WorkloadSpec:
    """fp32, batch 2, rows [3,5] on cache [17,40], 4 q heads on 1 kv head,
    head_dim 64, page 16, 2 layers (layer 1), packed permuted pages, width 8,
    counts U[1, min(8, pos+1)], distinct U[0,pos], tail 999999."""
    return WorkloadSpec(
        name="tiny_ragged_fp32", seed=seed, rows=[3, 5], cache_lengths=[17, 40],
        num_q_heads=4, num_kv_heads=1, head_dim=64, page_size=16, num_layers=2, layer_idx=1,
        dtype="f32", out_dtype="f32", selection_width=8,
        select=_sel_uniform_distinct("uniform"), tail=_tail_const(999999),
    )


def bf16_decode(seed: int = 2, batch: int = 64, cache_range=(1024, 8192), width: int = 2048,
                num_layers: int = 4, layer_idx: int = 2, name: str = "bf16_decode") -> WorkloadSpec:
    """bf16 decode: one new token per sequence, cache U[1024, 8192], 32 q heads
    on 8 kv heads, head_dim 128, page 128, 4 layers (layer 2), width 2048,
    counts = min(2048, pos+1), distinct U[0,pos] in random order, tail -1."""
    rng = np.random.default_rng(seed + 1000)
    cache = rng.integers(cache_range[0], cache_range[1] + 1, size=batch)
    return WorkloadSpec(
        name=name, seed=seed, rows=[1] * batch, cache_lengths=cache.tolist(),
        num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=128, num_layers=num_layers,
        layer_idx=layer_idx, dtype="bf16", out_dtype="bf16", selection_width=width,
        select=_sel_uniform_distinct("full"), tail=_tail_const(-1),
    )


def bf16_chunked_prefill(seed: int = 3, rows=(512, 1024, 256, 2048), cache=(0, 4096, 16384, 8192),
                         width: int = 2048) -> WorkloadSpec:
    """bf16 chunked prefill: rows [512,1024,256,2048] on cache [0,4096,16384,8192],
    64 q heads on 8 kv heads, head_dim 128, page 64, 1 layer, width 2048,
    counts = min(2048, pos+1); the 64 positions nearest pos plus distinct
    uniform picks from the rest, sorted ascending; tail -1."""
    return WorkloadSpec(
        name="bf16_chunked_prefill", seed=seed, rows=list(rows), cache_lengths=list(cache),
        num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64, num_layers=1, layer_idx=0,
        dtype="bf16", out_dtype="bf16", selection_width=width,
        select=_sel_local_plus_uniform(64), tail=_tail_const(-1),
    )


def bf16_long_decode(seed: int = 4, batch: int = 32, cache_range=(65536, 131072), runs: int = 64) -> WorkloadSpec:
    """bf16 long-context decode: batch 32, cache U[65536, 131072], 16 q heads on
    1 kv head, head_dim 128, page 64, 1 layer; selection = 64 distinct
    page-aligned runs of 64 (the run holding pos always in, clipped to pos),
    ascending; width 4096; tail -1."""
    rng = np.random.default_rng(seed + 1000)
    cache_l = rng.integers(cache_range[0], cache_range[1] + 1, size=batch)
    return WorkloadSpec(
        name="bf16_long_decode", seed=seed, rows=[1] * batch, cache_lengths=cache_l.tolist(),
        num_q_heads=16, num_kv_heads=1, head_dim=128, page_size=64, num_layers=1, layer_idx=0,
        dtype="bf16", out_dtype="bf16", selection_width=runs * 64,
        select=_sel_block_runs(runs, 64), tail=_tail_const(-1),
    )


def fp8_mixed(seed: int = 5, n_decode: int = 120, n_prefill: int = 8, prefill_rows: int = 512,
              cache_range=(256, 32768), width: int = 1024) -> WorkloadSpec:
    """FP8 e4m3 mixed batch: 120 decode sequences + 8 prefill sequences of 512
    rows placed by a seeded permutation, cache log-uniform in [256, 32768],
    32 q heads on 4 kv heads, head_dim 128, page 128, 2 layers (layer 0),
    page_stride = packed page + 4096 elements, bf16 output, width 1024,
    counts U[1, min(1024, pos+1)], distinct U[0,pos], tail random
    out-of-range ints."""
    rng = np.random.default_rng(seed + 1000)
    kinds = np.array([1] * n_decode + [prefill_rows] * n_prefill)
    rows = kinds[rng.permutation(kinds.size)]
    lo, hi = math.log(cache_range[0]), math.log(cache_range[1])
    cache = np.floor(np.exp(rng.uniform(lo, hi, size=kinds.size))).astype(np.int64)
    return WorkloadSpec(
        name="fp8_mixed", seed=seed, rows=rows.tolist(), cache_lengths=cache.tolist(),
        num_q_heads=32, num_kv_heads=4, head_dim=128, page_size=128, num_layers=2, layer_idx=0,
        dtype="e4m3", out_dtype="bf16", selection_width=width,
        select=_sel_uniform_distinct("uniform"), tail=_tail_out_of_range, page_pad=4096,
    )


WORKLOADS = {
    "tiny_ragged_fp32": tiny_ragged,
    "bf16_decode": bf16_decode,
    # the same gathers from a 1-layer cache (1.2 GB instead of 4.8 GB): a
    # smaller device footprint for profiler captures
    "bf16_decode_1layer": lambda: bf16_decode(num_layers=1, layer_idx=0, name="bf16_decode_1layer"),
    "bf16_chunked_prefill": bf16_chunked_prefill,
    # the same rows, counts and selection recipe with 4 and 16 query heads per kv head (the
    # row-group kernel's other group sizes): 32 q / 8 kv and 64 q / 4 kv
    "bf16_chunked_prefill_g4": lambda: dataclasses.replace(bf16_chunked_prefill(), name="bf16_chunked_prefill_g4",
                                                           num_q_heads=32),
    "bf16_chunked_prefill_g16": lambda: dataclasses.replace(bf16_chunked_prefill(), name="bf16_chunked_prefill_g16",
                                                            num_kv_heads=4),
    "bf16_long_decode": bf16_long_decode,
    "fp8_mixed": fp8_mixed,
}


def small_variants() -> dict:
    """Reduced copies of the four large workloads: each keeps its dtype, head
    layout, page size, selection recipe and tail rule, at sizes the oracle
    finishes in seconds while still spanning several 64-key tiles and a
    ragged last tile."""
    return {
        "bf16_decode_small": bf16_decode(seed=12, batch=6, cache_range=(150, 900), width=512),
        "bf16_prefill_small": bf16_chunked_prefill(seed=13, rows=(40, 9, 23), cache=(0, 300, 77), width=256),
        "bf16_long_decode_small": bf16_long_decode(seed=14, batch=3, cache_range=(3000, 9000), runs=12),
        "fp8_mixed_small": fp8_mixed(seed=15, n_decode=5, n_prefill=2, prefill_rows=17,
                                     cache_range=(40, 1500), width=200),
    }


def to_torch(x: QSAInputs, device, out_dtype: Optional[str] = None) -> dict:
    """Uploads ``x`` and returns the keyword arguments of
    ``binding.qsa_sparse_attention_ragged_paged`` (output freshly allocated).
    U32 operands travel as int32 tensors holding the same bits."""
    import torch

    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}

    def raw(a: np.ndarray, dtype: str):
        a = np.ascontiguousarray(a)
        if dtype == "f32":
            return torch.from_numpy(a)
        if dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        return torch.from_numpy(a).view(torch.float8_e4m3fn)

    def i32(a: np.ndarray):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(device)

    n, two, L, P, nkv, D = x.kv_shape
    flat = raw(x.kv_flat, x.dtype).to(device)
    kv = flat.as_strided(x.kv_shape, (x.page_pitch, L * P * nkv * D, P * nkv * D, nkv * D, D, 1))
    od = out_dtype or x.out_dtype
    return dict(
        output=torch.empty((x.total_q, x.num_q_heads, D), dtype=tdt[od], device=device),
        q=raw(x.q, x.dtype).to(device),
        input_row_offsets=i32(x.input_row_offsets),
        kv_blocks=kv,
        page_stride=x.page_stride,
        cache_lengths=i32(x.cache_lengths),
        kv_lookup_table=i32(x.kv_lookup_table),
        max_prompt_length=x.max_prompt_length,
        max_cache_length=x.max_cache_length,
        layer_idx=x.layer_idx,
        token_indices=i32(x.token_indices),
        counts=i32(x.counts),
        scale=x.scale,
        group=x.group,
    )


# ----------------------------------------------------------------------------
# block-granular (MSA-style) selection: d_indices [num_kv_heads, total_q, topk]
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class MSAInputs(QSAInputs):
    """A block-sparse call: the same paged cache, queries and page table, with
    ``d_indices[h, r, :]`` naming whole logical blocks (pages) of row r's
    sequence per kv head (``-1`` = unused).  ``token_indices``/``counts`` are
    empty: block ids replace them."""

    d_indices: Optional[np.ndarray] = None

    @property
    def topk(self) -> int:
        return int(self.d_indices.shape[2])

    def query_positions(self) -> np.ndarray:
        """Each row's position: cache_lengths[b] + (r - input_row_offsets[b])."""
        seq = self.row_sequence()
        off = self.input_row_offsets.astype(np.int64)
        return self.cache_lengths.astype(np.int64)[seq] + np.arange(self.total_q) - off[seq]

    def attended_keys(self) -> np.ndarray:
        """Keys attended per (kv head, row): positions <= the row's position
        inside its listed blocks (duplicates count twice)."""
        P = int(self.kv_shape[3])
        pos = self.query_positions()[None, :, None]
        blk = self.d_indices.astype(np.int64)
        return np.where(blk >= 0, np.clip(pos - blk * P + 1, 0, P), 0).sum(axis=2)

    def algorithmic_bytes(self) -> int:
        ekv = ELEM_BYTES[self.dtype]
        eo = ELEM_BYTES[self.out_dtype]
        n = int(self.attended_keys().sum())  # summed over kv heads already
        D = self.head_dim
        return (n * 2 * D * ekv + self.total_q * self.num_q_heads * D * (ekv + eo)
                + self.d_indices.size * 4)

    def attended_pairs(self) -> int:
        return int(self.attended_keys().sum())

    def distinct_kv_bytes(self) -> int:
        """K and V bytes of the distinct blocks listed per (sequence, kv head),
        each counted whole."""
        P = int(self.kv_shape[3])
        seq = self.row_sequence()
        blocks = 0
        for b in range(self.batch):
            rows = np.nonzero(seq == b)[0]
            for h in range(self.num_kv_heads):
                ids = self.d_indices[h, rows].reshape(-1)
                blocks += int(np.unique(ids[ids >= 0]).size)
        return blocks * P * 2 * self.head_dim * ELEM_BYTES[self.dtype]


@dataclasses.dataclass
class MSASpec:
    """Block-sparse workload recipe: per (kv head, row), the block holding the
    row's position plus ``topk - 1`` distinct uniform picks among the earlier
    blocks, in random order; ``-1`` fills the rest when fewer exist."""

    name: str
    seed: int
    rows: Sequence[int]
    cache_lengths: Sequence[int]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_layers: int
    layer_idx: int
    dtype: str
    out_dtype: str
    topk: int
    page_pad: Optional[int] = None

    def build(self, keep_logical: bool = False) -> MSAInputs:
        rng = np.random.default_rng(self.seed)
        B = len(self.rows)
        rows = np.asarray(self.rows, dtype=np.int64)
        cache = np.asarray(self.cache_lengths, dtype=np.int64)
        nq, nkv, D, P = self.num_q_heads, self.num_kv_heads, self.head_dim, self.page_size
        kv_len = cache + rows
        perm = rng.permutation(int((-(-kv_len // P)).sum()))
        total_q = int(rows.sum())
        q = encode(rng.standard_normal((total_q, nq, D), dtype=np.float32), self.dtype)
        lk, lv = [], []
        for b in range(B):
            n = int(kv_len[b])
            lk.append(encode(rng.standard_normal((n, nkv, D), dtype=np.float32), self.dtype))
            lv.append(encode(rng.standard_normal((n, nkv, D), dtype=np.float32), self.dtype))
        d_idx = np.full((nkv, total_q, self.topk), -1, dtype=np.int32)
        r = 0
        for b in range(B):
            for t in range(int(rows[b])):
                last = (int(cache[b]) + t) // P
                for h in range(nkv):
                    k = min(self.topk, last + 1)
                    others = rng.choice(last, size=k - 1, replace=False) if k > 1 else np.zeros(0, np.int64)
                    blocks = np.concatenate([others.astype(np.int64), [last]])
                    d_idx[h, r, :k] = blocks[rng.permutation(k)]
                r += 1
        base = assemble(self.name, self.dtype, self.out_dtype, q, lk, lv, rows, cache, P, self.num_layers,
                        self.layer_idx, np.zeros((total_q, 0), np.int32), np.zeros(total_q, np.int32),
                        1.0 / math.sqrt(D), page_perm=perm, page_pad=self.page_pad, keep_logical=keep_logical)
        return MSAInputs(**{f.name: getattr(base, f.name) for f in dataclasses.fields(QSAInputs)}, d_indices=d_idx)


def msa_bf16_decode(seed: int = 6, batch: int = 64, cache_range=(1024, 8192), topk: int = 32,
                    name: str = "msa_bf16_decode") -> MSASpec:
    """Block-sparse bf16 decode: 64 x 1 row, cache U[1024, 8192], 32 q heads on
    8 kv heads, head_dim 128, page (block) 64, 1 layer, topk 32 blocks per
    (kv head, row) = up to 2048 keys."""
    rng = np.random.default_rng(seed + 1000)
    cache = rng.integers(cache_range[0], cache_range[1] + 1, size=batch)
    return MSASpec(name=name, seed=seed, rows=[1] * batch, cache_lengths=cache.tolist(), num_q_heads=32,
                   num_kv_heads=8, head_dim=128, page_size=64, num_layers=1, layer_idx=0, dtype="bf16",
                   out_dtype="bf16", topk=topk)


def msa_bf16_prefill(seed: int = 7, rows=(128, 256, 64, 512), cache=(0, 4096, 16384, 8192), topk: int = 32,
                     name: str = "msa_bf16_prefill") -> MSASpec:
    """Block-sparse bf16 chunked prefill: rows [128,256,64,512] on cache
    [0,4096,16384,8192], 64 q heads on 8 kv heads, head_dim 128, block 64,
    topk 32 (causal inside the block holding each row's position)."""
    return MSASpec(name=name, seed=seed, rows=list(rows), cache_lengths=list(cache), num_q_heads=64,
                   num_kv_heads=8, head_dim=128, page_size=64, num_layers=1, layer_idx=0, dtype="bf16",
                   out_dtype="bf16", topk=topk)


def msa_fp8_decode(seed: int = 8, batch: int = 96, cache_range=(512, 16384), topk: int = 16,
                   name: str = "msa_fp8_decode") -> MSASpec:
    """Block-sparse scale-free FP8 e4m3 decode: 96 x 1 row, cache U[512,16384],
    32 q heads on 4 kv heads, head_dim 128, block 128, 2 layers (layer 1),
    padded pages, bf16 output, topk 16 blocks."""
    rng = np.random.default_rng(seed + 1000)
    cache = rng.integers(cache_range[0], cache_range[1] + 1, size=batch)
    return MSASpec(name=name, seed=seed, rows=[1] * batch, cache_lengths=cache.tolist(), num_q_heads=32,
                   num_kv_heads=4, head_dim=128, page_size=128, num_layers=2, layer_idx=1, dtype="e4m3",
                   out_dtype="bf16", topk=topk, page_pad=4096)


MSA_WORKLOADS = {
    "msa_bf16_decode": msa_bf16_decode,
    "msa_bf16_prefill": msa_bf16_prefill,
    "msa_fp8_decode": msa_fp8_decode,
}


def msa_small_variants() -> dict:
    """Block-sparse workloads at oracle-friendly sizes (several blocks, a
    partial last block, -1 padding where a row has fewer blocks than topk)."""
    return {
        "msa_bf16_decode_small": msa_bf16_decode(seed=16, batch=5, cache_range=(70, 900), topk=6),
        "msa_bf16_prefill_small": msa_bf16_prefill(seed=17, rows=(20, 7, 33), cache=(0, 130, 300), topk=5),
        "msa_fp8_decode_small": msa_fp8_decode(seed=18, batch=4, cache_range=(100, 1200), topk=4),
        # speculative-decode shape: 2, 3 and 4 new rows per sequence on cached
        # context, the last one straddling a block boundary (positions 255..258
        # with blocks of 64), so rows of one sequence differ in their causal block
        "msa_bf16_specdec_small": msa_bf16_prefill(seed=19, rows=(2, 3, 4), cache=(150, 700, 255), topk=6,
                                                   name="msa_bf16_specdec"),
    }


def to_torch_msa(x: MSAInputs, device, out_dtype: Optional[str] = None) -> dict:
    """Uploads a block-sparse call: the keyword arguments of
    ``binding.qsa_msa_attention_ragged_paged``."""
    import torch

    d = to_torch(x, device, out_dtype)
    d.pop("token_indices")
    d.pop("counts")
    d["d_indices"] = torch.from_numpy(np.ascontiguousarray(x.d_indices, dtype=np.int32)).to(device)
    return d


# ----------------------------------------------------------------------------
# block-key compression (QSACompressKeysPaged): raw index keys -> block keys
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class CompressInputs:
    """One block-key compression call, host arrays in raw storage.  ``cache``
    holds the raw keys in a one-head paged cache (K at axis-1 index 0)."""

    name: str
    dtype: str        # keys, gamma and output
    freq_dtype: str
    cache: QSAInputs  # kv_flat / kv_shape / page_stride / table / cache_lengths / layer_idx
    key_counts: np.ndarray  # [batch] int32
    gamma: np.ndarray       # [head_dim] raw storage
    freqs_cis: np.ndarray   # [positions, rotary_dim] raw storage: cos, sin pairs
    max_blocks: int
    ratio: int
    rotary_dim: int
    eps: float

    @property
    def batch(self) -> int:
        return int(self.key_counts.shape[0])

    @property
    def head_dim(self) -> int:
        return int(self.cache.kv_shape[5])

    def algorithmic_bytes(self) -> int:
        """Raw keys of complete blocks read once, block keys written, plus
        gamma and the rotary rows used."""
        e = ELEM_BYTES[self.dtype]
        D = self.head_dim
        nblk = np.minimum(np.maximum(self.key_counts, 0) // self.ratio, self.max_blocks)
        return int(nblk.sum() * self.ratio * D * e + self.batch * self.max_blocks * D * e + D * e
                   + min(int(nblk.max()) if nblk.size else 0, self.freqs_cis.shape[0]) * self.rotary_dim
                   * ELEM_BYTES[self.freq_dtype])


def rope_table(positions: int, rotary_dim: int, theta: float = 10000.0) -> np.ndarray:
    """[positions, rotary_dim] cos/sin pairs: angle pos * theta^(-2k/rotary_dim)
    for pair k (the usual rotary frequencies)."""
    k = np.arange(rotary_dim // 2, dtype=np.float64)
    ang = np.arange(positions, dtype=np.float64)[:, None] * theta ** (-2.0 * k / max(rotary_dim, 1))[None, :]
    out = np.empty((positions, rotary_dim), np.float64)
    out[:, 0::2] = np.cos(ang)
    out[:, 1::2] = np.sin(ang)
    return out


@dataclasses.dataclass
class CompressSpec:
    name: str
    seed: int
    key_counts: Sequence[int]
    head_dim: int = 128
    page_size: int = 64
    num_layers: int = 1
    layer_idx: int = 0
    ratio: int = 4
    rotary_dim: int = 64
    dtype: str = "bf16"
    freq_dtype: str = "f32"
    eps: float = 1e-6
    extra_blocks: int = 2  # rows past the longest sequence's last block (written as zeros)
    page_pad: Optional[int] = None

    def build(self, keep_logical: bool = False) -> CompressInputs:
        rng = np.random.default_rng(self.seed)
        counts = np.asarray(self.key_counts, dtype=np.int64)
        B, D, P = counts.size, self.head_dim, self.page_size
        n_keys = np.maximum(counts, 0)
        perm = rng.permutation(int((-(-n_keys // P)).sum()))
        keys = [encode(rng.standard_normal((int(n), 1, D), dtype=np.float32), self.dtype) for n in n_keys]
        vals = [encode(np.zeros((int(n), 1, D), dtype=np.float32), self.dtype) for n in n_keys]
        cache = assemble(self.name, self.dtype, self.dtype, np.zeros((0, 1, D), np.float32).astype(_STORAGE[self.dtype]),
                         keys, vals, [0] * B, n_keys, P, self.num_layers, self.layer_idx,
                         np.zeros((0, 0), np.int32), np.zeros(0, np.int32), 1.0, page_perm=perm,
                         page_pad=self.page_pad, keep_logical=keep_logical)
        max_blocks = int((n_keys // self.ratio).max()) + self.extra_blocks if B else 0
        gamma = encode((1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32), self.dtype)
        freqs = rope_table(max(max_blocks, 1), self.rotary_dim)
        freqs = freqs.astype(np.float32) if self.freq_dtype == "f32" else encode(freqs.astype(np.float32), self.freq_dtype)
        return CompressInputs(name=self.name, dtype=self.dtype, freq_dtype=self.freq_dtype, cache=cache,
                              key_counts=counts.astype(np.int32), gamma=gamma, freqs_cis=np.ascontiguousarray(freqs),
                              max_blocks=max_blocks, ratio=self.ratio, rotary_dim=self.rotary_dim, eps=self.eps)


def compress_bf16(seed: int = 9, batch: int = 64, count_range=(1024, 65536), ratio: int = 4,
                  name: str = "compress_bf16") -> CompressSpec:
    """Block-key compression, bf16: 64 sequences of U[1024, 65536] raw index
    keys (head_dim 128), page 64, ratio 4, rotary over 64 channels."""
    rng = np.random.default_rng(seed + 1000)
    counts = rng.integers(count_range[0], count_range[1] + 1, size=batch)
    return CompressSpec(name=name, seed=seed, key_counts=counts.tolist(), ratio=ratio)


COMPRESS_WORKLOADS = {"compress_bf16": compress_bf16}


def compress_small_variants() -> dict:
    return {
        "compress_bf16_small": compress_bf16(seed=19, batch=5, count_range=(0, 300), name="compress_bf16_small"),
        "compress_f32_small": dataclasses.replace(
            compress_bf16(seed=20, batch=4, count_range=(3, 200), ratio=3, name="compress_f32_small"),
            dtype="f32", rotary_dim=128, page_size=16, page_pad=64),
    }


def to_torch_compress(x: CompressInputs, device) -> dict:
    """Uploads a block-key compression call: the keyword arguments of
    ``binding.qsa_compress_keys_paged`` (block_keys freshly allocated)."""
    import torch

    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}

    def raw(a: np.ndarray, dtype: str):
        a = np.ascontiguousarray(a)
        if dtype == "f32":
            return torch.from_numpy(a.astype(np.float32, copy=False))
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)

    c = x.cache
    d = to_torch(c, device)
    return dict(
        block_keys=torch.empty((x.batch * x.max_blocks, x.head_dim), dtype=tdt[x.dtype], device=device),
        gamma=raw(x.gamma, x.dtype).to(device),
        freqs_cis=raw(x.freqs_cis, x.freq_dtype).to(device),
        key_counts=torch.from_numpy(np.ascontiguousarray(x.key_counts, dtype=np.int32)).to(device),
        kv_blocks=d["kv_blocks"], page_stride=c.page_stride, cache_lengths=d["cache_lengths"],
        kv_lookup_table=d["kv_lookup_table"], max_prompt_length=0, max_cache_length=c.max_cache_length,
        layer_idx=c.layer_idx, ratio=x.ratio, rotary_dim=x.rotary_dim, eps=x.eps,
    )


# ----------------------------------------------------------------------------
# latent sparse attention: sliding window + listed compressed entries + sinks
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class LatentInputs:
    """One latent sparse attention call: ``swa`` holds q, the row offsets and
    the token-paged window cache (one latent head); ``comp`` the entry-paged
    compressed cache (its cache_lengths = entries per sequence)."""

    name: str
    swa: QSAInputs
    comp: QSAInputs
    comp_indices: np.ndarray  # [total_q, num_comp] int32, -1 = unused
    attn_sink: np.ndarray     # [num_heads] float32
    window: int

    @property
    def dtype(self) -> str:
        return self.swa.dtype

    @property
    def total_q(self) -> int:
        return self.swa.total_q

    @property
    def num_heads(self) -> int:
        return self.swa.num_q_heads

    def query_positions(self) -> np.ndarray:
        x = self.swa
        seq = x.row_sequence()
        off = x.input_row_offsets.astype(np.int64)
        return x.cache_lengths.astype(np.int64)[seq] + np.arange(x.total_q) - off[seq]

    def attended_keys(self) -> np.ndarray:
        pos = self.query_positions()
        win = np.minimum(pos + 1, self.window)
        return win + (self.comp_indices >= 0).sum(axis=1)

    def algorithmic_bytes(self) -> int:
        """Each attended K and V row once per row (one latent head), q, the
        output, the entry lists and the sinks."""
        x = self.swa
        e, eo = ELEM_BYTES[x.dtype], ELEM_BYTES[x.out_dtype]
        D = x.head_dim
        n = int(self.attended_keys().sum())
        return (n * 2 * D * e + x.total_q * x.num_q_heads * D * (e + eo) + self.comp_indices.size * 4
                + self.attn_sink.size * 4)


@dataclasses.dataclass
class LatentSpec:
    name: str
    seed: int
    rows: Sequence[int]
    cache_lengths: Sequence[int]
    num_heads: int
    window: int
    num_comp: int
    comp_ratio: int = 4       # compressed entries per sequence = (cache + rows) // comp_ratio
    head_dim: int = 128
    page_size: int = 64
    comp_page_size: int = 64
    num_layers: int = 1
    layer_idx: int = 0
    dtype: str = "bf16"
    out_dtype: str = "bf16"

    def build(self, keep_logical: bool = False) -> LatentInputs:
        rng = np.random.default_rng(self.seed)
        B = len(self.rows)
        rows = np.asarray(self.rows, dtype=np.int64)
        cache = np.asarray(self.cache_lengths, dtype=np.int64)
        H, D = self.num_heads, self.head_dim
        kv_len = cache + rows
        n_comp = kv_len // self.comp_ratio
        total_q = int(rows.sum())
        q = encode(rng.standard_normal((total_q, H, D), dtype=np.float32), self.dtype)
        lk = [encode(rng.standard_normal((int(n), 1, D), dtype=np.float32), self.dtype) for n in kv_len]
        lv = [encode(rng.standard_normal((int(n), 1, D), dtype=np.float32), self.dtype) for n in kv_len]
        ck = [encode(rng.standard_normal((int(n), 1, D), dtype=np.float32), self.dtype) for n in n_comp]
        cv = [encode(rng.standard_normal((int(n), 1, D), dtype=np.float32), self.dtype) for n in n_comp]
        idx = np.full((total_q, self.num_comp), -1, dtype=np.int32)
        seq = np.repeat(np.arange(B), rows)
        for r in range(total_q):
            n = int(n_comp[seq[r]])
            k = min(self.num_comp, n)
            if k:
                idx[r, :k] = rng.choice(n, size=k, replace=False)
        sink = rng.standard_normal(H).astype(np.float32)
        swa = assemble(self.name, self.dtype, self.out_dtype, q, lk, lv, rows, cache, self.page_size,
                       self.num_layers, self.layer_idx, np.zeros((total_q, 0), np.int32),
                       np.zeros(total_q, np.int32), 1.0 / math.sqrt(D),
                       page_perm=rng.permutation(int((-(-kv_len // self.page_size)).sum())), keep_logical=keep_logical)
        comp = assemble(self.name + "_comp", self.dtype, self.out_dtype, np.zeros((0, H, D), q.dtype), ck, cv,
                        [0] * B, n_comp, self.comp_page_size, self.num_layers, self.layer_idx,
                        np.zeros((0, 0), np.int32), np.zeros(0, np.int32), 1.0,
                        page_perm=rng.permutation(int((-(-n_comp // self.comp_page_size)).sum())),
                        keep_logical=keep_logical)
        return LatentInputs(name=self.name, swa=swa, comp=comp, comp_indices=idx, attn_sink=sink, window=self.window)


def latent_bf16_decode(seed: int = 10, batch: int = 64, cache_range=(2048, 32768), num_heads: int = 16,
                       window: int = 128, num_comp: int = 512, name: str = "latent_bf16_decode") -> LatentSpec:
    """Latent sparse attention, bf16 decode: 64 x 1 row, cache U[2048, 32768],
    16 query heads on one latent head of 128, window 128 tokens, 512 listed
    compressed entries of (kv_len // 4) per sequence, per-head sinks."""
    rng = np.random.default_rng(seed + 1000)
    cache = rng.integers(cache_range[0], cache_range[1] + 1, size=batch)
    return LatentSpec(name=name, seed=seed, rows=[1] * batch, cache_lengths=cache.tolist(), num_heads=num_heads,
                      window=window, num_comp=num_comp)


def latent_bf16_prefill(seed: int = 11, rows=(256, 512, 128), cache=(0, 2048, 8192), num_heads: int = 64,
                        window: int = 128, num_comp: int = 256, name: str = "latent_bf16_prefill") -> LatentSpec:
    """Latent sparse attention, bf16 chunked prefill: rows [256,512,128] on
    cache [0,2048,8192], 64 query heads (four groups of 16 on the one latent
    head), window 128, 256 listed compressed entries, per-head sinks."""
    return LatentSpec(name=name, seed=seed, rows=list(rows), cache_lengths=list(cache), num_heads=num_heads,
                      window=window, num_comp=num_comp)


LATENT_WORKLOADS = {"latent_bf16_decode": latent_bf16_decode, "latent_bf16_prefill": latent_bf16_prefill}


def latent_small_variants() -> dict:
    return {
        "latent_bf16_decode_small": latent_bf16_decode(seed=21, batch=5, cache_range=(40, 700), window=48,
                                                       num_comp=40, name="latent_bf16_decode_small"),
        "latent_bf16_prefill_small": latent_bf16_prefill(seed=22, rows=(17, 30, 5), cache=(0, 90, 300), num_heads=32,
                                                         window=24, num_comp=30, name="latent_bf16_prefill_small"),
        "latent_fp8_small": dataclasses.replace(
            latent_bf16_decode(seed=23, batch=4, cache_range=(100, 900), window=64, num_comp=24, num_heads=8,
                               name="latent_fp8_small"), dtype="e4m3", page_size=32, comp_page_size=16),
    }


def to_torch_latent(x: LatentInputs, device, out_dtype: Optional[str] = None) -> dict:
    """Uploads a latent sparse attention call: the keyword arguments of
    ``binding.qsa_latent_attention_ragged_paged``."""
    import torch

    a = to_torch(x.swa, device, out_dtype)
    c = to_torch(x.comp, device)
    return dict(
        output=a["output"], q=a["q"], input_row_offsets=a["input_row_offsets"], swa_blocks=a["kv_blocks"],
        swa_page_stride=x.swa.page_stride, swa_cache_lengths=a["cache_lengths"], swa_lookup_table=a["kv_lookup_table"],
        comp_blocks=c["kv_blocks"], comp_page_stride=x.comp.page_stride, comp_cache_lengths=c["cache_lengths"],
        comp_lookup_table=c["kv_lookup_table"], layer_idx=x.swa.layer_idx,
        comp_indices=torch.from_numpy(np.ascontiguousarray(x.comp_indices, dtype=np.int32)).to(device),
        attn_sink=torch.from_numpy(np.ascontiguousarray(x.attn_sink, dtype=np.float32)).to(device),
        window=x.window, scale=x.swa.scale,
    )
