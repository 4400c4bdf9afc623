"""The C ABI without a GPU: the library loads, exports what include/qsa.h
declares, and rejects every malformed call with its status code before any
CUDA work ("Raises: Error: If the operand shapes disagree with the
parameters", QSASparseAttentionRaggedPaged)."""
import ctypes

import pytest

from index_gathered_sparse_gb300 import binding as B


@pytest.fixture(scope="module")
def lib():
    from index_gathered_sparse_gb300 import build

    build.build()
    return B.load_library()


def test_exports_every_declared_symbol(lib):
    names = B.exported_names()
    assert "qsa_sparse_attention_ragged_paged" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert B.qsa_version() == 1
    assert B.qsa_status_string(2) == "QSA_ERR_SHAPE"
    assert B.qsa_status_string(99) == "QSA_ERR_UNKNOWN"


FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced


def _t(shape, code, data=FAKE):
    d = B.qsa_tensor()
    d.data = data
    d.dtype = code
    d.ndim = len(shape)
    for i, s in enumerate(shape):
        d.shape[i] = s
    return d


def _args(**over):
    """A consistent call: batch 2, total_q 5, 8 q heads on 2 kv heads (group
    4), head_dim 128, 10 pages of 16 slots, 3 layers, selection width 32."""
    a = dict(
        output=_t((5, 8, 128), B.QSA_BF16), q=_t((5, 8, 128), B.QSA_BF16),
        input_row_offsets=_t((3,), B.QSA_U32), kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_BF16),
        page_stride=-1, cache_lengths=_t((2,), B.QSA_U32), kv_lookup_table=_t((2, 4), B.QSA_U32),
        max_prompt_length=4, max_cache_length=40, layer_idx=2, token_indices=_t((5, 32), B.QSA_I32),
        counts=_t((5,), B.QSA_I32), scale=0.125, group=4, stream=None,
    )
    a.update(over)
    return a


def _call(lib, **over):
    a = _args(**over)
    order = ["output", "q", "input_row_offsets", "kv_blocks", "page_stride", "cache_lengths", "kv_lookup_table",
             "max_prompt_length", "max_cache_length", "layer_idx", "token_indices", "counts", "scale", "group",
             "stream"]
    return lib.qsa_sparse_attention_ragged_paged(*[a[k] for k in order])


CASES = {
    "group_mismatch": (dict(group=3), 2),
    "zero_group": (dict(group=0), 2),
    "q_rank": (dict(q=_t((5, 8), B.QSA_BF16)), 2),
    "output_shape": (dict(output=_t((5, 8, 64), B.QSA_BF16)), 2),
    "kv_axis1": (dict(kv_blocks=_t((10, 3, 3, 16, 2, 128), B.QSA_BF16)), 2),
    "kv_head_dim": (dict(kv_blocks=_t((10, 2, 3, 16, 2, 64), B.QSA_BF16)), 2),
    "offsets_extent": (dict(input_row_offsets=_t((2,), B.QSA_U32)), 2),
    "table_rows": (dict(kv_lookup_table=_t((3, 4), B.QSA_U32)), 2),
    "indices_rows": (dict(token_indices=_t((4, 32), B.QSA_I32)), 2),
    "counts_extent": (dict(counts=_t((6,), B.QSA_I32)), 2),
    "rows_without_batch": (dict(cache_lengths=_t((0,), B.QSA_U32), input_row_offsets=_t((1,), B.QSA_U32),
                                kv_lookup_table=_t((0, 4), B.QSA_U32)), 2),
    "kv_dtype_differs": (dict(kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_F32)), 3),
    "q_integer": (dict(q=_t((5, 8, 128), B.QSA_I32), kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_I32)), 3),
    "output_fp8": (dict(output=_t((5, 8, 128), B.QSA_F8E4M3)), 3),
    "offsets_i32": (dict(input_row_offsets=_t((3,), B.QSA_I32)), 3),
    "indices_u32": (dict(token_indices=_t((5, 32), B.QSA_U32)), 3),
    "counts_f32": (dict(counts=_t((5,), B.QSA_F32)), 3),
    "null_q": (dict(q=_t((5, 8, 128), B.QSA_BF16, data=None)), 1),
    "null_kv": (dict(kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_BF16, data=None)), 1),
    "null_offsets": (dict(input_row_offsets=_t((3,), B.QSA_U32, data=None)), 1),
    "layer_out_of_range": (dict(layer_idx=3), 5),
    "page_stride_small": (dict(page_stride=2 * 3 * 16 * 2 * 128 - 8), 5),
    "page_stride_negative": (dict(page_stride=-2), 5),
    "head_dim_96": (dict(q=_t((5, 8, 96), B.QSA_BF16), output=_t((5, 8, 96), B.QSA_BF16),
                     kv_blocks=_t((10, 2, 3, 16, 2, 96), B.QSA_BF16)), 4),
    "group_17": (dict(q=_t((5, 34, 128), B.QSA_BF16), output=_t((5, 34, 128), B.QSA_BF16), group=17), 4),
    "misaligned_kv": (dict(kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_BF16, data=FAKE + 8)), 4),
    "page_stride_unaligned": (dict(page_stride=2 * 3 * 16 * 2 * 128 + 4), 4),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_rejects_bad_call_before_launch(lib, case):
    over, code = CASES[case]
    status = _call(lib, **over)
    assert status == code, (case, B.STATUS_NAMES.get(status), lib.qsa_last_error_message())
    assert lib.qsa_last_error_message()


def test_empty_call_is_a_no_op(lib):
    """total_q == 0 checks the descriptors and returns without touching CUDA."""
    st = _call(lib, output=_t((0, 8, 128), B.QSA_BF16, data=None), q=_t((0, 8, 128), B.QSA_BF16, data=None),
               token_indices=_t((0, 32), B.QSA_I32, data=None), counts=_t((0,), B.QSA_I32, data=None),
               input_row_offsets=_t((3,), B.QSA_U32))
    assert st == 0


def test_forced_kernel_limits(lib):
    opt = B.qsa_options(kernel=2)
    a = _args(q=_t((5, 8, 128), B.QSA_F32), kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_F32),
              output=_t((5, 8, 128), B.QSA_F32))
    order = ["output", "q", "input_row_offsets", "kv_blocks", "page_stride", "cache_lengths", "kv_lookup_table",
             "max_prompt_length", "max_cache_length", "layer_idx", "token_indices", "counts", "scale", "group",
             "stream"]
    st = lib.qsa_sparse_attention_ragged_paged_ex(*[a[k] for k in order], ctypes.byref(opt))
    assert st == 4  # FP32 has no tensor-core kernel (its 1e-4 tolerance rules out TF32)
    opt = B.qsa_options(kernel=1, splits=4)
    st = lib.qsa_sparse_attention_ragged_paged_ex(*[_args()[k] for k in order], ctypes.byref(opt))
    assert st == 4
    opt = B.qsa_options(kernel=7)
    st = lib.qsa_sparse_attention_ragged_paged_ex(*[_args()[k] for k in order], ctypes.byref(opt))
    assert st == 5


def test_launch_option_limits(lib):
    """The launch controls added for tests and sweeps are checked with the
    arguments, before anything is launched."""
    order = ["output", "q", "input_row_offsets", "kv_blocks", "page_stride", "cache_lengths", "kv_lookup_table",
             "max_prompt_length", "max_cache_length", "layer_idx", "token_indices", "counts", "scale", "group",
             "stream"]

    def ex(opt, **over):
        return lib.qsa_sparse_attention_ragged_paged_ex(*[_args(**over)[k] for k in order], ctypes.byref(opt))

    e4m3 = dict(q=_t((5, 8, 128), B.QSA_F8E4M3), kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_F8E4M3))
    cases = [
        (B.qsa_options(kernel=3, heads_per_unit=3), {}, 5),   # not 1, 2, 4 or 8
        (B.qsa_options(kernel=3, heads_per_unit=4), {}, 5),   # does not divide 2 kv heads
        (B.qsa_options(kernel=2, heads_per_unit=2), {}, 4),   # only the persistent kernel groups heads
        (B.qsa_options(kernel=1, test_stall=1), {}, 4),       # only the persistent kernel stalls
        (B.qsa_options(kernel=2, tcgen05=2), {}, 5),          # -1, 0 or 1
        (B.qsa_options(kernel=3, tcgen05=1), {}, 4),          # only kernel 2 has the tcgen05 consumer
        (B.qsa_options(kernel=2, tcgen05=1), e4m3, 4),        # which reads BF16 caches
        # the row-group kernel: BF16, head_dim 128, group 4, 8 or 16, a power-of-two page of >= 8 slots,
        # bitmaps of at most 1 Mi positions; none of the other kernels' controls
        (B.qsa_options(kernel=4), e4m3, 4),
        (B.qsa_options(kernel=4), dict(q=_t((5, 4, 128), B.QSA_BF16), output=_t((5, 4, 128), B.QSA_BF16), group=2), 4),
        (B.qsa_options(kernel=4), dict(kv_blocks=_t((10, 2, 3, 12, 2, 128), B.QSA_BF16)), 4),
        (B.qsa_options(kernel=4), dict(kv_blocks=_t((10, 2, 3, 4, 2, 128), B.QSA_BF16)), 4),
        (B.qsa_options(kernel=4), dict(max_cache_length=(1 << 20)), 4),
        (B.qsa_options(kernel=4, splits=2), {}, 4),
        (B.qsa_options(kernel=4, ctas=3), {}, 4),
        (B.qsa_options(kernel=4, heads_per_unit=2), {}, 4),
        (B.qsa_options(kernel=4, tcgen05=1), {}, 4),
        (B.qsa_options(kernel=5), {}, 5),
    ]
    for opt, over, code in cases:
        st = ex(opt, **over)
        assert st == code, (opt.kernel, opt.heads_per_unit, opt.test_stall, opt.tcgen05, B.STATUS_NAMES.get(st),
                            lib.qsa_last_error_message())


def test_plan_without_extents_never_plans_the_row_group_kernel(lib):
    """qsa_plan has no page size or length hints: forcing kernel 4 there is
    refused before any CUDA call; qsa_plan_ex checks its extra extents."""
    opt = B.qsa_options(kernel=4)
    k, s = ctypes.c_int32(), ctypes.c_int32()
    c, w = ctypes.c_int64(), ctypes.c_size_t()
    outs = (ctypes.byref(k), ctypes.byref(s), ctypes.byref(c), ctypes.byref(w))
    assert lib.qsa_plan(B.QSA_BF16, 64, 8, 128, 256, 8, ctypes.byref(opt), *outs) == 4
    assert b"qsa_plan_ex" in lib.qsa_last_error_message()
    assert lib.qsa_plan_ex(B.QSA_BF16, 64, 0, 8, 128, 64, 256, 8, 16, 100, ctypes.byref(opt), *outs) == 2  # no batch
    assert lib.qsa_plan_ex(B.QSA_BF16, 64, 2, 8, 128, 0, 256, 8, 16, 100, ctypes.byref(opt), *outs) == 2  # no page
    assert lib.qsa_plan_ex(B.QSA_BF16, 64, 2, 8, 128, 48, 256, 8, 16, 100, ctypes.byref(opt), *outs) == 4
