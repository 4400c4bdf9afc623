"""The block-sparse entry point's argument checks, without a GPU: every
malformed call returns its status code before any CUDA work."""
import ctypes

import pytest

from index_gathered_sparse_gb300 import binding as B

FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    from index_gathered_sparse_gb300 import build

    build.build()
    return B.load_library()


def _t(shape, code, data=FAKE):
    d = B.qsa_tensor()
    d.data = data
    d.dtype = code
    d.ndim = len(shape)
    for i, s in enumerate(shape):
        d.shape[i] = s
    return d


def _call(lib, kernel=0, **over):
    """A consistent call: total_q 5, 8 q heads on 2 kv heads, head_dim 128,
    10 pages of 16 slots, 3 layers, topk 4 blocks."""
    a = dict(
        output=_t((5, 8, 128), B.QSA_BF16), q=_t((5, 8, 128), B.QSA_BF16),
        input_row_offsets=_t((3,), B.QSA_U32), kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_BF16),
        page_stride=-1, cache_lengths=_t((2,), B.QSA_U32), kv_lookup_table=_t((2, 4), B.QSA_U32),
        max_prompt_length=4, max_cache_length=40, layer_idx=2, d_indices=_t((2, 5, 4), B.QSA_I32),
        scale=0.125, group=4, stream=None,
    )
    a.update(over)
    order = ["output", "q", "input_row_offsets", "kv_blocks", "page_stride", "cache_lengths", "kv_lookup_table",
             "max_prompt_length", "max_cache_length", "layer_idx", "d_indices", "scale", "group", "stream"]
    opt = B.qsa_options(kernel=kernel, splits=0, ctas=0)
    return lib.qsa_msa_attention_ragged_paged(*[a[k] for k in order], ctypes.byref(opt))


CASES = {
    "d_indices_rank": (dict(d_indices=_t((2, 5), B.QSA_I32)), 2),
    "d_indices_dtype": (dict(d_indices=_t((2, 5, 4), B.QSA_U32)), 3),
    "d_indices_heads": (dict(d_indices=_t((3, 5, 4), B.QSA_I32)), 2),
    "d_indices_rows": (dict(d_indices=_t((2, 6, 4), B.QSA_I32)), 2),
    "d_indices_null": (dict(d_indices=_t((2, 5, 4), B.QSA_I32, data=None)), 1),
    "group_mismatch": (dict(group=3), 2),
    "f32_cache": (dict(q=_t((5, 8, 128), B.QSA_F32), kv_blocks=_t((10, 2, 3, 16, 2, 128), B.QSA_F32)), 4),
    "head_dim_64": (dict(output=_t((5, 8, 64), B.QSA_BF16), q=_t((5, 8, 64), B.QSA_BF16),
                         kv_blocks=_t((10, 2, 3, 16, 2, 64), B.QSA_BF16)), 4),
    "layer_out_of_range": (dict(layer_idx=3), 5),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_rejects_malformed_call(lib, case):
    over, want = CASES[case]
    assert _call(lib, **over) == want, B.load_library().qsa_last_error_message().decode()


@pytest.mark.parametrize("kernel", [1, 3, 7])
def test_block_lists_run_on_kernel_2_only(lib, kernel):
    assert _call(lib, kernel=kernel) == 4
