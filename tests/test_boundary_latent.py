"""Latent sparse attention's argument checks, without a GPU."""
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


def _call(lib, kernel=0, ctas=0, **over):
    """A consistent call: batch 2, total_q 5, 32 heads (two groups of 16),
    head_dim 128, window 64, 10 entries per row (compressed-cache arrays and
    sinks as plain pointers)."""
    a = dict(
        output=_t((5, 32, 128), B.QSA_BF16), q=_t((5, 32, 128), B.QSA_BF16), input_row_offsets=_t((3,), B.QSA_U32),
        swa_blocks=_t((12, 2, 2, 64, 1, 128), B.QSA_BF16), swa_page_stride=-1, swa_cache_lengths=_t((2,), B.QSA_U32),
        swa_lookup_table=_t((2, 6), B.QSA_U32), comp_blocks=_t((4, 2, 2, 32, 1, 128), B.QSA_BF16),
        comp_page_stride=-1, comp_cache_lengths=FAKE, comp_lookup_table=FAKE, comp_max_pages=2,
        layer_idx=1, comp_indices=FAKE, num_comp=10, attn_sink=FAKE, window=64, scale=0.1,
        stream=None,
    )
    a.update(over)
    order = ["output", "q", "input_row_offsets", "swa_blocks", "swa_page_stride", "swa_cache_lengths",
             "swa_lookup_table", "comp_blocks", "comp_page_stride", "comp_cache_lengths", "comp_lookup_table",
             "comp_max_pages", "layer_idx", "comp_indices", "num_comp", "attn_sink", "window", "scale", "stream"]
    opt = B.qsa_options(kernel=kernel, splits=0, ctas=ctas)
    return lib.qsa_latent_attention_ragged_paged(*[a[k] for k in order], ctypes.byref(opt))


CASES = {
    "two_swa_heads": (dict(swa_blocks=_t((12, 2, 2, 64, 2, 128), B.QSA_BF16)), 2),
    "comp_head_dim": (dict(comp_blocks=_t((4, 2, 2, 32, 1, 64), B.QSA_BF16)), 2),
    "sink_null": (dict(attn_sink=None), 1),
    "null_entries": (dict(comp_indices=None), 1),
    "null_comp_lengths": (dict(comp_cache_lengths=None), 1),
    "negative_num_comp": (dict(num_comp=-1), 2),
    "cache_dtype_differs": (dict(comp_blocks=_t((4, 2, 2, 32, 1, 128), B.QSA_F8E4M3)), 3),
    "f32_q": (dict(q=_t((5, 32, 128), B.QSA_F32), output=_t((5, 32, 128), B.QSA_F32),
                   swa_blocks=_t((12, 2, 2, 64, 1, 128), B.QSA_F32), comp_blocks=_t((4, 2, 2, 32, 1, 128), B.QSA_F32)), 4),
    "heads_not_multiple_of_16": (dict(q=_t((5, 24, 128), B.QSA_BF16), output=_t((5, 24, 128), B.QSA_BF16),
                                      ), 4),
    "negative_window": (dict(window=-1), 5),
    "layer_past_comp_layers": (dict(comp_blocks=_t((4, 2, 1, 32, 1, 128), B.QSA_BF16)), 5),
    "null_q": (dict(q=_t((5, 32, 128), B.QSA_BF16, data=None)), 1),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_rejects_malformed_call(lib, case):
    over, want = CASES[case]
    assert _call(lib, **over) == want, B.load_library().qsa_last_error_message().decode()


def test_options(lib):
    assert _call(lib, kernel=3) == 4
    assert _call(lib, ctas=5) == 5
