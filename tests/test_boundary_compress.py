"""Block-key compression's argument checks, without a GPU: each malformed
call returns its status code before any CUDA work."""
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


def _call(lib, **over):
    """A consistent call: batch 3, max_blocks 10, head_dim 128, 20 pages of 64
    slots, 2 layers, ratio 4, rotary over 64 channels."""
    a = dict(
        block_keys=_t((30, 128), B.QSA_BF16), gamma=_t((128,), B.QSA_BF16), freqs_cis=_t((10, 64), B.QSA_F32),
        key_counts=_t((3,), B.QSA_I32), kv_blocks=_t((20, 2, 2, 64, 1, 128), B.QSA_BF16), page_stride=-1,
        cache_lengths=_t((3,), B.QSA_U32), kv_lookup_table=_t((3, 7), B.QSA_U32), max_prompt_length=0,
        max_cache_length=400, layer_idx=1, ratio=4, rotary_dim=64, eps=1e-6, stream=None,
    )
    a.update(over)
    order = ["block_keys", "gamma", "freqs_cis", "key_counts", "kv_blocks", "page_stride", "cache_lengths",
             "kv_lookup_table", "max_prompt_length", "max_cache_length", "layer_idx", "ratio", "rotary_dim", "eps",
             "stream"]
    return lib.qsa_compress_keys_paged(*[a[k] for k in order])


CASES = {
    "rows_not_multiple_of_batch": (dict(block_keys=_t((31, 128), B.QSA_BF16)), 2),
    "two_kv_heads": (dict(kv_blocks=_t((20, 2, 2, 64, 2, 128), B.QSA_BF16)), 2),
    "gamma_extent": (dict(gamma=_t((64,), B.QSA_BF16)), 2),
    "freqs_width": (dict(freqs_cis=_t((10, 32), B.QSA_F32)), 2),
    "freqs_too_few_positions": (dict(freqs_cis=_t((9, 64), B.QSA_F32)), 2),
    "table_rows": (dict(kv_lookup_table=_t((2, 7), B.QSA_U32)), 2),
    "fp8_keys": (dict(block_keys=_t((30, 128), B.QSA_F8E4M3), gamma=_t((128,), B.QSA_F8E4M3),
                      kv_blocks=_t((20, 2, 2, 64, 1, 128), B.QSA_F8E4M3)), 3),
    "gamma_dtype": (dict(gamma=_t((128,), B.QSA_F32)), 3),
    "counts_dtype": (dict(key_counts=_t((3,), B.QSA_U32)), 3),
    "ratio_zero": (dict(ratio=0), 5),
    "ratio_above_64": (dict(ratio=65), 4),
    "rotary_odd": (dict(rotary_dim=63, freqs_cis=_t((10, 63), B.QSA_F32)), 5),
    "rotary_too_wide": (dict(rotary_dim=130, freqs_cis=_t((10, 130), B.QSA_F32)), 5),
    "layer_out_of_range": (dict(layer_idx=2), 5),
    "negative_eps": (dict(eps=-1.0), 5),
    "head_dim_64": (dict(block_keys=_t((30, 64), B.QSA_BF16), gamma=_t((64,), B.QSA_BF16),
                         kv_blocks=_t((20, 2, 2, 64, 1, 64), B.QSA_BF16)), 4),
    "null_keys": (dict(block_keys=_t((30, 128), B.QSA_BF16, data=None)), 1),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_rejects_malformed_call(lib, case):
    over, want = CASES[case]
    assert _call(lib, **over) == want, B.load_library().qsa_last_error_message().decode()


def test_empty_output_is_a_no_op(lib):
    assert _call(lib, block_keys=_t((0, 128), B.QSA_BF16), freqs_cis=_t((0, 64), B.QSA_F32)) == 0
