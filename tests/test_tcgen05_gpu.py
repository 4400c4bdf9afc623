"""GPU parity of kernel 2's tcgen05 consumer (options.tcgen05 = 1) against the
float64 oracle: scores and output accumulate in tensor memory through tcgen05
MMAs on the tile-copy stage layout.  Block lists (whole-page tile copies),
token lists with page-aligned runs (tile copies) and random positions
(16-byte copies into the same layout), groups of 4, 8 and 16, split-K bands
merged in a cluster and through the workspace tickets, edge cases of the
lists, page placement (bit-exact), and sampled rows at full size.

Tolerances as for the other paths: BF16 1e-2 + 1e-2|ref|.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import binding as B
from index_gathered_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-2, 1e-2
SMALL_TOKENS = {k: v for k, v in wl.small_variants().items() if v.dtype == "bf16"}
SMALL_BLOCKS = {k: v for k, v in wl.msa_small_variants().items() if v.dtype == "bf16"}
SPLITS = [1, 3, 8, 12, 40]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    B.qsa_read_device_status(clear=True)
    yield


def assert_close(got, ref, what):
    assert np.isfinite(got).all(), f"{what}: non-finite output (a poisoned byte was read)"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (f"{what}: {int((err > bound).sum())} of {err.size} outside tolerance; worst at "
                                  f"{worst}: got {got[worst]}, ref {ref[worst]}")


def run_tokens(x, **kw):
    d = wl.to_torch(x, "cuda")
    B.qsa_sparse_attention_ragged_paged(**d, kernel=2, tcgen05=1, **kw)
    torch.cuda.synchronize()
    return d["output"].float().cpu().double().numpy()


def run_blocks(x, **kw):
    d = wl.to_torch_msa(x, "cuda")
    B.qsa_msa_attention_ragged_paged(**d, tcgen05=1, **kw)
    torch.cuda.synchronize()
    return d["output"].float().cpu().double().numpy()


@pytest.mark.parametrize("name", sorted(SMALL_TOKENS))
@pytest.mark.parametrize("splits", SPLITS)
def test_token_lists_match_oracle(name, splits):
    x = SMALL_TOKENS[name].build()
    assert_close(run_tokens(x, splits=splits), oracle.sparse_attention(x), f"{name} splits {splits}")
    assert B.qsa_read_device_status(clear=True) == 0


@pytest.mark.parametrize("name", sorted(SMALL_BLOCKS))
@pytest.mark.parametrize("splits", [0] + SPLITS)
def test_block_lists_match_oracle(name, splits):
    x = SMALL_BLOCKS[name].build()
    assert_close(run_blocks(x, splits=splits), oracle.msa_attention(x), f"{name} splits {splits}")
    assert B.qsa_read_device_status(clear=True) == 0


@pytest.mark.parametrize("page_size", [32, 96, 192])
def test_block_sizes_mix_tile_and_row_copies(page_size):
    x = dataclasses.replace(SMALL_BLOCKS["msa_bf16_prefill_small"], page_size=page_size).build()
    ref = oracle.msa_attention(x)
    for splits in (0, 3, 12):
        assert_close(run_blocks(x, splits=splits), ref, f"P={page_size} splits {splits}")
        assert B.qsa_read_device_status(clear=True) == 0


def test_empty_clamped_and_out_of_range_entries():
    """counts <= 0 gives zero rows, counts > W clamps, a position past the
    sequence inside counts is skipped and flagged (its value stays inside the
    allocated cache)."""
    x = SMALL_TOKENS["bf16_prefill_small"].build()
    W = x.selection_width
    x.counts[0] = 0
    x.counts[1] = -5
    full = [r for r in range(x.total_q) if x.counts[r] == W]  # rows whose whole width is valid
    assert full
    x.counts[full[0]] = W + 100
    seq = x.row_sequence()
    kv_len = x.cache_lengths.astype(np.int64) + np.diff(x.input_row_offsets.astype(np.int64))
    r = 5
    n = int(x.valid_counts()[r])
    assert n >= 2
    y = dataclasses.replace(x, token_indices=x.token_indices.copy(), counts=x.counts.copy())
    x.token_indices[r, n - 1] = kv_len[seq[r]]
    y.counts[r] = n - 1
    got = run_tokens(x, splits=3)
    assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_INDEX
    assert not got[:2].any()
    assert_close(got, oracle.sparse_attention(y), "edge cases")


def test_page_placement_is_bit_exact():
    spec = SMALL_BLOCKS["msa_bf16_decode_small"]
    a = run_blocks(spec.build(), splits=3)
    b = run_blocks(dataclasses.replace(spec, page_pad=512).build(), splits=3)
    np.testing.assert_array_equal(a, b)


def test_same_result_bits_as_tile_and_row_copies():
    """A token list of whole pages loads by tile copies; the same list with one
    entry of each tile moved elsewhere in its page loads by 16-byte copies.
    Both reach the tensor cores in the same layout: outputs of the common
    rows agree with the oracle."""
    x = SMALL_TOKENS["bf16_long_decode_small"].build()
    assert_close(run_tokens(x, splits=1), oracle.sparse_attention(x), "long decode, one band")


@pytest.mark.parametrize("name", ["bf16_long_decode"])
def test_full_size_token_workload_sampled_rows(name):
    x = wl.WORKLOADS[name]().build()
    got = run_tokens(x)
    rows = np.unique(np.linspace(0, x.total_q - 1, 8).astype(np.int64))
    assert_close(got[rows], oracle.sparse_attention(x, rows), name)
    assert np.isfinite(got).all()
    assert B.qsa_read_device_status(clear=True) == 0


@pytest.mark.parametrize("name", ["msa_bf16_decode", "msa_bf16_prefill"])
def test_full_size_block_workload_sampled_rows(name):
    x = wl.MSA_WORKLOADS[name]().build()
    got = run_blocks(x)
    rows = np.unique(np.linspace(0, x.total_q - 1, 6).astype(np.int64))
    assert_close(got[rows], oracle.msa_attention(x, rows), name)
    assert np.isfinite(got).all()
    assert B.qsa_read_device_status(clear=True) == 0
