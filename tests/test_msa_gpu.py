"""GPU parity of the block-sparse (MSA-style) entry point against the float64
block oracle, on the same seeded inputs: small variants under several split
counts, edge cases of the block lists, a missing page, page placement
(bit-exact), and sampled rows of the full-size block workloads.

Tolerances as for the token path: BF16 1e-2 + 1e-2|ref|, FP8 6e-2 + 3e-2|ref|.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import binding as B
from index_gathered_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-2), "e4m3": (6e-2, 3e-2)}
SMALL = wl.msa_small_variants()
LAUNCHES = [dict(), dict(splits=1), dict(splits=3), dict(splits=8)]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    B.qsa_read_device_status(clear=True)
    yield


def run_gpu(x, **kw) -> np.ndarray:
    d = wl.to_torch_msa(x, "cuda")
    B.qsa_msa_attention_ragged_paged(**d, **kw)
    torch.cuda.synchronize()
    return d["output"].float().cpu().double().numpy()


def assert_close(got, ref, dtype, what=""):
    atol, rtol = TOL[dtype]
    assert np.isfinite(got).all(), f"{what}: non-finite output (a poisoned byte was read)"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    assert (err <= bound).all(), f"{what}: {int((err > bound).sum())} of {err.size} outside tolerance"


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("launch", range(len(LAUNCHES)))
def test_small_block_workloads_match_oracle(name, launch):
    x = SMALL[name].build()
    assert_close(run_gpu(x, **LAUNCHES[launch]), oracle.msa_attention(x), x.dtype, f"{name} {LAUNCHES[launch]}")
    assert B.qsa_read_device_status(clear=True) == 0


@pytest.mark.parametrize("page_size", [32, 96, 192])
@pytest.mark.parametrize("base", ["msa_bf16_prefill_small", "msa_fp8_decode_small"])
def test_page_sizes_mix_tile_and_row_copies(base, page_size):
    """Blocks of 96 or 192 slots straddle the 64-key tiles: whole-page tiles
    (some starting mid-page) take tile copies, the straddling ones 16-byte
    copies; blocks of 32 slots take 16-byte copies only.  Bands merge in a
    cluster (3) or through the workspace tickets (12)."""
    x = dataclasses.replace(SMALL[base], page_size=page_size).build()
    ref = oracle.msa_attention(x)
    for kw in (dict(), dict(splits=3), dict(splits=12)):
        assert_close(run_gpu(x, **kw), ref, x.dtype, f"{base} P={page_size} {kw}")
        assert B.qsa_read_device_status(clear=True) == 0


def test_block_list_edge_cases():
    x = SMALL["msa_bf16_prefill_small"].build()
    P = x.kv_shape[3]
    pos = x.query_positions()
    d = x.d_indices.copy()
    d[0, 0, :] = -1  # kv head 0 of row 0 attends nothing: zero rows
    d[1, :, -1] = d[1, :, 0]  # a repeated block counts twice
    d[2, :, 0] = pos // P + 1  # a block wholly after the row's position adds nothing
    d[3, :, 1:3] = -1  # unused slots in the middle of a list
    y = dataclasses.replace(x, d_indices=d)
    for kw in (dict(), dict(splits=4)):
        got = run_gpu(y, **kw)
        assert_close(got, oracle.msa_attention(y), y.dtype, f"edge cases {kw}")
        assert not got[0, : x.group].any()
        assert B.qsa_read_device_status(clear=True) == 0


def test_missing_page_is_skipped_and_flagged():
    """A listed block whose table entry names no page of the kv_blocks
    descriptor is skipped and flagged.  The descriptor ends one page before
    the allocation and the entry names that last allocated (NaN-filled)
    page, so even a regressed check could not read outside the cache."""
    x = SMALL["msa_bf16_decode_small"].build()
    seq = x.row_sequence()
    b, blk = int(seq[1]), int(x.d_indices[0, 1, 0])
    tab = x.kv_lookup_table.copy()
    assert x.poison_page == x.kv_shape[0] - 1
    tab[b, blk] = x.poison_page
    bad = dataclasses.replace(x, kv_lookup_table=tab)
    d = wl.to_torch_msa(bad, "cuda")
    d["kv_blocks"] = d["kv_blocks"][: x.poison_page]  # the descriptor's pages stop before the poison page
    B.qsa_msa_attention_ragged_paged(**d)
    torch.cuda.synchronize()
    got = d["output"].float().cpu().double().numpy()
    assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_PAGE
    d = x.d_indices.copy()  # the expected result: that block unlisted wherever this sequence lists it
    rows = np.nonzero(seq == b)[0]
    sub = d[:, rows]
    sub[sub == blk] = -1
    d[:, rows] = sub
    assert_close(got, oracle.msa_attention(dataclasses.replace(x, d_indices=d)), x.dtype, "missing page")


def test_page_placement_is_bit_exact():
    spec = SMALL["msa_fp8_decode_small"]
    a = run_gpu(spec.build())
    b = run_gpu(dataclasses.replace(spec, page_pad=None).build())
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("name", sorted(wl.MSA_WORKLOADS))
def test_full_size_block_workload_sampled_rows(name):
    x = wl.MSA_WORKLOADS[name]().build()
    got = run_gpu(x)
    rows = np.unique(np.linspace(0, x.total_q - 1, 6).astype(np.int64))
    assert_close(got[rows], oracle.msa_attention(x, rows), x.dtype, name)
    assert B.qsa_read_device_status(clear=True) == 0
