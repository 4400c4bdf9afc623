"""GPU parity of block-key compression against the float64 oracle: small
variants (bf16 and f32 keys, ragged counts, incomplete blocks, zero rows),
a key with no page, page placement (bit-exact), and sampled rows of the
full-size workload.  Tolerances: BF16 1e-2 + 1e-2|ref|, F32 1e-4."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import binding as B
from index_gathered_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-2), "f32": (1e-4, 0.0)}
SMALL = wl.compress_small_variants()


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    B.qsa_read_device_status(clear=True)
    yield


def run_gpu(x) -> np.ndarray:
    d = wl.to_torch_compress(x, "cuda")
    B.qsa_compress_keys_paged(**d)
    torch.cuda.synchronize()
    return d["block_keys"].float().cpu().double().numpy()


def assert_close(got, ref, dtype, what):
    atol, rtol = TOL[dtype]
    assert np.isfinite(got).all(), what
    err, bound = np.abs(got - ref), atol + rtol * np.abs(ref)
    assert (err <= bound).all(), f"{what}: {int((err > bound).sum())} of {err.size} outside tolerance"


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_compress_matches_oracle(name):
    x = SMALL[name].build()
    got = run_gpu(x)
    ref = oracle.compress_keys(x)
    assert_close(got, ref, x.dtype, name)
    assert not got[np.all(ref == 0, axis=1)].any()  # incomplete and missing blocks: exact zero rows
    assert B.qsa_read_device_status(clear=True) == 0


@pytest.mark.parametrize("ratio,rotary", [(1, 128), (5, 0), (16, 64)])
def test_ratios_and_rotary_widths(ratio, rotary):
    x = dataclasses.replace(SMALL["compress_bf16_small"], ratio=ratio, rotary_dim=rotary).build()
    assert_close(run_gpu(x), oracle.compress_keys(x), x.dtype, f"ratio {ratio} rotary {rotary}")


def test_key_without_page_zeroes_its_block_and_flags():
    """The first page of sequence 1 names no page of the kv_blocks
    descriptor: its blocks are zero and flagged.  The descriptor ends one
    page before the allocation and the entry names that last allocated
    (NaN-filled) page, so even a regressed check could not read outside the
    cache."""
    x = SMALL["compress_f32_small"].build()
    tab = x.cache.kv_lookup_table.copy()
    assert x.cache.poison_page == x.cache.kv_shape[0] - 1
    tab[1, 0] = x.cache.poison_page
    y = dataclasses.replace(x, cache=dataclasses.replace(x.cache, kv_lookup_table=tab))
    d = wl.to_torch_compress(y, "cuda")
    d["kv_blocks"] = d["kv_blocks"][: x.cache.poison_page]  # the descriptor's pages stop before the poison page
    B.qsa_compress_keys_paged(**d)
    torch.cuda.synchronize()
    got = d["block_keys"].float().cpu().double().numpy()
    assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_PAGE
    ref = oracle.compress_keys(x)
    P = x.cache.kv_shape[3]
    hit = np.zeros(x.batch * x.max_blocks, bool)  # blocks of sequence 1 with a key on that page
    for i in range(x.max_blocks):
        hit[1 * x.max_blocks + i] = i * x.ratio < P
    assert not got[hit].any()
    assert_close(got[~hit], ref[~hit], x.dtype, "other blocks")


def test_page_placement_is_bit_exact():
    spec = SMALL["compress_bf16_small"]
    np.testing.assert_array_equal(run_gpu(spec.build()), run_gpu(dataclasses.replace(spec, page_pad=256).build()))


def test_full_size_compress_sampled_rows():
    x = wl.COMPRESS_WORKLOADS["compress_bf16"]().build()
    got = run_gpu(x)
    ref = oracle.compress_keys(x)  # the whole output: one pass over the raw keys in C
    rows = np.unique(np.linspace(0, got.shape[0] - 1, 4096).astype(np.int64))
    assert_close(got[rows], ref[rows], x.dtype, "compress_bf16")
    assert B.qsa_read_device_status(clear=True) == 0
