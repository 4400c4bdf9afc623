"""Pins of the block-key compression oracle, independent of its own code.

- Each block key equals the composition of library routines on the unpaged
  raw keys: torch mean over the block's keys -> torch rms_norm with gamma and
  eps -> a complex multiply (numpy) of channel pairs by cos + i sin.
- Closed forms and invariants: a rotation keeps every pair's length; with the
  identity rotation the output divided by gamma has mean square
  ms / (ms + eps); identical raw keys pool to themselves; incomplete and
  missing blocks are zero rows; page placement does not matter.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import workloads as wl

SMALL = wl.compress_small_variants()


@pytest.fixture(scope="module", autouse=True)
def _build():
    oracle.build()


def library_reference(x) -> np.ndarray:
    D, R = x.head_dim, x.rotary_dim
    gamma = torch.from_numpy(oracle.decode(x.gamma, x.dtype))
    fr = oracle.decode(x.freqs_cis, x.freq_dtype)
    out = np.zeros((x.batch * x.max_blocks, D))
    for b in range(x.batch):
        raw = torch.from_numpy(oracle.decode(x.cache.logical_k[b], x.dtype)[:, 0, :])
        for i in range(min(raw.shape[0] // x.ratio, x.max_blocks)):
            pooled = raw[i * x.ratio:(i + 1) * x.ratio].mean(dim=0)
            y = torch.nn.functional.rms_norm(pooled, (D,), weight=gamma, eps=x.eps).numpy()
            z = (y[0:R:2] + 1j * y[1:R:2]) * (fr[i, 0::2] + 1j * fr[i, 1::2])
            y = y.copy()
            y[0:R:2], y[1:R:2] = z.real, z.imag
            out[b * x.max_blocks + i] = y
    return out


@pytest.mark.parametrize("name", sorted(SMALL))
def test_matches_library_composition(name):
    x = SMALL[name].build(keep_logical=True)
    np.testing.assert_allclose(oracle.compress_keys(x), library_reference(x), rtol=1e-10, atol=1e-12)


def test_rotation_keeps_pair_lengths_and_identity_rotation_normalises():
    x = SMALL["compress_f32_small"].build()
    ident = np.zeros_like(x.freqs_cis)
    ident[:, 0::2] = 1.0
    a = oracle.compress_keys(x)
    b = oracle.compress_keys(dataclasses.replace(x, freqs_cis=ident))
    R = x.rotary_dim
    # the table is float32: cos^2 + sin^2 = 1 only to ~1e-7, which the rotation applies as given
    np.testing.assert_allclose(np.hypot(a[:, 0:R:2], a[:, 1:R:2]), np.hypot(b[:, 0:R:2], b[:, 1:R:2]), rtol=3e-7, atol=1e-12)
    gamma = oracle.decode(x.gamma, x.dtype)
    live = np.abs(b).sum(axis=1) > 0
    y = b[live] / gamma
    # y = x / sqrt(ms + eps) with ms the pooled key's mean square: mean(y^2) = ms / (ms + eps) < 1, -> 1
    m = (y ** 2).mean(axis=1)
    assert (m < 1).all() and (m > 1 - 1e-3).all()


def test_identical_keys_pool_to_themselves_and_missing_blocks_are_zero():
    spec = dataclasses.replace(SMALL["compress_f32_small"], ratio=4, rotary_dim=0)
    x = spec.build(keep_logical=True)
    # overwrite every raw key of sequence 0 with its first key: pooling returns it
    c = x.cache
    n, two, L, P, nkv, D = c.kv_shape
    kv = c.kv_view()
    first = None
    for j in range(int(x.key_counts[0])):
        page = c.kv_lookup_table[0, j // P]
        if first is None:
            first = kv[page, 0, c.layer_idx, j % P, 0].copy()
        kv[page, 0, c.layer_idx, j % P, 0] = first
    got = oracle.compress_keys(x)
    gamma = oracle.decode(x.gamma, x.dtype)
    f = oracle.decode(first, x.dtype)
    want = f / np.sqrt((f ** 2).mean() + x.eps) * gamma
    nblk = int(x.key_counts[0]) // x.ratio
    np.testing.assert_allclose(got[:nblk], np.broadcast_to(want, (nblk, D)), rtol=1e-12, atol=1e-14)
    # rows past each sequence's complete blocks are zero
    for b in range(x.batch):
        assert not got[b * x.max_blocks + int(x.key_counts[b]) // x.ratio:(b + 1) * x.max_blocks].any()


def test_no_keys_gives_zero_rows_and_page_placement_does_not_matter():
    spec = SMALL["compress_bf16_small"]
    a = spec.build()
    zero = dataclasses.replace(a, key_counts=np.zeros_like(a.key_counts))
    assert not oracle.compress_keys(zero).any()
    b = dataclasses.replace(spec, page_pad=128).build()
    np.testing.assert_array_equal(oracle.compress_keys(a), oracle.compress_keys(b))
