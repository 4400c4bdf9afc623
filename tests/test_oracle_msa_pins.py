"""Pins of the block-sparse (MSA-style) oracle against what the pages and the
mathematics fix, independently of the oracle's own code.

- Selecting every block up to the row's position is dense causal attention
  (PyTorch float64 scaled_dot_product_attention with a causal mask on the
  logical, unpaged K/V, kv heads repeated for GQA).
- A plain numpy brute force over the logical K/V (no pages, no page table)
  that expands each listed block into its positions <= the row's position.
- Invariances: block order, -1 padding anywhere, blocks wholly after the row's
  position, page placement; a repeated block weighs double; nothing attended
  gives a zero row; a selected page outside kv_blocks is an error.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import workloads as wl

SMALL = wl.msa_small_variants()


def _logical(x, b):
    k = oracle.decode(x.logical_k[b], x.dtype)
    v = oracle.decode(x.logical_v[b], x.dtype)
    return k, v


def brute_force(x) -> np.ndarray:
    """Each (row, kv head): the listed blocks' positions <= pos, in list order,
    read from the unpaged K/V; softmax over them in float64."""
    P = x.kv_shape[3]
    nkv, g = x.num_kv_heads, x.group
    seq = x.row_sequence()
    pos = x.query_positions()
    q = oracle.decode(x.q, x.dtype)
    out = np.zeros(q.shape)
    cache_kv = [_logical(x, b) for b in range(x.batch)]
    for r in range(x.total_q):
        k_all, v_all = cache_kv[seq[r]]
        for h in range(nkv):
            keys = [bb * P + s for bb in x.d_indices[h, r] if bb >= 0 for s in range(P) if bb * P + s <= pos[r]]
            if not keys:
                continue
            K, V = k_all[keys, h], v_all[keys, h]
            for i in range(g):
                sc = x.scale * (K @ q[r, h * g + i])
                w = np.exp(sc - sc.max())
                out[r, h * g + i] = (w / w.sum()) @ V
    return out


@pytest.fixture(scope="module", autouse=True)
def _build():
    oracle.build()


@pytest.mark.parametrize("name", sorted(SMALL))
def test_matches_brute_force(name):
    x = SMALL[name].build(keep_logical=True)
    np.testing.assert_allclose(oracle.msa_attention(x), brute_force(x), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_all_blocks_is_dense_causal_attention(name):
    x = SMALL[name].build(keep_logical=True)
    P = x.kv_shape[3]
    pos = x.query_positions()
    topk = int(pos.max()) // P + 1
    d = np.full((x.num_kv_heads, x.total_q, topk), -1, np.int32)
    for r in range(x.total_q):
        d[:, r, : pos[r] // P + 1] = np.arange(pos[r] // P + 1)
    x = dataclasses.replace(x, d_indices=d)
    got = oracle.msa_attention(x)
    q = oracle.decode(x.q, x.dtype)
    seq = x.row_sequence()
    off = x.input_row_offsets.astype(np.int64)
    for b in range(x.batch):
        rows = np.arange(off[b], off[b + 1])
        if rows.size == 0:
            continue
        k, v = _logical(x, b)  # [kv_len, nkv, D]
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(x.group, 0)  # [nq, kv_len, D]
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(x.group, 0)
        qt = torch.from_numpy(q[rows]).permute(1, 0, 2)  # [nq, rows, D]
        # causal with the queries at the end of the cache: row t sees 0 .. cache + t
        n_kv, n_q = kt.shape[1], qt.shape[1]
        mask = torch.arange(n_kv)[None, :] <= (torch.arange(n_q)[:, None] + (n_kv - n_q))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=x.scale)
        np.testing.assert_allclose(got[rows], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    assert (seq >= 0).all()


def test_invariances():
    x = SMALL["msa_bf16_prefill_small"].build()
    P = x.kv_shape[3]
    base = oracle.msa_attention(x)
    rng = np.random.default_rng(0)
    # block order inside each (kv head, row)
    d = x.d_indices.copy()
    for h in range(d.shape[0]):
        for r in range(d.shape[1]):
            d[h, r] = d[h, r, rng.permutation(d.shape[2])]
    np.testing.assert_allclose(oracle.msa_attention(dataclasses.replace(x, d_indices=d)), base, rtol=1e-12, atol=1e-14)
    # -1 slots inserted anywhere, and blocks wholly after the row's position
    pos = x.query_positions()
    extra = np.full(d.shape[:2] + (3,), -1, np.int32)
    extra[:, :, 1] = (pos // P + 1)[None, :]  # the block after the one holding pos: nothing in it is attended
    d2 = np.concatenate([extra[:, :, :1], x.d_indices, extra[:, :, 1:]], axis=2)
    np.testing.assert_array_equal(oracle.msa_attention(dataclasses.replace(x, d_indices=d2)), base)


def test_duplicate_block_weighs_double_and_empty_rows_are_zero():
    x = SMALL["msa_bf16_decode_small"].build(keep_logical=True)
    d = x.d_indices.copy()
    d[:, :, -1] = d[:, :, 0]  # repeat the first listed block in the last slot
    d[0, 0, :] = -1  # kv head 0 of row 0 attends nothing
    y = dataclasses.replace(x, d_indices=d)
    got = oracle.msa_attention(y)
    np.testing.assert_allclose(got, brute_force(y), rtol=1e-11, atol=1e-12)
    assert not got[0, : x.group].any()


def test_page_placement_does_not_matter():
    spec = SMALL["msa_fp8_decode_small"]
    a = spec.build()
    b = dataclasses.replace(spec, page_pad=None).build()  # packed pages, same draws
    np.testing.assert_array_equal(oracle.msa_attention(a), oracle.msa_attention(b))


def test_selected_page_outside_kv_blocks_is_an_error():
    x = SMALL["msa_bf16_decode_small"].build()
    tab = x.kv_lookup_table.copy()
    blk = int(x.d_indices[0, 2, 0])
    tab[x.row_sequence()[2], blk] = x.kv_shape[0] + 5
    with pytest.raises(oracle.OracleError):
        oracle.msa_attention(dataclasses.replace(x, kv_lookup_table=tab))
