"""Pins of the latent sparse attention oracle (sliding window + listed
compressed entries + per-head sinks), independent of its own code.

- Brute force on tiny inputs over the unpaged caches (no page tables).
- With every sink at -inf, a plain softmax attention: PyTorch float64 SDPA on
  the gathered keys; with a window covering the whole prefix and no entries,
  dense causal attention (SDPA with a causal mask).
- A sink only scales a head's output: out(sink) / out(-inf) is one factor in
  (0, 1) per (row, head), and a huge sink drives the output to zero.
- Invariances: entry order, -1 slots anywhere, page placement; an entry past
  the sequence's compressed entries is an error.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import workloads as wl

SMALL = wl.latent_small_variants()


@pytest.fixture(scope="module", autouse=True)
def _build():
    oracle.build()


def gathered(x, r):
    """K, V [n, D] attended by row r (window oldest first, then entries), from
    the unpaged caches."""
    seq = x.swa.row_sequence()[r]
    pos = x.query_positions()[r]
    dt = x.dtype
    k_w = oracle.decode(x.swa.logical_k[seq], dt)[:, 0]
    v_w = oracle.decode(x.swa.logical_v[seq], dt)[:, 0]
    k_c = oracle.decode(x.comp.logical_k[seq], dt)[:, 0]
    v_c = oracle.decode(x.comp.logical_v[seq], dt)[:, 0]
    win = np.arange(max(0, pos - x.window + 1), pos + 1)
    ent = [e for e in x.comp_indices[r] if e >= 0]
    return np.concatenate([k_w[win], k_c[ent]]), np.concatenate([v_w[win], v_c[ent]])


def brute_force(x) -> np.ndarray:
    q = oracle.decode(x.swa.q, x.dtype)
    out = np.zeros(q.shape)
    for r in range(x.total_q):
        K, V = gathered(x, r)
        for h in range(x.num_heads):
            s = x.swa.scale * (K @ q[r, h])
            m = max(s.max(initial=-np.inf), float(x.attn_sink[h]))
            w = np.exp(s - m)
            out[r, h] = (w @ V) / (w.sum() + np.exp(float(x.attn_sink[h]) - m))
    return out


@pytest.mark.parametrize("name", sorted(SMALL))
def test_matches_brute_force(name):
    x = SMALL[name].build(keep_logical=True)
    np.testing.assert_allclose(oracle.latent_attention(x), brute_force(x), rtol=1e-11, atol=1e-12)


def test_without_sinks_is_softmax_attention_on_the_gathered_keys():
    x = SMALL["latent_bf16_prefill_small"].build(keep_logical=True)
    x = dataclasses.replace(x, attn_sink=np.full(x.num_heads, -np.inf, np.float32))
    got = oracle.latent_attention(x)
    q = oracle.decode(x.swa.q, x.dtype)
    for r in range(x.total_q):
        K, V = gathered(x, r)
        kt = torch.from_numpy(K)[None].expand(x.num_heads, -1, -1)  # [H, n, D]
        vt = torch.from_numpy(V)[None].expand(x.num_heads, -1, -1)
        qt = torch.from_numpy(q[r])[:, None]  # [H, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=x.swa.scale)[:, 0]
        np.testing.assert_allclose(got[r], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_full_window_without_entries_is_dense_causal_attention():
    spec = dataclasses.replace(SMALL["latent_bf16_prefill_small"], window=10_000, num_comp=0)
    x = spec.build(keep_logical=True)
    x = dataclasses.replace(x, attn_sink=np.full(x.num_heads, -np.inf, np.float32))
    got = oracle.latent_attention(x)
    q = oracle.decode(x.swa.q, x.dtype)
    off = x.swa.input_row_offsets.astype(np.int64)
    for b in range(x.swa.batch):
        rows = np.arange(off[b], off[b + 1])
        if rows.size == 0:
            continue
        k = torch.from_numpy(oracle.decode(x.swa.logical_k[b], x.dtype)[:, 0])[None].expand(x.num_heads, -1, -1)
        v = torch.from_numpy(oracle.decode(x.swa.logical_v[b], x.dtype)[:, 0])[None].expand(x.num_heads, -1, -1)
        qt = torch.from_numpy(q[rows]).permute(1, 0, 2)
        n_kv, n_q = k.shape[1], qt.shape[1]
        mask = torch.arange(n_kv)[None, :] <= (torch.arange(n_q)[:, None] + (n_kv - n_q))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, k, v, attn_mask=mask, scale=x.swa.scale)
        np.testing.assert_allclose(got[rows], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_sink_only_scales_each_head():
    x = SMALL["latent_bf16_decode_small"].build()
    with_sink = oracle.latent_attention(x)
    plain = oracle.latent_attention(dataclasses.replace(x, attn_sink=np.full(x.num_heads, -np.inf, np.float32)))
    ratio = with_sink / plain
    f = ratio[..., :1]
    np.testing.assert_allclose(ratio, np.broadcast_to(f, ratio.shape), rtol=1e-9)
    assert ((f > 0) & (f < 1)).all()
    huge = oracle.latent_attention(dataclasses.replace(x, attn_sink=np.full(x.num_heads, 1e4, np.float32)))
    assert np.abs(huge).max() < 1e-300


def test_invariances_and_errors():
    spec = SMALL["latent_bf16_prefill_small"]
    x = spec.build()
    base = oracle.latent_attention(x)
    rng = np.random.default_rng(0)
    ci = x.comp_indices.copy()
    for r in range(ci.shape[0]):
        ci[r] = ci[r, rng.permutation(ci.shape[1])]  # moves -1 slots into the middle too
    np.testing.assert_allclose(oracle.latent_attention(dataclasses.replace(x, comp_indices=ci)), base,
                               rtol=1e-12, atol=1e-14)
    y = dataclasses.replace(spec, page_size=16, comp_page_size=32).build()  # same draws, other paging
    np.testing.assert_array_equal(oracle.latent_attention(y), base)
    bad = x.comp_indices.copy()
    bad[3, 0] = int(x.comp.cache_lengths[x.swa.row_sequence()[3]])
    with pytest.raises(oracle.OracleError):
        oracle.latent_attention(dataclasses.replace(x, comp_indices=bad))
