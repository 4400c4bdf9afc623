"""Pins of the float64 CPU oracle to things other than itself.

Each check ties the oracle to the QSASparseAttentionRaggedPaged page (gather-GQA
over the selected token indices, valid entries first, nothing past counts
read, softmax(scale * q.K_sel) . V_sel) through an independent route: a
hand-worked example, PyTorch's float64 scaled_dot_product_attention on the
logical (never paged) K/V, closed forms, invariances and PyTorch's own dtype
decoders.  A dropped term, a wrong sign, index, layer or K/V axis, or a
transposed head mapping in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from index_gathered_sparse_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _decode_torch(raw: np.ndarray, dtype: str) -> torch.Tensor:
    """Raw storage -> float64 through PyTorch's own dtype conversions."""
    t = torch.from_numpy(np.ascontiguousarray(raw))
    if dtype == "f32":
        return t.double()
    if dtype == "bf16":
        return t.view(torch.int16).view(torch.bfloat16).double()
    return t.view(torch.float8_e4m3fn).double()


def _sdpa_reference(x: wl.QSAInputs, rows) -> np.ndarray:
    """Per (row, kv head): gather the selected rows of the *logical* K/V and
    call PyTorch's float64 scaled_dot_product_attention."""
    g, nkv, D = x.group, x.num_kv_heads, x.head_dim
    seq = x.row_sequence()
    n_all = x.valid_counts()
    out = np.zeros((len(rows), x.num_q_heads, D))
    qd = _decode_torch(x.q, x.dtype)
    for k, r in enumerate(rows):
        b = seq[r]
        n = int(n_all[r])
        if n == 0:
            continue
        idx = torch.from_numpy(x.token_indices[r, :n].astype(np.int64))
        K = _decode_torch(x.logical_k[b], x.dtype)[idx]  # [n, nkv, D]
        V = _decode_torch(x.logical_v[b], x.dtype)[idx]
        for h in range(nkv):
            Q = qd[r, h * g : (h + 1) * g, :]  # query heads h*g .. h*g+g-1 share kv head h
            o = torch.nn.functional.scaled_dot_product_attention(
                Q[None], K[:, h, :][None], V[:, h, :][None], scale=x.scale
            )[0]
            out[k, h * g : (h + 1) * g, :] = o.numpy()
    return out


# --------------------------------------------------------------------------
# decoders
# --------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_for_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle_mod.decode(codes, "e4m3")
    ref = _decode_torch(codes, "e4m3").numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    # the format's fixed points: max normal 448, min subnormal 2^-9, 0x7F / 0xFF NaN
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0**-9 and np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])


def test_bf16_decode_matches_torch(oracle_mod):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**16, size=4096, dtype=np.uint16)
    mine = oracle_mod.decode(bits, "bf16")
    ref = _decode_torch(bits, "bf16").numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


# --------------------------------------------------------------------------
# hand-worked example
# --------------------------------------------------------------------------

def _golden_inputs(page_pad=None, perm=None):
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    nkv, D = g["num_kv_heads"], g["head_dim"]
    k = np.asarray(g["logical_k"], np.float32).reshape(-1, nkv, D)
    v = np.asarray(g["logical_v"], np.float32).reshape(-1, nkv, D)
    q = np.asarray(g["q"], np.float32)
    # the fixture fixes its own page assignment (logical 0 -> physical 1, 1 -> 0)
    table_perm = np.asarray(g["kv_lookup_table"][0]) if perm is None else perm
    x = wl.assemble("golden", "f32", "f32", q, [k], [v], rows=[1], cache_lengths=g["cache_lengths"],
                    page_size=g["page_size"], num_layers=g["num_layers"], layer_idx=g["layer_idx"],
                    token_indices=np.asarray(g["token_indices"]), counts=np.asarray(g["counts"]),
                    scale=g["scale"], page_perm=table_perm, page_pad=page_pad)
    assert x.kv_lookup_table[0].tolist() == list(table_perm)
    return x, g


def test_worked_example(oracle_mod):
    x, g = _golden_inputs()
    out = oracle_mod.sparse_attention(x)
    np.testing.assert_allclose(out, np.asarray(g["expected"]), atol=g["tolerance"], rtol=0)


def test_worked_example_paging_invariance(oracle_mod):
    """Physical placement (page order, padding between pages) never changes the result."""
    base = oracle_mod.sparse_attention(_golden_inputs()[0])
    for pad, perm in ((None, np.array([0, 1])), (48, np.array([1, 0])), (16, np.array([0, 1]))):
        other = oracle_mod.sparse_attention(_golden_inputs(page_pad=pad, perm=perm)[0])
        assert np.array_equal(base, other)


# --------------------------------------------------------------------------
# brute force on the logical K/V (paging never enters it)
# --------------------------------------------------------------------------

SMALL = {"tiny_ragged_fp32": lambda: wl.tiny_ragged()}
SMALL.update({k: (lambda s=s: s) for k, s in wl.small_variants().items()})


@pytest.mark.parametrize("name", sorted(SMALL))
def test_matches_sdpa_on_logical_kv(oracle_mod, name):
    x = SMALL[name]().build(keep_logical=True)
    rows = np.arange(x.total_q)
    if x.total_q > 24:  # a spread of rows keeps the CPU suite short
        rows = np.unique(np.linspace(0, x.total_q - 1, 24).astype(np.int64))
    out = oracle_mod.sparse_attention(x, rows)
    ref = _sdpa_reference(x, rows)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=1e-12)


def _dense_selection_inputs(dtype="f32", shuffle=True, seed=7):
    """Every row selects all of 0..pos (shuffled): dense causal attention."""
    rng = np.random.default_rng(seed)
    rows, cache = [5, 7, 1], [0, 9, 4]
    nq, nkv, D, P = 4, 2, 64, 4
    kv_len = [r + c for r, c in zip(rows, cache)]
    W = max(kv_len)
    q = wl.encode(rng.standard_normal((sum(rows), nq, D), dtype=np.float32), dtype)
    ks = [wl.encode(rng.standard_normal((n, nkv, D), dtype=np.float32), dtype) for n in kv_len]
    vs = [wl.encode(rng.standard_normal((n, nkv, D), dtype=np.float32), dtype) for n in kv_len]
    idx = np.full((sum(rows), W), -1, np.int32)
    cnt = np.zeros(sum(rows), np.int32)
    r = 0
    for b in range(len(rows)):
        for t in range(rows[b]):
            pos = cache[b] + t
            sel = rng.permutation(pos + 1) if shuffle else np.arange(pos + 1)
            idx[r, : pos + 1] = sel
            cnt[r] = pos + 1
            r += 1
    perm = rng.permutation(sum(-(-n // P) for n in kv_len))
    return wl.assemble("dense", dtype, "f32", q, ks, vs, rows, cache, P, 2, 1, idx, cnt, 1 / math.sqrt(D),
                       page_perm=perm, keep_logical=True), rows, cache


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_full_selection_is_dense_causal_attention(oracle_mod, dtype):
    """Selecting all of 0..pos reproduces causal flash attention (the
    mo.mha.ragged.no_cache math with a causal mask) computed densely, with GQA
    done by repeating each kv head over its group of query heads."""
    x, rows, cache = _dense_selection_inputs(dtype)
    out = oracle_mod.sparse_attention(x)
    g = x.group
    off = x.input_row_offsets
    for b in range(len(rows)):
        Q = _decode_torch(x.q[off[b] : off[b + 1]], dtype).transpose(0, 1)  # [nq, R, D]
        K = _decode_torch(x.logical_k[b], dtype).repeat_interleave(g, dim=1).transpose(0, 1)
        V = _decode_torch(x.logical_v[b], dtype).repeat_interleave(g, dim=1).transpose(0, 1)
        t = torch.arange(rows[b])[:, None]
        j = torch.arange(K.shape[1])[None, :]
        mask = j <= cache[b] + t  # bottom-right aligned causal mask
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=x.scale)
        np.testing.assert_allclose(out[off[b] : off[b + 1]], ref.transpose(0, 1).numpy(), atol=1e-12, rtol=1e-12)


# --------------------------------------------------------------------------
# closed forms and invariances
# --------------------------------------------------------------------------

def _tiny():
    return wl.tiny_ragged().build(keep_logical=True)


def test_count_one_returns_that_v_row(oracle_mod):
    x = _tiny()
    x.counts[:] = 1
    out = oracle_mod.sparse_attention(x)
    seq = x.row_sequence()
    for r in range(x.total_q):
        v = oracle_mod.decode(x.logical_v[seq[r]][x.token_indices[r, 0]], "f32")  # [nkv, D]
        for head in range(x.num_q_heads):
            assert np.array_equal(out[r, head], v[head // x.group])


def test_zero_query_gives_mean_of_selected_v(oracle_mod):
    x = _tiny()
    x.q[:] = 0
    out = oracle_mod.sparse_attention(x)
    seq = x.row_sequence()
    for r in range(x.total_q):
        n = x.counts[r]
        v = oracle_mod.decode(x.logical_v[seq[r]][x.token_indices[r, :n]], "f32")  # [n, nkv, D]
        mean = v.sum(axis=0) / n
        for head in range(x.num_q_heads):
            np.testing.assert_allclose(out[r, head], mean[head // x.group], atol=1e-14, rtol=1e-13)


def test_huge_scale_picks_the_argmax_key(oracle_mod):
    x = _tiny()
    x.scale = 1e6
    out = oracle_mod.sparse_attention(x)
    seq = x.row_sequence()
    q = oracle_mod.decode(x.q, "f32")
    for r in range(x.total_q):
        n = x.counts[r]
        K = oracle_mod.decode(x.logical_k[seq[r]][x.token_indices[r, :n]], "f32")[:, 0, :]
        V = oracle_mod.decode(x.logical_v[seq[r]][x.token_indices[r, :n]], "f32")[:, 0, :]
        for head in range(x.num_q_heads):
            s = K @ q[r, head]
            top = np.sort(s)[::-1]
            if n > 1 and top[0] - top[1] < 1e-4:
                continue  # a near-tie has no single winner
            np.testing.assert_allclose(out[r, head], V[np.argmax(s)], atol=1e-12)


@pytest.mark.parametrize("name", ["tiny_ragged_fp32", "fp8_mixed_small"])
def test_valid_prefix_order_does_not_matter(oracle_mod, name):
    x = SMALL[name]().build()
    base = oracle_mod.sparse_attention(x)
    rng = np.random.default_rng(3)
    n = x.valid_counts()
    for r in range(x.total_q):
        x.token_indices[r, : n[r]] = rng.permutation(x.token_indices[r, : n[r]])
    np.testing.assert_allclose(oracle_mod.sparse_attention(x), base, atol=1e-12, rtol=1e-12)


def test_entries_past_counts_are_never_read(oracle_mod):
    x = SMALL["fp8_mixed_small"]().build()
    base = oracle_mod.sparse_attention(x)
    n = x.valid_counts()
    rng = np.random.default_rng(4)
    for fill in (lambda k: np.full(k, 2**31 - 1), lambda k: np.full(k, -7), lambda k: rng.integers(0, 5, k)):
        for r in range(x.total_q):
            x.token_indices[r, n[r] :] = fill(x.selection_width - n[r])
        assert np.array_equal(oracle_mod.sparse_attention(x), base)


def test_only_layer_idx_is_read(oracle_mod):
    """Every other layer, the page padding and the unused pages are NaN: any
    stray read would poison the output."""
    x = SMALL["fp8_mixed_small"]().build()
    assert x.page_stride != -1
    out = oracle_mod.sparse_attention(x)
    assert np.isfinite(out).all()


def test_grouped_heads_match_repeated_kv_heads(oracle_mod):
    """GQA: running with kv heads repeated `group` times (group 1, plain MHA)
    gives the same result as the grouped layout."""
    x = SMALL["bf16_decode_small"]().build(keep_logical=True)
    g = x.group
    ks = [np.repeat(k, g, axis=1) for k in x.logical_k]
    vs = [np.repeat(v, g, axis=1) for v in x.logical_v]
    rows = np.diff(x.input_row_offsets.astype(np.int64))
    mha = wl.assemble("mha", x.dtype, x.out_dtype, x.q, ks, vs, rows, x.cache_lengths, x.kv_shape[3],
                      x.kv_shape[2], x.layer_idx, x.token_indices, x.counts, x.scale)
    assert mha.group == 1
    np.testing.assert_allclose(oracle_mod.sparse_attention(mha), oracle_mod.sparse_attention(x), atol=1e-13, rtol=0)


# --------------------------------------------------------------------------
# edge readings (empty, clamped, duplicated, out of range)
# --------------------------------------------------------------------------

def test_non_positive_counts_give_a_zero_row(oracle_mod):
    x = _tiny()
    x.counts[0] = 0
    x.counts[3] = -5
    out = oracle_mod.sparse_attention(x)
    assert np.array_equal(out[0], np.zeros_like(out[0])) and np.array_equal(out[3], np.zeros_like(out[3]))
    assert np.isfinite(out).all()


def test_counts_above_width_clamp_to_width(oracle_mod):
    x = SMALL["bf16_decode_small"]().build()
    r = int(np.argmax(x.counts))
    assert x.counts[r] == x.selection_width
    base = oracle_mod.sparse_attention(x, [r])
    x.counts[r] = x.selection_width + 100
    assert np.array_equal(oracle_mod.sparse_attention(x, [r]), base)


def test_duplicate_index_counts_twice(oracle_mod):
    """softmax over the listed entries: a repeated index is its own term.
    With q=0 every term weighs the same, so the result is the weighted mean."""
    x = _tiny()
    x.q[:] = 0
    r = 7  # pos = 40 + 4
    x.token_indices[r, :3] = [5, 5, 9]
    x.counts[r] = 3
    out = oracle_mod.sparse_attention(x, [r])
    v = oracle_mod.decode(x.logical_v[1][[5, 9]], "f32")[:, 0, :]
    np.testing.assert_allclose(out[0, 0], (2 * v[0] + v[1]) / 3, atol=1e-14)


def test_out_of_range_index_inside_counts_is_an_error(oracle_mod):
    x = _tiny()
    x.token_indices[2, 0] = 10**6
    with pytest.raises(oracle_mod.OracleError) as e:
        oracle_mod.sparse_attention(x)
    assert e.value.row == 2
    x = _tiny()
    x.token_indices[4, 0] = -1
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.sparse_attention(x)


def test_index_at_last_valid_position(oracle_mod):
    """The newest key of the step (pos itself, cache_lengths + t) is valid."""
    x = _tiny()
    seq = x.row_sequence()
    for r in range(x.total_q):
        t = r - x.input_row_offsets[seq[r]]
        x.token_indices[r, 0] = int(x.cache_lengths[seq[r]]) + int(t)
    oracle_mod.sparse_attention(x)
