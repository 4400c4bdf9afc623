"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs, element by element.

Tolerances (max |err| <= atol + rtol * |ref|): BF16 1e-2 + 1e-2|ref|,
FP8 e4m3 6e-2 + 3e-2|ref|, FP32 1e-4.  Which cache positions are read is
checked bit-exactly: every byte no selection may read is NaN, skipped
positions are reported in the device status word, and changing anything a
call must not read (tail entries, page placement, other layers) leaves the
output bits unchanged.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import binding as B
from index_gathered_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-4, 0.0), "bf16": (1e-2, 1e-2), "e4m3": (6e-2, 3e-2)}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    B.qsa_read_device_status(clear=True)
    yield


def run_gpu(x: wl.QSAInputs, **kw) -> np.ndarray:
    d = wl.to_torch(x, "cuda")
    B.qsa_sparse_attention_ragged_paged(**d, **kw)
    torch.cuda.synchronize()
    return d["output"].float().cpu().double().numpy()


def assert_close(got, ref, dtype, what=""):
    atol, rtol = TOL[dtype]
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output (a poisoned byte was read)"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (
        f"{what}: {int((err > bound).sum())} of {err.size} outside tolerance; worst at {worst}: "
        f"got {got[worst]}, ref {ref[worst]}")


def status_clean():
    return B.qsa_read_device_status(clear=True) == 0


SMALL = dict(wl.small_variants())
SMALL["tiny_ragged_fp32"] = wl.tiny_ragged()


def _launches(dtype):
    if dtype == "f32":
        return [dict(kernel=1)]
    # auto (the persistent stream-K kernel), the CUDA-core kernel, the per-unit
    # tensor-core kernel without split-K, with bands merged inside a cluster
    # (3, 8) and through the workspace tickets (12, 40: more bands than a
    # cluster holds, some of them empty), and stream-K grids small and large
    # enough that units are shared by several CTAs
    return [dict(), dict(kernel=1), dict(kernel=2, splits=1), dict(kernel=2, splits=3), dict(kernel=2, splits=8),
            dict(kernel=2, splits=12), dict(kernel=2, splits=40),
            dict(kernel=3, ctas=1), dict(kernel=3, ctas=7), dict(kernel=3, ctas=64), dict(kernel=3, ctas=1000)]


CASES = [(n, i) for n in sorted(SMALL) for i in range(len(_launches(SMALL[n].dtype)))]

# units of the persistent kernel with a forced number of kv heads: eight (2 KB
# of K per key for BF16, one consumer warp per head) where num_kv_heads and
# group allow, one and two everywhere, each on split and unsplit grids
HPU_CASES = []
for _n in sorted(SMALL):
    _s = SMALL[_n]
    if _s.dtype == "f32":
        continue
    _g = _s.num_q_heads // _s.num_kv_heads
    for _h in (1, 2, 8):
        if _s.num_kv_heads % _h or (_h == 8 and _g > 8):
            continue
        for _c in (0, 7, 1000):
            HPU_CASES.append((_n, _h, _c))


@pytest.mark.parametrize("name,launch", CASES)
def test_small_workloads_match_oracle(name, launch):
    x = SMALL[name].build()
    kw = _launches(x.dtype)[launch]
    got = run_gpu(x, **kw)
    ref = oracle.sparse_attention(x)
    assert_close(got, ref, x.dtype, f"{name} {kw}")
    assert status_clean()


@pytest.mark.parametrize("name,hpu,ctas", HPU_CASES)
def test_heads_per_unit_match_oracle(name, hpu, ctas):
    x = SMALL[name].build()
    kw = dict(kernel=3, heads_per_unit=hpu, ctas=ctas)
    assert_close(run_gpu(x, **kw), oracle.sparse_attention(x), x.dtype, f"{name} {kw}")
    assert status_clean()


def test_give_up_path_reports_timeout_and_keeps_the_stream_usable():
    """A test-only launch makes the persistent kernel's producers issue no K/V
    copies, so every consumer wait gives up after a few thousand polls (no
    copy is in flight when a CTA leaves) and the call reports
    QSA_STATUS_TIMEOUT.  The CTAs still arrive on the tickets of the units
    they share, so the next calls on the same stream, with the same grid and
    workspace, match the oracle again."""
    x = SMALL["bf16_decode_small"].build()
    ref = oracle.sparse_attention(x)
    for ctas in (7, 64):  # more units than CTAs (scanned split), then units spread over several CTAs
        B.qsa_read_device_status(clear=True)
        run_gpu(x, kernel=3, ctas=ctas, test_stall=1)
        assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_TIMEOUT
        for _ in range(2):
            assert_close(run_gpu(x, kernel=3, ctas=ctas), ref, "bf16", f"after a give-up, ctas {ctas}")
            assert status_clean()


def test_worked_example_on_gpu():
    import json
    import os

    with open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")) as f:
        g = json.load(f)
    nkv, D = g["num_kv_heads"], g["head_dim"]
    # the CUDA kernels need head_dim 64 or 128: embed the 2-wide example in 64 zeros-padded channels
    pad = 64
    k = np.zeros((4, nkv, pad), np.float32)
    v = np.zeros((4, nkv, pad), np.float32)
    q = np.zeros((1, 2, pad), np.float32)
    k[:, :, :D] = np.asarray(g["logical_k"], np.float32).reshape(-1, nkv, D)
    v[:, :, :D] = np.asarray(g["logical_v"], np.float32).reshape(-1, nkv, D)
    q[:, :, :D] = np.asarray(g["q"], np.float32)
    x = wl.assemble("golden", "f32", "f32", q, [k], [v], [1], g["cache_lengths"], g["page_size"], g["num_layers"],
                    g["layer_idx"], np.asarray(g["token_indices"]), np.asarray(g["counts"]), g["scale"],
                    page_perm=np.asarray(g["kv_lookup_table"][0]))
    got = run_gpu(x)
    np.testing.assert_allclose(got[..., :D], np.asarray(g["expected"]), atol=g["tolerance"], rtol=0)
    assert np.array_equal(got[..., D:], np.zeros_like(got[..., D:]))


def _dense_bf16(seed=21):
    """bf16, head_dim 128, group 8: every row selects all of 0..pos."""
    rng = np.random.default_rng(seed)
    rows, cache = [37, 5, 70], [0, 150, 30]
    nq, nkv, D, P = 16, 2, 128, 16
    kv_len = [r + c for r, c in zip(rows, cache)]
    W = max(kv_len)
    q = wl.encode(rng.standard_normal((sum(rows), nq, D), dtype=np.float32), "bf16")
    ks = [wl.encode(rng.standard_normal((n, nkv, D), dtype=np.float32), "bf16") for n in kv_len]
    vs = [wl.encode(rng.standard_normal((n, nkv, D), dtype=np.float32), "bf16") for n in kv_len]
    idx = np.full((sum(rows), W), -1, np.int32)
    cnt = np.zeros(sum(rows), np.int32)
    r = 0
    for b in range(len(rows)):
        for t in range(rows[b]):
            pos = cache[b] + t
            idx[r, : pos + 1] = rng.permutation(pos + 1)
            cnt[r] = pos + 1
            r += 1
    perm = rng.permutation(sum(-(-n // P) for n in kv_len))
    return wl.assemble("dense_bf16", "bf16", "bf16", q, ks, vs, rows, cache, P, 1, 0, idx, cnt, 1 / math.sqrt(D),
                       page_perm=perm)


@pytest.mark.parametrize("launch", [dict(), dict(kernel=1), dict(kernel=2, splits=2), dict(kernel=3, ctas=5)])
def test_full_selection_bf16(launch):
    x = _dense_bf16()
    assert_close(run_gpu(x, **launch), oracle.sparse_attention(x), "bf16", f"dense {launch}")
    assert status_clean()


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_output_dtypes(out_dtype):
    x = SMALL["fp8_mixed_small"].build()
    d = wl.to_torch(x, "cuda", out_dtype=out_dtype)
    B.qsa_sparse_attention_ragged_paged(**d)
    torch.cuda.synchronize()
    assert_close(d["output"].double().cpu().numpy(), oracle.sparse_attention(x), "e4m3", out_dtype)


def test_head_dim_64_and_odd_groups():
    """Shapes only the CUDA-core kernel runs: head_dim 64, groups 1, 2, 3, 5."""
    for dtype, g in (("bf16", 1), ("bf16", 3), ("e4m3", 2), ("f32", 5)):
        spec = wl.bf16_decode(seed=30 + g, batch=3, cache_range=(60, 300), width=96)
        spec.num_kv_heads, spec.num_q_heads, spec.head_dim = 2, 2 * g, 64
        spec.dtype, spec.out_dtype = dtype, "f32"
        x = spec.build()
        assert_close(run_gpu(x), oracle.sparse_attention(x), dtype, f"{dtype} g{g}")


def test_odd_groups_on_tensor_cores_with_split_k():
    """Groups 3, 5 and 7 pad the 8-wide head tile; split-K partials of an odd
    group must still start 16-byte aligned."""
    for g in (3, 5, 7):
        spec = wl.bf16_decode(seed=60 + g, batch=4, cache_range=(300, 900), width=384)
        spec.num_kv_heads, spec.num_q_heads = 2, 2 * g
        x = spec.build()
        for kw in (dict(kernel=2, splits=1), dict(kernel=2, splits=3), dict(kernel=2, splits=6), dict(),
                   dict(kernel=3, ctas=3)):
            assert_close(run_gpu(x, **kw), oracle.sparse_attention(x), "bf16", f"g{g} {kw}")


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
@pytest.mark.parametrize("nkv", [1, 2, 3, 4, 6, 8, 12])
def test_kv_head_groupings(dtype, nkv):
    """Units of 4, 2 or 1 adjacent kv heads (by divisibility of num_kv_heads)
    in the persistent kernel, at grid sizes that share units between CTAs."""
    spec = wl.bf16_decode(seed=70 + nkv, batch=3, cache_range=(200, 700), width=320)
    spec.num_kv_heads, spec.num_q_heads = nkv, 4 * nkv
    spec.dtype = dtype
    x = spec.build()
    ref = oracle.sparse_attention(x)
    for kw in (dict(), dict(kernel=3, ctas=2), dict(kernel=3, ctas=11)):
        assert_close(run_gpu(x, **kw), ref, dtype, f"nkv{nkv} {kw}")
    assert status_clean()


def test_group_16_and_12_on_tensor_cores():
    for g in (16, 12):
        spec = wl.bf16_long_decode(seed=40 + g, batch=2, cache_range=(2000, 4000), runs=5)
        spec.num_q_heads = g * spec.num_kv_heads
        x = spec.build()
        for kw in (dict(), dict(kernel=2, splits=1), dict(kernel=3, ctas=4)):
            assert_close(run_gpu(x, **kw), oracle.sparse_attention(x), "bf16", f"g{g} {kw}")


# ---------------------------------------------------------------------------
# which positions are read: bit-exact
# ---------------------------------------------------------------------------

def test_tail_entries_never_change_a_bit():
    x = SMALL["bf16_decode_small"].build()
    n = x.valid_counts()
    for launch in (dict(), dict(kernel=1), dict(kernel=2, splits=4), dict(kernel=3, ctas=5)):
        base = run_gpu(x, **launch)
        y = SMALL["bf16_decode_small"].build()
        rng = np.random.default_rng(9)
        for r in range(y.total_q):
            y.token_indices[r, n[r]:] = rng.integers(-(2**31), 2**31 - 1, size=y.selection_width - n[r])
        assert np.array_equal(run_gpu(y, **launch), base)
    assert status_clean()


def test_page_placement_never_changes_a_bit():
    spec = SMALL["bf16_prefill_small"]
    x = spec.build(keep_logical=True)
    base = run_gpu(x)
    rows = np.diff(x.input_row_offsets.astype(np.int64))
    total_pages = x.kv_shape[0] - 1
    for pad, seed in ((None, 1), (4096, 2), (16, 3)):
        perm = np.random.default_rng(seed).permutation(total_pages)
        y = wl.assemble("moved", x.dtype, x.out_dtype, x.q, x.logical_k, x.logical_v, rows, x.cache_lengths,
                        x.kv_shape[3], x.kv_shape[2], x.layer_idx, x.token_indices, x.counts, x.scale,
                        page_perm=perm, page_pad=pad)
        assert np.array_equal(run_gpu(y), base), (pad, seed)


def test_other_layers_never_read():
    x = SMALL["bf16_decode_small"].build()
    base = run_gpu(x)
    kv6 = x.kv_view()
    L = x.kv_shape[2]
    for layer in range(L):
        if layer != x.layer_idx:
            kv6[:, :, layer] = np.uint16(0x3F80)  # 1.0 instead of NaN
    assert np.array_equal(run_gpu(x), base)


def test_empty_and_clamped_counts():
    x = SMALL["fp8_mixed_small"].build()
    x.counts[:3] = 0
    x.counts[3] = -9
    # counts past the width clamp to the width, so the whole row must then hold
    # valid positions: repeat the valid prefix over the tail
    n4 = int(x.counts[4])
    x.token_indices[4, n4:] = np.resize(x.token_indices[4, :n4], x.selection_width - n4)
    x.counts[4] = x.selection_width + 1000
    ref = oracle.sparse_attention(x)
    for launch in (dict(), dict(kernel=1), dict(kernel=2, splits=5), dict(kernel=3, ctas=9), dict(kernel=3, ctas=2)):
        got = run_gpu(x, **launch)
        assert np.array_equal(got[:4], np.zeros_like(got[:4]))
        assert_close(got, ref, "e4m3", str(launch))
    assert status_clean()


def test_zero_width_selection():
    spec = wl.bf16_decode(seed=50, batch=2, cache_range=(10, 20), width=0)
    spec.select = lambda rng, pos, W, P: np.zeros(0, np.int64)
    x = spec.build()
    got = run_gpu(x)
    assert np.array_equal(got, np.zeros_like(got))


def test_out_of_range_positions_are_skipped_and_reported():
    """Positions inside counts but at or past the sequence's length are
    skipped and flagged.  The bad values lie in [kv_len, max_pages * page_size):
    their table entries name the sequence's last page (slots past kv_len)
    or the poison page, both allocated and NaN-filled, so even a kernel whose
    range check regressed could only read NaN inside the cache, never outside
    any tensor.  (No negative value has that property, so negative positions
    are left to the same comparison, pos < 0 || pos >= kv_len.)"""
    x = SMALL["bf16_decode_small"].build()
    n = x.valid_counts()
    P, max_pages = x.kv_shape[3], x.kv_lookup_table.shape[1]
    seq = x.row_sequence()
    kv_len = x.cache_lengths.astype(np.int64) + np.diff(x.input_row_offsets.astype(np.int64))
    bad_rows = [r for r in range(x.total_q) if kv_len[seq[r]] + P < max_pages * P and n[r] >= 3][:3]
    assert len(bad_rows) == 3
    for r in bad_rows:
        x.token_indices[r, 1] = kv_len[seq[r]]          # the first position past the sequence
        x.token_indices[r, n[r] - 1] = kv_len[seq[r]] + P - 1  # a later page of the table row
    assert (x.token_indices[bad_rows][:, [1]] < max_pages * P).all()
    # expected: the same rows with those entries removed
    y = SMALL["bf16_decode_small"].build()
    for r in bad_rows:
        keep = [j for j in range(n[r]) if j not in (1, n[r] - 1)]
        sel = x.token_indices[r, keep].copy()
        y.token_indices[r, : len(sel)] = sel
        y.counts[r] = len(sel)
    ref = oracle.sparse_attention(y)
    for launch in (dict(), dict(kernel=1), dict(kernel=2, splits=3), dict(kernel=3, ctas=4),
                   dict(kernel=3, heads_per_unit=8)):
        B.qsa_read_device_status(clear=True)
        got = run_gpu(x, **launch)
        assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_INDEX
        assert_close(got, ref, "bf16", str(launch))


def test_bad_page_table_entry_is_skipped_and_reported():
    """A table entry naming no page of the kv_blocks descriptor is skipped and
    flagged.  The descriptor ends one page before the allocation and the bad
    entry names that last allocated (NaN-filled) page, so even a regressed
    check could not read outside the cache."""
    x = SMALL["bf16_decode_small"].build()
    r = 1
    b = x.row_sequence()[r]
    p = int(x.token_indices[r, 0])
    lp = p // x.kv_shape[3]
    assert x.poison_page == x.kv_shape[0] - 1
    x.kv_lookup_table[b, lp] = x.poison_page
    # expected: row r's keys on that page removed (no other row of sequence b exists in this decode batch)
    assert (x.row_sequence() == b).sum() == 1
    y = SMALL["bf16_decode_small"].build()
    sel = [int(v) for v in y.token_indices[r, : y.counts[r]] if int(v) // x.kv_shape[3] != lp]
    y.token_indices[r, : len(sel)] = sel
    y.counts[r] = len(sel)
    ref = oracle.sparse_attention(y)
    for launch in (dict(), dict(kernel=2), dict(kernel=1), dict(kernel=3, heads_per_unit=8)):
        d = wl.to_torch(x, "cuda")
        d["kv_blocks"] = d["kv_blocks"][: x.poison_page]  # the descriptor's pages stop before the poison page
        B.qsa_read_device_status(clear=True)
        B.qsa_sparse_attention_ragged_paged(**d, **launch)
        torch.cuda.synchronize()
        got = d["output"].float().cpu().double().numpy()
        assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_PAGE
        assert_close(got, ref, "bf16", f"bad page {launch}")


def test_rows_outside_every_sequence_are_zero_and_reported():
    """input_row_offsets that stop short of total_q: the trailing rows belong
    to no sequence, come out zero and raise QSA_STATUS_BAD_ROW."""
    x = SMALL["bf16_prefill_small"].build()  # its last sequence has 23 rows
    x.input_row_offsets[-1] -= 2  # still nondecreasing: rows total_q-2, total_q-1 are orphaned
    assert (np.diff(x.input_row_offsets.astype(np.int64)) >= 0).all()
    ref = oracle.sparse_attention(x, np.arange(x.total_q - 2))
    for launch in (dict(), dict(kernel=2), dict(kernel=1)):
        B.qsa_read_device_status(clear=True)
        got = run_gpu(x, **launch)
        assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_ROW
        assert np.array_equal(got[-2:], np.zeros_like(got[-2:]))
        assert_close(got[:-2], ref, "bf16", str(launch))


# ---------------------------------------------------------------------------
# the four large workloads at full size, in the bench's launch configuration,
# on sampled rows the oracle computes one by one
# ---------------------------------------------------------------------------

FULL = ["bf16_decode", "bf16_chunked_prefill", "bf16_chunked_prefill_g4", "bf16_chunked_prefill_g16",
        "bf16_long_decode", "fp8_mixed", "tiny_ragged_fp32"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled_rows(name):
    x = wl.WORKLOADS[name]().build()
    got = run_gpu(x)
    n = x.total_q
    rows = np.unique(np.concatenate([np.linspace(0, n - 1, min(n, 12)).astype(np.int64), [0, n - 1]]))
    ref = oracle.sparse_attention(x, rows)
    assert_close(got[rows], ref, x.dtype, name)
    assert np.isfinite(got).all()
    assert status_clean()


@pytest.mark.parametrize("ctas", [0, 7, 1000])
def test_fp8_eight_head_units_match_oracle(ctas):
    """FP8 with 8 kv heads (1 KB of K per key for eight heads): the persistent
    kernel's eight-head units, on split and unsplit grids."""
    import dataclasses

    spec = dataclasses.replace(wl.small_variants()["fp8_mixed_small"], num_q_heads=64, num_kv_heads=8)
    x = spec.build()
    kw = dict(kernel=3, heads_per_unit=8, ctas=ctas)
    assert_close(run_gpu(x, **kw), oracle.sparse_attention(x), "e4m3", f"fp8 eight-head units {kw}")
    assert status_clean()
