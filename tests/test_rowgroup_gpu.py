"""Kernel 4, the row-group kernel (R = 128 / group consecutive rows of a
sequence per CTA and kv head, dense page tiles masked to each row's own
positions, tcgen05 contractions), against the float64 oracle element by
element, with the tolerances of the other BF16 parity tests (1e-2 + 1e-2|ref|).

Every byte no selection may read is NaN in these caches (slots past a
sequence, unowned pages, other layers), and the kernel reads whole pages: the
tests check that none of it reaches an output, that positions inside a
sequence which no row selects may hold NaN too, and that the cases the
bitmaps cannot hold (repeated positions, sequences longer than the length
hints) take the kernel's exact path with the same results.
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


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    B.qsa_read_device_status(clear=True)
    yield


def spec(name, seed, rows, cache, width, nq=64, nkv=8, page=64, out="bf16"):
    """The chunked-prefill recipe (the 64 nearest positions plus distinct
    uniform picks, sorted, tail -1) on other shapes."""
    s = wl.bf16_chunked_prefill(seed=seed, rows=rows, cache=cache, width=width)
    return dataclasses.replace(s, name=name, num_q_heads=nq, num_kv_heads=nkv, page_size=page, out_dtype=out)


CASES = {
    # group 8: 16 rows per group; ragged groups, a one-row sequence, a sequence without cache
    "g8_p64": spec("g8_p64", 31, (40, 9, 23, 1), (0, 300, 77, 5), 256),
    # group 4: 32 rows per group, pages of 16 slots (eight copies per tile line)
    "g4_p16": spec("g4_p16", 32, (70, 33), (20, 150), 200, nq=32, nkv=8, page=16),
    # group 16: 8 rows per group, pages of one tile
    "g16_p128": spec("g16_p128", 33, (20, 13, 8), (100, 0, 500), 300, nq=32, nkv=2, page=128),
    # pages of two tiles (a tile starts inside a page), F32 output
    "g8_p256_f32": spec("g8_p256_f32", 34, (50, 17), (700, 40), 400, nq=16, nkv=2, page=256, out="f32"),
    # the smallest page the kernel takes
    "g8_p8": spec("g8_p8", 35, (40, 12), (60, 33), 96, nq=16, nkv=2, page=8),
}


def plan(x, **kw):
    code = B.QSA_BF16
    return B.qsa_plan(code, x.total_q, x.num_kv_heads, x.head_dim, x.selection_width, x.group, batch=x.batch,
                      page_size=x.kv_shape[3], max_prompt_length=x.max_prompt_length,
                      max_cache_length=x.max_cache_length, **kw)


def run(x, d=None, **kw):
    d = d or wl.to_torch(x, "cuda")
    B.qsa_sparse_attention_ragged_paged(**d, **kw)
    torch.cuda.synchronize()
    return d["output"].float().cpu().double().numpy()


def assert_close(got, ref, what=""):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output (a poisoned byte reached it)"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (f"{what}: {int((err > bound).sum())} of {err.size} outside tolerance; worst at "
                                  f"{worst}: got {got[worst]}, ref {ref[worst]}")


@pytest.mark.parametrize("name", sorted(CASES))
def test_row_groups_match_oracle(name):
    x = CASES[name].build()
    assert plan(x)["kernel"] == 4, "these prefill shapes are the row-group kernel's by default"
    ref = oracle.sparse_attention(x)
    for kw in (dict(), dict(kernel=4)):
        got = run(x, **kw)
        assert_close(got, ref, f"{name} {kw}")
    assert B.qsa_read_device_status(clear=True) == 0


def test_agrees_with_the_persistent_kernel():
    """The same call on kernel 3 and kernel 4: both within the tolerance of
    the oracle, and of each other."""
    x = CASES["g8_p64"].build()
    a, b = run(x, kernel=3), run(x, kernel=4)
    assert np.abs(a - b).max() <= 2 * (ATOL + RTOL * np.abs(a).max())


def _poison_unselected(x):
    """NaN in K and V at every position of [0, kv_len) that no row of its
    sequence selects (the oracle never reads them; the kernel loads them with
    their pages)."""
    kv6 = x.kv_view()
    P = x.kv_shape[3]
    seq = x.row_sequence()
    kv_len = x.cache_lengths.astype(np.int64) + np.diff(x.input_row_offsets.astype(np.int64))
    nan = np.uint16(0x7FC0)
    n_poisoned = 0
    for b in range(x.batch):
        rows = np.nonzero(seq == b)[0]
        sel = set()
        for r in rows:
            sel.update(int(v) for v in x.token_indices[r, : x.counts[r]])
        for pos in range(int(kv_len[b])):
            if pos in sel:
                continue
            page = int(x.kv_lookup_table[b, pos // P])
            kv6[page, :, x.layer_idx, pos % P] = nan
            n_poisoned += 1
    return n_poisoned


SPARSE = {
    # few rows on long contexts: their selections leave most positions unselected
    "sparse_g8": spec("sparse_g8", 36, (20, 6), (3000, 1500), 128),
    "g16_p128": CASES["g16_p128"],
}


@pytest.mark.parametrize("name", sorted(SPARSE))
def test_unselected_positions_may_hold_nan(name):
    x = SPARSE[name].build()
    ref = oracle.sparse_attention(x)
    assert _poison_unselected(x) > 0
    got = run(x, kernel=4)
    assert_close(got, ref, f"{name} with NaN at unselected positions")
    assert B.qsa_read_device_status(clear=True) == 0


def test_repeated_positions_take_the_exact_path():
    """A repeated index is its own softmax term: the groups holding such a row
    run on the kernel's CUDA-core path, the others on the tensor cores."""
    x = CASES["g8_p64"].build()
    for r in (3, 41, 60):
        n = int(x.counts[r])
        assert n >= 4
        x.token_indices[r, 1] = x.token_indices[r, 0]
        x.token_indices[r, n - 1] = x.token_indices[r, 2]
    ref = oracle.sparse_attention(x)
    got = run(x, kernel=4)
    assert_close(got, ref, "repeated positions")
    assert B.qsa_read_device_status(clear=True) == 0


def test_short_length_hints_take_the_exact_path():
    """Bitmaps sized from hints shorter than a sequence cannot hold it: that
    sequence's groups take the exact path; results do not depend on hints."""
    x = CASES["g8_p64"].build()
    ref = oracle.sparse_attention(x)
    for mp, mc in ((x.max_prompt_length, 0), (1, 1), (0, 0)):
        d = wl.to_torch(x, "cuda")
        d["max_prompt_length"], d["max_cache_length"] = mp, mc
        got = run(x, d, kernel=4)
        assert_close(got, ref, f"hints {mp}, {mc}")
    assert B.qsa_read_device_status(clear=True) == 0


def test_empty_and_clamped_rows():
    x = CASES["g8_p64"].build()
    x.counts[0] = 0
    x.counts[17] = -5
    x.counts[18] = 0
    # a whole group of empty rows (rows 16..31 of the first sequence)
    x.counts[16:32] = 0
    ref = oracle.sparse_attention(x)
    got = run(x, kernel=4)
    for r in (0, 17, 18, 20):
        assert np.array_equal(got[r], np.zeros_like(got[r]))
    assert_close(got, ref, "empty rows")


def test_out_of_range_positions_are_skipped_and_reported():
    """Positions in [kv_len, max_pages * page_size) inside counts: skipped
    and flagged (their table entries name allocated, NaN-filled pages)."""
    x = CASES["g8_p64"].build()
    P, max_pages = x.kv_shape[3], x.kv_lookup_table.shape[1]
    seq = x.row_sequence()
    kv_len = x.cache_lengths.astype(np.int64) + np.diff(x.input_row_offsets.astype(np.int64))
    y = CASES["g8_p64"].build()
    bad_rows = [r for r in range(x.total_q) if kv_len[seq[r]] < max_pages * P and x.counts[r] >= 3][:4]
    assert len(bad_rows) == 4
    for r in bad_rows:
        n = int(x.counts[r])
        x.token_indices[r, 1] = kv_len[seq[r]]
        keep = [j for j in range(n) if j != 1]
        sel = x.token_indices[r, keep].copy()
        y.token_indices[r, : len(sel)] = sel
        y.counts[r] = len(sel)
    ref = oracle.sparse_attention(y)
    B.qsa_read_device_status(clear=True)
    got = run(x, kernel=4)
    assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_INDEX
    assert_close(got, ref, "out-of-range positions")


def test_bad_page_table_entry_is_skipped_and_reported():
    """A table entry naming no page of the descriptor (it ends one page before
    the allocation's NaN-filled last page): every row of that sequence loses
    the keys on that page, and the call flags it."""
    x = CASES["g8_p64"].build()
    P = x.kv_shape[3]
    b = 1  # 9 rows on 300 cached positions
    lp = 2
    assert x.poison_page == x.kv_shape[0] - 1
    x.kv_lookup_table[b, lp] = x.poison_page
    y = CASES["g8_p64"].build()
    seq = y.row_sequence()
    for r in np.nonzero(seq == b)[0]:
        sel = [int(v) for v in y.token_indices[r, : y.counts[r]] if int(v) // P != lp]
        y.token_indices[r, : len(sel)] = sel
        y.counts[r] = len(sel)
    ref = oracle.sparse_attention(y)
    d = wl.to_torch(x, "cuda")
    d["kv_blocks"] = d["kv_blocks"][: x.poison_page]
    B.qsa_read_device_status(clear=True)
    got = run(x, d, kernel=4)
    assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_PAGE
    assert_close(got, ref, "bad page")


def test_output_never_depends_on_page_placement():
    """The same logical cache on a different page permutation gives the same
    output bits."""
    s = CASES["g8_p64"]
    x = s.build()
    a = run(x, kernel=4)
    n_pages = x.kv_shape[0] - 1
    perm = np.random.default_rng(5).permutation(n_pages)
    y = s.build()
    kv6x, kv6y = x.kv_view(), y.kv_view()
    table = y.kv_lookup_table.copy()
    kv6y[perm] = kv6x[:n_pages]
    for b in range(y.batch):
        for lp in range(table.shape[1]):
            if x.kv_lookup_table[b, lp] < n_pages:
                table[b, lp] = perm[x.kv_lookup_table[b, lp]]
    y.kv_lookup_table[:] = table
    bb = run(y, kernel=4)
    assert np.array_equal(a, bb)


def test_reference_moves_within_and_across_tiles():
    """Scores that climb by more than 2^8 (in base 2) every 16 positions: the
    lazy reference maximum moves inside tiles (the first half's P, already in
    tensor memory, is rescaled) and across tiles (O is rescaled), on every row;
    results still match the oracle."""
    x = CASES["g8_p64"].build()
    P = x.kv_shape[3]
    kv6 = x.kv_view()
    kv_len = x.cache_lengths.astype(np.int64) + np.diff(x.input_row_offsets.astype(np.int64))
    x.q[:] = wl.encode(np.full(x.q.shape, 0.5, np.float32), "bf16")
    D, nkv = x.head_dim, x.num_kv_heads
    for b in range(x.batch):
        for pos in range(int(kv_len[b])):
            # q.k = 64 (pos // 16): 8.16 more (base 2, scale 1/sqrt(128)) per step of 16
            page = int(x.kv_lookup_table[b, pos // P])
            kv6[page, 0, x.layer_idx, pos % P] = wl.encode(np.full((nkv, D), float(pos // 16), np.float32), "bf16")
    assert abs(x.scale * 64 * np.log2(np.e) - 8.16) < 0.01
    ref = oracle.sparse_attention(x)
    got = run(x, kernel=4)
    assert_close(got, ref, "climbing scores")
    assert B.qsa_read_device_status(clear=True) == 0


def test_more_sequences_than_threads():
    """400 sequences, more than the kernel's 352 threads: groups are numbered
    in sequence order instead of longest first, and every row still matches."""
    rows = tuple([17] * 400)
    cache = tuple(int(c) for c in np.arange(400) % 61)
    x = spec("many_seqs", 37, rows, cache, 64).build()
    assert plan(x)["kernel"] == 4
    sample = np.unique(np.linspace(0, x.total_q - 1, 40).astype(np.int64))
    ref = oracle.sparse_attention(x, sample)
    got = run(x, kernel=4)
    assert_close(got[sample], ref, "400 sequences")
    assert np.isfinite(got).all()
    assert B.qsa_read_device_status(clear=True) == 0


@pytest.mark.parametrize("factor", [-1.0, 0.0])
def test_negative_and_zero_scale(factor):
    """The kernel runs the softmax on raw scores times |scale log2(e)| and
    applies a negative scale by negating Q (exact in BF16); a zero scale is a
    uniform softmax over each row's own keys."""
    x = CASES["g8_p64"].build()
    x.scale = float(x.scale) * factor
    ref = oracle.sparse_attention(x)
    got = run(x, kernel=4)
    assert_close(got, ref, f"scale x {factor}")
    assert B.qsa_read_device_status(clear=True) == 0
