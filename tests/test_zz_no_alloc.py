"""The allocation-free entry point against the default one and the oracle.

qsa_sparse_attention_ragged_paged_noalloc keeps its scratch in a fixed device
array shared by every call; two calls in a row must each reproduce the default
entry point's output and the float64 oracle (within the parity tolerances)
and raise no status bit.  A call whose scratch would not fit is refused
before anything is enqueued, and status bits reach the caller's word.  This
file runs last so that it also sees the scratch after everything the other
GPU tests left behind.
"""
import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import binding as B
from index_gathered_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-2), "e4m3": (6e-2, 3e-2)}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    yield


def _close(got: torch.Tensor, ref: torch.Tensor, dtype: str, what: str) -> None:
    atol, rtol = TOL[dtype]
    g = got.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    bound = atol + rtol * np.abs(r)
    err = np.abs(g - r)
    assert (err <= bound).all(), f"{what}: {int((err > bound).sum())} of {err.size} outside tolerance"


@pytest.mark.parametrize("name", ["bf16_decode_small", "bf16_long_decode_small", "fp8_mixed_small",
                                  "bf16_prefill_small"])
def test_noalloc_matches_default_entry_point(name):
    x = wl.small_variants()[name].build()
    d = wl.to_torch(x, "cuda")
    B.qsa_sparse_attention_ragged_paged(**d)
    torch.cuda.synchronize()
    ref = d["output"].clone()
    exact = torch.from_numpy(oracle.sparse_attention(x))
    for call in range(2):
        d["output"].fill_(float("nan"))
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.qsa_sparse_attention_ragged_paged_noalloc(**d, status_flags=flags)
        torch.cuda.synchronize()
        _close(d["output"], ref, x.dtype, f"{name} call {call + 1} vs the default entry point")
        _close(d["output"], exact, x.dtype, f"{name} call {call + 1} vs the oracle")
        assert int(flags.item()) == 0


def test_noalloc_reports_status_bits_in_the_callers_word():
    """A position inside counts past its sequence (in [kv_len, max_pages *
    page_size): it stays inside the allocated, NaN-filled cache) is skipped
    and BAD_INDEX lands in status_flags; the rest matches the oracle."""
    x = wl.small_variants()["bf16_decode_small"].build()
    P, max_pages = x.kv_shape[3], x.kv_lookup_table.shape[1]
    kv_len = x.cache_lengths.astype(np.int64) + 1
    r = next(r for r in range(x.total_q) if kv_len[r] < max_pages * P and x.counts[r] >= 2)
    y = wl.small_variants()["bf16_decode_small"].build()
    x.token_indices[r, 0] = kv_len[r]
    y.token_indices[r, : y.counts[r] - 1] = y.token_indices[r, 1 : y.counts[r]].copy()
    y.counts[r] -= 1
    d = wl.to_torch(x, "cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.qsa_sparse_attention_ragged_paged_noalloc(**d, status_flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) & B.QSA_STATUS_BAD_INDEX
    _close(d["output"], torch.from_numpy(oracle.sparse_attention(y)), x.dtype, "bad index")


def test_noalloc_refuses_calls_beyond_its_scratch():
    """One kv head and about 4.2 M query rows need more arrival tickets than
    the fixed scratch holds: QSA_ERR_UNSUPPORTED, and nothing is enqueued (a
    NaN-filled output stays untouched)."""
    rows, D = 4_200_000, 128
    dev = "cuda"
    bf = torch.bfloat16
    q = torch.zeros((rows, 1, D), dtype=bf, device=dev)
    out = torch.full((rows, 1, D), float("nan"), dtype=bf, device=dev)
    kv = torch.zeros((1, 2, 1, 16, 1, D), dtype=bf, device=dev)
    offs = torch.tensor([0, rows], dtype=torch.int32, device=dev)
    cache = torch.zeros(1, dtype=torch.int32, device=dev)
    table = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    idx = torch.zeros((rows, 1), dtype=torch.int32, device=dev)
    cnt = torch.zeros(rows, dtype=torch.int32, device=dev)
    with pytest.raises(B.QSAError) as ei:
        B.qsa_sparse_attention_ragged_paged_noalloc(out, q, offs, kv, -1, cache, table, rows, 0, 0, idx, cnt,
                                                    D ** -0.5, 1)
    assert ei.value.status == 4 and "scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert bool(torch.isnan(out).all())


def test_noalloc_rejects_f32():
    x = wl.tiny_ragged().build()
    d = wl.to_torch(x, "cuda")
    if d["q"].dtype != torch.float32:
        pytest.skip("tiny case is not F32")
    with pytest.raises(B.QSAError) as ei:
        B.qsa_sparse_attention_ragged_paged_noalloc(**d)
    assert ei.value.status == 4
