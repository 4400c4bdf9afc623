"""GPU parity of latent sparse attention (window + listed compressed entries
+ per-head sinks) against the float64 latent oracle: small variants under
several split counts, sinks at -inf, window only / entries only, an entry
past the sequence's entries (flagged and skipped), page placement
(bit-exact), and sampled rows of the full-size latent workloads.
Tolerances: BF16 1e-2 + 1e-2|ref|, FP8 6e-2 + 3e-2|ref|."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from index_gathered_sparse_gb300 import binding as B
from index_gathered_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-2), "e4m3": (6e-2, 3e-2)}
SMALL = wl.latent_small_variants()
LAUNCHES = [dict(), dict(splits=1), dict(splits=3)]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
    oracle.build()
    assert torch.cuda.is_available()
    B.qsa_read_device_status(clear=True)
    yield


def run_gpu(x, **kw) -> np.ndarray:
    d = wl.to_torch_latent(x, "cuda")
    B.qsa_latent_attention_ragged_paged(**d, **kw)
    torch.cuda.synchronize()
    return d["output"].float().cpu().double().numpy()


def assert_close(got, ref, dtype, what):
    atol, rtol = TOL[dtype]
    assert np.isfinite(got).all(), f"{what}: non-finite output (a poisoned byte was read)"
    err, bound = np.abs(got - ref), atol + rtol * np.abs(ref)
    assert (err <= bound).all(), f"{what}: {int((err > bound).sum())} of {err.size} outside tolerance"


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("launch", range(len(LAUNCHES)))
def test_small_latent_matches_oracle(name, launch):
    x = SMALL[name].build()
    assert_close(run_gpu(x, **LAUNCHES[launch]), oracle.latent_attention(x), x.dtype, f"{name} {LAUNCHES[launch]}")
    assert B.qsa_read_device_status(clear=True) == 0


@pytest.mark.parametrize("num_heads", [64, 128])
def test_head_groups_in_fours(num_heads):
    """64 or 128 query heads (4 or 8 groups of 16): with one band a CTA serves
    four groups of a row, one warp per group over every key; with three bands
    each group is its own unit again.  Both match the oracle."""
    x = dataclasses.replace(SMALL["latent_bf16_prefill_small"], num_heads=num_heads).build()
    ref = oracle.latent_attention(x)
    for kw in (dict(), dict(splits=1), dict(splits=3)):
        assert_close(run_gpu(x, **kw), ref, x.dtype, f"{num_heads} heads {kw}")
        assert B.qsa_read_device_status(clear=True) == 0


def test_without_sinks_and_single_sources():
    spec = SMALL["latent_bf16_prefill_small"]
    x = spec.build()
    no_sink = dataclasses.replace(x, attn_sink=np.full(x.num_heads, -np.inf, np.float32))
    assert_close(run_gpu(no_sink), oracle.latent_attention(no_sink), x.dtype, "no sinks")
    win_only = dataclasses.replace(x, comp_indices=np.full_like(x.comp_indices, -1))
    assert_close(run_gpu(win_only, splits=2), oracle.latent_attention(win_only), x.dtype, "window only")
    ent_only = dataclasses.replace(spec, window=0).build()
    assert_close(run_gpu(ent_only), oracle.latent_attention(ent_only), x.dtype, "entries only")
    assert B.qsa_read_device_status(clear=True) == 0


def test_entry_past_the_sequence_is_skipped_and_flagged():
    x = SMALL["latent_bf16_decode_small"].build()
    bad = x.comp_indices.copy()
    seq = x.swa.row_sequence()
    bad[2, 1] = int(x.comp.cache_lengths[seq[2]]) + 5
    got = run_gpu(dataclasses.replace(x, comp_indices=bad))
    assert B.qsa_read_device_status(clear=True) & B.QSA_STATUS_BAD_INDEX
    ok = bad.copy()
    ok[2, 1] = -1
    assert_close(got, oracle.latent_attention(dataclasses.replace(x, comp_indices=ok)), x.dtype, "bad entry")


def test_page_placement_is_bit_exact():
    spec = SMALL["latent_bf16_prefill_small"]
    a = run_gpu(spec.build())
    b = run_gpu(dataclasses.replace(spec, page_size=16, comp_page_size=32).build())
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("name", sorted(wl.LATENT_WORKLOADS))
def test_full_size_latent_sampled_rows(name):
    x = wl.LATENT_WORKLOADS[name]().build()
    got = run_gpu(x)
    rows = np.unique(np.linspace(0, x.total_q - 1, 6).astype(np.int64))
    assert_close(got[rows], oracle.latent_attention(x, rows), x.dtype, name)
    assert B.qsa_read_device_status(clear=True) == 0
