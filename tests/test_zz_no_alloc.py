"""The allocation-free entry point against the default one.

qsa_sparse_attention_ragged_paged_noalloc keeps its scratch in a fixed device
array shared by every call; two calls in a row must each reproduce the default
entry point's output (within the parity tolerances) and raise no status bit.
This file runs last so that it also sees the scratch after everything the
other GPU tests left behind.
"""
import numpy as np
import pytest
import torch

from index_gathered_sparse_gb300 import binding as B
from index_gathered_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": (1e-2, 1e-2), "e4m3": (6e-2, 3e-2)}


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
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
    for call in range(2):
        d["output"].fill_(float("nan"))
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.qsa_sparse_attention_ragged_paged_noalloc(**d, status_flags=flags)
        torch.cuda.synchronize()
        _close(d["output"], ref, x.dtype, f"{name} call {call + 1}")
        assert int(flags.item()) == 0


def test_noalloc_rejects_f32():
    x = wl.tiny_ragged().build()
    d = wl.to_torch(x, "cuda")
    if d["q"].dtype != torch.float32:
        pytest.skip("tiny case is not F32")
    with pytest.raises(B.QSAError) as ei:
        B.qsa_sparse_attention_ragged_paged_noalloc(**d)
    assert ei.value.status == 4
