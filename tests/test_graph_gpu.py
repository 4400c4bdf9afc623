"""GPU: qsa_sparse_attention_ragged_paged(_ex) and
qsa_msa_attention_ragged_paged inside a captured CUDA graph.  After the
workspace of the capturing stream is reserved (qsa_plan's figure) and one
warm-up call has run on it, a call captured with torch.cuda.graph and
replayed writes the same output bits as a direct call.  Cases cover each launch form: the persistent
kernel, kernel 2 with bands merged inside a thread-block cluster
(cudaLaunchKernelEx) and through the workspace tickets, block lists
with tile copies (a tensor map encoded on the host at capture time), and
the row-group kernel (two launches; its bitmaps in the workspace).
"""
import numpy as np
import pytest
import torch

from index_gathered_sparse_gb300 import binding as B
from index_gathered_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    from index_gathered_sparse_gb300 import build

    build.build()
    assert torch.cuda.is_available()
    B.qsa_read_device_status(clear=True)
    yield


CASES = {
    "persistent": ("bf16_decode_small", dict()),
    "cluster_bands": ("bf16_long_decode_small", dict(kernel=2, splits=6)),
    "ticket_bands": ("bf16_long_decode_small", dict(kernel=2, splits=12)),
    "block_tiles": ("msa_bf16_decode_small", dict(splits=3)),
    "row_groups": ("bf16_prefill_small", dict(kernel=4)),
}


def _inputs(name):
    small = {**wl.small_variants(), **wl.msa_small_variants()}
    x = small[name].build()
    if name.startswith("msa"):
        return x, wl.to_torch_msa(x, "cuda"), B.qsa_msa_attention_ragged_paged
    return x, wl.to_torch(x, "cuda"), B.qsa_sparse_attention_ragged_paged


@pytest.mark.parametrize("case", sorted(CASES))
def test_graph_replay_matches_direct_call(case):
    name, kw = CASES[case]
    x, d, fn = _inputs(name)
    fn(**d, **kw)
    torch.cuda.synchronize()
    direct = d["output"].clone()

    s = torch.cuda.Stream()
    code = {"bf16": B.QSA_BF16, "e4m3": B.QSA_F8E4M3}[x.dtype]
    if name.startswith("msa"):
        plan = B.qsa_plan(code, x.total_q, x.num_kv_heads, x.head_dim, x.topk * x.kv_shape[3], x.group,
                          kernel=2, splits=kw.get("splits", 0), block_lists=True)
    else:
        plan = B.qsa_plan(code, x.total_q, x.num_kv_heads, x.head_dim, x.selection_width, x.group,
                          kernel=kw.get("kernel", 0), splits=kw.get("splits", 0), batch=x.batch,
                          page_size=x.kv_shape[3], max_prompt_length=x.max_prompt_length,
                          max_cache_length=x.max_cache_length)
    B.qsa_reserve_workspace(plan["workspace_bytes"], stream=s.cuda_stream)
    with torch.cuda.stream(s):
        fn(**d, **kw)  # warm-up on the capturing stream (status word, kernel attributes)
    s.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(**d, **kw)
    d["output"].zero_()
    torch.cuda.synchronize()
    for _ in range(2):  # replays re-arm the split-K tickets themselves
        g.replay()
    torch.cuda.synchronize()
    got = d["output"]
    assert torch.equal(got.view(torch.uint8) if got.dtype != torch.float32 else got.view(torch.int32),
                       direct.view(torch.uint8) if direct.dtype != torch.float32 else direct.view(torch.int32))
    assert B.qsa_read_device_status(clear=True) == 0
