"""Host-side logic of bench.py (no GPU): the kernel-source hash that gates
the recorded ncu traffic ignores comments, blank lines and runs of spaces
but not code, and the recorded traffic is reported only under the hash it
was taken with."""
import json
import os
import shutil

import numpy as np

import bench


def test_code_only_drops_comments_keeps_literals():
    src = ('int a = 1;  // trailing\n'
           '/* block\n   comment */ const char* s = "x // kept /* kept */";\n'
           '\n'
           "char q = '\"';  x = \"esc \\\" // kept\";\n")
    out = bench._code_only(src)
    assert "trailing" not in out and "block" not in out and "comment" not in out
    assert '"x // kept /* kept */"' in out
    assert "'\"'" in out and '"esc \\" // kept"' in out
    assert "\n\n" not in out and "  " not in out


def _hash_of(tmp_path, files, monkeypatch):
    root = tmp_path / "r"
    csrc = root / "index_gathered_sparse_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for n, t in files.items():
        (csrc / n).write_text(t)
    monkeypatch.setattr(bench, "ROOT", str(root))
    return bench.kernel_source_hash(), root


def test_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    base = {"k.cu": "__global__ void k(int* p) { p[0] = 1; }\n"}
    h0, _ = _hash_of(tmp_path / "a", base, monkeypatch)
    h1, _ = _hash_of(tmp_path / "b", {"k.cu": "// a comment\n__global__ void k(int* p) {  /* c */ p[0] = 1; }\n\n"},
                     monkeypatch)
    h2, _ = _hash_of(tmp_path / "c", {"k.cu": "__global__ void k(int* p) { p[0] = 2; }\n"}, monkeypatch)
    assert h0 == h1
    assert h0 != h2


def test_recorded_traffic_follows_the_hash(tmp_path, monkeypatch):
    h, root = _hash_of(tmp_path, {"k.cu": "int x;\n"}, monkeypatch)
    (root / "profiles").mkdir()
    rec = {"w": {"kernel_hash": h, "dram_bytes_per_launch": 123}, "old": {"kernel_hash": "0" * 16,
                                                                         "dram_bytes_per_launch": 7}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("w") == 123
    assert bench.recorded_traffic("old") is None
    assert bench.recorded_traffic("missing") is None


def test_committed_traffic_matches_the_sources():
    """The records in profiles/ were taken on the current kernel code."""
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")) as f:
        rec = json.load(f)
    h = bench.kernel_source_hash()
    assert rec and all(e["kernel_hash"] == h for e in rec.values())


def test_roofline_bound_follows_l2_reuse():
    """Selections whose repeats are L2 hits (prefill rows of one sequence)
    take the tensor bound, with flops = 4 * group * head_dim per attended
    (key, kv head) pair; one row per sequence (decode) takes the HBM bound."""
    from index_gathered_sparse_gb300 import workloads as wl

    small = wl.small_variants()
    pre = small["bf16_prefill_small"].build()
    r = bench.roofline(pre, 2.0, "k", 1000)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["l2_reuse"] > 2
    flops = 4 * pre.group * pre.head_dim * int(pre.valid_counts().sum()) * pre.num_kv_heads
    assert r["flops_per_launch"] == flops
    assert abs(r["achieved"] - flops / 2e-3 / 1e12) < 1e-9 and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    assert r["dram"]["traffic"] == 1000 and abs(r["dram"]["achieved"] - 1000 / 2e-3 / 1e9) < 1e-9
    dec = small["bf16_decode_small"].build()
    r = bench.roofline(dec, 2.0, "k", None)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["dram"] is None
    assert abs(r["achieved"] - dec.algorithmic_bytes() / 2e-3 / 1e9) < 1e-6
    fp8 = small["fp8_mixed_small"].build()
    r = bench.roofline(fp8, 2.0, "k", None)
    if r["bound"] == "tensor":  # fp8: q.K at twice the bf16 rate, p.V at the f16 rate
        assert abs(r["peak"] - bench.measured_peaks()["bf16_tflops_sustained"] * 4 / 3) < 1e-9


def test_cpu_baseline_reports_threads_and_one_thread():
    from index_gathered_sparse_gb300 import workloads as wl

    x = wl.tiny_ragged().build()
    cpu = bench.cpu_baseline(x, 1.0, 2)
    assert cpu["kind"] == "oracle" and cpu["cores"] == 2 and cpu["value"] > 0
    assert cpu["one_thread"]["cores"] == 1 and cpu["one_thread"]["value"] > 0
    assert bench.host_cores() >= 1


def test_group_variants_of_chunked_prefill():
    """The group-4 and group-16 workloads keep the headline's rows, counts and
    page tables (their random picks follow the changed head counts)."""
    from index_gathered_sparse_gb300 import workloads as wl

    base = wl.WORKLOADS["bf16_chunked_prefill"]().build()
    for name, nq, nkv in (("bf16_chunked_prefill_g4", 32, 8), ("bf16_chunked_prefill_g16", 64, 4)):
        x = wl.WORKLOADS[name]().build()
        assert (x.num_q_heads, x.num_kv_heads, x.group) == (nq, nkv, nq // nkv)
        assert np.array_equal(x.input_row_offsets, base.input_row_offsets)
        assert np.array_equal(x.counts, base.counts) and np.array_equal(x.kv_lookup_table, base.kv_lookup_table)
