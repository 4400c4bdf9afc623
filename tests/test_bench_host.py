"""Host-side logic of bench.py (no GPU): the kernel-source hash that gates
the recorded ncu traffic ignores comments, blank lines and runs of spaces
but not code, and the recorded traffic is reported only under the hash it
was taken with."""
import json
import os
import shutil

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
