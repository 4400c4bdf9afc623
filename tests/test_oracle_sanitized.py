"""The C oracle under AddressSanitizer and UndefinedBehaviorSanitizer (no
GPU): a copy built with -fsanitize=address,undefined runs every oracle
function on the small workloads in a child process with the sanitizer
runtimes preloaded; any out-of-bounds access, use after free or undefined
operation aborts the child."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r})
import oracle, oracle.oracle as O
O._LIB = {lib!r}
O.build = oracle.build = lambda force=False: O._LIB
from index_gathered_sparse_gb300 import workloads as wl
n = 0
for name, spec in sorted(wl.small_variants().items()):
    oracle.sparse_attention(spec.build()); n += 1
oracle.sparse_attention(wl.tiny_ragged().build()); n += 1
for name, spec in sorted(wl.msa_small_variants().items()):
    oracle.msa_attention(spec.build()); n += 1
for name, spec in sorted(wl.latent_small_variants().items()):
    oracle.latent_attention(spec.build()); n += 1
for name, spec in sorted(wl.compress_small_variants().items()):
    oracle.compress_keys(spec.build()); n += 1
print("calls", n)
"""


def _runtime(name):
    try:
        p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True, check=True).stdout.strip()
    except (OSError, subprocess.CalledProcessError):
        return None
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_is_clean_under_asan_and_ubsan(tmp_path):
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not asan or not ubsan:
        pytest.skip("sanitizer runtimes not installed")
    lib = str(tmp_path / "libqsa_oracle_san.so")
    subprocess.run(["gcc", "-O1", "-g", "-std=c99", "-fPIC", "-shared", "-fsanitize=address,undefined",
                    "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer", "-o", lib,
                    os.path.join(ROOT, "oracle", "qsa_oracle.c"), "-lm"], check=True)
    env = dict(os.environ, LD_PRELOAD=f"{asan}:{ubsan}", ASAN_OPTIONS="detect_leaks=0:abort_on_error=1")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, lib=lib)], env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-4000:]
    assert "calls" in r.stdout
    assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, r.stderr[-4000:]
