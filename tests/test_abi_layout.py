"""The ctypes structures of the binding match the C header (no GPU): a probe
compiled with the host C compiler against include/qsa.h prints the size and
every field offset of qsa_tensor and qsa_options, and the binding's
ctypes.Structure definitions must agree field by field."""
import ctypes
import os
import shutil
import subprocess

import pytest

from index_gathered_sparse_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "qsa.h"
#define F(T, f) printf(#T " " #f " %zu\n", offsetof(T, f))
int main(void) {
  printf("qsa_tensor size %zu\n", sizeof(qsa_tensor));
  F(qsa_tensor, data); F(qsa_tensor, dtype); F(qsa_tensor, ndim); F(qsa_tensor, shape);
  printf("qsa_options size %zu\n", sizeof(qsa_options));
  F(qsa_options, kernel); F(qsa_options, splits); F(qsa_options, ctas); F(qsa_options, block_lists);
  F(qsa_options, heads_per_unit); F(qsa_options, test_stall); F(qsa_options, tcgen05);
  F(qsa_options, reserved);
  return 0;
}
"""


@pytest.fixture(scope="module")
def layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    d = tmp_path_factory.mktemp("abi")
    src, exe = d / "probe.c", d / "probe"
    src.write_text(PROBE)
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    res = {}
    for line in out.splitlines():
        t, f, v = line.split()
        res[(t, f)] = int(v)
    return res


@pytest.mark.parametrize("cls", [B.qsa_tensor, B.qsa_options])
def test_ctypes_struct_matches_header(layout, cls):
    name = cls.__name__
    assert ctypes.sizeof(cls) == layout[(name, "size")]
    for fname, _ in cls._fields_:
        assert getattr(cls, fname).offset == layout[(name, fname)], f"{name}.{fname}"
