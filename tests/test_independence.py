"""The library and the oracle are independent, and the library has no other
path: nothing under the package or include/ loads, includes or imports the
oracle; the oracle names neither the package nor its header; and without its
shared library the binding raises instead of computing anything.
"""

import os
import re

import pytest

import paged_kv_cache_reshape_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CODE = (".py", ".cu", ".cuh", ".h", ".c", ".cpp")


def _files(*dirs):
    for d in dirs:
        for base, _, names in os.walk(os.path.join(ROOT, d)):
            if "__pycache__" in base:
                continue
            for n in names:
                if n.endswith(CODE):
                    yield os.path.join(base, n)


def test_library_does_not_reach_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s*[<\"].*oracle)|liboracle|oracle\.c\b", re.M)
    hits = [f for f in _files("paged_kv_cache_reshape_gb300", "include") if pat.search(open(f).read())]
    assert not hits, f"library files reaching the oracle: {hits}"


def test_oracle_does_not_reach_the_library():
    pat = re.compile(r"paged_kv_cache_reshape_gb300|libpa_gb300|#\s*include\s*[<\"][^>\"]*pa\.h|\bcsrc\b")
    hits = [f for f in _files("oracle") if pat.search(open(f).read())]
    assert not hits, f"oracle files reaching the library: {hits}"


def test_binding_raises_without_its_library(monkeypatch, tmp_path):
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(pa, "LIB_PATH", str(tmp_path / "libpa_gb300.so"))
    with pytest.raises(RuntimeError, match="missing"):
        pa.lib()
