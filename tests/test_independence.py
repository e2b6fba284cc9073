"""The oracle and the CUDA path share no code (no GPU): no product file names
the oracle, no oracle file names the product, ``bench.py`` reaches the oracle
only from its CPU legs, and the binding refuses to run without its library."""
import ast
import os
import re

import pytest

from conftest import ROOT

PKG = os.path.join(ROOT, "persistent_megakernel_decode_gb300")
ORACLE = os.path.join(ROOT, "oracle")
SRC_EXT = (".py", ".c", ".h", ".cpp", ".cu", ".cuh")


def _sources(top):
    for d, dirs, files in os.walk(top):
        dirs[:] = [x for x in dirs if not x.startswith(("_lib", "__pycache__"))]
        for f in files:
            if f.endswith(SRC_EXT):
                yield os.path.join(d, f)


def test_product_never_imports_or_includes_the_oracle():
    pat = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b|#\s*include\s*[<\"].*oracle)", re.M)
    for p in _sources(PKG):
        assert not pat.search(open(p).read()), p


def test_oracle_never_imports_or_includes_the_product():
    pat = re.compile(r"^\s*(from\s+persistent_megakernel_decode_gb300\b|import\s+persistent_megakernel_decode_gb300\b"
                     r"|#\s*include\s*[<\"].*(csrc|mk\.h|mk_internal|planner))", re.M)
    for p in _sources(ORACLE):
        assert not pat.search(open(p).read()), p


# bench.py functions that may import the oracle: the CPU baseline legs and the
# reference arm
CPU_LEGS = {"cpu_oracle_rate", "run_glm", "run_glm_reference"}


def test_bench_reaches_the_oracle_only_from_its_cpu_legs():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())

    def imports_oracle(node):
        for n in ast.walk(node):
            if isinstance(n, ast.ImportFrom) and (n.module or "").split(".")[0] == "oracle":
                return True
            if isinstance(n, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in n.names):
                return True
        return False

    for node in tree.body:
        if isinstance(node, ast.FunctionDef):
            if imports_oracle(node):
                assert node.name in CPU_LEGS, node.name
        else:
            assert not imports_oracle(node)


def test_binding_fails_loudly_without_its_library(monkeypatch):
    from persistent_megakernel_decode_gb300 import runtime as rt
    monkeypatch.setattr(rt, "_lib", None)
    monkeypatch.setattr(rt, "LIB_PATH", os.path.join(ROOT, "no-such-dir", "libmk.so"))
    with pytest.raises(RuntimeError, match="libmk.so not found"):
        rt.load()
