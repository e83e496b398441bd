"""The oracle and the CUDA path share nothing, and the product path has no fallback.

Static checks over the committed sources (CPU only):
- nothing in the package (binding, build script, kernels) imports, includes or names a file of
  the oracle; outside tests/ only the build/smoke entry and the benchmark's CPU legs import it;
- the oracle imports nothing of the package and includes no header of the kernels;
- the seeded input generators import neither side;
- the binding refuses to run when the library is missing instead of computing anything itself.
"""
import ast
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "packed_weight_gemv_gb300"


def _py_files(rel_dir):
    out = []
    for dirpath, _, files in os.walk(os.path.join(ROOT, rel_dir)):
        if "__pycache__" in dirpath or os.sep + "_lib" in dirpath:
            continue
        out += [os.path.join(dirpath, f) for f in files if f.endswith(".py")]
    return sorted(out)


def _imported_roots(path):
    tree = ast.parse(open(path, encoding="utf-8").read(), filename=path)
    roots = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            roots |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.level == 0 and node.module:
            roots.add(node.module.split(".")[0])
    return roots


def _local_includes(path):
    return re.findall(r'^\s*#\s*include\s+"([^"]+)"', open(path, encoding="utf-8").read(), re.M)


def test_package_never_imports_the_oracle():
    files = _py_files(PKG)
    assert files, "package sources not found"
    for f in files:
        assert "oracle" not in _imported_roots(f), f


def test_kernels_include_nothing_of_the_oracle_or_the_generators():
    csrc = os.path.join(ROOT, PKG, "csrc")
    own = set(os.listdir(csrc)) | {"nt.h"}
    for name in os.listdir(csrc):
        if name.endswith((".cu", ".cuh", ".h", ".cpp")):
            for inc in _local_includes(os.path.join(csrc, name)):
                assert inc in own, f"{name} includes {inc}"


def test_only_tests_entry_and_benchmark_import_the_oracle():
    allowed = {"bench.py", "__graft_entry__.py"}
    for f in _py_files("."):
        rel = os.path.relpath(f, ROOT)
        parts = rel.split(os.sep)
        top = parts[0] if len(parts) > 1 else ""
        if top in ("tests", "oracle", "baseline") or top.startswith(("_", ".")) or top.endswith("_out"):
            continue  # the tests, the oracle itself, the reference install, scratch folders
        if "oracle" in _imported_roots(f):
            assert rel in allowed, rel


def test_oracle_imports_nothing_of_the_package():
    for f in _py_files("oracle"):
        assert PKG not in _imported_roots(f), f
    c = os.path.join(ROOT, "oracle", "oracle.c")
    assert _local_includes(c) == [], "the oracle's C source includes a project header"


def test_input_generators_import_neither_side():
    for f in _py_files("synth"):
        roots = _imported_roots(f)
        assert "oracle" not in roots and PKG not in roots, f
    assert _local_includes(os.path.join(ROOT, "synth", "synth.c")) == []


def test_binding_refuses_to_run_without_the_library(tmp_path):
    code = ("import sys\n"
            "from packed_weight_gemv_gb300 import nt\n"
            f"nt.load_library({str(tmp_path / 'libnt.so')!r})\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "is missing" in r.stderr
