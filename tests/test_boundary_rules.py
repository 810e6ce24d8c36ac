"""Who may use the oracle, and what the two sides share (host only, no GPU).

The oracle is test infrastructure: the package (the binding, the harness, the host logic) never
imports it; bench.py reaches it only from its CPU-baseline leg and its reference arm; the oracle
never imports the package's compute side, and its C part includes no header of the CUDA library.
The seeded input generators (paged_mla_kv_gb300/synth.py) are the one module both may use, and
they import neither side.  The binding fails loudly, rather than falling back, when the library
has not been built.
"""
import ast
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_mla_kv_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _py_files(d):
    for base, dirs, files in os.walk(d):
        dirs[:] = [x for x in dirs if x not in ("_build", "__pycache__")]
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(base, f)


def _imports(path):
    """(line, top-level module or relative marker, enclosing scopes) of every import in a file."""
    tree = ast.parse(open(path).read(), path)
    out = []

    def walk(node, scopes):
        for c in ast.iter_child_nodes(node):
            s = scopes + [c.name] if isinstance(c, (ast.FunctionDef, ast.ClassDef)) else scopes
            if isinstance(c, ast.Import):
                out.extend((c.lineno, a.name.split(".")[0], s) for a in c.names)
            elif isinstance(c, ast.ImportFrom):
                mod = "." * c.level + (c.module or "")
                if c.level and not c.module:
                    out.extend((c.lineno, "." + a.name, s) for a in c.names)
                else:
                    out.append((c.lineno, mod.split(".")[0] if not c.level else mod, s))
            walk(c, s)

    walk(tree, [])
    return out


def test_package_never_imports_the_oracle():
    for f in _py_files(PKG):
        for line, mod, _ in _imports(f):
            assert mod != "oracle", f"{f}:{line} imports the oracle"


def test_oracle_never_imports_the_package():
    for f in _py_files(ORACLE):
        for line, mod, _ in _imports(f):
            assert mod != "paged_mla_kv_gb300", f"{f}:{line} imports the package"


def test_input_generators_import_neither_side():
    for line, mod, _ in _imports(os.path.join(PKG, "synth.py")):
        assert mod not in ("oracle", "paged_mla_kv_gb300") and not mod.startswith("."), \
            f"synth.py:{line} imports {mod}"


def test_bench_reaches_the_oracle_only_from_its_baseline_legs():
    legs = {"OracleSample", "TopkOracleSample", "reference_arm"}
    found = 0
    for line, mod, scopes in _imports(os.path.join(ROOT, "bench.py")):
        if mod == "oracle":
            found += 1
            assert scopes and scopes[0] in legs, f"bench.py:{line} imports the oracle from {scopes}"
    assert found > 0
    # the sample classes are built only by the reference arm and after the timed region
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef) and fn.name not in legs:
            for c in ast.walk(fn):
                if isinstance(c, ast.Call) and isinstance(c.func, ast.Name) and c.func.id.endswith("OracleSample"):
                    assert c.func.id in ("OracleSample", "TopkOracleSample")
                    # each such call is guarded by the cpu-baseline switch
                    src = ast.get_source_segment(open(os.path.join(ROOT, "bench.py")).read(), fn)
                    assert "no_cpu_baseline" in src, fn.name


def test_oracle_c_shares_no_header_with_the_library():
    for f in os.listdir(ORACLE):
        if f.endswith((".c", ".h")):
            for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', open(os.path.join(ORACLE, f)).read()):
                assert "tf_" not in inc and "csrc" not in inc and "include/" not in inc, (f, inc)
    for f in os.listdir(os.path.join(PKG, "csrc")):
        src = open(os.path.join(PKG, "csrc", f), errors="replace").read()
        assert "oracle" not in " ".join(re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', src)), f


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    from paged_mla_kv_gb300 import binding as B
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "libtf_paged_mla.so"))
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()
