"""Static checks that the oracle and the CUDA path stay apart.

The oracle is test infrastructure: the product package (Python binding,
workloads, generators, CUDA sources) must not import, include or name it,
the oracle must not import the product package, and the two programs that
may run it (bench.py's CPU baseline and reference arm, the entry module's
smoke check) import it only inside those functions, never at module level.
CPU only; reads source files."""
import ast
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "sparse_attention_decode_qsa_gb300")


def _sources(top, exts):
    for d, dirs, files in os.walk(top):
        dirs[:] = [x for x in dirs if not x.startswith(("_build", "__pycache__"))]
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _imported_modules(tree):
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield node, a.name
        elif isinstance(node, ast.ImportFrom) and node.module:
            yield node, node.module


def test_product_package_never_reaches_the_oracle():
    py = list(_sources(PKG, (".py",)))
    assert py, "no package sources found"
    for path in py:
        tree = ast.parse(open(path).read(), path)
        for _, mod in _imported_modules(tree):
            assert not (mod == "oracle" or mod.startswith("oracle.") or "qsa_oracle" in mod), \
                f"{os.path.relpath(path, ROOT)} imports {mod}"
        assert "qsa_oracle" not in open(path).read(), os.path.relpath(path, ROOT)
    native = list(_sources(os.path.join(PKG, "csrc"), (".cu", ".cuh", ".h", ".cpp")))
    native += list(_sources(os.path.join(ROOT, "include"), (".h",)))
    assert native, "no native sources found"
    for path in native:
        text = open(path).read()
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', text):
            assert "oracle" not in inc, f"{os.path.relpath(path, ROOT)} includes {inc}"


def test_oracle_never_imports_the_product():
    for path in _sources(os.path.join(ROOT, "oracle"), (".py",)):
        tree = ast.parse(open(path).read(), path)
        for _, mod in _imported_modules(tree):
            assert not mod.startswith("sparse_attention_decode_qsa_gb300"), \
                f"{os.path.relpath(path, ROOT)} imports {mod}"
            assert mod not in ("torch", "bench", "__graft_entry__"), \
                f"{os.path.relpath(path, ROOT)} imports {mod}"


def test_oracle_imported_only_inside_the_allowed_functions():
    allowed = {"bench.py": {"_oracle_sample"}, "__graft_entry__.py": {"smoke"}}
    for name, funcs in allowed.items():
        path = os.path.join(ROOT, name)
        tree = ast.parse(open(path).read(), path)
        # module-level statements (outside any function) never import it
        for node in tree.body:
            if isinstance(node, (ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)):
                continue
            for _, mod in _imported_modules(node):
                assert not mod.startswith("oracle"), f"{name}: module-level import of {mod}"
        seen = set()
        for fn in ast.walk(tree):
            if not isinstance(fn, (ast.FunctionDef, ast.AsyncFunctionDef)):
                continue
            for _, mod in _imported_modules(fn):
                if mod.startswith("oracle"):
                    seen.add(fn.name)
        assert seen and seen <= funcs, (name, seen)
