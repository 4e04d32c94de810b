"""CPU checks of the separation between the CUDA path and its float64 oracle,
read from the sources (no import of either side):

* the oracle imports only numpy, scipy and the standard library;
* the product package (its Python binding, build script and CUDA sources)
  never names the oracle;
* the seeded input generators that both sides share import neither;
* bench.py touches the oracle only in ``oracle_sample``, called by the
  reference arm and the CPU-baseline leg, and __graft_entry__.py only in
  ``smoke``, in both cases inside the function, never at import time;
* no tracked code file refers to the git-ignored scratch folder ``_work``."""
import ast
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "headwise_chunked_attention_gb300"
STDLIB_OK = {"__future__", "math", "typing", "dataclasses", "functools", "itertools",
             "collections", "os", "sys"}


def py_files(folder):
    base = os.path.join(ROOT, folder)
    return sorted(os.path.join(base, f) for f in os.listdir(base) if f.endswith(".py"))


def imports(path):
    """(top-level module name, relative level, enclosing function or None) of
    every import statement in the file."""
    tree = ast.parse(open(path).read(), path)
    out = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else fn
            if isinstance(child, ast.Import):
                out.extend((a.name.split(".")[0], 0, fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom):
                out.append(((child.module or "").split(".")[0], child.level, fn))
            visit(child, name)

    visit(tree, None)
    return out


def test_oracle_imports_only_numpy_scipy_and_the_standard_library():
    for path in py_files("oracle"):
        for mod, level, _ in imports(path):
            if level:            # the oracle's own modules
                continue
            assert mod in STDLIB_OK | {"numpy", "scipy"}, (os.path.basename(path), mod)


def test_product_package_never_names_the_oracle():
    base = os.path.join(ROOT, PKG)
    for path in py_files(PKG):
        for mod, _, _ in imports(path):
            assert mod != "oracle", os.path.basename(path)
    for sub, _, files in os.walk(base):
        for f in files:
            if f.endswith((".cu", ".cuh", ".h", ".cpp", ".c")):
                src = open(os.path.join(sub, f)).read()
                assert not re.search(r"#\s*include\s*[<\"][^>\"]*oracle", src), f
    for f in os.listdir(os.path.join(ROOT, "include")):
        assert "oracle" not in open(os.path.join(ROOT, "include", f)).read(), f


def test_shared_input_generators_import_neither_side():
    for mod, level, _ in imports(os.path.join(ROOT, "workloads.py")):
        assert level == 0 and mod not in ("oracle", PKG), mod


def test_bench_and_entry_touch_the_oracle_only_where_allowed():
    allowed = {"bench.py": {"oracle_sample"}, "__graft_entry__.py": {"smoke"}}
    for name, fns in allowed.items():
        found = [fn for mod, _, fn in imports(os.path.join(ROOT, name)) if mod == "oracle"]
        assert found and set(found) <= fns, (name, found)
    # and oracle_sample is called by the reference arm and the measurement's
    # CPU-baseline leg alone
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    callers = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.FunctionDef):
            for sub in ast.walk(node):
                if isinstance(sub, ast.Call) and getattr(sub.func, "id", None) == "oracle_sample":
                    callers.add(node.name)
    assert callers == {"run_reference", "measure"}, callers


def test_no_tracked_code_refers_to_the_scratch_folder():
    try:
        files = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True,
                               check=True).stdout.split()
    except (OSError, subprocess.CalledProcessError):
        files = []
    code = [f for f in files if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp", ".sh"))]
    if not code:   # not a git checkout (a copy of the tree): walk it instead
        for sub, dirs, fs in os.walk(ROOT):
            dirs[:] = [d for d in dirs if not d.startswith((".", "_work", "gpurun_out", "_build"))]
            code += [os.path.relpath(os.path.join(sub, f), ROOT) for f in fs
                     if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp", ".sh"))]
    pat = re.compile(r"(^|[^A-Za-z0-9_])_work(/|['\"]|$)")
    for f in code:
        if f == os.path.join("tests", "test_layering.py"):
            continue
        for i, line in enumerate(open(os.path.join(ROOT, f), errors="replace"), 1):
            assert not pat.search(line), f"{f}:{i}"
