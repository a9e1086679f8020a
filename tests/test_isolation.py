"""The product path and the oracle stay apart (CPU, static checks).

The CUDA library and its binding never import, link or read the oracle; the
oracle never imports the product; the benchmark touches the oracle only in its
CPU-baseline and reference legs.
"""

import ast
import glob
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp8_fine_grained_19_b300")


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    found = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            found += [a.name.split(".")[0] for a in node.names]
        elif isinstance(node, ast.ImportFrom) and node.module:
            found.append(node.module.split(".")[0])
    return found


def test_product_never_imports_the_oracle():
    for path in glob.glob(os.path.join(PKG, "**", "*.py"), recursive=True):
        assert "oracle" not in _imports(path), path


def test_native_sources_do_not_mention_the_oracle():
    for ext in ("cu", "cuh", "h"):
        for path in glob.glob(os.path.join(PKG, "**", f"*.{ext}"), recursive=True) + \
                glob.glob(os.path.join(ROOT, "include", f"*.{ext}")):
            assert "oracle" not in open(path).read().lower(), path


def test_oracle_never_imports_the_product():
    for path in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        imps = _imports(path)
        assert "fp8_fine_grained_19_b300" not in imps and "torch" not in imps, path


def test_bench_uses_the_oracle_only_in_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read())
    allowed = {"oracle_sample", "run_reference"}

    def walk(node, func):
        for child in ast.iter_child_nodes(node):
            name = child.name if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)) else func
            if isinstance(child, (ast.Import, ast.ImportFrom)):
                mods = [a.name for a in child.names] if isinstance(child, ast.Import) else [child.module or ""]
                if any(m.split(".")[0] == "oracle" for m in mods):
                    assert func in allowed, f"oracle imported in {func}"
            walk(child, name)

    walk(tree, None)
