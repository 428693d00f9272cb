"""The product path never reaches the oracle (CPU, static).

The package (the binding, the build script, the synthetic-input generators) must not
import anything under oracle/, and the oracle must not import the package's compute
path. bench.py may use the oracle only in its CPU-baseline and reference-arm
functions; __graft_entry__ only in build() (importing the checker) and smoke().
"""
import ast
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _imports(tree):
    """(module name, enclosing function name or None) for every import."""
    out = []

    def visit(node, fn):
        for child in ast.iter_child_nodes(node):
            if isinstance(child, (ast.FunctionDef, ast.AsyncFunctionDef)):
                visit(child, child.name)
                continue
            if isinstance(child, ast.Import):
                out.extend((a.name, fn) for a in child.names)
            elif isinstance(child, ast.ImportFrom) and child.module:
                out.extend((child.module + "." + a.name, fn) for a in child.names)
                out.append((child.module, fn))
            visit(child, fn)

    visit(tree, None)
    return out


def _parse(path):
    with open(path) as f:
        return ast.parse(f.read(), path)


def test_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "transformer_forward_gpt_b300")
    for name in os.listdir(pkg):
        if name.endswith(".py"):
            for mod, _ in _imports(_parse(os.path.join(pkg, name))):
                assert not mod.startswith("oracle"), f"{name} imports {mod}"


def test_oracle_never_imports_the_compute_path():
    allowed = {"transformer_forward_gpt_b300.synth"}   # seeded inputs only, no arithmetic
    odir = os.path.join(ROOT, "oracle")
    for name in os.listdir(odir):
        if name.endswith(".py"):
            for mod, _ in _imports(_parse(os.path.join(odir, name))):
                if mod.startswith("transformer_forward_gpt_b300"):
                    assert mod in allowed, f"oracle/{name} imports {mod}"


def test_bench_and_entry_use_the_oracle_only_where_allowed():
    rules = {"bench.py": {"oracle_prefill_sample", "oracle_decode_sample", "cpu_baseline",
                          "run_reference"},
             "__graft_entry__.py": {"build", "smoke"}}
    for name, fns in rules.items():
        for mod, fn in _imports(_parse(os.path.join(ROOT, name))):
            if mod.startswith("oracle"):
                assert fn in fns, f"{name}: oracle imported in {fn}"
