"""Static checks of bench.py that need no GPU: every name a function reads is defined somewhere it
can see (a parameter, a local, a module-level name or a builtin). Most of the benchmark only runs on
a GPU machine, so a name left behind by a refactor would otherwise surface only there."""
import ast
import builtins
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _names_bound_in(fn):
    bound = set()
    for node in ast.walk(fn):
        if isinstance(node, ast.arg):
            bound.add(node.arg)
        elif isinstance(node, ast.Name) and isinstance(node.ctx, (ast.Store, ast.Del)):
            bound.add(node.id)
        elif isinstance(node, (ast.FunctionDef, ast.AsyncFunctionDef, ast.ClassDef)) and node is not fn:
            bound.add(node.name)
        elif isinstance(node, (ast.Import, ast.ImportFrom)):
            bound.update((a.asname or a.name).split(".")[0] for a in node.names)
    return bound


def test_bench_functions_read_only_defined_names():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    module = set(dir(builtins))
    for node in tree.body:
        if isinstance(node, (ast.FunctionDef, ast.ClassDef)):
            module.add(node.name)
        elif isinstance(node, ast.Assign):
            module.update(t.id for t in node.targets if isinstance(t, ast.Name))
        elif isinstance(node, (ast.Import, ast.ImportFrom)):
            module.update((a.asname or a.name).split(".")[0] for a in node.names)
    problems = []
    for fn in (n for n in tree.body if isinstance(n, ast.FunctionDef)):
        read = {n.id for n in ast.walk(fn) if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Load)}
        missing = sorted(read - _names_bound_in(fn) - module)
        if missing:
            problems.append(f"{fn.name}: {missing}")
    assert not problems, "; ".join(problems)
