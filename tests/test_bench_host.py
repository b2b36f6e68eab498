"""bench.py on the host (no GPU): every name a function reads is defined
somewhere it can see (a parameter, a local, an enclosing function, the
module, or a builtin), and the command line parses.  The timed paths need a
GPU; this catches the mistakes that would only show there."""

import ast
import builtins
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bound(node):
    out = set()
    for n in ast.walk(node):
        if isinstance(n, ast.Name) and isinstance(n.ctx, (ast.Store, ast.Del)):
            out.add(n.id)
        elif isinstance(n, (ast.FunctionDef, ast.AsyncFunctionDef, ast.Lambda)):
            a = n.args
            out |= {x.arg for x in a.posonlyargs + a.args + a.kwonlyargs}
            if a.vararg:
                out.add(a.vararg.arg)
            if a.kwarg:
                out.add(a.kwarg.arg)
            if not isinstance(n, ast.Lambda):
                out.add(n.name)
        elif isinstance(n, (ast.Import, ast.ImportFrom)):
            out |= {(al.asname or al.name).split(".")[0] for al in n.names}
        elif isinstance(n, ast.ExceptHandler) and n.name:
            out.add(n.name)
        elif isinstance(n, ast.ClassDef):
            out.add(n.name)
    return out


def test_bench_functions_read_only_defined_names():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    module = set(dir(builtins)) | {"__file__", "__name__"}
    for n in tree.body:
        if isinstance(n, (ast.FunctionDef, ast.ClassDef)):
            module.add(n.name)
        elif isinstance(n, (ast.Import, ast.ImportFrom)):
            module |= {(al.asname or al.name).split(".")[0] for al in n.names}
        else:
            module |= _bound(n)
    missing = []
    for fn in [n for n in tree.body if isinstance(n, (ast.FunctionDef, ast.ClassDef))]:
        seen = module | _bound(fn)
        for n in ast.walk(fn):
            if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Load) and n.id not in seen:
                missing.append((fn.name, n.id, n.lineno))
    assert not missing, missing


def test_bench_help_parses():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and "--workload" in r.stdout
