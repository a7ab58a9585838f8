"""The product path never loads the oracle: the library package imports and
runs without it, its sources do not name it, and in bench.py only the CPU
legs (the timed oracle baseline and the reference arm) import it."""
import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "int4_weight_only_w4_gb300")


def test_package_sources_do_not_import_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "w4_oracle" not in text, f


def test_binding_import_does_not_load_the_oracle():
    code = ("import sys; import int4_weight_only_w4_gb300.synthetic; "
            "import importlib.util as u; "
            "spec = u.find_spec('int4_weight_only_w4_gb300.w4'); "
            "print('oracle' in sys.modules)")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "False"


def test_bench_imports_the_oracle_only_in_cpu_legs():
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    users = set()
    for fn in ast.walk(tree):
        if isinstance(fn, (ast.FunctionDef, ast.ClassDef)):
            for node in ast.walk(fn):
                if isinstance(node, ast.Import) and any(a.name == "oracle" for a in node.names):
                    users.add(fn.name)
    top = [n for n in tree.body if isinstance(n, ast.Import)
           and any(a.name == "oracle" for a in n.names)]
    assert not top, "bench.py imports the oracle at module level"
    # OracleSampler (and its methods) serves cpu_baseline and the reference
    # arm only
    assert users <= {"OracleSampler", "next_gemv", "per_config", "omp_chain",
                     "check_outputs"}, users
    callers = set()
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.Call) and getattr(node.func, "id", None) == "OracleSampler":
                    callers.add(fn.name)
    assert callers == {"cpu_baseline", "reference_arm"}, callers

