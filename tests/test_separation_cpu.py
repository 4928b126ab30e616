"""The oracle and the CUDA path stay apart (no GPU needed).

The oracle is test infrastructure: only the tests, the smoke check and the bench's
CPU-baseline and reference legs may use it, and the product path must fail loudly
rather than fall back to it.  These checks read the sources and import the product
modules in a fresh interpreter.
"""
from __future__ import annotations

import ast
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "int4_group_quantized_kvq_gb300")
CSRC = os.path.join(PKG, "csrc")
ORACLE = os.path.join(ROOT, "oracle")


def _py_files(top: str) -> list[str]:
    out = []
    for d, _, files in os.walk(top):
        if "__pycache__" in d:
            continue
        out += [os.path.join(d, f) for f in files if f.endswith(".py")]
    return out


def _imported_modules(path: str) -> list[tuple[str, ast.AST]]:
    tree = ast.parse(open(path).read(), path)
    mods = []
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods += [(a.name, node) for a in node.names]
        elif isinstance(node, ast.ImportFrom) and node.module:
            mods.append((node.module, node))
    return mods


def test_product_modules_never_import_the_oracle():
    files = _py_files(PKG) + _py_files(os.path.join(ROOT, "workloads"))
    assert files
    for f in files:
        for mod, _ in _imported_modules(f):
            assert mod.split(".")[0] != "oracle", f"{f} imports {mod}"
        assert "kvq_oracle" not in open(f).read(), f"{f} names the oracle library"


def test_sources_share_no_headers():
    incl = re.compile(r'^\s*#\s*include\s*[<"]([^>"]+)[>"]', re.M)
    cuda_files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    cuda_files += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    oracle_files = [os.path.join(ORACLE, f) for f in os.listdir(ORACLE) if f.endswith((".c", ".h"))]
    assert cuda_files and oracle_files
    cuda_names = {os.path.basename(f) for f in cuda_files}
    oracle_names = {os.path.basename(f) for f in oracle_files}
    for f in cuda_files:
        for inc in incl.findall(open(f).read()):
            assert "oracle" not in inc and os.path.basename(inc) not in oracle_names, f"{f} includes {inc}"
    for f in oracle_files:
        for inc in incl.findall(open(f).read()):
            assert "kvq.h" not in inc and os.path.basename(inc) not in cuda_names, f"{f} includes {inc}"
            assert not inc.endswith((".cuh", ".cu")), f"{f} includes {inc}"


def test_bench_uses_the_oracle_only_in_its_host_legs():
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read(), path)
    allowed = {"OracleSample", "time_oracle_quantize"}
    seen = set()

    def visit(node, owner):
        for child in ast.iter_child_nodes(node):
            name = owner
            if isinstance(child, (ast.FunctionDef, ast.ClassDef)):
                name = child.name if owner is None else owner
            if isinstance(child, ast.Import) and any(a.name.split(".")[0] == "oracle" for a in child.names):
                assert name in allowed, f"bench.py imports the oracle in {name}"
                seen.add(name)
            if isinstance(child, ast.ImportFrom) and (child.module or "").split(".")[0] == "oracle":
                assert name in allowed, f"bench.py imports from the oracle in {name}"
                seen.add(name)
            visit(child, name)

    visit(tree, None)
    assert seen == allowed
    # the host legs are called only by the CPU-baseline block of the kernel arm and by the
    # reference arm (and by one another)
    legs = {"OracleSample", "plan_oracle_sample", "time_oracle", "time_oracle_quantize"}
    callers: dict[str, set[str]] = {}
    for top in tree.body:
        if isinstance(top, (ast.FunctionDef, ast.ClassDef)):
            for node in ast.walk(top):
                if isinstance(node, ast.Call) and isinstance(node.func, ast.Name) and node.func.id in legs:
                    callers.setdefault(node.func.id, set()).add(top.name)
    assert callers.keys() == legs
    assert set().union(*callers.values()) <= legs | {"run_kvq", "run_reference"}


def test_importing_the_product_loads_no_oracle():
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import int4_group_quantized_kvq_gb300, workloads, bench\n"
            "assert 'oracle' not in sys.modules, sorted(m for m in sys.modules if 'oracle' in m)\n"
            "print('ok')\n") % ROOT
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stderr


def test_binding_fails_loudly_without_its_library():
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from int4_group_quantized_kvq_gb300 import binding\n"
            "binding.LIB_PATH = '/nonexistent/libkvq.so'\n"
            "binding._lib = None\n"
            "try:\n"
            "    binding.lib()\n"
            "except ImportError as e:\n"
            "    print('raised', 'missing' in str(e))\n") % ROOT
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "raised True", (r.stdout, r.stderr)
