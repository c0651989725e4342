"""The product path has no fallback and never reaches the oracle (CPU only).

The library is the only place the computation runs: if it is not built, the
binding refuses to work rather than falling back to a CPU or torch path, and
nothing in the package (the binding, the graph helpers, the context-parallel
helpers, the input generator) imports the oracle or links its code.
"""
import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "split_kv_decode_gb300")


def test_missing_library_fails_loudly():
    code = (
        "import sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "from split_kv_decode_gb300 import _native as N\n"
        "N.LIB_PATH = '/nonexistent/libsplitkv.so'\n"
        "from split_kv_decode_gb300 import api as A\n"
        "try:\n"
        "    A.decode_attn_version()\n"
        "except RuntimeError as e:\n"
        "    print('refused:', e)\n"
        "    sys.exit(0)\n"
        "sys.exit(1)\n"
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "not built" in r.stdout


def _imported_modules(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom) and node.module:
            yield node.module


def test_package_sources_never_import_the_oracle_or_the_tests():
    for f in sorted(os.listdir(PKG)):
        if f.endswith(".py"):
            for m in _imported_modules(os.path.join(PKG, f)):
                top = m.split(".")[0]
                assert top not in ("oracle", "tests"), f"{f} imports {m}"


def test_importing_the_package_loads_no_oracle():
    code = (
        "import sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import split_kv_decode_gb300.api, split_kv_decode_gb300.graphs\n"
        "import split_kv_decode_gb300.dcp, split_kv_decode_gb300.workloads\n"
        "bad = sorted(m for m in sys.modules if m.split('.')[0] in ('oracle', 'tests'))\n"
        "print(bad)\n"
        "sys.exit(1 if bad else 0)\n"
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr


def test_the_library_exports_no_oracle_code():
    from split_kv_decode_gb300 import build as B
    from split_kv_decode_gb300 import _native as N
    B.build()
    lib = N.load()
    for name in ("orc_attention", "orc_attention_split", "orc_merge", "orc_max_threads"):
        assert not hasattr(lib, name), name
