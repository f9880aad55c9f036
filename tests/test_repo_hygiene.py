"""Checks of the tree: the product never reaches the oracle and has no
fallback when its library is missing, and every committed ncu command leaves
the GPU clocks alone."""
import ast
import os
import re
import subprocess
import sys

from conftest import ROOT

PKG = os.path.join(ROOT, "turboquant_compressed_kv_tq_gb300")


def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield a.name
        elif isinstance(node, ast.ImportFrom):
            yield node.module or ""


def test_product_package_never_imports_the_oracle():
    # the oracle is test infrastructure: the package, its binding and its
    # build never import it, so no product call can route through it
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith(".py"):
                p = os.path.join(dirpath, f)
                mods = list(_imports(p))
                assert not any(m == "oracle" or m.startswith("oracle.") for m in mods), p
                assert "tq_oracle" not in open(p).read(), p


def test_native_sources_share_nothing_with_the_oracle():
    # the CUDA path and the C oracle are independent: no include, no symbol
    csrc = os.path.join(PKG, "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        assert "tq_oracle" not in text and "tqo_" not in text, f
    oracle_c = open(os.path.join(ROOT, "oracle", "tq_oracle.c")).read()
    assert not re.search(r'#include\s+"(?!tq_oracle\.h)', oracle_c)


def test_profile_commands_leave_clocks_alone():
    prof = os.path.join(ROOT, "profiles")
    for f in sorted(os.listdir(prof)):
        text = open(os.path.join(prof, f)).read()
        # join continuation lines, then look at every ncu invocation
        joined = re.sub(r"\\\n\s*", " ", text)
        for line in joined.splitlines():
            if re.search(r"(^|\s)ncu\s+-", line) and "-i " not in line:
                assert "--clock-control none" in line, (f, line)


def test_missing_library_fails_loudly():
    # without libtq.so every call raises: there is no fallback path
    code = ("import turboquant_compressed_kv_tq_gb300 as tq\n"
            "from turboquant_compressed_kv_tq_gb300 import _lib, build\n"
            "build.LIB = '/nonexistent/libtq.so'\n"
            "try:\n"
            "    tq.tq_abi_version()\n"
            "except RuntimeError as e:\n"
            "    print('raised', 'not built' in str(e))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "raised True", (r.stdout, r.stderr)
