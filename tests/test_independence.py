"""The product path and the oracle stay apart (no GPU needed).

The CUDA library and its binding never import, load or call the oracle, the two share no source
file, and the binding refuses to run without the compiled library instead of falling back to
anything else.
"""
import ast
import glob
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_gqa_block_gb300")


def _imports(path):
    tree = ast.parse(open(path).read(), path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module:
            names.add(node.module.split(".")[0])
    return names


def test_package_never_imports_the_oracle_or_the_tests():
    for path in glob.glob(os.path.join(PKG, "*.py")):
        assert not ({"oracle", "tests"} & _imports(path)), path


def test_cuda_sources_never_mention_the_oracle():
    for path in glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(path, errors="replace").read()
        assert "oracle" not in text, path


def test_the_oracle_shares_no_source_with_the_cuda_path():
    csrc = open(os.path.join(ROOT, "oracle", "pda_oracle.c")).read()
    assert "#include \"" not in csrc            # only system headers
    assert "pda_" not in csrc.replace("pda_oracle", "")


def test_binding_refuses_to_run_without_the_library(tmp_path):
    # a fresh interpreter whose binding points at a library that does not exist
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "import paged_kv_gqa_block_gb300 as pda\n"
        "pda.LIB_PATH = %r\n"
        "try:\n"
        "    pda.plan(1, 1, 8, 16, 4)\n"
        "except RuntimeError as e:\n"
        "    print('refused:', e)\n"
        "    sys.exit(0)\n"
        "sys.exit(3)\n" % (ROOT, str(tmp_path / "missing" / "libpda.so"))
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "is not built" in r.stdout
