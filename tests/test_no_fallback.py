"""The product path has no fallback: without the CUDA library every entry
point raises, and the package never imports the oracle."""
import ast
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "block_scaled_precision_04_gb300")


def test_missing_library_raises():
    code = (
        "import block_scaled_precision_04_gb300 as bsg\n"
        "bsg.LIB = '/nonexistent/libbsgemm.so'\n"
        "bsg._lib = None\n"
        "for f in (lambda: bsg.library(), lambda: bsg.bsg_problem_check(bsg.make_problem(4, 4, 32, 1)),\n"
        "          lambda: bsg.bsg_quant_check(bsg.make_quant_problem(4, 32))):\n"
        "    try:\n"
        "        f()\n"
        "    except RuntimeError as e:\n"
        "        assert 'no fallback' in str(e), e\n"
        "    else:\n"
        "        raise SystemExit('no error without the library')\n"
        "print('ok')\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stderr


def test_package_never_imports_the_oracle():
    for name in os.listdir(PKG):
        if not name.endswith(".py"):
            continue
        tree = ast.parse(open(os.path.join(PKG, name)).read())
        for node in ast.walk(tree):
            mods = []
            if isinstance(node, ast.Import):
                mods = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                mods = [node.module or ""]
            assert not any(m.split(".")[0] == "oracle" for m in mods), (name, mods)
